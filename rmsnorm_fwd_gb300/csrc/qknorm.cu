// qknorm.cu -- per-head QK norm ("CuTeDSL at Perplexity", section "QK
// Norm"): every head of q and of k is RMS-normalised over head_dim with the q
// or k weight plus WEIGHT_BIAS, in place, in one launch for both tensors.
//
// A head is a short row (64..256 elements), so TPR lanes of one warp own it
// (the page uses a half warp with one 16-byte vector per lane for a
// 128-element bf16 head; on GB300 8 lanes with two vectors each measure
// faster), NV 16-byte vectors per lane, and 256 / TPR heads share a block.
// Head h of token t: h < q_heads -> q + t * q_token_stride + h * head_dim,
// else k (strides let q and k be views into a fused QKV buffer).  The
// reduction is the butterfly shuffle over the TPR lanes; the statistic never
// leaves registers.
#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace {

// out = (x * r) * (w + bias), two elements per packed fp32x2 instruction
// (each result rounded as its scalar form), rounded to the element type.
template <int DT>
__device__ inline void scale_bias2(Vec<16> &out, const Vec<16> &xv, const Vec<16> &wv, float r,
                                   float bias)
{
    const uint64_t r2 = f2(r, r), b2 = f2(bias, bias);
    float f[8];
#pragma unroll
    for (int p = 0; p < 8 / Elem<DT>::kSize; ++p) {
        const uint64_t v = mul2(mul2(widen_pair<DT, 16>(xv, p), r2),
                                add2(widen_pair<DT, 16>(wv, p), b2));
        f2split(v, f[2 * p], f[2 * p + 1]);
    }
#pragma unroll
    for (int k = 0; k < Vec<16>::kWords; ++k)
        out.w[k] = Elem<DT>::kPerWord == 2 ? Elem<DT>::narrow(f[2 * k], f[2 * k + 1])
                                           : Elem<DT>::narrow(f[k], 0.f);
}

__device__ inline void vzero16(Vec<16> &v)
{
#pragma unroll
    for (int k = 0; k < 4; ++k)
        v.w[k] = 0u;
}

template <int DT, int TPR, int NV, int RPG>
__global__ void __launch_bounds__(256, 6) // <= 40 registers: 6 resident blocks
qk_norm_kernel(void *q, void *k, const void *__restrict__ qw, const void *__restrict__ kw,
               int64_t tokens, int32_t q_heads, int32_t k_heads, int32_t head_dim,
               int64_t q_stride, int64_t k_stride, float bias, float eps)
{
    using E = Elem<DT>;
    constexpr int VPE = 16 / E::kSize;
    constexpr int GROUPS = 256 / TPR;

    pdl_begin();
    const int nvec = head_dim / VPE;
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const int heads = q_heads + k_heads;
    const int64_t total = tokens * heads;
    const bool small = total < (int64_t(1) << 31); // 32-bit head index arithmetic
    const float n = static_cast<float>(head_dim);

    // Each group takes RPG heads per iteration (heads g, g + GROUPS, ... of
    // the block's window), so a lane has RPG * NV loads in flight.
    for (int64_t base = static_cast<int64_t>(blockIdx.x) * GROUPS * RPG; base < total;
         base += static_cast<int64_t>(gridDim.x) * GROUPS * RPG) {
        char *ht[RPG];
        bool active[RPG];
        Vec<16> xv[RPG][NV], wv[RPG][NV];
#pragma unroll
        for (int r = 0; r < RPG; ++r) {
            const int64_t row = base + g + r * GROUPS;
            active[r] = row < total;
            int64_t tok;
            int h;
            if (small) {
                const uint32_t rr = active[r] ? static_cast<uint32_t>(row) : 0u;
                const uint32_t tt = rr / static_cast<uint32_t>(heads);
                tok = tt;
                h = static_cast<int>(rr - tt * static_cast<uint32_t>(heads));
            } else {
                tok = active[r] ? row / heads : 0;
                h = active[r] ? static_cast<int>(row - tok * heads) : 0;
            }
            const bool isq = h < q_heads;
            char *head = isq ? static_cast<char *>(q) +
                                   (tok * q_stride + int64_t(h) * head_dim) * E::kSize
                             : static_cast<char *>(k) +
                                   (tok * k_stride + int64_t(h - q_heads) * head_dim) * E::kSize;
            ht[r] = head + t * 16;
            // The head's weight slice comes with it (an L1 hit after the
            // first heads), instead of holding both q and k slices in
            // registers across the loop.
            const char *wt = static_cast<const char *>(isq ? qw : kw) + t * 16;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (active[r] && t + j * TPR < nvec) {
                    ld_stream<0>(xv[r][j], ht[r] + j * TPR * 16);
                    ld_weight(wv[r][j], wt + j * TPR * 16);
                } else {
                    vzero16(xv[r][j]);
                    vzero16(wv[r][j]);
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RPG; ++r) {
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < NV; ++j)
                s = sumsq_mixed<DT, 16>(xv[r][j], s);
            s = group_allreduce<TPR>(s);
            const float rf = row_factor(s, n, eps);
            if constexpr (kRangeGuard<DT>) {
                // Range guard (device_common.cuh), warp-uniform: the groups
                // of a warp reduce with whole-warp shuffles.  The heads are
                // done again from memory (none of them is written yet), one
                // vector at a time, so the registers above are not kept
                // alive for this rare path.
                const bool redo = sum_needs_rescale(s, eps);
                if (__any_sync(0xFFFFFFFFu, redo)) {
                    const int64_t hrow = base + g + r * GROUPS;
                    const bool hq = active[r] && static_cast<int>(hrow % heads) < q_heads;
                    const char *wt = static_cast<const char *>(hq ? qw : kw) + t * 16;
                    const float kk = rescale_k(s);
                    float sk = 0.f;
#pragma unroll 1
                    for (int j = 0; j < NV; ++j) {
                        if (active[r] && t + j * TPR < nvec) {
                            Vec<16> xk;
                            ld_stream<0>(xk, ht[r] + j * TPR * 16);
                            sk = sumsq_k<DT, 16>(xk, kk, sk);
                        }
                    }
                    const Factor f = rescaled_factor(group_allreduce<TPR>(sk), kk, n, eps);
                    const float rr = redo ? f.r : rf;
                    const bool up = redo && f.up;
#pragma unroll 1
                    for (int j = 0; j < NV; ++j) {
                        if (active[r] && t + j * TPR < nvec) {
                            Vec<16> xk, wk, o;
                            ld_stream<0>(xk, ht[r] + j * TPR * 16);
                            ld_weight(wk, wt + j * TPR * 16);
                            if (up)
                                scale_up<DT, 16>(xk);
                            scale_bias2<DT>(o, xk, wk, rr, bias);
                            st_stream<0>(ht[r] + j * TPR * 16, o);
                        }
                    }
                    continue;
                }
            }
#pragma unroll
            for (int j = 0; j < NV; ++j)
                reuse_barrier(xv[r][j]);
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (active[r] && t + j * TPR < nvec) {
                    Vec<16> o;
                    scale_bias2<DT>(o, xv[r][j], wv[r][j], rf, bias);
                    st_stream<0>(ht[r] + j * TPR * 16, o);
                }
            }
        }
    }
}

// Any alignment / head size: a warp per head, scalar accesses, two passes
// (the second re-reads the head from L1).
template <int DT>
__global__ void __launch_bounds__(256)
qk_norm_scalar_kernel(void *q, void *k, const void *__restrict__ qw, const void *__restrict__ kw,
                      int64_t tokens, int32_t q_heads, int32_t k_heads, int32_t head_dim,
                      int64_t q_stride, int64_t k_stride, float bias, float eps)
{
    using E = Elem<DT>;
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int heads = q_heads + k_heads;
    const int64_t total = tokens * heads;
    const float n = static_cast<float>(head_dim);
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps + (threadIdx.x >> 5); row < total;
         row += static_cast<int64_t>(gridDim.x) * warps) {
        const int64_t tok = row / heads;
        const int h = static_cast<int>(row - tok * heads);
        const bool isq = h < q_heads;
        void *base = isq ? q : k;
        const void *w = isq ? qw : kw;
        const int64_t off =
            isq ? tok * q_stride + int64_t(h) * head_dim : tok * k_stride + int64_t(h - q_heads) * head_dim;
        float s = 0.f;
        for (int d = lane; d < head_dim; d += 32) {
            const float v = E::widen1(base, off + d);
            s = fmaf(v, v, s);
        }
        s = group_allreduce<32>(s);
        float r = row_factor(s, n, eps);
        float pre = 1.f; // 2^100 when the range guard scales x up (exact)
        if constexpr (kRangeGuard<DT>) {
            if (sum_needs_rescale(s, eps)) { // warp-uniform; a third pass over the head
                const float kk = rescale_k(s);
                float sk = 0.f;
                for (int d = lane; d < head_dim; d += 32) {
                    const float v = E::widen1(base, off + d) * kk;
                    sk = fmaf(v, v, sk);
                }
                const Factor f = rescaled_factor(group_allreduce<32>(sk), kk, n, eps);
                r = f.r;
                pre = f.up ? 0x1p100f : 1.f;
            }
        }
        for (int d = lane; d < head_dim; d += 32) {
            const float v = E::widen1(base, off + d) * pre;
            E::store1(base, off + d, (v * r) * (E::widen1(w, d) + bias));
        }
    }
}

template <int DT, int TPR, int NV, int RPG>
cudaError_t launch_qk(const QkArgs &a)
{
    return launch_kernel(qk_norm_kernel<DT, TPR, NV, RPG>, a.grid, 256, 0, a.base, a.q, a.k, a.qw,
                         a.kw, a.tokens, a.q_heads, a.k_heads, a.head_dim, a.q_stride,
                         a.k_stride, a.bias, a.eps);
}

template <int DT>
cudaError_t launch_qk_scalar(const QkArgs &a)
{
    return launch_kernel(qk_norm_scalar_kernel<DT>, a.grid, 256, 0, a.base, a.q, a.k, a.qw, a.kw,
                         a.tokens, a.q_heads, a.k_heads, a.head_dim, a.q_stride, a.k_stride,
                         a.bias, a.eps);
}

#define QK_ENTRY(DT, TPR, NV, RPG) QkKernel{DT, TPR, NV, RPG, &launch_qk<DT, TPR, NV, RPG>}
#define QK_SET(DT)                                                                             \
    QK_ENTRY(DT, 4, 1, 1), QK_ENTRY(DT, 4, 1, 4), QK_ENTRY(DT, 4, 2, 1), QK_ENTRY(DT, 4, 2, 2), \
        QK_ENTRY(DT, 8, 1, 1), QK_ENTRY(DT, 8, 1, 2), QK_ENTRY(DT, 8, 1, 4),                  \
        QK_ENTRY(DT, 8, 2, 1), QK_ENTRY(DT, 8, 2, 2), QK_ENTRY(DT, 16, 1, 1),                 \
        QK_ENTRY(DT, 16, 1, 2), QK_ENTRY(DT, 16, 1, 4), QK_ENTRY(DT, 16, 2, 1),               \
        QK_ENTRY(DT, 16, 2, 2), QK_ENTRY(DT, 32, 1, 1), QK_ENTRY(DT, 32, 1, 2),               \
        QK_ENTRY(DT, 32, 2, 1), QK_ENTRY(DT, 32, 4, 1), QkKernel{DT, 0, 0, 1, &launch_qk_scalar<DT>}

const QkKernel kTable[] = {QK_SET(RMSNORM_F32), QK_SET(RMSNORM_BF16), QK_SET(RMSNORM_F16)};

} // namespace

const QkKernel *qk_kernels(int *n)
{
    *n = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

} // namespace rmsnorm
