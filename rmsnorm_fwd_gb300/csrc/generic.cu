// generic.cu -- RMSNorm for any hidden size and any element alignment.
//
// One thread block per row (grid-stride), scalar element accesses, two
// passes over the row: the first accumulates the fp32 sum of squares, the
// block reduces it (warp shuffles, then one float per warp through shared
// memory), the second re-reads x (now in L1/L2) and writes y.  This is the
// fallback for rows whose byte length or pointers do not allow 16-byte
// vectors; the arithmetic is the same as the vector kernels' (sum of
// squares, divide by the count, add epsilon, rsqrt, then (x * r) * w rounded
// to the element type -- "Build a GPU compiler from scratch ... (Emmy)",
// section "Tensor IR"; "CuTeDSL at Perplexity", section "QK Norm").
#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace {

// EPI: RMSNORM_EPI_PLAIN, or RMSNORM_EPI_BIAS (the weight plus `bias`).
template <int DT, int EPI>
__global__ void __launch_bounds__(1024)
generic_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                    int32_t hidden, float eps, float bias)
{
    using E = Elem<DT>;
    __shared__ float part[2][32];
    __shared__ float rare[32]; // the range guard's own reduction
    pdl_begin();
    const int t = threadIdx.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = blockDim.x >> 5;
    const float n = static_cast<float>(hidden);

    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const int64_t base = row * hidden;
        float s = 0.f;
        for (int j = t; j < hidden; j += blockDim.x) {
            const float v = E::widen1(x, base + j);
            s = fmaf(v, v, s);
        }
        s = group_allreduce<32>(s);
        if (lane == 0)
            part[it & 1][warp] = s;
        // Also orders every pass-one read of this row before any pass-two
        // write (in-place calls).
        __syncthreads();
        float tot = lane < nwarps ? part[it & 1][lane] : 0.f;
        tot = group_allreduce<32>(tot);
        float r = row_factor(tot, n, eps);
        float pre = 1.f; // 2^100 when the range guard scales x up (exact)
        if constexpr (kRangeGuard<DT>) {
            if (sum_needs_rescale(tot, eps)) { // block-uniform; a third pass over the row
                const float kk = rescale_k(tot);
                float sk = 0.f;
                for (int j = t; j < hidden; j += blockDim.x) {
                    const float v = E::widen1(x, base + j) * kk;
                    sk = fmaf(v, v, sk);
                }
                sk = group_allreduce<32>(sk);
                if (lane == 0)
                    rare[warp] = sk;
                __syncthreads();
                sk = group_allreduce<32>(lane < nwarps ? rare[lane] : 0.f);
                __syncthreads();
                const Factor f = rescaled_factor(sk, kk, n, eps);
                r = f.r;
                pre = f.up ? 0x1p100f : 1.f;
            }
        }
        for (int j = t; j < hidden; j += blockDim.x) {
            const float v = E::widen1(x, base + j) * pre;
            if constexpr (EPI == RMSNORM_EPI_BIAS)
                E::store1(y, base + j, (v * r) * (E::widen1(w, j) + bias));
            else
                E::store1(y, base + j, (v * r) * E::widen1(w, j));
        }
    }
}

template <int DT, int EPI>
cudaError_t launch_generic(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    return launch_kernel(generic_rows_kernel<DT, EPI>, p.grid, p.block_threads, 0, a, a.x, a.w,
                         a.y, a.rows, a.hidden, a.eps, a.bias);
}

#define GENERIC_ENTRY(DT, EPI)                                                                 \
    KernelDesc{RMSNORM_VARIANT_GENERIC, DT, 0, 0, 0, 0, 0, 0, &launch_generic<DT, EPI>,        \
               reinterpret_cast<const void *>(&generic_rows_kernel<DT, EPI>), EPI}

const KernelDesc kTable[] = {
    GENERIC_ENTRY(RMSNORM_F32, RMSNORM_EPI_PLAIN), GENERIC_ENTRY(RMSNORM_BF16, RMSNORM_EPI_PLAIN),
    GENERIC_ENTRY(RMSNORM_F16, RMSNORM_EPI_PLAIN), GENERIC_ENTRY(RMSNORM_F32, RMSNORM_EPI_BIAS),
    GENERIC_ENTRY(RMSNORM_BF16, RMSNORM_EPI_BIAS), GENERIC_ENTRY(RMSNORM_F16, RMSNORM_EPI_BIAS)};

} // namespace

const KernelDesc *generic_kernels(int *n)
{
    *n = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

} // namespace rmsnorm
