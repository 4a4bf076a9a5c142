// gridrow.cu -- a few very long rows spread over every SM, with one grid
// barrier between the sum of squares and the scaling.
//
// "CuTeDSL at Perplexity", section "Grid synchronization": to spread work
// over as many blocks as possible, all participating blocks synchronise
// through global memory; that is only safe when every block is resident at
// once (no more blocks than the SMs hold), which a cooperative launch
// enforces, and the barrier costs about as much as splitting the work into
// two launches.  Here it serves decode rows longer than a thread-block
// cluster holds in registers (above 512 KiB).
//
// The rows' 16-byte vectors, taken one row after the other, are cut into G
// equal ranges, one per block (a block may cover a part of one row or parts
// of a few).
//   Phase 1: the block's sum of squares of its part of each row it touches,
//            written to partial[row * G + b] (the rest of partial is zero).
//   Barrier: one thread per block adds one to an arrival counter (release)
//            and waits, bounded by %globaltimer, until all G have arrived
//            (acquire).  A wait that runs out records RMSNORM_ERR_DEVICE_TIMEOUT
//            in the status word and its block skips phase 2 (y is left as it
//            was); it never hangs.
//   Phase 2: every block sums the partials of a row -- those of the blocks
//            whose ranges meet it, all written in phase 1 of this call -- in
//            the same order, so every block forms the bit-identical row
//            factor, re-reads its range of x (an L2 hit: phase 1 just read
//            it) and writes y.
//   Exit:    each block adds one to a departure counter; the last block to
//            leave sets both counters back to zero for the next call.
#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace {

__device__ inline uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ inline uint32_t ld_acquire(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ inline uint32_t add_release(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__device__ inline uint32_t add_acq_rel(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__device__ inline double ld_l2(const double *p)
{
    double v;
    asm volatile("ld.global.cg.f64 %0, [%1];" : "=d"(v) : "l"(p) : "memory");
    return v;
}

template <int VB>
__device__ inline void vzero(Vec<VB> &v)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        v.w[k] = 0u;
}

// Block-wide sum (every thread gets it); `part` holds one float per warp.
__device__ inline float block_sum(float s, float *part)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    s = group_allreduce<32>(s);
    if (lane == 0)
        part[warp] = s;
    __syncthreads();
    float tot = lane < nwarps ? part[lane] : 0.f;
    tot = group_allreduce<32>(tot);
    __syncthreads(); // part is reused by the next call
    return tot;
}

// Block-wide sum of doubles (every thread gets it, formed in the same order
// in every block); `part` holds one double per warp.
__device__ inline double block_sum_f64(double d, double *part)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        d += __shfl_xor_sync(0xFFFFFFFFu, d, off, 32);
    if (lane == 0)
        part[warp] = d;
    __syncthreads();
    double tot = lane < nwarps ? part[lane] : 0.0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        tot += __shfl_xor_sync(0xFFFFFFFFu, tot, off, 32);
    __syncthreads();
    return tot;
}

template <int DT>
__global__ void __launch_bounds__(512, 2)
grid_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                 int32_t hidden, float eps, double *partial, uint32_t *counters, int *status,
                 uint64_t limit_ns, uint32_t flags)
{
    using E = Elem<DT>;
    constexpr int VB = 16;
    constexpr int VPE = VB / E::kSize;
    constexpr int U = 4;
    __shared__ float part[32];
    __shared__ double part64[32];
    __shared__ int passed;

    const int G = gridDim.x;
    const int b = blockIdx.x;
    const int t = threadIdx.x;
    const int tpr = blockDim.x;
    const int64_t nvec = hidden / VPE;
    // Block b owns the range [f0, f1) of the rows' vectors taken one row
    // after the other (an equal share of all of them, so a few rows each of
    // some blocks or a part of one row each).
    const int64_t total = rows * nvec;
    const int64_t share = (total + G - 1) / G;
    const int64_t f0 = min(total, b * share);
    const int64_t f1 = min(total, f0 + share);
    const int64_t row_lo = f0 / nvec;
    const int64_t row_hi = f1 > f0 ? (f1 - 1) / nvec : row_lo - 1; // last row touched
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const float n = static_cast<float>(hidden);

    // ---- phase 1: this block's partial sum of squares of every row it touches
    for (int64_t row = row_lo; row <= row_hi; ++row) {
        const int v0 = static_cast<int>(max(f0, row * nvec) - row * nvec);
        const int v1 = static_cast<int>(min(f1, (row + 1) * nvec) - row * nvec);
        const char *xr = static_cast<const char *>(x) + row * row_bytes;
        float s = 0.f;
        for (int v = v0 + t; v < v1; v += U * tpr) {
            Vec<VB> xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int vv = v + u * tpr;
                if (vv < v1)
                    ld_stream<1>(xv[u], xr + static_cast<int64_t>(vv) * VB);
                else
                    vzero(xv[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                s = sumsq<DT, VB>(xv[u], s);
        }
        s = block_sum(s, part);
        double sd = s;
        if constexpr (kRangeGuard<DT>) {
            // Range guard (device_common.cuh) on this block's part of the
            // row: formed again from k x, read again (an L2 hit), and kept
            // exactly as Sk / k^2 in binary64.
            if (sum_needs_rescale(s, eps)) {
                const float kk = rescale_k(s);
                float sk = 0.f;
                for (int v = v0 + t; v < v1; v += U * tpr) {
                    Vec<VB> xv[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int vv = v + u * tpr;
                        if (vv < v1)
                            ld_stream<0>(xv[u], xr + static_cast<int64_t>(vv) * VB);
                        else
                            vzero(xv[u]);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        sk = sumsq_k<DT, VB>(xv[u], kk, sk);
                }
                const double kd = kk;
                sd = static_cast<double>(block_sum(sk, part)) / (kd * kd);
            }
        }
        if (t == 0)
            partial[row * G + b] = sd;
    }

    // ---- grid barrier (counters[0]: arrivals, counters[1]: departures)
    __syncthreads();
    if (t == 0) {
        // kFlagWithholdCopies (failure-detection test only): block 0 does not
        // arrive, so every wait runs out.
        if (!((flags & kFlagWithholdCopies) && b == 0))
            add_release(&counters[0], 1u); // orders this block's partials before it
        int ok = 1;
        if (ld_acquire(&counters[0]) < static_cast<uint32_t>(G)) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire(&counters[0]) < static_cast<uint32_t>(G)) {
                if (globaltimer_ns() - t0 > limit_ns) {
                    ok = 0;
                    atomicCAS(status, 0, static_cast<int>(RMSNORM_ERR_DEVICE_TIMEOUT));
                    break;
                }
            }
        }
        passed = ok;
    }
    __syncthreads();

    // ---- phase 2: each touched row's factor from all G partials, then scale
    // and store this block's part of it
    if (passed) {
        const char *wb = static_cast<const char *>(w);
        for (int64_t row = row_lo; row <= row_hi; ++row) {
            // The partials in the same order in every block: in fp32 (each is
            // an fp32 sum unless the range guard rescaled it), and again in
            // binary64 when a partial or the fp32 total is out of fp32's
            // trusted range (block-uniform).
            const int b_lo = static_cast<int>(row * nvec / share);
            const int b_hi = static_cast<int>(min(static_cast<int64_t>(G - 1), ((row + 1) * nvec - 1) / share));
            double ad = 0.0;
            for (int i = b_lo + t; i <= b_hi; i += tpr)
                ad += ld_l2(partial + row * G + i);
            const float tot = block_sum(static_cast<float>(ad), part);
            float r = row_factor(tot, n, eps);
            bool up = false;
            if constexpr (kRangeGuard<DT>) {
                const float af = static_cast<float>(ad);
                const bool wide = static_cast<double>(af) != ad || sum_needs_rescale(tot, eps);
                if (__syncthreads_or(wide)) {
                    float Sk, kk;
                    wide_total(block_sum_f64(ad, part64), eps, Sk, kk);
                    const Factor f = rescaled_factor(Sk, kk, n, eps);
                    r = f.r;
                    up = f.up;
                }
            }
            const int v0 = static_cast<int>(max(f0, row * nvec) - row * nvec);
            const int v1 = static_cast<int>(min(f1, (row + 1) * nvec) - row * nvec);
            const char *xr = static_cast<const char *>(x) + row * row_bytes;
            char *yr = static_cast<char *>(y) + row * row_bytes;
            if (kRangeGuard<DT> && up) {
                // The range guard's rows of subnormals (x scaled up by 2^100
                // before the scaling): one vector at a time, so the loop below
                // carries no test for them.
#pragma unroll 1
                for (int v = v0 + t; v < v1; v += tpr) {
                    Vec<VB> xk, wk, o;
                    ld_stream<0>(xk, xr + static_cast<int64_t>(v) * VB);
                    ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                    scale_up<DT, VB>(xk);
                    scale<DT, VB>(o, xk, wk, r);
                    st_stream<1>(yr + static_cast<int64_t>(v) * VB, o);
                }
                continue;
            }
            for (int v = v0 + t; v < v1; v += U * tpr) {
                Vec<VB> xv[U], wv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int vv = v + u * tpr;
                    if (vv < v1) {
                        ld_stream<0>(xv[u], xr + static_cast<int64_t>(vv) * VB);
                        ld_weight(wv[u], wb + static_cast<int64_t>(vv) * VB);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int vv = v + u * tpr;
                    if (vv < v1) {
                        Vec<VB> o;
                        scale<DT, VB>(o, xv[u], wv[u], r);
                        st_stream<1>(yr + static_cast<int64_t>(vv) * VB, o);
                    }
                }
            }
        }
    }

    // ---- departure: the last block out clears the counters (every block
    // has passed or given up on the barrier and read its partials by now)
    __syncthreads();
    if (t == 0 && add_acq_rel(&counters[1], 1u) == static_cast<uint32_t>(G) - 1u) {
        counters[0] = 0u;
        counters[1] = 0u;
    }
}

template <int DT>
cudaError_t launch_grid(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(p.block_threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative; // every block resident at once, or no launch
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // scratch: two counters (zero between calls), then rows * G partials
    uint32_t *counters = static_cast<uint32_t *>(a.scratch);
    double *partial = reinterpret_cast<double *>(static_cast<char *>(a.scratch) + kGridCounterBytes);
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, grid_rows_kernel<DT>, a.x, a.w, a.y, a.rows, a.hidden, a.eps,
                           partial, counters, a.status, a.wait_limit_ns, a.flags);
    return err != cudaSuccess ? err : cudaGetLastError();
}

#define GRID_ENTRY(DT)                                                                         \
    KernelDesc{RMSNORM_VARIANT_GRID, DT, 16, 0, 0, 512, 2, 1, &launch_grid<DT>,               \
               reinterpret_cast<const void *>(&grid_rows_kernel<DT>)}

const KernelDesc kTable[] = {GRID_ENTRY(RMSNORM_F32), GRID_ENTRY(RMSNORM_BF16),
                             GRID_ENTRY(RMSNORM_F16)};

} // namespace

const KernelDesc *grid_kernels(int *n)
{
    *n = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

} // namespace rmsnorm
