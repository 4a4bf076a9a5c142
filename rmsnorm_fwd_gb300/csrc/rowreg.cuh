// rowreg.cuh -- register-resident RMSNorm kernels: a group of lanes per row
// (warp-per-row) and a thread block per row (block-per-row, also used with a
// capped grid for decode shapes).
//
// One pass over HBM: every thread loads its slice of the row as 16- or
// 32-byte vectors into registers, accumulates the squares in fp32, the row
// total is formed with warp butterfly shuffles (plus one float per warp
// through shared memory for the block-per-row body), and the same registers
// are scaled and stored.  The statistic never leaves the chip ("Build a GPU
// compiler from scratch ... (Emmy)", section "Loop IR"; "CuTeDSL at
// Perplexity", section "QK Norm", for the shuffle reduction over the lanes
// that share a row and for packing several rows into one warp).
//
// Thread t of a row group owns vectors t, t + TPR, t + 2*TPR, ... so each
// warp-wide access is contiguous.  The number of warps per block is a
// compile-time constant for the warp-per-row body and an upper bound
// (__launch_bounds__) for the block-per-row body ("CuTeDSL at Perplexity",
// section "Prefill and decode specialization").
#pragma once

#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace rowreg {

template <int VB>
__device__ inline void vzero(Vec<VB> &v)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        v.w[k] = 0u;
}

// ---------------------------------------------------------------- warp-per-row

// TPR lanes (4..32, power of two) per row, BLOCK/TPR rows per block per
// iteration, grid-stride over rows.  Row r is handled in the iteration in
// which its group's base row reaches it; the loop bound is block-uniform so
// every lane takes part in every shuffle.
template <int DT, int VB, int TPR, int NV, int BLOCK>
__global__ void __launch_bounds__(BLOCK)
warp_rows_kernel(const void *__restrict__ x, const void *__restrict__ w, void *y, int64_t rows,
                 int32_t hidden, float eps)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;     // elements per vector
    constexpr int GROUPS = BLOCK / TPR;    // rows per block per iteration
    constexpr bool W_HELD = NV * VB <= 64; // keep the weight slice in registers

    const int nvec = hidden / VPE;
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const float n = static_cast<float>(hidden);
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const char *xb = static_cast<const char *>(x);
    const char *wb = static_cast<const char *>(w);
    char *yb = static_cast<char *>(y);

    Vec<VB> wv[W_HELD ? NV : 1];
    if (W_HELD) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * TPR;
            if (v < nvec)
                ld_weight(wv[k], wb + static_cast<int64_t>(v) * VB);
            else
                vzero(wv[k]);
        }
    }

    for (int64_t base = static_cast<int64_t>(blockIdx.x) * GROUPS; base < rows;
         base += static_cast<int64_t>(gridDim.x) * GROUPS) {
        const int64_t row = base + g;
        const bool active = row < rows;
        const char *xr = xb + row * row_bytes;
        char *yr = yb + row * row_bytes;

        Vec<VB> xv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * TPR;
            if (active && v < nvec)
                ld_stream(xv[k], xr + static_cast<int64_t>(v) * VB);
            else
                vzero(xv[k]);
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            s = sumsq<DT, VB>(xv[k], s);
        s = group_allreduce<TPR>(s);
        const float r = row_factor(s, n, eps);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * TPR;
            if (active && v < nvec) {
                Vec<VB> o;
                if (W_HELD) {
                    scale<DT, VB>(o, xv[k], wv[W_HELD ? k : 0], r);
                } else {
                    Vec<VB> wk;
                    ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                    scale<DT, VB>(o, xv[k], wk, r);
                }
                st_stream(yr + static_cast<int64_t>(v) * VB, o);
            }
        }
    }
}

// ---------------------------------------------------------------- block-per-row

// blockDim.x threads (a multiple of 32, <= MAXT) per row, grid-stride over
// rows.  Warp totals go through a double-buffered shared array so one
// __syncthreads per row suffices.
template <int DT, int VB, int NV, int MAXT>
__global__ void __launch_bounds__(MAXT)
cta_rows_kernel(const void *__restrict__ x, const void *__restrict__ w, void *y, int64_t rows,
                int32_t hidden, float eps)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;
    constexpr bool W_HELD = NV * VB <= 64;
    __shared__ float part[2][32];

    const int nvec = hidden / VPE;
    const int t = threadIdx.x;
    const int tpr = blockDim.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = tpr >> 5;
    const float n = static_cast<float>(hidden);
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const char *xb = static_cast<const char *>(x);
    const char *wb = static_cast<const char *>(w);
    char *yb = static_cast<char *>(y);

    Vec<VB> wv[W_HELD ? NV : 1];
    if (W_HELD) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * tpr;
            if (v < nvec)
                ld_weight(wv[k], wb + static_cast<int64_t>(v) * VB);
            else
                vzero(wv[k]);
        }
    }

    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const char *xr = xb + row * row_bytes;
        char *yr = yb + row * row_bytes;
        Vec<VB> xv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * tpr;
            if (v < nvec)
                ld_stream(xv[k], xr + static_cast<int64_t>(v) * VB);
            else
                vzero(xv[k]);
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            s = sumsq<DT, VB>(xv[k], s);
        s = group_allreduce<32>(s);
        if (lane == 0)
            part[it & 1][warp] = s;
        __syncthreads();
        float tot = lane < nwarps ? part[it & 1][lane] : 0.f;
        tot = group_allreduce<32>(tot);
        const float r = row_factor(tot, n, eps);

#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = t + k * tpr;
            if (v < nvec) {
                Vec<VB> o;
                if (W_HELD) {
                    scale<DT, VB>(o, xv[k], wv[W_HELD ? k : 0], r);
                } else {
                    Vec<VB> wk;
                    ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                    scale<DT, VB>(o, xv[k], wk, r);
                }
                st_stream(yr + static_cast<int64_t>(v) * VB, o);
            }
        }
    }
}

// ---------------------------------------------------------------- launchers

template <int DT, int VB, int TPR, int NV, int BLOCK>
cudaError_t launch_warp(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    warp_rows_kernel<DT, VB, TPR, NV, BLOCK><<<p.grid, BLOCK, 0, a.stream>>>(
        a.x, a.w, a.y, a.rows, a.hidden, a.eps);
    return cudaGetLastError();
}

template <int DT, int VB, int NV, int MAXT>
cudaError_t launch_cta(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    cta_rows_kernel<DT, VB, NV, MAXT><<<p.grid, p.block_threads, 0, a.stream>>>(
        a.x, a.w, a.y, a.rows, a.hidden, a.eps);
    return cudaGetLastError();
}

constexpr int kWarpBlock = 256;

#define WARP_ENTRY(DT, VB, TPR, NV)                                                            \
    KernelDesc{RMSNORM_VARIANT_WARP_PER_ROW, DT, VB, TPR, NV, kWarpBlock,                     \
               &launch_warp<DT, VB, TPR, NV, kWarpBlock>,                                      \
               reinterpret_cast<const void *>(&warp_rows_kernel<DT, VB, TPR, NV, kWarpBlock>)}

#define CTA_ENTRY(DT, VB, NV, MAXT)                                                            \
    KernelDesc{RMSNORM_VARIANT_CTA_PER_ROW, DT, VB, 0, NV, MAXT, &launch_cta<DT, VB, NV, MAXT>, \
               reinterpret_cast<const void *>(&cta_rows_kernel<DT, VB, NV, MAXT>)}

#define ROWREG_SET(DT)                                                                         \
    WARP_ENTRY(DT, 16, 4, 1), WARP_ENTRY(DT, 16, 8, 1), WARP_ENTRY(DT, 16, 8, 2),             \
        WARP_ENTRY(DT, 16, 16, 1), WARP_ENTRY(DT, 16, 16, 2), WARP_ENTRY(DT, 16, 32, 1),      \
        WARP_ENTRY(DT, 16, 32, 2), WARP_ENTRY(DT, 16, 32, 4), WARP_ENTRY(DT, 16, 32, 8),      \
        WARP_ENTRY(DT, 16, 32, 16), WARP_ENTRY(DT, 32, 32, 1), WARP_ENTRY(DT, 32, 32, 2),     \
        WARP_ENTRY(DT, 32, 32, 4), WARP_ENTRY(DT, 32, 32, 8), CTA_ENTRY(DT, 16, 1, 1024),     \
        CTA_ENTRY(DT, 16, 2, 1024), CTA_ENTRY(DT, 16, 3, 1024), CTA_ENTRY(DT, 16, 4, 1024),   \
        CTA_ENTRY(DT, 16, 6, 512), CTA_ENTRY(DT, 16, 8, 512), CTA_ENTRY(DT, 32, 1, 1024),     \
        CTA_ENTRY(DT, 32, 2, 1024), CTA_ENTRY(DT, 32, 4, 512)

} // namespace rowreg
} // namespace rmsnorm
