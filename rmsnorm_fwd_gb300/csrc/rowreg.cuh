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
//
// Occupancy is what sets the bandwidth of an HBM-bound row kernel: a block
// cannot store a row before all of it has arrived, so the bytes in flight per
// SM are (resident rows) x (row bytes).  MINB > 0 asks the compiler for at
// least MINB resident blocks per SM (a register cap) and, with more than one
// vector per thread, loads the weight after the reduction instead of holding
// it in registers across rows.
//
// EPI selects what the kernels write (rmsnorm_epilogue_t): the plain output,
// the weight plus a bias, or a block-scaled output (MXFP8 / MXFP4 / NVFP4
// codes and scales, q_emit in device_common.cuh).  Only the plain
// instantiations feed the plain entry points; the others are separate
// template instances with their own table entries.
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

// ---------------------------------------------------------------- range guard

// v, hidden from the compiler's value numbering: the range guard's redo
// recomputes its row pointers from it instead of keeping the main path's
// alive across the reduction (they are dead there on the main path).
__device__ inline int64_t opaque(int64_t v)
{
    asm volatile("mov.b64 %0, %0;" : "+l"(v));
    return v;
}

// Block-wide total of the warp totals `s` for the range guard's redo: one
// float per warp through its own shared array, with a barrier on each side
// of the read so it never meets the main reduction's double buffer.
__device__ inline float block_total_rare(float s, float *sh, int lane, int warp, int nwarps)
{
    if (lane == 0)
        sh[warp] = s;
    __syncthreads();
    const float tot = group_allreduce<32>(lane < nwarps ? sh[lane] : 0.f);
    __syncthreads();
    return tot;
}

// One vector of a row, scaled by rr and written: the plain, weight-bias or
// block-scaled output (every lane of the warp calls it for the block-scaled
// ones, in the (x * r) * w order; `live`: the vector is part of the row).
template <int DT, int VB, int CP, int EPI, bool PACKED>
__device__ inline void emit_vec(const Vec<VB> &xk, const Vec<VB> &wk, float rr, float bias,
                                const QParams &qp, bool live, bool leader, char *yp, uint8_t *sp)
{
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;
    if constexpr (MX) {
        q_emit<DT, VB, EPI - RMSNORM_EPI_MXFP8, false>(xk, wk, rr, qp, live, leader, yp, sp);
    } else if (live) {
        Vec<VB> o;
        if constexpr (EPI == RMSNORM_EPI_BIAS)
            scale_bias<DT, VB>(o, xk, wk, rr, bias);
        else if constexpr (PACKED)
            scale_packed<DT, VB>(o, xk, wk, rr);
        else
            scale<DT, VB>(o, xk, wk, rr);
        st_stream<CP>(yp, o);
    }
}

// The exact-product form's fallback (q_emit): the vectors t + j * tpr, j < NV,
// of lane t of a group of tpr lanes written again in the (x * r) * w order,
// from x and w read again (rolled, so that the common path's register
// allocation is not raised for it).  Every lane of the warp calls it.
template <int DT, int VB, int NV, int Q>
__device__ __forceinline__ void q_redo(const char *xr, const char *wt, char *yr, uint8_t *sr, int t,
                                    int tpr, int nvec, bool active, float r, const QParams &qp)
{
    constexpr int LPB = QGeo<DT, VB, Q>::kLanes;
    constexpr int OB = QGeo<DT, VB, Q>::kCodeBytes;
#pragma unroll 1
    for (int j = 0; j < NV; ++j) {
        const bool live = active && t + j * tpr < nvec;
        Vec<VB> xk, wk;
        if (live) {
            ld_stream<0>(xk, xr + j * tpr * VB);
            ld_weight(wk, wt + j * tpr * VB);
        } else {
            vzero(xk);
            vzero(wk);
        }
        q_emit<DT, VB, Q, false>(xk, wk, r, qp, live, t % LPB == 0, yr + j * tpr * OB,
                                 sr + (t + j * tpr) / LPB);
    }
}

// The range guard's redo of one row (device_common.cuh): the row is read
// again from memory (nothing of it is written yet), its sum formed from k x,
// and the whole row scaled and written, one vector at a time (rolled loops,
// the weight read again), so that the register bodies' allocation is not
// raised for it.  Lane t of a group of `tpr` lanes (a warp
// group, WARP, or the whole block) owns vectors t + j * tpr, j < NV.
// `redo`: this group's row needs it (WARP: the other groups of the warp come
// along for the shuffles and write their rows with the plain factor `r`).
template <int DT, int VB, int NV, int TPR, int CP, int EPI, bool PACKED>
__device__ __forceinline__ void redo_row(const char *xr, const char *wt, char *yr, uint8_t *sr,
                                      int t, int tpr, int nvec, bool active, bool redo, float s,
                                      float r, float n, float eps, float bias, QParams qp,
                                      float *sh)
{
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;
    constexpr int Q = MX ? EPI - RMSNORM_EPI_MXFP8 : 0;
    constexpr int LPB = QGeo<DT, VB, Q>::kLanes;
    constexpr int OB = MX ? QGeo<DT, VB, Q>::kCodeBytes : VB;
    const float kk = rescale_k(s);
    float sk = 0.f;
#pragma unroll 1
    for (int j = 0; j < NV; ++j) {
        if (active && t + j * tpr < nvec) {
            Vec<VB> xk;
            ld_stream<0>(xk, xr + j * tpr * VB);
            sk = sumsq_k<DT, VB>(xk, kk, sk);
        }
    }
    if constexpr (TPR > 0) {
        sk = group_allreduce<TPR>(sk);
    } else {
        const int lane = t & 31;
        sk = block_total_rare(group_allreduce<32>(sk), sh, lane, t >> 5, tpr >> 5);
    }
    const Factor f = rescaled_factor(sk, kk, n, eps);
    const float rr = redo ? f.r : r;
    const bool up = redo && f.up;
#pragma unroll 1
    for (int j = 0; j < NV; ++j) {
        const bool live = active && t + j * tpr < nvec;
        Vec<VB> xk, wk;
        if (live) {
            ld_stream<0>(xk, xr + j * tpr * VB);
            ld_weight(wk, wt + j * tpr * VB);
            if (up)
                scale_up<DT, VB>(xk);
        } else {
            vzero(xk);
            vzero(wk);
        }
        emit_vec<DT, VB, CP, EPI, PACKED>(xk, wk, rr, bias, qp, live, t % LPB == 0,
                                          yr + j * tpr * OB, sr + (t + j * tpr) / LPB);
    }
}

// ---------------------------------------------------------------- warp-per-row

// TPR lanes (4..32, power of two) per row, BLOCK/TPR rows per block per
// iteration, grid-stride over rows.  The loop bound is block-uniform so every
// lane takes part in every shuffle.
template <int DT, int VB, int TPR, int NV, int BLOCK, int MINB, int CP, int EPI, bool XW = false>
__global__ void __launch_bounds__(BLOCK, MINB > 0 ? MINB : 1)
warp_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                 int32_t hidden, float eps, float bias, uint8_t *scales, float gscale)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;                     // elements per vector
    constexpr int GROUPS = BLOCK / TPR;                    // rows per block per iteration
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;          // a block-scaled output
    constexpr int Q = MX ? EPI - RMSNORM_EPI_MXFP8 : 0;    // its format (QFmt)
    constexpr int LPB = QGeo<DT, VB, Q>::kLanes;           // lanes per scale block
    constexpr int OB = MX ? QGeo<DT, VB, Q>::kCodeBytes : VB; // output bytes per vector
    static_assert(!MX || TPR % LPB == 0, "a scale block must not straddle two rows");
    // Weight slice kept in registers (loaded before the row, off the
    // reduction's critical path): always for one vector per thread, else
    // only without a register cap.
    constexpr bool W_HELD = NV * VB <= 64 && (NV == 1 || MINB == 0);

    pdl_begin();
    const QParams qp = q_params(bias, gscale);
    const int nvec = hidden / VPE;
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    const RowCount rc = row_count(hidden);
    const float n = rc.n;
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const int64_t out_row = MX ? int64_t(hidden) * QFmt<Q>::kBits / 8 : row_bytes; // per row
    const char *wt = static_cast<const char *>(w) + t * VB;

    Vec<VB> wv[W_HELD ? NV : 1];
    if (W_HELD) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (t + k * TPR < nvec)
                ld_weight(wv[k], wt + k * TPR * VB);
            else
                vzero(wv[k]);
        }
    }

    for (int64_t base = static_cast<int64_t>(blockIdx.x) * GROUPS; base < rows;
         base += static_cast<int64_t>(gridDim.x) * GROUPS) {
        const int64_t row = base + g;
        const bool active = row < rows;
        const char *xr = static_cast<const char *>(x) + row * row_bytes + t * VB;
        char *yr = static_cast<char *>(y) + row * out_row + t * OB;

        Vec<VB> xv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (active && t + k * TPR < nvec)
                ld_stream<CP>(xv[k], xr + k * TPR * VB);
            else
                vzero(xv[k]);
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            s = MX ? sumsq_mixed<DT, VB>(xv[k], s) : sumsq<DT, VB>(xv[k], s);
        s = group_allreduce<TPR>(s);
        const float r = MX ? row_factor(s, rc, eps) : row_factor(s, n, eps);
        if constexpr (kRangeGuard<DT>) {
            // Range guard, warp-uniform (the groups of a warp reduce with
            // whole-warp shuffles): rare rows are redone from memory.
            const bool redo = sum_needs_rescale(s, eps);
            if (__any_sync(0xFFFFFFFFu, redo)) {
                const int64_t row2 = opaque(row);
                redo_row<DT, VB, NV, TPR, CP, EPI, false>(
                    static_cast<const char *>(x) + row2 * row_bytes + t * VB, wt, yr,
                    MX ? scales + row2 * (hidden / QFmt<Q>::kBlock) : nullptr, t, TPR, nvec,
                    active, redo, s, r, n, eps, bias, qp, nullptr);
                continue;
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k)
            reuse_barrier(xv[k]);

        bool bad = false; // exact-product blocks to write again (q_emit)
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if constexpr (MX) {
                const bool live = active && t + k * TPR < nvec;
                Vec<VB> wk;
                if (W_HELD)
                    wk = wv[W_HELD ? k : 0];
                else if (live)
                    ld_weight(wk, wt + k * TPR * VB);
                else
                    vzero(wk);
                const bool b = q_emit<DT, VB, Q, XW>(
                    xv[k], wk, r, qp, live, t % LPB == 0, yr + k * TPR * OB,
                    scales + row * (hidden / QFmt<Q>::kBlock) + (t + k * TPR) / LPB);
                bad |= b && live;
            } else if (active && t + k * TPR < nvec) {
                Vec<VB> o;
                Vec<VB> wk;
                if (W_HELD)
                    wk = wv[W_HELD ? k : 0];
                else
                    ld_weight(wk, wt + k * TPR * VB);
                if constexpr (EPI == RMSNORM_EPI_BIAS)
                    scale_bias<DT, VB>(o, xv[k], wk, r, bias);
                else
                    scale<DT, VB>(o, xv[k], wk, r);
                st_stream<CP>(yr + k * TPR * VB, o);
            }
        }
        if (XW && __any_sync(0xFFFFFFFFu, bad)) {
            const int64_t row2 = opaque(row);
            q_redo<DT, VB, NV, Q>(static_cast<const char *>(x) + row2 * row_bytes + t * VB, wt,
                                  static_cast<char *>(y) + row2 * out_row + t * OB,
                                  scales + row2 * (hidden / QFmt<Q>::kBlock), t, TPR, nvec,
                                  active, r, qp);
        }
    }
}

// ---------------------------------------------------------------- block-per-row

// blockDim.x threads (a multiple of 32, <= MAXT) per row, grid-stride over
// rows.  Warp totals go through a double-buffered shared array so one
// __syncthreads per row suffices.  TPRC > 0 fixes blockDim.x = TPRC at
// compile time (vector offsets become immediates).
template <int DT, int VB, int NV, int MAXT, int MINB, int CP, int TPRC, int EPI, bool XW = false>
__global__ void __launch_bounds__(MAXT, MINB > 0 ? MINB : 1)
cta_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                int32_t hidden, float eps, float bias, uint8_t *scales, float gscale)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;
    constexpr int Q = MX ? EPI - RMSNORM_EPI_MXFP8 : 0;
    constexpr int LPB = QGeo<DT, VB, Q>::kLanes;
    constexpr int OB = MX ? QGeo<DT, VB, Q>::kCodeBytes : VB;
    constexpr bool W_HELD = NV * VB <= 64 && (NV == 1 || MINB == 0); // as above
    __shared__ float part[2][32];
    __shared__ float rare[32]; // the range guard's own reduction

    pdl_begin();
    const QParams qp = q_params(bias, gscale);
    const int nvec = hidden / VPE;
    const int t = threadIdx.x;
    const int tpr = TPRC > 0 ? TPRC : blockDim.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = tpr >> 5;
    const int stride = tpr * VB; // bytes between a thread's consecutive vectors
    const RowCount rc = row_count(hidden);
    const float n = rc.n;
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const int64_t out_row = MX ? int64_t(hidden) * QFmt<Q>::kBits / 8 : row_bytes;
    const char *wt = static_cast<const char *>(w) + t * VB;

    Vec<VB> wv[W_HELD ? NV : 1];
    if (W_HELD) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (t + k * tpr < nvec)
                ld_weight(wv[k], wt + k * stride);
            else
                vzero(wv[k]);
        }
    }

    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const char *xr = static_cast<const char *>(x) + row * row_bytes + t * VB;
        char *yr = static_cast<char *>(y) + row * out_row + t * OB;
        Vec<VB> xv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (t + k * tpr < nvec)
                ld_stream<CP>(xv[k], xr + k * stride);
            else
                vzero(xv[k]);
        }
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
            s = sumsq_mixed<DT, VB>(xv[k], s);
        s = group_allreduce<32>(s);
        if (TPRC != 32) {
            if (lane == 0)
                part[it & 1][warp] = s;
            __syncthreads();
            const float tot = lane < nwarps ? part[it & 1][lane] : 0.f;
            s = group_allreduce<32>(tot);
        }
        const float r = MX ? row_factor(s, rc, eps) : row_factor(s, n, eps);
        if constexpr (kRangeGuard<DT>) {
            // Range guard, block-uniform (every warp holds the same s): a
            // rare row is redone from memory.
            if (sum_needs_rescale(s, eps)) {
                const int64_t row2 = opaque(row);
                redo_row<DT, VB, NV, TPRC == 32 ? 32 : 0, CP, EPI, true>(
                    static_cast<const char *>(x) + row2 * row_bytes + t * VB, wt, yr,
                    MX ? scales + row2 * (hidden / QFmt<Q>::kBlock) : nullptr, t, tpr, nvec, true,
                    true, s, r, n, eps, bias, qp, rare);
                continue;
            }
        }
#pragma unroll
        for (int k = 0; k < NV; ++k)
            reuse_barrier(xv[k]);

        bool bad = false; // exact-product blocks to write again (q_emit)
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if constexpr (MX) {
                const bool live = t + k * tpr < nvec;
                Vec<VB> wk;
                if (W_HELD)
                    wk = wv[W_HELD ? k : 0];
                else if (live)
                    ld_weight(wk, wt + k * stride);
                else
                    vzero(wk);
                const bool b = q_emit<DT, VB, Q, XW>(
                    xv[k], wk, r, qp, live, t % LPB == 0, yr + k * tpr * OB,
                    scales + row * (hidden / QFmt<Q>::kBlock) + (t + k * tpr) / LPB);
                bad |= b && live;
            } else if (t + k * tpr < nvec) {
                Vec<VB> o;
                Vec<VB> wk;
                if (W_HELD)
                    wk = wv[W_HELD ? k : 0];
                else
                    ld_weight(wk, wt + k * stride);
                if constexpr (EPI == RMSNORM_EPI_BIAS)
                    scale_bias_packed<DT, VB>(o, xv[k], wk, r, bias);
                else
                    scale_packed<DT, VB>(o, xv[k], wk, r);
                st_stream<CP>(yr + k * stride, o);
            }
        }
        if (XW && __any_sync(0xFFFFFFFFu, bad)) {
            const int64_t row2 = opaque(row);
            q_redo<DT, VB, NV, Q>(static_cast<const char *>(x) + row2 * row_bytes + t * VB, wt,
                                  static_cast<char *>(y) + row2 * out_row + t * OB,
                                  scales + row2 * (hidden / QFmt<Q>::kBlock), t, tpr, nvec, true,
                                  r, qp);
        }
    }
}

// ---------------------------------------------------------------- looped rows

// Rows of any length (16-byte multiple): a block per row, grid-stride, the
// row streamed twice in chunks of 4 vectors per thread -- the first pass sums
// the squares, the second re-reads the row (an L2 hit: the resident blocks'
// rows are a few tens of MB against a 129 MB L2), scales and stores.  DRAM
// sees x once and y once.  For rows longer than the register bodies hold.
template <int DT, int VB, int MAXT, int MINB, int CP, int EPI, bool XW = false>
__global__ void __launch_bounds__(MAXT, MINB > 0 ? MINB : 1)
cta_loop_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                int32_t hidden, float eps, float bias, uint8_t *scales, float gscale)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;
    constexpr int U = 4; // vectors in flight per thread per step
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;
    constexpr int Q = MX ? EPI - RMSNORM_EPI_MXFP8 : 0;
    constexpr int LPB = QGeo<DT, VB, Q>::kLanes;
    constexpr int OB = QGeo<DT, VB, Q>::kCodeBytes;
    __shared__ float part[2][32];
    __shared__ float rare[32]; // the range guard's own reduction

    pdl_begin();
    const QParams qp = q_params(bias, gscale);
    const int nvec = hidden / VPE;
    const int t = threadIdx.x;
    const int tpr = blockDim.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = tpr >> 5;
    const RowCount rc = row_count(hidden);
    const float n = rc.n;
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const char *wb = static_cast<const char *>(w);

    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
        const char *xr = static_cast<const char *>(x) + row * row_bytes;
        char *yr = static_cast<char *>(y) +
                   row * (MX ? int64_t(hidden) * QFmt<Q>::kBits / 8 : row_bytes);
        float s = 0.f;
        for (int v0 = t; v0 < nvec; v0 += U * tpr) {
            Vec<VB> xv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * tpr;
                if (v < nvec)
                    ld_stream<CP>(xv[u], xr + static_cast<int64_t>(v) * VB);
                else
                    vzero(xv[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
                s = MX ? sumsq_mixed<DT, VB>(xv[u], s) : sumsq<DT, VB>(xv[u], s);
        }
        s = group_allreduce<32>(s);
        if (lane == 0)
            part[it & 1][warp] = s;
        // Also orders every first-pass read of this row before any write of
        // it (in-place calls).
        __syncthreads();
        const float tot = group_allreduce<32>(lane < nwarps ? part[it & 1][lane] : 0.f);
        float r = MX ? row_factor(tot, rc, eps) : row_factor(tot, n, eps);
        bool up = false;
        if constexpr (kRangeGuard<DT>) {
            if (sum_needs_rescale(tot, eps)) { // block-uniform; a third pass over the row
                const float kk = rescale_k(tot);
                float sk = 0.f;
                for (int v0 = t; v0 < nvec; v0 += U * tpr) {
                    Vec<VB> xv[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int v = v0 + u * tpr;
                        if (v < nvec)
                            ld_stream<0>(xv[u], xr + static_cast<int64_t>(v) * VB);
                        else
                            vzero(xv[u]);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        sk = sumsq_k<DT, VB>(xv[u], kk, sk);
                }
                const Factor f = rescaled_factor(
                    block_total_rare(group_allreduce<32>(sk), rare, lane, warp, nwarps), kk, n,
                    eps);
                r = f.r;
                up = f.up;
            }
        }

        if (kRangeGuard<DT> && up) {
            // The range guard's rows of subnormals (x scaled up by 2^100 before
            // the scaling): a second pass of its own, one vector at a time, so
            // the loops below carry no test for them.
            if constexpr (MX) {
                uint8_t *sr = scales + row * (hidden / QFmt<Q>::kBlock);
#pragma unroll 1
                for (int v0 = t & ~31; v0 < nvec; v0 += tpr) {
                    const int v = v0 + lane;
                    Vec<VB> xk, wk;
                    if (v < nvec) {
                        ld_stream<0>(xk, xr + static_cast<int64_t>(v) * VB);
                        ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                        scale_up<DT, VB>(xk);
                    } else {
                        vzero(xk);
                        vzero(wk);
                    }
                    q_emit<DT, VB, Q, false>(xk, wk, r, qp, v < nvec, lane % LPB == 0,
                                             yr + static_cast<int64_t>(v) * OB, sr + v / LPB);
                }
            } else {
#pragma unroll 1
                for (int v = t; v < nvec; v += tpr) {
                    Vec<VB> xk, wk, o;
                    ld_stream<0>(xk, xr + static_cast<int64_t>(v) * VB);
                    ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                    scale_up<DT, VB>(xk);
                    if constexpr (EPI == RMSNORM_EPI_BIAS)
                        scale_bias<DT, VB>(o, xk, wk, r, bias);
                    else
                        scale<DT, VB>(o, xk, wk, r);
                    st_stream<CP>(yr + static_cast<int64_t>(v) * VB, o);
                }
            }
            continue;
        }

        if constexpr (MX) {
            // Warp-uniform trip count (the block maximum is a shuffle over
            // the whole warp): lane l of the warp starting at vector v0
            // takes vector v0 + l, the same vectors as below.
            uint8_t *sr = scales + row * (hidden / QFmt<Q>::kBlock);
            for (int v0 = t & ~31; v0 < nvec; v0 += U * tpr) {
                Vec<VB> xv[U], wv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + lane + u * tpr;
                    if (v < nvec) {
                        ld_stream<0>(xv[u], xr + static_cast<int64_t>(v) * VB);
                        ld_weight(wv[u], wb + static_cast<int64_t>(v) * VB);
                    } else {
                        vzero(xv[u]);
                        vzero(wv[u]);
                    }
                }
                bool bad = false; // exact-product blocks to write again (q_emit)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + lane + u * tpr;
                    const bool b = q_emit<DT, VB, Q, XW>(xv[u], wv[u], r, qp, v < nvec,
                                                         lane % LPB == 0,
                                                         yr + static_cast<int64_t>(v) * OB,
                                                         sr + v / LPB);
                    bad |= b && v < nvec;
                }
                if (XW && __any_sync(0xFFFFFFFFu, bad)) {
                    // q_redo takes lane-based pointers (lane + j * tpr, j < U,
                    // from v0) and the row's scale base
                    const int64_t vl = v0 + lane;
                    q_redo<DT, VB, U, Q>(xr + vl * VB, wb + vl * VB, yr + vl * OB,
                                         sr + v0 / LPB, lane, tpr, nvec - v0, true, r, qp);
                }
            }
        } else {
            for (int v0 = t; v0 < nvec; v0 += U * tpr) {
                Vec<VB> xv[U], wv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * tpr;
                    if (v < nvec) {
                        ld_stream<0>(xv[u], xr + static_cast<int64_t>(v) * VB);
                        ld_weight(wv[u], wb + static_cast<int64_t>(v) * VB);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int v = v0 + u * tpr;
                    if (v < nvec) {
                        Vec<VB> o;
                        if constexpr (EPI == RMSNORM_EPI_BIAS)
                            scale_bias<DT, VB>(o, xv[u], wv[u], r, bias);
                        else
                            scale<DT, VB>(o, xv[u], wv[u], r);
                        st_stream<CP>(yr + static_cast<int64_t>(v) * VB, o);
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- launchers

// Each launcher takes the exact-product instantiation of a block-scaled
// body when the call allows it (LaunchArgs::xw), else the general one.
template <int DT, int VB, int TPR, int NV, int BLOCK, int MINB, int CP, int EPI>
cudaError_t launch_warp(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, p.grid, BLOCK, 0, a, a.x, a.w, a.y, a.rows, a.hidden, a.eps,
                             a.bias, static_cast<uint8_t *>(a.scales), a.gscale);
    };
    if constexpr (kHasExactProducts<DT, EPI>)
        if (a.xw)
            return go(warp_rows_kernel<DT, VB, TPR, NV, BLOCK, MINB, CP, EPI, true>);
    return go(warp_rows_kernel<DT, VB, TPR, NV, BLOCK, MINB, CP, EPI>);
}

template <int DT, int VB, int NV, int MAXT, int MINB, int CP, int TPRC, int EPI>
cudaError_t launch_cta(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, p.grid, p.block_threads, 0, a, a.x, a.w, a.y, a.rows,
                             a.hidden, a.eps, a.bias, static_cast<uint8_t *>(a.scales), a.gscale);
    };
    if constexpr (kHasExactProducts<DT, EPI>)
        if (a.xw)
            return go(cta_rows_kernel<DT, VB, NV, MAXT, MINB, CP, TPRC, EPI, true>);
    return go(cta_rows_kernel<DT, VB, NV, MAXT, MINB, CP, TPRC, EPI>);
}

template <int DT, int VB, int MAXT, int MINB, int CP, int EPI>
cudaError_t launch_loop(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, p.grid, p.block_threads, 0, a, a.x, a.w, a.y, a.rows,
                             a.hidden, a.eps, a.bias, static_cast<uint8_t *>(a.scales), a.gscale);
    };
    if constexpr (kHasExactProducts<DT, EPI>)
        if (a.xw)
            return go(cta_loop_kernel<DT, VB, MAXT, MINB, CP, EPI, true>);
    return go(cta_loop_kernel<DT, VB, MAXT, MINB, CP, EPI>);
}

constexpr int kWarpBlock = 256;

#define WARP_ENTRY(DT, VB, TPR, NV, MINB, CP, EPI)                                             \
    KernelDesc{RMSNORM_VARIANT_WARP_PER_ROW, DT, VB, TPR, NV, kWarpBlock, MINB, CP,           \
               &launch_warp<DT, VB, TPR, NV, kWarpBlock, MINB, CP, EPI>,                       \
               reinterpret_cast<const void *>(                                                 \
                   &warp_rows_kernel<DT, VB, TPR, NV, kWarpBlock, MINB, CP, EPI>),             \
               EPI}

#define CTA_ENTRY(DT, VB, NV, MAXT, MINB, CP, EPI)                                             \
    KernelDesc{RMSNORM_VARIANT_CTA_PER_ROW, DT, VB, 0, NV, MAXT, MINB, CP,                    \
               &launch_cta<DT, VB, NV, MAXT, MINB, CP, 0, EPI>,                                \
               reinterpret_cast<const void *>(                                                 \
                   &cta_rows_kernel<DT, VB, NV, MAXT, MINB, CP, 0, EPI>),                      \
               EPI}

// Looped block-per-row (vectors per thread 0 = "any row length").
#define LOOP_ENTRY(DT, VB, MAXT, MINB, CP, EPI)                                                \
    KernelDesc{RMSNORM_VARIANT_CTA_PER_ROW, DT, VB, 0, 0, MAXT, MINB, CP,                     \
               &launch_loop<DT, VB, MAXT, MINB, CP, EPI>,                                      \
               reinterpret_cast<const void *>(&cta_loop_kernel<DT, VB, MAXT, MINB, CP, EPI>),  \
               EPI}

// Block of exactly TPR threads (compile time).
#define CTAF_ENTRY(DT, VB, TPR, NV, MINB, CP, EPI)                                             \
    KernelDesc{RMSNORM_VARIANT_CTA_PER_ROW, DT, VB, TPR, NV, TPR, MINB, CP,                   \
               &launch_cta<DT, VB, NV, TPR, MINB, CP, TPR, EPI>,                               \
               reinterpret_cast<const void *>(                                                 \
                   &cta_rows_kernel<DT, VB, NV, TPR, MINB, CP, TPR, EPI>),                     \
               EPI}

// The instantiations every element type gets, per epilogue.
//   warp-per-row: (VB, TPR, NV, MINB, CP)
//   block-per-row, runtime block size <= MAXT: (VB, NV, MAXT, MINB, CP)
//   block-per-row, block size fixed at TPR: (VB, TPR, NV, MINB, CP)
// MINB caps registers so at least MINB blocks of MAXT threads fit on an SM
// (65536 registers): MAXT x MINB = 2048 -> 32 registers per thread.  The
// selector (select.cpp) names these entries by their parameters.  The
// 4-lane warp body is left out of the block-scaled sets (a 32-element f32
// block spans 8 lanes).
#define ROWREG_SET_WIDE(DT, EPI)                                                               \
    WARP_ENTRY(DT, 16, 8, 1, 0, 0, EPI), WARP_ENTRY(DT, 16, 8, 2, 0, 0, EPI),                  \
        WARP_ENTRY(DT, 16, 16, 1, 0, 0, EPI), WARP_ENTRY(DT, 16, 16, 2, 0, 0, EPI),            \
        WARP_ENTRY(DT, 16, 32, 1, 0, 0, EPI), WARP_ENTRY(DT, 16, 32, 2, 0, 0, EPI),            \
        WARP_ENTRY(DT, 16, 32, 4, 0, 0, EPI), WARP_ENTRY(DT, 16, 32, 2, 8, 0, EPI),            \
        WARP_ENTRY(DT, 16, 32, 4, 8, 0, EPI), WARP_ENTRY(DT, 32, 32, 1, 0, 0, EPI),            \
        WARP_ENTRY(DT, 32, 32, 2, 0, 0, EPI), CTA_ENTRY(DT, 16, 1, 1024, 2, 1, EPI),           \
        CTA_ENTRY(DT, 32, 1, 1024, 1, 1, EPI), CTA_ENTRY(DT, 16, 2, 1024, 2, 1, EPI),          \
        CTA_ENTRY(DT, 32, 2, 1024, 0, 1, EPI), CTA_ENTRY(DT, 16, 4, 1024, 0, 1, EPI),          \
        CTA_ENTRY(DT, 32, 4, 512, 0, 1, EPI), CTA_ENTRY(DT, 16, 2, 256, 8, 1, EPI),            \
        CTA_ENTRY(DT, 16, 3, 512, 3, 1, EPI), CTA_ENTRY(DT, 16, 4, 256, 6, 1, EPI),            \
        CTA_ENTRY(DT, 16, 4, 512, 2, 1, EPI), CTA_ENTRY(DT, 16, 8, 512, 0, 1, EPI),            \
        CTAF_ENTRY(DT, 16, 512, 1, 0, 0, EPI), LOOP_ENTRY(DT, 16, 512, 2, 1, EPI),             \
        CTA_ENTRY(DT, 32, 2, 256, 6, 1, EPI), CTA_ENTRY(DT, 32, 4, 320, 2, 1, EPI)

#define ROWREG_SET(DT, EPI) WARP_ENTRY(DT, 16, 4, 1, 0, 0, EPI), ROWREG_SET_WIDE(DT, EPI)

// The block-scaled outputs add blocks of a compile-time size (vector offsets
// and warp count known to the compiler; a single warp reduces with shuffles
// only) with four 32-byte vectors per thread: one warp (up to 128 registers,
// for 16 resident blocks per SM), 64, 96 or 128 threads (register-capped at
// 64: 16, 10 or 8 resident blocks): rows of up to 128, 256, 384 or 512 such
// vectors.
#define ROWREG_SET_Q(DT, EPI)                                                                  \
    ROWREG_SET_WIDE(DT, EPI), CTAF_ENTRY(DT, 32, 32, 4, 16, 1, EPI),                           \
        CTAF_ENTRY(DT, 32, 64, 4, 16, 1, EPI), CTAF_ENTRY(DT, 32, 96, 4, 10, 1, EPI),          \
        CTAF_ENTRY(DT, 32, 128, 4, 8, 1, EPI)

} // namespace rowreg
} // namespace rmsnorm
