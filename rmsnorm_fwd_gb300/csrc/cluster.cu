// cluster.cu -- one row split over a thread-block cluster, for rows too long
// for one SM to move quickly when there are few of them (decode).
//
// "CuTeDSL at Perplexity", section "Prefill and decode specialization":
// with fewer rows than SMs a row should not be left to one block on one SM;
// section "Grid synchronization" names the launch-latency tools (programmatic
// dependent launch) the decode path leans on.  Here the C blocks of a
// cluster (C = 2, 4 or 8, on C SMs of one GPU processing cluster) each take
// a contiguous slice of one row: they load it into registers, reduce their
// slice's sum of squares (warp shuffles, then one float per warp through
// shared memory), publish the block total in their own shared memory, meet
// at a cluster barrier, and every block reads all C totals through
// distributed shared memory (mapa + ld.shared::cluster) in rank order -- the
// same order in every block, so every block forms the bit-identical row
// factor -- then scales and stores its slice.  A second cluster barrier
// keeps each block's shared memory alive until every peer has read it.
// No multicast, no spin-waits: the only waits are the hardware cluster
// barriers, which every thread of every block reaches exactly twice (four
// times on the range guard's path, which every block of the cluster takes
// or skips together).
#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace {

__device__ inline uint32_t cta_smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ inline uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ inline uint32_t cluster_size()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

// The float at shared address `local` in block `rank` of this cluster.
__device__ inline float ld_peer(uint32_t local, uint32_t rank)
{
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// The two floats at shared address `local` in block `rank` of this cluster.
__device__ inline float2 ld_peer2(uint32_t local, uint32_t rank)
{
    uint32_t remote;
    float2 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"(remote)
                 : "memory");
    return v;
}

// Butterfly sum of a double over the 32 lanes (every lane gets the total,
// formed in the same order in every block).
__device__ inline double warp_sum_f64(double d)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        d += __shfl_xor_sync(0xFFFFFFFFu, d, off, 32);
    return d;
}

template <int VB>
__device__ inline void vzero(Vec<VB> &v)
{
#pragma unroll
    for (int k = 0; k < Vec<VB>::kWords; ++k)
        v.w[k] = 0u;
}

// Row r = blockIdx.x / C; block rank c of the cluster owns vectors
// [c * S, min((c + 1) * S, nvec)) with S = ceil(nvec / C); thread t holds
// vectors c * S + t + k * blockDim.x, k < NV.  blockDim.x * NV >= S.
template <int DT, int VB, int NV>
__global__ void __launch_bounds__(1024)
cluster_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                    int32_t hidden, float eps)
{
    using E = Elem<DT>;
    constexpr int VPE = VB / E::kSize;
    __shared__ float part[32];
    __shared__ float block_total;
    __shared__ __align__(8) float2 block_pair; // range guard: (sum of (k x)^2 over the slice, k)

    pdl_begin();
    const uint32_t C = cluster_size();
    const uint32_t c = cluster_rank();
    const int64_t row = blockIdx.x / C;
    const int nvec = hidden / VPE;
    const int S = (nvec + static_cast<int>(C) - 1) / static_cast<int>(C);
    const int v0 = static_cast<int>(c) * S;
    const int v1 = min(nvec, v0 + S);
    const int t = threadIdx.x;
    const int tpr = blockDim.x;
    const int lane = t & 31;
    const int warp = t >> 5;
    const int nwarps = tpr >> 5;
    const bool live_row = row < rows; // always true for a well-formed grid
    const int64_t row_bytes = static_cast<int64_t>(hidden) * E::kSize;
    const char *xr = static_cast<const char *>(x) + (live_row ? row : 0) * row_bytes;
    char *yr = static_cast<char *>(y) + (live_row ? row : 0) * row_bytes;
    const char *wb = static_cast<const char *>(w);

    Vec<VB> xv[NV];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = v0 + t + k * tpr;
        if (live_row && v < v1)
            ld_stream<1>(xv[k], xr + static_cast<int64_t>(v) * VB);
        else
            vzero(xv[k]);
    }
#pragma unroll
    for (int k = 0; k < NV; ++k)
        s = sumsq<DT, VB>(xv[k], s);
    s = group_allreduce<32>(s);
    if (lane == 0)
        part[warp] = s;
    __syncthreads();
    if (warp == 0) {
        float b = lane < nwarps ? part[lane] : 0.f;
        b = group_allreduce<32>(b);
        if (lane == 0)
            block_total = b;
    }
    // Every block's total is visible to the whole cluster past this barrier.
    cluster_sync_all();
    float tot = static_cast<uint32_t>(lane) < C ? ld_peer(cta_smem_addr(&block_total), lane) : 0.f;
    tot = group_allreduce<32>(tot);
    // No block leaves (or lets its shared memory go) before every peer has
    // read its total: arrive now, wait at the end.  Relaxed: the peer reads
    // above have completed (their values are used), and nothing written
    // here needs to be seen through this barrier.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    const float nf = static_cast<float>(hidden);
    const float r = row_factor(tot, nf, eps);
    if constexpr (kRangeGuard<DT>) {
        // Range guard (device_common.cuh), taken by every block of the
        // cluster together (they all hold the same total).  Each block forms
        // its slice's sum again from k x where its own plain sum left fp32's
        // trusted range, the blocks exchange (Sk, k) in a second round, and
        // every block adds Sk / k^2 in binary64 in rank order (exact
        // scalings by powers of two; the same value in every block).  The
        // slice is then read again from memory (nothing of it is written
        // yet), one vector at a time, so the registers above are not kept
        // alive for this rare path.
        if (sum_needs_rescale(tot, eps)) {
            const float bt = block_total; // this block's own plain sum
            float bk = 1.f, bs = bt;
            if (sum_needs_rescale(bt, eps)) { // block-uniform
                bk = rescale_k(bt);
                float sk = 0.f;
#pragma unroll 1
                for (int k = 0; k < NV; ++k) {
                    const int v = v0 + t + k * tpr;
                    if (live_row && v < v1) {
                        Vec<VB> xk;
                        ld_stream<0>(xk, xr + static_cast<int64_t>(v) * VB);
                        sk = sumsq_k<DT, VB>(xk, bk, sk);
                    }
                }
                sk = group_allreduce<32>(sk);
                if (lane == 0)
                    part[warp] = sk; // part's last readers passed the cluster barrier
                __syncthreads();
                bs = group_allreduce<32>(lane < nwarps ? part[lane] : 0.f);
            }
            if (t == 0)
                block_pair = make_float2(bs, bk);
            // Close the first round (every peer has read block_total), then
            // one full cluster barrier makes every block's pair visible.
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
            cluster_sync_all();
            const float2 pk = static_cast<uint32_t>(lane) < C
                                  ? ld_peer2(cta_smem_addr(&block_pair), lane)
                                  : make_float2(0.f, 1.f);
            asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
            const double kd = pk.y;
            float Sk, kk;
            wide_total(warp_sum_f64(static_cast<double>(pk.x) / (kd * kd)), eps, Sk, kk);
            const Factor f = rescaled_factor(Sk, kk, nf, eps);
#pragma unroll 1
            for (int k = 0; k < NV; ++k) {
                const int v = v0 + t + k * tpr;
                if (live_row && v < v1) {
                    Vec<VB> xk, wk, o;
                    ld_stream<0>(xk, xr + static_cast<int64_t>(v) * VB);
                    ld_weight(wk, wb + static_cast<int64_t>(v) * VB);
                    if (f.up)
                        scale_up<DT, VB>(xk);
                    scale<DT, VB>(o, xk, wk, f.r);
                    st_stream<1>(yr + static_cast<int64_t>(v) * VB, o);
                }
            }
            asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < NV; ++k)
        reuse_barrier(xv[k]);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = v0 + t + k * tpr;
        if (live_row && v < v1) {
            Vec<VB> wv, o;
            ld_weight(wv, wb + static_cast<int64_t>(v) * VB);
            scale<DT, VB>(o, xv[k], wv, r);
            st_stream<1>(yr + static_cast<int64_t>(v) * VB, o);
        }
    }
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DT, int VB, int NV>
cudaError_t launch_cluster(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(p.block_threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(p.stages); // blocks per row
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
    if (a.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, cluster_rows_kernel<DT, VB, NV>, a.x, a.w,
                                               a.y, a.rows, a.hidden, a.eps);
    return err != cudaSuccess ? err : cudaGetLastError();
}

#define CLUSTER_ENTRY(DT, VB, NV)                                                              \
    KernelDesc{RMSNORM_VARIANT_CLUSTER, DT, VB, 0, NV, 1024, 0, 1, &launch_cluster<DT, VB, NV>, \
               reinterpret_cast<const void *>(&cluster_rows_kernel<DT, VB, NV>)}

#define CLUSTER_SET(DT)                                                                        \
    CLUSTER_ENTRY(DT, 16, 1), CLUSTER_ENTRY(DT, 16, 2), CLUSTER_ENTRY(DT, 16, 4),              \
        CLUSTER_ENTRY(DT, 32, 1), CLUSTER_ENTRY(DT, 32, 2)

const KernelDesc kTable[] = {CLUSTER_SET(RMSNORM_F32), CLUSTER_SET(RMSNORM_BF16),
                             CLUSTER_SET(RMSNORM_F16)};

} // namespace

const KernelDesc *cluster_kernels(int *n)
{
    *n = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

} // namespace rmsnorm
