// staged.cu -- RMSNorm with rows staged in shared memory by bulk copies.
//
// Persistent blocks (grid <= SMs x blocks per SM).  Warp 0, lane 0 is the
// producer: it streams each of its block's rows global -> shared with one
// cp.async.bulk into a ring of `stages` slots, each slot guarded by a "full"
// mbarrier (completed by the copy's transaction bytes) and an "empty"
// mbarrier (completed by the consumer).  Warps 1..C are consumers, one row at
// a time each: wait for the slot, sum the squares from shared memory in
// fp32, reduce across the warp with shuffles, r = rsqrt(S / hidden + eps),
// then read the slot again, scale by r and the weight (staged once per block
// in its own slot), store y with 16-byte vector stores, and release the
// slot.  HBM sees one read of x, one write of y and one read of the weight
// per block; the row statistic stays in registers ("Build a GPU compiler
// from scratch ... (Emmy)", sections "Tensor IR" and "Loop IR").
//
// Slot s holds rows k = s, s + stages, ...; group g of G takes k = g, g + G,
// ...; `stages` is a multiple of G so each slot always has the same group and
// mbarrier parity waits are never ambiguous.  The warps of a group agree on
// every wait's outcome at their named barrier before anyone writes, so a
// wait that runs out in one warp stops the whole group together.
//
// Every spin-wait is bounded by `limit_ns` of %globaltimer.  A wait that runs
// out records RMSNORM_ERR_DEVICE_TIMEOUT in the status word, raises the
// block's abort flag, and the producer then waits (again bounded) for every
// copy it issued before the block exits, so no copy lands in shared memory
// that has been handed to another block.  Nothing here traps.
#include <mutex>

#include "internal.h"
#include "device_common.cuh"

namespace rmsnorm {
namespace {

__device__ inline uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ inline void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ inline bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ inline void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// y row <- shared slot, tracked in this thread's bulk-async group.
__device__ inline void bulk_copy_s2g(void *dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ inline void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ inline void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Named barrier `id` over `threads` threads (whole warps).
__device__ inline void group_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ inline uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ inline void record_timeout(int *status)
{
    atomicCAS(status, 0, static_cast<int>(RMSNORM_ERR_DEVICE_TIMEOUT));
}

// Single-thread bounded wait.  Returns false if the limit ran out or (when
// abort_flag is non-null) the block's abort flag went up.
__device__ inline bool wait_one(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                const volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (abort_flag && *abort_flag)
            return false;
        if (globaltimer() - t0 > limit_ns)
            return false;
    }
}

// Whole-warp bounded wait: every lane observes the phase (acquire) before
// any lane reads the slot; lane 0 decides, for the warp, when to give up.
__device__ inline bool wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                 const volatile int *abort_flag, int lane)
{
    uint64_t t0 = 0;
    bool timing = false;
    for (;;) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xFFFFFFFFu, done))
            return true;
        int give_up = 0;
        if (lane == 0) {
            const uint64_t now = globaltimer();
            if (!timing) {
                t0 = now;
                timing = true;
            }
            give_up = (*abort_flag != 0) || (now - t0 > limit_ns);
        }
        if (__shfl_sync(0xFFFFFFFFu, give_up, 0))
            return false;
    }
}

// TMA_STORE: the consumer writes y back into its slot and one lane streams
// the row to global memory with a bulk copy; the slot is handed back to the
// producer once that copy has finished reading it.  Otherwise y is stored
// from registers with 16-byte vector stores.
//
// BLOCK_STATUS: `status` points at one word per block instead of one word
// per call; each block zeroes its own word when it starts, and a group whose
// wait ran out writes its remaining rows of y as NaN so the failure is
// visible in the output.
//
// EPI: the output (rmsnorm_epilogue_t).  BIAS adds `bias` to the weight;
// the block-scaled outputs (never with TMA_STORE: their codes are smaller
// than the slot) write codes and scales with q_store, in a warp-uniform loop
// so every lane of a warp takes part in each scale block's shuffles.
template <int DT, bool TMA_STORE, bool BLOCK_STATUS = false, int EPI = RMSNORM_EPI_PLAIN,
          bool XW = false>
__global__ void __launch_bounds__(32 * 17)
staged_rows_kernel(const void *x, const void *__restrict__ w, void *y, int64_t rows,
                   int32_t hidden, float eps, int32_t stages, int32_t wpr, int *status,
                   uint64_t limit_ns, uint32_t flags, float bias, uint8_t *scales, float gscale)
{
    using E = Elem<DT>;
    constexpr bool MX = EPI >= RMSNORM_EPI_MXFP8;
    constexpr int Q = MX ? EPI - RMSNORM_EPI_MXFP8 : 0;
    static_assert(!(MX && TMA_STORE), "block-scaled outputs are stored from registers");
    static_assert(!(BLOCK_STATUS && EPI != RMSNORM_EPI_PLAIN), "status-per-block: plain only");
    extern __shared__ __align__(128) unsigned char smem[];

    const int32_t row_bytes = hidden * E::kSize;
    const StagedLayout L = staged_layout(row_bytes, stages);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    // full[s] = bars[s], empty[s] = bars[stages + s], weight = bars[2 * stages]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 2 * stages + 1);
    float *red = reinterpret_cast<float *>(bars + 2 * stages + 2);  // [2][16] partial sums
    int *agree = reinterpret_cast<int *>(red + 32);                  // [2][16] wait outcomes
    unsigned char *wsm = smem + L.bar_bytes;
    unsigned char *slots = wsm + L.slot_stride;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int consumers = (blockDim.x >> 5) - 1;
    const int groups = consumers / wpr;
    const int64_t my_rows =
        rows > blockIdx.x ? (rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    pdl_begin();
    const QParams qp = q_params(bias, gscale);
    if (BLOCK_STATUS) {
        status += blockIdx.x;
        if (threadIdx.x == 0)
            *status = 0;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[stages + s]), TMA_STORE ? 1 : wpr);
        }
        mbar_init(smem_u32(&bars[2 * stages]), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const uint32_t wbar = smem_u32(&bars[2 * stages]);

    if (warp == 0) {
        if (lane != 0)
            return;
        // ---------------- producer
        mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(row_bytes));
        bulk_copy_g2s(smem_u32(wsm), w, static_cast<uint32_t>(row_bytes), wbar);

        const char *xb = static_cast<const char *>(x);
        int64_t issued = 0;
        if (!(flags & kFlagWithholdCopies)) {
            for (int64_t k = 0; k < my_rows; ++k) {
                const int s = static_cast<int>(k % stages);
                if (k >= stages) {
                    const uint32_t par = static_cast<uint32_t>(((k / stages) - 1) & 1);
                    if (!wait_one(smem_u32(&bars[stages + s]), par, limit_ns, abort_flag)) {
                        if (!*abort_flag)
                            record_timeout(status);
                        *abort_flag = 1;
                        break;
                    }
                }
                if (*abort_flag)
                    break;
                const int64_t row = blockIdx.x + k * static_cast<int64_t>(gridDim.x);
                const uint32_t fb = smem_u32(&bars[s]);
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(row_bytes));
                bulk_copy_g2s(smem_u32(slots + static_cast<int64_t>(s) * L.slot_stride),
                              xb + row * row_bytes, static_cast<uint32_t>(row_bytes), fb);
                issued = k + 1;
            }
        }
        // Drain: every copy this block issued has landed before it exits.
        if (!wait_one(wbar, 0, limit_ns, nullptr))
            record_timeout(status);
        const int64_t first = issued > stages ? issued - stages : 0;
        for (int64_t k = first; k < issued; ++k) {
            const int s = static_cast<int>(k % stages);
            if (!wait_one(smem_u32(&bars[s]), static_cast<uint32_t>((k / stages) & 1), limit_ns,
                          nullptr))
                record_timeout(status);
        }
        return;
    }

    // ---------------- consumers: warp c = wi-th warp of group g
    const int c = warp - 1;
    const int g = c / wpr;
    const int wi = c % wpr;
    const int gsize = 32 * wpr;
    const int gl = wi * 32 + lane; // thread index within the group
    const bool issuer = wi == 0 && lane == 0;
    const int nvec = row_bytes / 16;
    const float n = static_cast<float>(hidden);
    char *yb = static_cast<char *>(y);
    int prev_slot = -1; // TMA_STORE: slot whose bulk store may still be reading it

    const bool have_weight = wait_warp(wbar, 0, limit_ns, abort_flag, lane);
    int it = 0;
    int64_t failed_at = -1; // BLOCK_STATUS: first of this group's rows left uncomputed
    for (int64_t k = g; k < my_rows; k += groups, ++it) {
        const int s = static_cast<int>(k % stages);
        const uint32_t par = static_cast<uint32_t>((k / stages) & 1);
        bool ok = have_weight && wait_warp(smem_u32(&bars[s]), par, limit_ns, abort_flag, lane);
        const unsigned char *src = slots + static_cast<int64_t>(s) * L.slot_stride;

        float acc = 0.f;
        if (ok) {
#pragma unroll 4
            for (int v = gl; v < nvec; v += gsize) {
                const Vec<16> xv = *reinterpret_cast<const Vec<16> *>(src + v * 16);
                acc = sumsq<DT, 16>(xv, acc);
            }
        }
        acc = group_allreduce<32>(acc);
        if (wpr > 1) {
            if (lane == 0) {
                red[(it & 1) * 16 + c] = acc;
                agree[(it & 1) * 16 + c] = ok ? 1 : 0;
            }
            group_sync(1 + g, gsize);
            const int base = (it & 1) * 16 + g * wpr;
            acc = lane < wpr ? red[base + lane] : 0.f;
            const int bad = lane < wpr ? (agree[base + lane] == 0) : 0;
            acc = group_allreduce<32>(acc);
            ok = !__any_sync(0xFFFFFFFFu, bad);
        }
        if (!ok) { // the whole group leaves together, before writing anything
            if (lane == 0) {
                if (!*abort_flag)
                    record_timeout(status);
                *abort_flag = 1;
            }
            failed_at = k;
            break;
        }
        float r = row_factor(acc, n, eps);
        if constexpr (kRangeGuard<DT>) {
            if (sum_needs_rescale(acc, eps)) { // group-uniform: the range guard's redo
                const float kk = rescale_k(acc);
                float sk = 0.f;
                for (int v = gl; v < nvec; v += gsize)
                    sk = sumsq_k<DT, 16>(*reinterpret_cast<const Vec<16> *>(src + v * 16), kk, sk);
                sk = group_allreduce<32>(sk);
                if (wpr > 1) {
                    // The other half of the double buffer: its last readers
                    // (the previous row) are past this row's barrier; the
                    // second barrier keeps the next row's writes after these
                    // reads.
                    if (lane == 0)
                        red[((it + 1) & 1) * 16 + c] = sk;
                    group_sync(1 + g, gsize);
                    const int base = ((it + 1) & 1) * 16 + g * wpr;
                    sk = group_allreduce<32>(lane < wpr ? red[base + lane] : 0.f);
                    group_sync(1 + g, gsize);
                }
                const Factor f = rescaled_factor(sk, kk, n, eps);
                r = f.r;
                if (f.up) {
                    // x scaled up by 2^100 in place in the slot: each thread
                    // scales the vectors it alone reads back below (the same
                    // vectors in every write-back mode).
                    unsigned char *slot = slots + static_cast<int64_t>(s) * L.slot_stride;
                    for (int v = gl; v < nvec; v += gsize) {
                        Vec<16> *p = reinterpret_cast<Vec<16> *>(slot + v * 16);
                        Vec<16> xv = *p;
                        scale_up<DT, 16>(xv);
                        *p = xv;
                    }
                }
            }
        }

        const int64_t row = blockIdx.x + k * static_cast<int64_t>(gridDim.x);
        char *yr = yb + row * row_bytes;
        if (TMA_STORE) {
            unsigned char *dst = slots + static_cast<int64_t>(s) * L.slot_stride;
#pragma unroll 4
            for (int v = gl; v < nvec; v += gsize) {
                const Vec<16> xv = *reinterpret_cast<const Vec<16> *>(dst + v * 16);
                const Vec<16> wv = *reinterpret_cast<const Vec<16> *>(wsm + v * 16);
                Vec<16> o;
                if constexpr (EPI == RMSNORM_EPI_BIAS)
                    scale_bias<DT, 16>(o, xv, wv, r, bias);
                else
                    scale<DT, 16>(o, xv, wv, r);
                *reinterpret_cast<Vec<16> *>(dst + v * 16) = o;
            }
            // The slot's new contents must be visible to the bulk copy (async proxy).
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (wpr > 1)
                group_sync(1 + g, gsize);
            else
                __syncwarp();
            if (issuer) {
                bulk_copy_s2g(yr, smem_u32(dst), static_cast<uint32_t>(row_bytes));
                // The group's previous copy has finished reading its slot: release it.
                bulk_wait_read<1>();
                if (prev_slot >= 0)
                    mbar_arrive(smem_u32(&bars[stages + prev_slot]));
            }
            prev_slot = s;
        } else if constexpr (MX) {
            using G = QGeo<DT, 16, Q>;
            char *qr = yb + row * (static_cast<int64_t>(hidden) * QFmt<Q>::kBits / 8);
            uint8_t *sr = scales + row * (hidden / QFmt<Q>::kBlock);
            // lane l of the warp starting at vector vb takes vector vb + l:
            // the same vectors as gl, gl + gsize, ...
            for (int vb = wi * 32; vb < nvec; vb += gsize) {
                const int v = vb + lane;
                const bool live = v < nvec;
                Vec<16> xv, wv;
                if (live) {
                    xv = *reinterpret_cast<const Vec<16> *>(src + v * 16);
                    wv = *reinterpret_cast<const Vec<16> *>(wsm + v * 16);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        xv.w[k] = wv.w[k] = 0u;
                }
                const bool b = q_emit<DT, 16, Q, XW>(xv, wv, r, qp, live, lane % G::kLanes == 0,
                                                     qr + static_cast<int64_t>(v) * G::kCodeBytes,
                                                     sr + v / G::kLanes);
                if (XW && __any_sync(0xFFFFFFFFu, b && live)) {
                    // exact-product blocks outside their range: this vector again in
                    // the (x * r) * w order, from the slot
                    if (live) {
                        xv = *reinterpret_cast<const Vec<16> *>(src + v * 16);
                        wv = *reinterpret_cast<const Vec<16> *>(wsm + v * 16);
                    }
                    q_emit<DT, 16, Q, false>(xv, wv, r, qp, live, lane % G::kLanes == 0,
                                             qr + static_cast<int64_t>(v) * G::kCodeBytes,
                                             sr + v / G::kLanes);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[stages + s]));
        } else {
#pragma unroll 4
            for (int v = gl; v < nvec; v += gsize) {
                const Vec<16> xv = *reinterpret_cast<const Vec<16> *>(src + v * 16);
                const Vec<16> wv = *reinterpret_cast<const Vec<16> *>(wsm + v * 16);
                Vec<16> o;
                if constexpr (EPI == RMSNORM_EPI_BIAS)
                    scale_bias<DT, 16>(o, xv, wv, r, bias);
                else
                    scale<DT, 16>(o, xv, wv, r);
                st_stream<1>(yr + static_cast<int64_t>(v) * 16, o);
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&bars[stages + s]));
        }
    }
    if (TMA_STORE && issuer) {
        bulk_wait_all(); // every y row of this group written before the block exits
        if (prev_slot >= 0)
            mbar_arrive(smem_u32(&bars[stages + prev_slot]));
    }
    if (BLOCK_STATUS && failed_at >= 0) {
        Vec<16> nan;
        const uint32_t q = E::kSize == 4 ? 0x7FC00000u
                                         : (DT == RMSNORM_BF16 ? 0x7FC07FC0u : 0x7E007E00u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            nan.w[i] = q;
        for (int64_t k = failed_at; k < my_rows; k += groups) {
            char *yr = yb + (blockIdx.x + k * static_cast<int64_t>(gridDim.x)) * row_bytes;
            for (int v = gl; v < nvec; v += gsize)
                st_stream<0>(yr + static_cast<int64_t>(v) * 16, nan);
        }
    }
}

template <int DT, bool TS, int EPI>
cudaError_t launch_staged(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    auto go = [&](auto kernel) {
        return launch_kernel(kernel, p.grid, p.block_threads, p.smem_bytes, a, a.x, a.w, a.y,
                             a.rows, a.hidden, a.eps, p.stages, p.threads_per_row / 32, a.status,
                             a.wait_limit_ns, a.flags, a.bias, static_cast<uint8_t *>(a.scales),
                             a.gscale);
    };
    // the exact-product instantiation of a block-scaled output when the call allows it
    if constexpr (kHasExactProducts<DT, EPI>)
        if (a.xw)
            return go(staged_rows_kernel<DT, TS, false, EPI, true>);
    return go(staged_rows_kernel<DT, TS, false, EPI>);
}

// The exact-product instantiation launch_staged may pick (null where there is none).
template <int DT, bool TS, int EPI>
const void *staged_xw_func()
{
    if constexpr (kHasExactProducts<DT, EPI>)
        return reinterpret_cast<const void *>(&staged_rows_kernel<DT, TS, false, EPI, true>);
    else
        return nullptr;
}

#define STAGED_ENTRY(DT, TS, EPI)                                                              \
    KernelDesc{RMSNORM_VARIANT_STAGED, DT, 16, 32, 0, 0, 0, TS ? 3 : 0,                       \
               &launch_staged<DT, TS, EPI>,                                                    \
               reinterpret_cast<const void *>(&staged_rows_kernel<DT, TS, false, EPI>), EPI,    \
               staged_xw_func<DT, TS, EPI>()}

// Plain and weight-bias outputs with both write-back modes; the block-scaled
// outputs with register stores only.
#define STAGED_SET(DT)                                                                         \
    STAGED_ENTRY(DT, false, RMSNORM_EPI_PLAIN), STAGED_ENTRY(DT, true, RMSNORM_EPI_PLAIN),     \
        STAGED_ENTRY(DT, false, RMSNORM_EPI_BIAS), STAGED_ENTRY(DT, true, RMSNORM_EPI_BIAS),   \
        STAGED_ENTRY(DT, false, RMSNORM_EPI_MXFP8), STAGED_ENTRY(DT, false, RMSNORM_EPI_MXFP4), \
        STAGED_ENTRY(DT, false, RMSNORM_EPI_NVFP4)

const KernelDesc kTable[] = {STAGED_SET(RMSNORM_F32), STAGED_SET(RMSNORM_BF16),
                             STAGED_SET(RMSNORM_F16)};

// ---------------------------------------------------------------- no allocation

// Status words of rmsnorm_fwd_staged_noalloc: one per block of a launch,
// 4 KiB per device, held by every device that loads the library until the
// process exits.
constexpr int kNoAllocMaxBlocks = 1024;
static __device__ __align__(256) int g_noalloc_status[kNoAllocMaxBlocks];

struct NoAllocDevice {
    bool ready = false;
    int *status = nullptr; // device address of g_noalloc_status on this device
    int sm_count = 0;
    int smem_optin = 0;
};

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

template <int DT>
cudaError_t launch_staged_noalloc(const rmsnorm_plan_t &p, const LaunchArgs &a)
{
    staged_rows_kernel<DT, false, true><<<p.grid, p.block_threads, p.smem_bytes, a.stream>>>(
        a.x, a.w, a.y, a.rows, a.hidden, a.eps, p.stages, p.threads_per_row / 32, a.status,
        a.wait_limit_ns, a.flags, -0.0f, nullptr, 1.0f);
    return cudaGetLastError();
}

const void *noalloc_kernel(int dtype)
{
    switch (dtype) {
    case RMSNORM_F32:
        return reinterpret_cast<const void *>(&staged_rows_kernel<RMSNORM_F32, false, true>);
    case RMSNORM_BF16:
        return reinterpret_cast<const void *>(&staged_rows_kernel<RMSNORM_BF16, false, true>);
    default:
        return reinterpret_cast<const void *>(&staged_rows_kernel<RMSNORM_F16, false, true>);
    }
}

// One-time set-up of the current device, with that device current: the
// status array's device address (the array's name in host code is only a
// stand-in), the device limits, and the kernels' shared-memory opt-in.
// Makes no allocation.
int noalloc_setup(NoAllocDevice *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return RMSNORM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return RMSNORM_ERR_CUDA;
        if (major != 10 || minor != 3)
            return RMSNORM_ERR_UNSUPPORTED_DEVICE;
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_status) != cudaSuccess || ptr == nullptr)
            return RMSNORM_ERR_CUDA;
        for (int dt = RMSNORM_F32; dt <= RMSNORM_F16; ++dt)
            if (cudaFuncSetAttribute(noalloc_kernel(dt),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin) != cudaSuccess)
                return RMSNORM_ERR_CUDA;
        d.status = static_cast<int *>(ptr);
        d.sm_count = sms;
        d.smem_optin = optin;
        d.ready = true;
    }
    *out = d;
    return RMSNORM_OK;
}

} // namespace

const KernelDesc *staged_kernels(int *n)
{
    *n = static_cast<int>(sizeof(kTable) / sizeof(kTable[0]));
    return kTable;
}

} // namespace rmsnorm

namespace rmsnorm {
namespace {

// The allocation-free launch.  flags / limit_ns: the bounded waits'
// settings (kFlagWithholdCopies and a short limit only from the
// failure-detection test hook).
int noalloc_call(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                 float eps, int dtype, void *stream, uint32_t flags, uint64_t limit_ns)
{
    int rc = check_call_args(x, weight, y, rows, hidden, eps, dtype);
    if (rc != RMSNORM_OK)
        return rc;
    NoAllocDevice d;
    rc = noalloc_setup(&d);
    if (rc != RMSNORM_OK)
        return rc;
    if (rows == 0)
        return RMSNORM_OK;
    rmsnorm_plan_t p;
    rc = plan_launch(x, weight, y, rows, hidden, dtype, d.sm_count, d.smem_optin,
                     RMSNORM_VARIANT_STAGED, &p);
    if (rc != RMSNORM_OK)
        return rc == RMSNORM_ERR_VARIANT ? RMSNORM_ERR_TOO_LARGE : rc;
    if (p.grid > kNoAllocMaxBlocks)
        return RMSNORM_ERR_TOO_LARGE;
    LaunchArgs a;
    a.x = x;
    a.w = weight;
    a.y = y;
    a.rows = rows;
    a.hidden = static_cast<int32_t>(hidden);
    a.eps = eps;
    a.status = d.status;
    a.wait_limit_ns = limit_ns;
    a.flags = flags;
    a.stream = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    switch (dtype) {
    case RMSNORM_F32:
        err = launch_staged_noalloc<RMSNORM_F32>(p, a);
        break;
    case RMSNORM_BF16:
        err = launch_staged_noalloc<RMSNORM_BF16>(p, a);
        break;
    default:
        err = launch_staged_noalloc<RMSNORM_F16>(p, a);
        break;
    }
    return err == cudaSuccess ? RMSNORM_OK : RMSNORM_ERR_CUDA;
}

} // namespace
} // namespace rmsnorm

extern "C" int rmsnorm_fwd_staged_noalloc(const void *x, const void *weight, void *y,
                                          int64_t rows, int64_t hidden, float eps, int dtype,
                                          void *stream)
{
    return rmsnorm::noalloc_call(x, weight, y, rows, hidden, eps, dtype, stream, 0u,
                                 1000000000ull);
}

extern "C" int rmsnorm_test_staged_noalloc_timeout(const void *x, const void *weight, void *y,
                                                   int64_t rows, int64_t hidden, int dtype,
                                                   uint64_t limit_ns, void *stream)
{
    return rmsnorm::noalloc_call(x, weight, y, rows, hidden, 1e-6f, dtype, stream,
                                 rmsnorm::kFlagWithholdCopies, limit_ns);
}

extern "C" int rmsnorm_noalloc_block_status(int *host_out, int n)
{
    using namespace rmsnorm;
    if (!host_out || n < 0 || n > kNoAllocMaxBlocks)
        return RMSNORM_ERR_INVALID_ARG;
    NoAllocDevice d;
    const int rc = noalloc_setup(&d);
    if (rc != RMSNORM_OK)
        return rc;
    if (n == 0)
        return RMSNORM_OK;
    return cudaMemcpy(host_out, d.status, static_cast<size_t>(n) * sizeof(int),
                      cudaMemcpyDeviceToHost) == cudaSuccess
               ? RMSNORM_OK
               : RMSNORM_ERR_CUDA;
}
