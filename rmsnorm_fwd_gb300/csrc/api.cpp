// api.cpp -- the C ABI (include/rmsnorm.h): per-device contexts, argument
// validation, plan selection and the launch.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "host_link.h"
#include "internal.h"

namespace rmsnorm {

const KernelDesc *kernel_table(int *n)
{
    constexpr int kCap = 512;
    static KernelDesc table[kCap];
    static int count = [] {
        int c = 0;
        const KernelDesc *(*parts[])(int *) = {
            rowreg_kernels_f32,     rowreg_kernels_bf16,     rowreg_kernels_f16,
            staged_kernels,         generic_kernels,         rowreg_epi_kernels_f32,
            rowreg_epi_kernels_bf16, rowreg_epi_kernels_f16, cluster_kernels,
            rowreg_fp4_kernels_f32, rowreg_fp4_kernels_bf16, rowreg_fp4_kernels_f16,
            grid_kernels};
        for (auto part : parts) {
            int m = 0;
            const KernelDesc *t = part(&m);
            for (int i = 0; i < m && c < kCap; ++i)
                table[c++] = t[i];
        }
        return c;
    }();
    *n = count;
    return table;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull; // one second

// Host-buffer pipeline resources of one device (created on first use).
constexpr int kPipeBuffers = 3;
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr; // upload / download streams
    cudaEvent_t entry = nullptr;              // caller stream at entry
    cudaEvent_t loaded[kPipeBuffers] = {};    // upload of a buffer done
    cudaEvent_t computed[kPipeBuffers] = {};  // kernel on a buffer done
    cudaEvent_t drained[kPipeBuffers] = {};   // download of a buffer done (buffer free)
};

struct DeviceCtx {
    int refs = 0;
    int sm_count = 0;
    int smem_optin = 0;
    int *status = nullptr; // device word
    HostPipe *pipe = nullptr;
    // Grid variant: its counters and partial sums, allocated once (the
    // counters are left at zero by every launch), and the event its last
    // launch recorded, which the next one's stream waits on.
    void *grid_scratch = nullptr;
    cudaEvent_t grid_done = nullptr;
};

std::mutex g_mu;
DeviceCtx g_ctx[kMaxDevices];
std::mutex g_grid_mu[kMaxDevices]; // one grid-variant launch enqueues at a time per device

// Bytes of the grid variant's scratch on a device with `sms` SMs.
size_t grid_scratch_bytes(int sms)
{
    return static_cast<size_t>(kGridCounterBytes) +
           static_cast<size_t>(kGridMaxRows) * static_cast<size_t>(sms) *
               static_cast<size_t>(kGridBlocksPerSm) * sizeof(double);
}
std::mutex g_pipe_mu[kMaxDevices]; // one host-buffer call enqueues at a time per device

// Releases whatever make_pipe created, also after it failed part way.
void destroy_pipe(HostPipe *hp)
{
    if (!hp)
        return;
    for (cudaStream_t s : {hp->in, hp->out})
        if (s)
            cudaStreamDestroy(s);
    if (hp->entry)
        cudaEventDestroy(hp->entry);
    for (int b = 0; b < kPipeBuffers; ++b)
        for (cudaEvent_t e : {hp->loaded[b], hp->computed[b], hp->drained[b]})
            if (e)
                cudaEventDestroy(e);
    delete hp;
}

// True when [p, p + bytes) is page-locked host memory that the current
// device reaches at the same addresses.
bool host_mapped(const void *p, int64_t bytes)
{
    const char *c = static_cast<const char *>(p);
    for (const char *q : {c, c + bytes - 1}) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
            cudaGetLastError(); // clear the error this query may leave behind
            return false;
        }
        if (a.type != cudaMemoryTypeHost || a.devicePointer != q)
            return false;
    }
    return true;
}

int make_pipe(HostPipe *hp)
{
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->entry, ef) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    for (int b = 0; b < kPipeBuffers; ++b)
        if (cudaEventCreateWithFlags(&hp->loaded[b], ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp->computed[b], ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp->drained[b], ef) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}
std::atomic<uint64_t> g_wait_limit{kDefaultWaitLimitNs};
std::atomic<int> g_pdl{-1}; // -1: not set yet (RMSNORM_PDL decides), 0 off, 1 on

bool pdl_enabled()
{
    int v = g_pdl.load();
    if (v < 0) {
        const char *e = std::getenv("RMSNORM_PDL");
        v = (e && e[0] == '0') ? 0 : 1;
        int expected = -1;
        g_pdl.compare_exchange_strong(expected, v);
        v = g_pdl.load();
    }
    return v == 1;
}
thread_local int t_last_variant = 0;

// RMSNORM_FORCE_VARIANT: a variant name (warp_per_row, cta_per_row, staged,
// persistent, generic, cluster, grid) or its number; read once.  It replaces
// the automatic choice of every call that asks for one, so a program can be
// timed or checked on one body without code changes; a shape that body
// cannot take returns RMSNORM_ERR_VARIANT, as a forced rmsnorm_fwd_ex does.
int forced_variant()
{
    static const int v = [] {
        const char *e = std::getenv("RMSNORM_FORCE_VARIANT");
        if (!e || !e[0])
            return int(RMSNORM_VARIANT_AUTO);
        static const struct {
            const char *name;
            int v;
        } kNames[] = {{"warp_per_row", RMSNORM_VARIANT_WARP_PER_ROW},
                      {"cta_per_row", RMSNORM_VARIANT_CTA_PER_ROW},
                      {"staged", RMSNORM_VARIANT_STAGED},
                      {"persistent", RMSNORM_VARIANT_PERSISTENT},
                      {"generic", RMSNORM_VARIANT_GENERIC},
                      {"cluster", RMSNORM_VARIANT_CLUSTER},
                      {"grid", RMSNORM_VARIANT_GRID}};
        for (const auto &n : kNames)
            if (std::strcmp(e, n.name) == 0)
                return n.v;
        char *end = nullptr;
        const long k = std::strtol(e, &end, 10);
        if (end != e && *end == 0 && k >= RMSNORM_VARIANT_WARP_PER_ROW &&
            k <= RMSNORM_VARIANT_GRID)
            return int(k);
        std::fprintf(stderr, "rmsnorm: RMSNORM_FORCE_VARIANT=%s not understood; ignored\n", e);
        return int(RMSNORM_VARIANT_AUTO);
    }();
    return v;
}

bool log_enabled()
{
    static const bool on = [] {
        const char *e = std::getenv("RMSNORM_LOG");
        return e && e[0] == '1';
    }();
    return on;
}

// Looks up the current device's context (copy taken under the lock).
int current_ctx(DeviceCtx *out, int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return RMSNORM_ERR_NOT_INITIALIZED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ctx[dev].refs <= 0)
        return RMSNORM_ERR_NOT_INITIALIZED;
    *out = g_ctx[dev];
    if (dev_out)
        *dev_out = dev;
    return RMSNORM_OK;
}

bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

int check_args(const void *x, const void *w, void *y, int64_t rows, int64_t hidden, float eps,
               int dtype, int epi = RMSNORM_EPI_PLAIN, float bias = -0.0f,
               const void *scales = nullptr, float gscale = 1.0f)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || hidden <= 0 || !(eps >= 0.f) || !std::isfinite(eps) || !std::isfinite(bias))
        return RMSNORM_ERR_INVALID_ARG;
    if (epi < RMSNORM_EPI_PLAIN || epi > RMSNORM_EPI_NVFP4)
        return RMSNORM_ERR_INVALID_ARG;
    const bool mx = epi >= RMSNORM_EPI_MXFP8; // a block-scaled output
    const int block = epi == RMSNORM_EPI_NVFP4 ? 16 : 32;
    const int bits = epi == RMSNORM_EPI_MXFP8 ? 8 : 4;
    if (mx && hidden % block != 0)
        return RMSNORM_ERR_INVALID_ARG;
    if (epi == RMSNORM_EPI_NVFP4 && !(gscale > 0.f && std::isfinite(gscale)))
        return RMSNORM_ERR_INVALID_ARG;
    if (!w || (rows > 0 && (!x || !y || (mx && !scales))))
        return RMSNORM_ERR_INVALID_ARG;
    if (rows > 0) {
        const int64_t es = dtype == RMSNORM_F32 ? 4 : 2;
        if (rows > INT64_MAX / 4 / hidden)
            return RMSNORM_ERR_INVALID_ARG;
        const int64_t bytes = rows * hidden * es;
        if (mx) { // codes and scales are new buffers: no overlap with anything
            const int64_t qb = rows * hidden * bits / 8, sb = rows * (hidden / block);
            if (ranges_overlap(x, bytes, y, qb) || ranges_overlap(w, hidden * es, y, qb) ||
                ranges_overlap(x, bytes, scales, sb) ||
                ranges_overlap(w, hidden * es, scales, sb) || ranges_overlap(y, qb, scales, sb))
                return RMSNORM_ERR_ALIASING;
            return RMSNORM_OK;
        }
        if (y != x && ranges_overlap(x, bytes, y, bytes))
            return RMSNORM_ERR_ALIASING;
        if (ranges_overlap(w, hidden * es, y, bytes))
            return RMSNORM_ERR_ALIASING;
    }
    return RMSNORM_OK;
}

int launch(const void *x, const void *w, void *y, int64_t rows, int64_t hidden, float eps,
           int dtype, void *stream, int variant, rmsnorm_plan_t *plan, uint32_t flags,
           uint64_t limit_ns, int epi = RMSNORM_EPI_PLAIN, float bias = -0.0f,
           void *scales = nullptr, float gscale = 1.0f)
{
    int rc = check_args(x, w, y, rows, hidden, eps, dtype, epi, bias, scales, gscale);
    if (rc != RMSNORM_OK)
        return rc;
    DeviceCtx ctx;
    int dev = 0;
    rc = current_ctx(&ctx, &dev);
    if (rc != RMSNORM_OK)
        return rc;
    if (rows == 0) {
        if (plan && plan->variant == RMSNORM_VARIANT_AUTO)
            *plan = rmsnorm_plan_t{};
        return RMSNORM_OK;
    }

    rmsnorm_plan_t p;
    if (plan && plan->variant != RMSNORM_VARIANT_AUTO) {
        p = *plan;
        rc = validate_plan(p, x, w, y, rows, hidden, dtype, ctx.sm_count, ctx.smem_optin, epi);
    } else {
        if (variant == RMSNORM_VARIANT_AUTO)
            variant = forced_variant();
        rc = plan_launch(x, w, y, rows, hidden, dtype, ctx.sm_count, ctx.smem_optin, variant, &p,
                         epi);
    }
    if (rc != RMSNORM_OK)
        return rc;

    int n = 0;
    const KernelDesc *table = kernel_table(&n);
    const KernelDesc &d = table[p.kernel_index];
    LaunchArgs a;
    a.x = x;
    a.w = w;
    a.y = y;
    a.rows = rows;
    a.hidden = static_cast<int32_t>(hidden);
    a.eps = eps;
    a.status = ctx.status;
    a.wait_limit_ns = limit_ns;
    a.flags = flags;
    a.stream = static_cast<cudaStream_t>(stream);
    a.pdl = pdl_enabled();
    a.bias = bias;
    a.scales = scales;
    a.gscale = gscale;
    a.xw = quant_exact_products(dtype, epi, bias, gscale);
    if (log_enabled())
        std::fprintf(stderr,
                     "rmsnorm: rows=%lld hidden=%lld dtype=%d epi=%d -> variant=%d vec=%d tpr=%d "
                     "nv=%d block=%d grid=%d stages=%d smem=%d kernel=%d\n",
                     static_cast<long long>(rows), static_cast<long long>(hidden), dtype, epi,
                     p.variant, p.vec_bytes, p.threads_per_row, p.vecs_per_thread,
                     p.block_threads, p.grid, p.stages, p.smem_bytes, p.kernel_index);
    if (d.variant == RMSNORM_VARIANT_GRID) {
        // The context's scratch, shared by every grid-variant call on the
        // device: each launch waits for the previous one (its event) and
        // records its own, so calls on different streams take turns.  A
        // launch being captured into a CUDA graph is ordered by the graph's
        // own dependencies instead (an event recorded outside a capture
        // cannot be waited on inside it).
        if (static_cast<size_t>(kGridCounterBytes) +
                static_cast<size_t>(rows) * static_cast<size_t>(p.grid) * sizeof(double) >
            grid_scratch_bytes(ctx.sm_count))
            return RMSNORM_ERR_INVALID_ARG; // validate_plan bounds rows and grid: unreachable
        std::lock_guard<std::mutex> lk(g_grid_mu[dev]);
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(a.stream, &cs) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        const bool capturing = cs != cudaStreamCaptureStatusNone;
        a.scratch = ctx.grid_scratch;
        if ((!capturing && cudaStreamWaitEvent(a.stream, ctx.grid_done, 0) != cudaSuccess) ||
            d.launch(p, a) != cudaSuccess ||
            (!capturing && cudaEventRecord(ctx.grid_done, a.stream) != cudaSuccess))
            return RMSNORM_ERR_CUDA;
    } else if (d.launch(p, a) != cudaSuccess) {
        return RMSNORM_ERR_CUDA;
    }
    t_last_variant = p.variant;
    if (plan && plan->variant == RMSNORM_VARIANT_AUTO)
        *plan = p;
    return RMSNORM_OK;
}

} // namespace

int check_call_args(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                    float eps, int dtype)
{
    return check_args(x, w, const_cast<void *>(y), rows, hidden, eps, dtype);
}

} // namespace rmsnorm

using namespace rmsnorm;

extern "C" {

int rmsnorm_create(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return RMSNORM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceCtx &c = g_ctx[dev];
    if (c.refs > 0) {
        ++c.refs;
        return RMSNORM_OK;
    }
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return RMSNORM_ERR_CUDA;
    // The kernels are compiled for sm_103a only.
    if (major != 10 || minor != 3)
        return RMSNORM_ERR_UNSUPPORTED_DEVICE;
    // Everything the context owns on the device, allocated here and only
    // here: the status word and the grid variant's scratch (zeroed: its
    // counters start at zero).
    int *status = nullptr;
    void *scratch = nullptr;
    cudaEvent_t grid_done = nullptr;
    auto fail = [&] {
        cudaFree(status);
        cudaFree(scratch);
        if (grid_done)
            cudaEventDestroy(grid_done);
        return RMSNORM_ERR_CUDA;
    };
    const size_t sbytes = grid_scratch_bytes(sms);
    if (cudaMalloc(&status, sizeof(int)) != cudaSuccess ||
        cudaMemset(status, 0, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&scratch, sbytes) != cudaSuccess ||
        cudaMemset(scratch, 0, sbytes) != cudaSuccess ||
        cudaEventCreateWithFlags(&grid_done, cudaEventDisableTiming) != cudaSuccess)
        return fail();
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    for (int i = 0; i < n; ++i) {
        if (t[i].variant != RMSNORM_VARIANT_STAGED)
            continue;
        if (cudaFuncSetAttribute(t[i].func, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
                cudaSuccess ||
            (t[i].func_xw != nullptr &&
             cudaFuncSetAttribute(t[i].func_xw, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  optin) != cudaSuccess))
            return fail();
    }
    // The zeroed words are in place before any launch reads them (the
    // memsets run on the legacy stream; launches may use non-blocking ones).
    if (cudaStreamSynchronize(cudaStreamLegacy) != cudaSuccess)
        return fail();
    c.sm_count = sms;
    c.smem_optin = optin;
    c.status = status;
    c.grid_scratch = scratch;
    c.grid_done = grid_done;
    c.refs = 1;
    return RMSNORM_OK;
}

int rmsnorm_destroy(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return RMSNORM_ERR_NOT_INITIALIZED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceCtx &c = g_ctx[dev];
    if (c.refs <= 0)
        return RMSNORM_ERR_NOT_INITIALIZED;
    if (--c.refs == 0) {
        std::lock_guard<std::mutex> plk(g_pipe_mu[dev]);
        std::lock_guard<std::mutex> glk(g_grid_mu[dev]);
        cudaFree(c.status);
        cudaFree(c.grid_scratch);
        cudaEventDestroy(c.grid_done);
        destroy_pipe(c.pipe);
        c = DeviceCtx{};
    }
    return RMSNORM_OK;
}

int rmsnorm_fwd(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                float eps, int dtype, void *stream)
{
    return launch(x, weight, y, rows, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                  0u, g_wait_limit.load());
}

int rmsnorm_fwd_ex(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                   float eps, int dtype, void *stream, int variant, rmsnorm_plan_t *plan)
{
    return launch(x, weight, y, rows, hidden, eps, dtype, stream, variant, plan, 0u,
                  g_wait_limit.load());
}

int rmsnorm_fwd_bias(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                     float weight_bias, float eps, int dtype, void *stream)
{
    return launch(x, weight, y, rows, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                  0u, g_wait_limit.load(), RMSNORM_EPI_BIAS, weight_bias, nullptr);
}

int rmsnorm_fwd_mxfp8(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float weight_bias, float eps, int dtype, void *stream)
{
    return launch(x, weight, q, rows, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                  0u, g_wait_limit.load(), RMSNORM_EPI_MXFP8, weight_bias, scales);
}

int rmsnorm_fwd_mxfp4(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float weight_bias, float eps, int dtype, void *stream)
{
    return launch(x, weight, q, rows, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                  0u, g_wait_limit.load(), RMSNORM_EPI_MXFP4, weight_bias, scales);
}

int rmsnorm_fwd_nvfp4(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float global_scale, float weight_bias, float eps,
                      int dtype, void *stream)
{
    return launch(x, weight, q, rows, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                  0u, g_wait_limit.load(), RMSNORM_EPI_NVFP4, weight_bias, scales,
                  global_scale);
}

int rmsnorm_fwd_epilogue_ex(const void *x, const void *weight, void *y, void *scales,
                            int64_t rows, int64_t hidden, int epilogue, float weight_bias,
                            float global_scale, float eps, int dtype, void *stream, int variant,
                            rmsnorm_plan_t *plan)
{
    return launch(x, weight, y, rows, hidden, eps, dtype, stream, variant, plan, 0u,
                  g_wait_limit.load(), epilogue,
                  epilogue == RMSNORM_EPI_PLAIN ? -0.0f : weight_bias,
                  epilogue >= RMSNORM_EPI_MXFP8 ? scales : nullptr,
                  epilogue == RMSNORM_EPI_NVFP4 ? global_scale : 1.0f);
}

// Whether two strided head sets can share a byte: set A is
// {a + t * sa + [0, la)} and set B {b + t * sb + [0, lb)} for t < tokens (bytes).
bool strided_overlap(uintptr_t a, int64_t sa, int64_t la, uintptr_t b, int64_t sb, int64_t lb,
                     int64_t tokens)
{
    if (tokens <= 0 || la <= 0 || lb <= 0)
        return false;
    const int64_t ea = (tokens - 1) * sa + la, eb = (tokens - 1) * sb + lb;
    if (!ranges_overlap(reinterpret_cast<const void *>(a), ea, reinterpret_cast<const void *>(b),
                        eb))
        return false; // the whole extents are apart
    if (sa != sb || sa <= 0)
        return true; // interleaved with different strides: refuse
    // Equal strides P: some pair of tokens collides iff d + m P lies in
    // (-lb, la) for an integer |m| < tokens, with d = b - a.
    const int64_t d = static_cast<int64_t>(b - a), P = sa;
    auto floor_div = [](int64_t x, int64_t y) { return x >= 0 ? x / y : -((-x + y - 1) / y); };
    int64_t m_lo = floor_div(-lb - d, P) + 1;           // smallest m with d + mP > -lb
    int64_t m_hi = -floor_div(-(la - d), P) - 1;        // largest m with d + mP < la
    m_lo = std::max(m_lo, -(tokens - 1));
    m_hi = std::min(m_hi, tokens - 1);
    return m_lo <= m_hi;
}

// Whether the interval [w, w + wb) meets {a + t * P + [0, la)}, t < tokens.
bool interval_hits_strided(uintptr_t a, int64_t P, int64_t la, int64_t tokens, uintptr_t w,
                           int64_t wb)
{
    if (tokens <= 0 || la <= 0 || wb <= 0)
        return false;
    const int64_t d = static_cast<int64_t>(w - a);
    if (P <= 0) // a single interval
        return d < la && -d < wb;
    // t P < d + wb and d < t P + la, for an integer t in [0, tokens)
    auto floor_div = [](int64_t x, int64_t y) { return x >= 0 ? x / y : -((-x + y - 1) / y); };
    int64_t t_lo = floor_div(d - la, P) + 1;   // smallest t with t P > d - la
    int64_t t_hi = -floor_div(-(d + wb), P) - 1; // largest t with t P < d + wb
    t_lo = std::max<int64_t>(t_lo, 0);
    t_hi = std::min<int64_t>(t_hi, tokens - 1);
    return t_lo <= t_hi;
}

int rmsnorm_fwd_host(const void *x_host, const void *weight, void *y_host, int64_t rows,
                     int64_t hidden, float eps, int dtype, void *workspace,
                     size_t workspace_bytes, int64_t chunk_rows, void *stream)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || hidden <= 0 || !(eps >= 0.f) || !std::isfinite(eps) || chunk_rows < 0)
        return RMSNORM_ERR_INVALID_ARG;
    if (!weight || (rows > 0 && (!x_host || !y_host || !workspace)))
        return RMSNORM_ERR_INVALID_ARG;
    const int64_t es = dtype == RMSNORM_F32 ? 4 : 2;
    if (rows > INT64_MAX / 4 / hidden)
        return RMSNORM_ERR_INVALID_ARG;
    const int64_t row_bytes = hidden * es;
    if (rows > 0 && ranges_overlap(x_host, rows * row_bytes, y_host, rows * row_bytes) &&
        x_host != y_host)
        return RMSNORM_ERR_ALIASING;
    int dev = 0;
    DeviceCtx ctx;
    int rc = current_ctx(&ctx, &dev);
    if (rc != RMSNORM_OK)
        return rc;
    if (rows == 0)
        return RMSNORM_OK;

    // Buffers: up to three slices of the workspace, 256-byte aligned.
    const int64_t ws = static_cast<int64_t>(workspace_bytes);
    int nbuf = kPipeBuffers;
    int64_t per = 0;
    for (; nbuf >= 1; --nbuf) {
        per = (ws / nbuf) / 256 * 256;
        if (per >= row_bytes)
            break;
    }
    if (nbuf < 1)
        return RMSNORM_ERR_INVALID_ARG; // the workspace holds less than one row
    int64_t chunk = per / row_bytes;
    if (chunk_rows > 0)
        chunk = std::min(chunk, chunk_rows);
    else // about 16 chunks, so filling and draining the pipeline stay small
        chunk = std::min(chunk, std::max<int64_t>(1, (rows + 15) / 16));

    // Page-locked, device-mapped host buffers: the kernel reads x and writes
    // y in host memory directly (over the CPU-GPU link), no staging.
    if (host_mapped(x_host, rows * row_bytes) && host_mapped(y_host, rows * row_bytes)) {
        rmsnorm_plan_t p;
        rc = plan_host_link(x_host, weight, y_host, rows, hidden, dtype, ctx.sm_count,
                            ctx.smem_optin, &p);
        if (rc != RMSNORM_OK)
            return rc;
        return launch(x_host, weight, y_host, rows, hidden, eps, dtype, stream,
                      RMSNORM_VARIANT_AUTO, &p, 0u, g_wait_limit.load());
    }

    std::lock_guard<std::mutex> plk(g_pipe_mu[dev]);
    HostPipe *hp = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DeviceCtx &c = g_ctx[dev];
        if (c.refs <= 0)
            return RMSNORM_ERR_NOT_INITIALIZED;
        if (!c.pipe) {
            c.pipe = new HostPipe;
            if (make_pipe(c.pipe) != RMSNORM_OK) {
                destroy_pipe(c.pipe);
                c.pipe = nullptr;
                return RMSNORM_ERR_CUDA;
            }
        }
        hp = c.pipe;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // Everything already on the caller's stream (the workspace's last users,
    // the weight's producer) happens first.
    if (cudaEventRecord(hp->entry, cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->in, hp->entry, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->entry, 0) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    const char *xh = static_cast<const char *>(x_host);
    char *yh = static_cast<char *>(y_host);
    char *wsb = static_cast<char *>(workspace);
    int64_t i = 0;
    for (int64_t r0 = 0; r0 < rows; r0 += chunk, ++i) {
        const int b = static_cast<int>(i % nbuf);
        const int64_t n = std::min(chunk, rows - r0);
        const size_t bytes = static_cast<size_t>(n * row_bytes);
        char *buf = wsb + b * per;
        // upload (after the buffer's previous download)
        if ((i >= nbuf && cudaStreamWaitEvent(hp->in, hp->drained[b], 0) != cudaSuccess) ||
            cudaMemcpyAsync(buf, xh + r0 * row_bytes, bytes, cudaMemcpyHostToDevice, hp->in) !=
                cudaSuccess ||
            cudaEventRecord(hp->loaded[b], hp->in) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        // normalise in place on the caller's stream
        if (cudaStreamWaitEvent(cs, hp->loaded[b], 0) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        rc = launch(buf, weight, buf, n, hidden, eps, dtype, stream, RMSNORM_VARIANT_AUTO, nullptr,
                    0u, g_wait_limit.load());
        if (rc != RMSNORM_OK)
            return rc;
        if (cudaEventRecord(hp->computed[b], cs) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
        // download
        if (cudaStreamWaitEvent(hp->out, hp->computed[b], 0) != cudaSuccess ||
            cudaMemcpyAsync(yh + r0 * row_bytes, buf, bytes, cudaMemcpyDeviceToHost, hp->out) !=
                cudaSuccess ||
            cudaEventRecord(hp->drained[b], hp->out) != cudaSuccess)
            return RMSNORM_ERR_CUDA;
    }
    // The caller's stream resumes after the last download.
    const int last = static_cast<int>((i - 1) % nbuf);
    if (cudaStreamWaitEvent(cs, hp->drained[last], 0) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

int rmsnorm_qk_norm_ex(void *q, void *k, const void *q_weight, const void *k_weight,
                       int64_t tokens, int64_t q_heads, int64_t k_heads, int64_t head_dim,
                       int64_t q_token_stride, int64_t k_token_stride, float weight_bias,
                       float eps, int dtype, void *stream, rmsnorm_qk_plan_t *plan)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_UNSUPPORTED_DTYPE;
    if (tokens < 0 || q_heads < 0 || k_heads < 0 || head_dim <= 0 || head_dim > (1 << 20) ||
        q_heads > (1 << 20) || k_heads > (1 << 20) || !(eps >= 0.f) || !std::isfinite(eps) ||
        !std::isfinite(weight_bias) || q_token_stride < 0 || k_token_stride < 0)
        return RMSNORM_ERR_INVALID_ARG;
    const int64_t qs = q_token_stride ? q_token_stride : q_heads * head_dim;
    const int64_t ks = k_token_stride ? k_token_stride : k_heads * head_dim;
    if (qs < q_heads * head_dim || ks < k_heads * head_dim)
        return RMSNORM_ERR_INVALID_ARG;
    if ((q_heads > 0 && (!q || !q_weight)) || (k_heads > 0 && (!k || !k_weight)))
        return RMSNORM_ERR_INVALID_ARG;
    if (tokens > 0 && (tokens > INT64_MAX / 8 / std::max<int64_t>(qs, 1) ||
                       tokens > INT64_MAX / 8 / std::max<int64_t>(ks, 1)))
        return RMSNORM_ERR_INVALID_ARG;
    const int64_t es = dtype == RMSNORM_F32 ? 4 : 2;
    const uintptr_t qa = reinterpret_cast<uintptr_t>(q), ka = reinterpret_cast<uintptr_t>(k);
    if (q_heads > 0 && k_heads > 0 &&
        strided_overlap(qa, qs * es, q_heads * head_dim * es, ka, ks * es, k_heads * head_dim * es,
                        tokens))
        return RMSNORM_ERR_ALIASING;
    // The weights are read-only inputs: they may not sit inside a head q or k
    // writes.
    const int64_t wbytes = head_dim * es;
    for (const void *wp : {q_weight, k_weight}) {
        if (!wp)
            continue;
        const uintptr_t wa = reinterpret_cast<uintptr_t>(wp);
        if ((q_heads > 0 && interval_hits_strided(qa, qs * es, q_heads * head_dim * es, tokens, wa,
                                                  wbytes)) ||
            (k_heads > 0 && interval_hits_strided(ka, ks * es, k_heads * head_dim * es, tokens, wa,
                                                  wbytes)))
            return RMSNORM_ERR_ALIASING;
    }
    DeviceCtx ctx;
    int rc = current_ctx(&ctx, nullptr);
    if (rc != RMSNORM_OK)
        return rc;
    const int64_t heads = q_heads + k_heads;
    if (tokens == 0 || heads == 0)
        return RMSNORM_OK;

    // Vector body when every head starts on a 16-byte boundary.
    auto al = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool vec = (head_dim * es) % 16 == 0 && (qs * es) % 16 == 0 && (ks * es) % 16 == 0 &&
                     (q_heads == 0 || (al(q) && al(q_weight))) &&
                     (k_heads == 0 || (al(k) && al(k_weight)));
    const int64_t total = tokens * heads;
    int n = 0;
    const QkKernel *t = qk_kernels(&n);
    const QkKernel *kern = nullptr;
    int64_t grid = 0;
    const bool explicit_plan = plan && plan->lanes_per_head != 0;
    if (explicit_plan) {
        // A caller's plan (tuning sweeps): the vector body it names must cover
        // the head and the heads must be 16-byte aligned; -1 lanes = scalar.
        const int lanes = plan->lanes_per_head < 0 ? 0 : plan->lanes_per_head;
        for (int i = 0; i < n; ++i)
            if (t[i].dtype == dtype && t[i].tpr == lanes && t[i].nv == plan->vecs_per_lane &&
                t[i].rpg == plan->heads_per_group)
                kern = &t[i];
        if (!kern || plan->grid < 1)
            return RMSNORM_ERR_VARIANT;
        if (kern->tpr > 0 && (!vec || int64_t(kern->tpr) * kern->nv * 16 < head_dim * es))
            return RMSNORM_ERR_VARIANT;
        grid = plan->grid;
    } else {
        // Automatic (from a sweep of every compiled shape on GB300): two
        // 16-byte vectors per lane (8 lanes for a 128-element bf16 head, 16
        // for 256), one head per group, one pass over all heads.
        int tpr = 0, nv = 0, rpg = 1;
        if (vec) {
            const int64_t nvec = head_dim * es / 16;
            static const int kOpt[][3] = {{4, 1, 1}, {4, 2, 1}, {8, 2, 1}, {16, 2, 1},
                                          {32, 2, 1}, {32, 4, 1}};
            for (const auto &o : kOpt)
                if (int64_t(o[0]) * o[1] >= nvec) {
                    tpr = o[0];
                    nv = o[1];
                    rpg = o[2];
                    break;
                }
        }
        for (int i = 0; i < n; ++i)
            if (t[i].dtype == dtype && t[i].tpr == tpr && t[i].nv == (tpr ? nv : 0) &&
                t[i].rpg == (tpr ? rpg : 1))
                kern = &t[i];
        if (!kern)
            return RMSNORM_ERR_VARIANT;
        const int64_t per_block = kern->tpr ? int64_t(256 / kern->tpr) * kern->rpg : 8;
        grid = std::min<int64_t>((total + per_block - 1) / per_block, INT_MAX);
        if (plan) {
            plan->lanes_per_head = kern->tpr ? kern->tpr : -1;
            plan->vecs_per_lane = kern->nv;
            plan->heads_per_group = kern->rpg;
            plan->grid = static_cast<int32_t>(grid);
        }
    }
    QkArgs a;
    a.base = LaunchArgs{};
    a.base.stream = static_cast<cudaStream_t>(stream);
    a.base.pdl = pdl_enabled();
    a.q = q;
    a.k = k;
    a.qw = q_weight;
    a.kw = k_weight;
    a.tokens = tokens;
    a.q_heads = static_cast<int32_t>(q_heads);
    a.k_heads = static_cast<int32_t>(k_heads);
    a.head_dim = static_cast<int32_t>(head_dim);
    a.q_stride = qs;
    a.k_stride = ks;
    a.bias = weight_bias;
    a.eps = eps;
    a.grid = static_cast<int>(grid);
    if (kern->launch(a) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    return RMSNORM_OK;
}

int rmsnorm_qk_norm(void *q, void *k, const void *q_weight, const void *k_weight, int64_t tokens,
                    int64_t q_heads, int64_t k_heads, int64_t head_dim, int64_t q_token_stride,
                    int64_t k_token_stride, float weight_bias, float eps, int dtype, void *stream)
{
    return rmsnorm_qk_norm_ex(q, k, q_weight, k_weight, tokens, q_heads, k_heads, head_dim,
                              q_token_stride, k_token_stride, weight_bias, eps, dtype, stream,
                              nullptr);
}

int rmsnorm_plan(const void *x, const void *weight, const void *y, int64_t rows, int64_t hidden,
                 int dtype, int sm_count, int smem_optin, int variant, rmsnorm_plan_t *out)
{
    return plan_launch(x, weight, y, rows, hidden, dtype, sm_count, smem_optin, variant, out);
}

int rmsnorm_plan_host_mapped(const void *x_host, const void *weight, const void *y_host,
                             int64_t rows, int64_t hidden, int dtype, int sm_count,
                             int smem_optin, rmsnorm_plan_t *out)
{
    if (!out)
        return RMSNORM_ERR_INVALID_ARG;
    return plan_host_link(x_host, weight, y_host, rows, hidden, dtype, sm_count, smem_optin, out);
}

int rmsnorm_validate_plan(const rmsnorm_plan_t *plan, const void *x, const void *weight,
                          const void *y, int64_t rows, int64_t hidden, int dtype, int sm_count,
                          int smem_optin)
{
    if (!plan)
        return RMSNORM_ERR_INVALID_ARG;
    return validate_plan(*plan, x, weight, y, rows, hidden, dtype, sm_count, smem_optin);
}

int rmsnorm_plan_epilogue(const void *x, const void *weight, const void *y, int64_t rows,
                          int64_t hidden, int dtype, int epilogue, int sm_count, int smem_optin,
                          int variant, rmsnorm_plan_t *out)
{
    return plan_launch(x, weight, y, rows, hidden, dtype, sm_count, smem_optin, variant, out,
                       epilogue);
}

int rmsnorm_validate_plan_epilogue(const rmsnorm_plan_t *plan, const void *x,
                                   const void *weight, const void *y, int64_t rows,
                                   int64_t hidden, int dtype, int epilogue, int sm_count,
                                   int smem_optin)
{
    if (!plan)
        return RMSNORM_ERR_INVALID_ARG;
    return validate_plan(*plan, x, weight, y, rows, hidden, dtype, sm_count, smem_optin,
                         epilogue);
}

int rmsnorm_device_limits(int *sm_count, int *smem_optin)
{
    if (!sm_count || !smem_optin)
        return RMSNORM_ERR_INVALID_ARG;
    DeviceCtx ctx;
    int rc = current_ctx(&ctx, nullptr);
    if (rc != RMSNORM_OK)
        return rc;
    *sm_count = ctx.sm_count;
    *smem_optin = ctx.smem_optin;
    return RMSNORM_OK;
}

int rmsnorm_kernel_count(void)
{
    int n = 0;
    kernel_table(&n);
    return n;
}

int rmsnorm_kernel_info(int index, rmsnorm_kernel_info_t *out)
{
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    if (!out || index < 0 || index >= n)
        return RMSNORM_ERR_INVALID_ARG;
    const KernelDesc &d = t[index];
    out->variant = d.variant;
    out->dtype = d.dtype;
    out->vec_bytes = d.vec_bytes;
    out->tpr = d.tpr;
    out->nv = d.nv;
    out->block = d.block;
    out->min_blocks = d.minb;
    out->cache_policy = d.cache;
    out->epilogue = d.epi;
    return RMSNORM_OK;
}

int rmsnorm_last_variant(void)
{
    return t_last_variant;
}

int rmsnorm_get_device_status(int *status)
{
    if (!status)
        return RMSNORM_ERR_INVALID_ARG;
    DeviceCtx ctx;
    int rc = current_ctx(&ctx, nullptr);
    if (rc != RMSNORM_OK)
        return rc;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ctx.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (cudaMemset(ctx.status, 0, sizeof(int)) != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess)
        return RMSNORM_ERR_CUDA;
    *status = v;
    return RMSNORM_OK;
}

int rmsnorm_set_wait_limit_ns(uint64_t limit_ns)
{
    g_wait_limit.store(limit_ns ? limit_ns : kDefaultWaitLimitNs);
    return RMSNORM_OK;
}

int rmsnorm_set_pdl(int enable)
{
    if (enable != 0 && enable != 1)
        return RMSNORM_ERR_INVALID_ARG;
    g_pdl.store(enable);
    return RMSNORM_OK;
}

int rmsnorm_get_pdl(void)
{
    return pdl_enabled() ? 1 : 0;
}

int rmsnorm_test_staged_timeout(const void *x, const void *weight, void *y, int64_t rows,
                                int64_t hidden, int dtype, uint64_t limit_ns, void *stream)
{
    if (rows <= 0 || limit_ns == 0)
        return RMSNORM_ERR_INVALID_ARG;
    return launch(x, weight, y, rows, hidden, 0.f, dtype, stream, RMSNORM_VARIANT_STAGED, nullptr,
                  kFlagWithholdCopies, limit_ns);
}

int rmsnorm_test_grid_timeout(const void *x, const void *weight, void *y, int64_t rows,
                              int64_t hidden, int dtype, uint64_t limit_ns, void *stream)
{
    if (rows <= 0 || limit_ns == 0)
        return RMSNORM_ERR_INVALID_ARG;
    return launch(x, weight, y, rows, hidden, 0.f, dtype, stream, RMSNORM_VARIANT_GRID, nullptr,
                  kFlagWithholdCopies, limit_ns);
}

const char *rmsnorm_status_string(int status)
{
    switch (status) {
    case RMSNORM_OK:
        return "ok";
    case RMSNORM_ERR_INVALID_ARG:
        return "invalid argument";
    case RMSNORM_ERR_UNSUPPORTED_DTYPE:
        return "unsupported dtype";
    case RMSNORM_ERR_NOT_INITIALIZED:
        return "no context on the current device (call rmsnorm_create)";
    case RMSNORM_ERR_ALIASING:
        return "y partially overlaps x or overlaps weight";
    case RMSNORM_ERR_CUDA:
        return "CUDA runtime error";
    case RMSNORM_ERR_DEVICE_TIMEOUT:
        return "a bounded device-side wait ran out";
    case RMSNORM_ERR_MISALIGNED:
        return "pointers or row length not aligned for the forced vector variant";
    case RMSNORM_ERR_UNSUPPORTED_DEVICE:
        return "device is not compute capability 10.3 (sm_103a)";
    case RMSNORM_ERR_VARIANT:
        return "the forced variant or plan cannot take this shape";
    case RMSNORM_ERR_TOO_LARGE:
        return "beyond the static scratch of the allocation-free entry point";
    default:
        return "unknown status";
    }
}

int rmsnorm_version(void)
{
    return (1 << 16) | 0;
}

} // extern "C"
