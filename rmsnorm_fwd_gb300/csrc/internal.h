// internal.h -- shared between the host side (api.cpp, select.cpp) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "rmsnorm.h"

#if defined(__CUDACC__)
#define RMSNORM_HD __host__ __device__
#else
#define RMSNORM_HD
#endif

namespace rmsnorm {

// Everything one launch needs besides the plan.
struct LaunchArgs {
    const void *x;
    const void *w;
    void *y;
    int64_t rows;
    int32_t hidden;
    float eps;
    int *status;            // device status word (staged variant's bounded waits)
    uint64_t wait_limit_ns; // bound on every spin-wait, %globaltimer ns
    uint32_t flags;         // kFlagWithholdCopies: failure-detection test only
    cudaStream_t stream;
    bool pdl = false;       // launch with a programmatic dependency on the stream's last kernel
    float bias = -0.0f;     // weight offset (every epilogue but PLAIN); -0 adds nothing
    void *scales = nullptr; // block-scaled epilogues: the scales; y holds the codes
    float gscale = 1.0f;    // NVFP4: the per-tensor scale
    void *scratch = nullptr; // grid variant: counters + partial sums (the context's, from create)
    bool xw = false;        // block-scaled output formed from exact x * w products (q_store)
};

// Whether a block-scaled output of 16-bit elements may form its values from
// the exact products x * w (q_store's second instantiation): the weight
// offset is -0 (adds nothing, zeros' signs included) and, for NVFP4, every
// scale value times the per-tensor scale g and its reciprocal are normal
// floats (g in [2^-117, 2^100]).
inline bool quant_exact_products(int dtype, int epi, float bias, float gscale)
{
    if (dtype == RMSNORM_F32 || epi < RMSNORM_EPI_MXFP8)
        return false;
    uint32_t bits;
    std::memcpy(&bits, &bias, sizeof bits);
    if (bits != 0x80000000u)
        return false;
    return epi != RMSNORM_EPI_NVFP4 || (gscale >= 0x1p-117f && gscale <= 0x1p100f);
}

// Instantiations with the exact-product form exist for 16-bit elements'
// block-scaled outputs only.
template <int DT, int EPI>
constexpr bool kHasExactProducts = DT != RMSNORM_F32 && EPI >= RMSNORM_EPI_MXFP8;

#if defined(__CUDACC__)
// Launches `kernel` on a.stream, with the programmatic-stream-serialization
// attribute when a.pdl is set (the kernels wait for their predecessor before
// touching memory, so the attribute only lets launches overlap).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int grid, int block, int smem,
                          const LaunchArgs &a, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    if (a.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    return err != cudaSuccess ? err : cudaGetLastError();
}
#endif

constexpr uint32_t kFlagWithholdCopies = 1u;

using LaunchFn = cudaError_t (*)(const rmsnorm_plan_t &, const LaunchArgs &);

// One compiled kernel instantiation.
struct KernelDesc {
    int32_t variant;     // WARP_PER_ROW, CTA_PER_ROW (also PERSISTENT), STAGED, GENERIC, CLUSTER
    int32_t dtype;       // rmsnorm_dtype_t
    int32_t vec_bytes;   // 16 / 32; 0 = scalar
    int32_t tpr;         // threads per row, compile time (warp kernels); 0 = runtime
    int32_t nv;          // vectors per thread, compile time; 0 = runtime loop
    int32_t block;       // threads per block, compile time; 0 = runtime
    int32_t minb;        // occupancy floor asked of the compiler (blocks per SM); 0 = none
    int32_t cache;       // memory path: 0 plain, 1 L2 256B prefetch, 2 streaming (.cs),
                         // 3 staged rows stored by bulk copies
    LaunchFn launch;
    const void *func;    // the __global__ function (attributes)
    int32_t epi = RMSNORM_EPI_PLAIN; // what it writes (rmsnorm_epilogue_t)
    const void *func_xw = nullptr; // its exact-product instantiation where the launcher has one
                                   // and it needs attributes set (staged: dynamic shared memory)
};

// Per translation unit tables, concatenated by kernel_table().
const KernelDesc *rowreg_kernels_f32(int *n);
const KernelDesc *rowreg_kernels_bf16(int *n);
const KernelDesc *rowreg_kernels_f16(int *n);
const KernelDesc *rowreg_epi_kernels_f32(int *n); // BIAS and MXFP8 epilogues
const KernelDesc *rowreg_epi_kernels_bf16(int *n);
const KernelDesc *rowreg_epi_kernels_f16(int *n);
const KernelDesc *rowreg_fp4_kernels_f32(int *n); // MXFP4 and NVFP4 epilogues
const KernelDesc *rowreg_fp4_kernels_bf16(int *n);
const KernelDesc *rowreg_fp4_kernels_f16(int *n);
const KernelDesc *staged_kernels(int *n);
const KernelDesc *cluster_kernels(int *n);
const KernelDesc *grid_kernels(int *n);

// Grid variant scratch: two 32-bit counters padded to 16 bytes, then
// rows * grid partial sums in binary64.
constexpr int64_t kGridCounterBytes = 16;
constexpr int kGridBlocksPerSm = 2;  // 512-thread blocks, <= 64 registers
constexpr int64_t kGridMaxRows = 64; // bounds the scratch: rows * grid doubles
const KernelDesc *generic_kernels(int *n);

const KernelDesc *kernel_table(int *n);

// Staged variant's shared-memory layout (host and device agree on it).
struct StagedLayout {
    int32_t row_bytes;   // hidden * element size (multiple of 16)
    int32_t slot_stride; // row_bytes rounded up to 128
    int32_t bar_bytes;   // mbarriers (2 per slot + weight + abort flag) and the
                         // consumer groups' reduction scratch, rounded to 128
    int32_t smem_bytes;  // total dynamic shared memory
};

RMSNORM_HD inline StagedLayout staged_layout(int32_t row_bytes, int32_t stages)
{
    StagedLayout L;
    L.row_bytes = row_bytes;
    L.slot_stride = (row_bytes + 127) / 128 * 128;
    L.bar_bytes = ((2 * stages + 2) * 8 + 256 + 127) / 128 * 128;
    L.smem_bytes = L.bar_bytes + L.slot_stride * (stages + 1); // +1: the weight row
    return L;
}

// Per-head QK norm (qknorm.cu).
struct QkArgs {
    LaunchArgs base; // stream and launch attributes
    void *q;
    void *k;
    const void *qw;
    const void *kw;
    int64_t tokens;
    int32_t q_heads;
    int32_t k_heads;
    int32_t head_dim;
    int64_t q_stride; // elements between tokens
    int64_t k_stride;
    float bias;
    float eps;
    int grid;
};
using QkLaunchFn = cudaError_t (*)(const QkArgs &);
struct QkKernel {
    int32_t dtype;
    int32_t tpr; // lanes per head; 0 = scalar warp-per-head body
    int32_t nv;  // 16-byte vectors per lane
    int32_t rpg; // heads a lane group takes per iteration
    QkLaunchFn launch;
};
const QkKernel *qk_kernels(int *n);

// Host-side selector (select.cpp).
int plan_launch(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                int dtype, int sm_count, int smem_optin, int variant, rmsnorm_plan_t *out,
                int epi = RMSNORM_EPI_PLAIN);

// Argument checks shared by every launching entry point (api.cpp).
int check_call_args(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                    float eps, int dtype);

// Checks a caller-supplied plan against the shape and the kernel table.
int validate_plan(const rmsnorm_plan_t &p, const void *x, const void *w, const void *y,
                  int64_t rows, int64_t hidden, int dtype, int sm_count, int smem_optin,
                  int epi = RMSNORM_EPI_PLAIN);

} // namespace rmsnorm
