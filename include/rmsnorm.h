/*
 * rmsnorm.h -- C ABI of the GB300 (sm_103a) row-wise RMSNorm forward library
 * (librmsnorm.so).
 *
 * The operation.  "Build a GPU compiler from scratch: from PyTorch to CUDA via
 * multi-level IR (Emmy)", introduction and section "Tensor IR": for every row
 * take the mean of the squared elements, add epsilon, take the reciprocal
 * square root, and scale every element by that factor and by its learned
 * weight; section "Loop IR": all of it is one fused kernel whose row
 * statistic never leaves the chip.  "CuTeDSL at Perplexity", section "QK
 * Norm": the squares are summed in fp32, the factor is rsqrt(sum/n + EPS),
 * each output is weight * (x * factor) cast back to the input's element type,
 * and the store may overwrite the input.
 *
 *   y[i, j] = round( (x[i, j] * r_i) * w[j] ),   r_i = rsqrt( sum_j x[i, j]^2 / hidden + eps )
 *
 * computed in fp32 on the device and rounded to the element type with
 * round-to-nearest-even.  Variants of the output (the "epilogues": a weight
 * offset, MXFP8 / MXFP4 / NVFP4 block-scaled codes) and the per-head QK norm
 * are declared further down, each with its own definition.
 *
 * Memory layout.  x and y are row-major [rows, hidden], contiguous (row
 * stride = hidden elements); weight is [hidden].  x, weight and y share one
 * element type.  All three are DEVICE pointers owned by the caller; the
 * library never frees or retains them.  The only memory the library itself
 * allocates is its per-device context, at rmsnorm_create: a 4-byte device
 * status word, the grid variant's fixed scratch and host-side state.  No
 * call after rmsnorm_create allocates device memory.
 *
 * Aliasing.  y == x (exactly in place) is allowed.  Any other overlap between
 * y and x, or between y and weight, is rejected with RMSNORM_ERR_ALIASING.
 *
 * Asynchrony and errors.  rmsnorm_fwd only validates and enqueues at most
 * one kernel on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 * default stream); it never synchronises.  Argument errors are reported
 * before anything is enqueued.  A launch failure returns RMSNORM_ERR_CUDA.
 * Device-side faults the kernels can detect themselves (a bounded wait that
 * ran out) are recorded in the device status word, read with
 * rmsnorm_get_device_status.  No function throws across this boundary and
 * none aborts the process.
 *
 * Threads.  All functions may be called from any host thread; the context
 * table is guarded by a mutex.  Contexts are per CUDA device: create on each
 * device you use, with that device current.
 */
#ifndef RMSNORM_H
#define RMSNORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type shared by x, weight and y. */
typedef enum {
    RMSNORM_F32 = 0,  /* IEEE binary32 */
    RMSNORM_BF16 = 1, /* bfloat16 */
    RMSNORM_F16 = 2   /* IEEE binary16 */
} rmsnorm_dtype_t;

typedef enum {
    RMSNORM_OK = 0,
    RMSNORM_ERR_INVALID_ARG = 1,        /* null pointer, rows < 0, hidden <= 0, eps < 0 or NaN, bad plan */
    RMSNORM_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype not one of rmsnorm_dtype_t */
    RMSNORM_ERR_NOT_INITIALIZED = 3,    /* no rmsnorm_create on the current device */
    RMSNORM_ERR_ALIASING = 4,           /* y partially overlaps x, or overlaps weight */
    RMSNORM_ERR_CUDA = 5,               /* a CUDA runtime call or a launch failed */
    RMSNORM_ERR_DEVICE_TIMEOUT = 6,     /* a kernel's bounded wait ran out (device status word) */
    RMSNORM_ERR_MISALIGNED = 7,         /* a forced vector variant got pointers it cannot load */
    RMSNORM_ERR_UNSUPPORTED_DEVICE = 8, /* current device is not compute capability 10.3 */
    RMSNORM_ERR_VARIANT = 9,            /* forced variant cannot take this shape */
    RMSNORM_ERR_TOO_LARGE = 10          /* beyond the static scratch of rmsnorm_fwd_staged_noalloc */
} rmsnorm_status_t;

/* What a row kernel writes (see rmsnorm_fwd_bias and rmsnorm_fwd_mxfp8). */
typedef enum {
    RMSNORM_EPI_PLAIN = 0, /* y = round((x * r) * w) in the element type */
    RMSNORM_EPI_BIAS = 1,  /* y = round((x * r) * (w + weight_bias)) in the element type */
    RMSNORM_EPI_MXFP8 = 2, /* (x * r) * (w + weight_bias) as MXFP8: E4M3 codes + E8M0 scales */
    RMSNORM_EPI_MXFP4 = 3, /* ... as MXFP4: packed E2M1 codes + E8M0 scales per 32 */
    RMSNORM_EPI_NVFP4 = 4  /* ... as NVFP4: packed E2M1 codes + E4M3 scales per 16 */
} rmsnorm_epilogue_t;

/* Kernel variants.  AUTO lets the selector choose from (rows, hidden, dtype,
 * pointer alignment, SM count). */
typedef enum {
    RMSNORM_VARIANT_AUTO = 0,
    /* A group of 4..32 lanes of one warp per row; the row stays in registers;
     * the reduction is warp shuffles only.  Small hidden. */
    RMSNORM_VARIANT_WARP_PER_ROW = 1,
    /* One thread block per row; the row stays in registers; warp shuffles,
     * then one float per warp through shared memory.  Medium/large hidden. */
    RMSNORM_VARIANT_CTA_PER_ROW = 2,
    /* Persistent blocks (one or two per SM) stream whole rows global ->
     * shared with cp.async.bulk into a ring of slots guarded by mbarriers
     * (bounded waits); one consumer warp per row.  Large hidden. */
    RMSNORM_VARIANT_STAGED = 3,
    /* Decode shapes: the block-per-row body with grid <= SM count and a
     * grid-stride row loop. */
    RMSNORM_VARIANT_PERSISTENT = 4,
    /* Any hidden and any element alignment: scalar loads, two passes over
     * the row (the second from cache).  Fallback for ragged shapes. */
    RMSNORM_VARIANT_GENERIC = 5,
    /* Decode shapes with long rows: each row split over a thread-block
     * cluster of 2, 4 or 8 blocks (on as many SMs); the blocks' partial sums
     * meet through distributed shared memory.  Plain output only. */
    RMSNORM_VARIANT_CLUSTER = 6,
    /* Decode shapes with rows longer than a cluster holds: every row spread
     * over all SMs (a cooperative launch of 2 blocks per SM), one grid
     * barrier through global memory between the sums and the scaling
     * (bounded wait; a wait that runs out records RMSNORM_ERR_DEVICE_TIMEOUT).
     * Its counters and partial sums live in the context's fixed scratch,
     * shared by every grid-variant call on the device: each such call makes
     * its stream wait for the previous one (an event the context records
     * after each), so calls on different streams take turns.  Calls captured
     * into a CUDA graph are ordered by the graph alone: a replay must not
     * overlap another grid-variant call.  Plain output only; at most 64
     * rows. */
    RMSNORM_VARIANT_GRID = 7
} rmsnorm_variant_t;

/* A launch plan: what the selector chose.  Filled by rmsnorm_plan. */
typedef struct {
    int32_t variant;         /* rmsnorm_variant_t (never AUTO) */
    int32_t vec_bytes;       /* bytes per vector access: 16 or 32; 0 = scalar */
    int32_t threads_per_row; /* threads cooperating on one row (staged: 32) */
    int32_t vecs_per_thread; /* register-resident vectors per thread per row */
    int32_t block_threads;   /* threads per block */
    int32_t rows_per_block;  /* rows a block works on at once */
    int32_t stages;          /* staged: row slots in shared memory; cluster: blocks per row
                              * (the cluster size, 2, 4 or 8); else 0 */
    int32_t grid;            /* blocks launched (0 when rows == 0) */
    int32_t smem_bytes;      /* dynamic shared memory per block */
    int32_t kernel_index;    /* internal instantiation index */
} rmsnorm_plan_t;

/* Create (or add a reference to) the context of the CURRENT CUDA device:
 * queries SM count, shared memory limits and compute capability (must be
 * 10.3; the kernels are built for sm_103a), and allocates everything the
 * library will ever hold on the device: the device status word and the grid
 * variant's fixed scratch (16 + 64 rows * 2 blocks per SM * SMs * 8 bytes,
 * about 156 KB on a 152-SM GB300), both zeroed.  It waits for those zeroing
 * copies (the legacy default stream), so call it outside any stream capture.
 * Idempotent and reference counted.  Returns RMSNORM_OK,
 * RMSNORM_ERR_UNSUPPORTED_DEVICE or RMSNORM_ERR_CUDA. */
int rmsnorm_create(void);

/* Drop one reference to the current device's context; at zero the status
 * word and the scratch are freed.  Returns RMSNORM_ERR_NOT_INITIALIZED if
 * there is none. */
int rmsnorm_destroy(void);

/* y = RMSNorm(x) * weight, per row (see the top of this file).
 *   x       device pointer, [rows, hidden] elements of `dtype`
 *   weight  device pointer, [hidden] elements of `dtype`
 *   y       device pointer, [rows, hidden]; may equal x
 *   rows    >= 0 (0 returns RMSNORM_OK and launches nothing)
 *   hidden  >= 1
 *   eps     >= 0, finite (added to the mean square before the rsqrt)
 *   dtype   rmsnorm_dtype_t
 *   stream  cudaStream_t (as void*); NULL = legacy default stream
 * Enqueues one kernel; does not synchronise. */
int rmsnorm_fwd(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                float eps, int dtype, void *stream);

/* rmsnorm_fwd with a forced variant (RMSNORM_VARIANT_AUTO = selector's choice)
 * and an optional plan override: when `plan` is non-NULL and plan->variant
 * is not AUTO, that exact plan is launched after validation against the
 * shape (benchmark sweeps); when `plan` is non-NULL and plan->variant is
 * AUTO, the chosen plan is written back into it.
 *
 * The environment variable RMSNORM_FORCE_VARIANT (a variant name without
 * its prefix -- warp_per_row, cta_per_row, staged, persistent, generic,
 * cluster, grid -- or its number), read once per process, replaces the
 * automatic choice of every device call that asks for one (rmsnorm_fwd, the
 * epilogue calls, and this call with variant AUTO and no explicit plan), so
 * a program can be run on one body without code changes; a shape that body
 * cannot take returns RMSNORM_ERR_VARIANT or RMSNORM_ERR_MISALIGNED.  The
 * host-only planners (rmsnorm_plan, rmsnorm_plan_epilogue) ignore it. */
int rmsnorm_fwd_ex(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                   float eps, int dtype, void *stream, int variant, rmsnorm_plan_t *plan);

/* ---- epilogues ("CuTeDSL at Perplexity": section "QK Norm" for the weight
 * offset WEIGHT_BIAS; section "Blackwell support" for the MXFP8 / MXFP4 /
 * NVFP4 block formats whose absolute maxima are taken over 16 or 32
 * elements) ---------------------------------------------------------------- */

/* Row normalisation with a weight offset, as the per-head kernel applies it:
 *
 *   y[i, j] = round( (x[i, j] * r_i) * (w[j] + weight_bias) )
 *
 * with w[j] + weight_bias formed in fp32 (weight_bias = -0.0f gives exactly
 * rmsnorm_fwd's result; +0.0f may differ from it only in the sign of zero
 * outputs of zero weights).  Arguments, layout, aliasing (y == x allowed),
 * errors and asynchrony as rmsnorm_fwd.  weight_bias must be finite. */
int rmsnorm_fwd_bias(const void *x, const void *weight, void *y, int64_t rows, int64_t hidden,
                     float weight_bias, float eps, int dtype, void *stream);

/* Fused RMSNorm -> MXFP8.  The normalised values v[i, j] = (x[i, j] * r_i) *
 * (w[j] + weight_bias), held in fp32, leave as the OCP Microscaling (MX)
 * v1.0 format MXFP8 with E4M3 elements (the pages name the format; its
 * definition is the MX specification's):
 *
 *   for every 32 consecutive elements of a row (block b = j / 32):
 *     s = floor(log2(max |v|)) - 8, clamped to [-127, 127]  (8 = E4M3's largest exponent)
 *     scales[i, b] = s + 127        (E8M0; 0xFF when the block holds a NaN or an infinity;
 *                                    an all-zero block gets s = -127)
 *     q[i, j] = E4M3( v[i, j] / 2^s )   (nearest-even, saturating at +-448)
 *
 *   x      [rows, hidden] of `dtype` (device), 16-byte aligned
 *   weight [hidden] of `dtype` (device), 16-byte aligned
 *   q      [rows, hidden] bytes (device, E4M3 codes), 16-byte aligned
 *   scales [rows, hidden / 32] bytes (device, E8M0 codes), row-major, any alignment
 *
 * hidden must be a multiple of 32 (RMSNORM_ERR_INVALID_ARG otherwise);
 * misaligned x / weight / q give RMSNORM_ERR_MISALIGNED (there is no scalar
 * MX body).  q and scales may not overlap each other, x or weight
 * (RMSNORM_ERR_ALIASING).  Otherwise as rmsnorm_fwd.
 *
 * weight_bias = -0.0f means no offset (w exactly; +0.0f turns a -0 weight
 * into +0, which shows in the sign of that element's zero code).  With
 * -0.0f and bf16 / f16 elements the device forms the same values as
 * (x * w) * r, x * w exact (a faster path; the results agree with the
 * definition above within the 1e-5 relative band the decisions are checked
 * with); a block whose products leave [2^-100, 2^100) is formed in the
 * order above.  This holds for all three block-scaled formats. */
int rmsnorm_fwd_mxfp8(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float weight_bias, float eps, int dtype, void *stream);

/* Fused RMSNorm -> MXFP4: as rmsnorm_fwd_mxfp8 with E2M1 elements (OCP MX
 * v1.0): per 32 elements s = floor(log2(max |v|)) - 2 (2 = E2M1's largest
 * exponent), clamped to [-127, 127], scales[i, b] = s + 127 (0xFF for a
 * NaN / Inf block, 0 for an all-zero block); each element v / 2^s rounded to
 * E2M1 (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; nearest-even, saturating at
 * +-6).  q is [rows, hidden / 2] bytes, two 4-bit codes per byte, element
 * 2k in the low nibble of byte k; scales [rows, hidden / 32].  hidden must
 * be a multiple of 32.  Pointer, aliasing and error rules as
 * rmsnorm_fwd_mxfp8. */
int rmsnorm_fwd_mxfp4(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float weight_bias, float eps, int dtype, void *stream);

/* Fused RMSNorm -> NVFP4 (NVIDIA's description of the format: E2M1
 * elements, an E4M3 scale per 16 elements, a per-tensor fp32 scale g =
 * global_scale, a value standing for code * scale * g):
 *
 *   per 16 consecutive elements of a row (block b = j / 16):
 *     scales[i, b] = E4M3( max |v| / (6 * g) )     (nearest-even, saturating at 448;
 *                                                    0x7F when the block holds a NaN)
 *     q[i, j]      = E2M1( v[i, j] / (value(scales[i, b]) * g) )   (0 when the scale is 0)
 *
 * The device forms 1 / (6 g) and 1 / (value * g) once per block and
 * multiplies.  q is [rows, hidden / 2] bytes packed as for MXFP4; scales
 * [rows, hidden / 16] bytes.  hidden must be a multiple of 16, global_scale
 * positive and finite (RMSNORM_ERR_INVALID_ARG otherwise). */
int rmsnorm_fwd_nvfp4(const void *x, const void *weight, void *q, void *scales, int64_t rows,
                      int64_t hidden, float global_scale, float weight_bias, float eps,
                      int dtype, void *stream);

/* Any epilogue with a forced variant or an explicit plan (as rmsnorm_fwd_ex;
 * `scales` is used by the block-scaled epilogues only, `weight_bias` by all
 * but PLAIN, `global_scale` by NVFP4 only).  The bulk-copy staged and the
 * cluster variants exist for RMSNORM_EPI_PLAIN only: the automatic choice
 * uses the register or looped bodies instead, and forcing them returns
 * RMSNORM_ERR_VARIANT. */
int rmsnorm_fwd_epilogue_ex(const void *x, const void *weight, void *y, void *scales,
                            int64_t rows, int64_t hidden, int epilogue, float weight_bias,
                            float global_scale, float eps, int dtype, void *stream, int variant,
                            rmsnorm_plan_t *plan);

/* The selector for an epilogue (host only, as rmsnorm_plan). */
int rmsnorm_plan_epilogue(const void *x, const void *weight, const void *y, int64_t rows,
                          int64_t hidden, int dtype, int epilogue, int sm_count, int smem_optin,
                          int variant, rmsnorm_plan_t *out);

/* Host-only check of an explicit plan for an epilogue (as rmsnorm_validate_plan). */
int rmsnorm_validate_plan_epilogue(const rmsnorm_plan_t *plan, const void *x,
                                   const void *weight, const void *y, int64_t rows,
                                   int64_t hidden, int dtype, int epilogue, int sm_count,
                                   int smem_optin);

/* y = RMSNorm(x) * weight for x and y in HOST memory.  When both buffers
 * are page-locked host memory mapped into the device's address space (for
 * example from cudaHostAlloc or cudaHostRegister), the kernel reads x and
 * writes y there directly over the CPU-GPU link (NVLink-C2C on GB300), with
 * no staging and no use of the workspace, in the launch shape
 * rmsnorm_plan_host_mapped gives.  Otherwise rows are processed in
 * chunks through a device workspace the caller provides, with the upload of
 * one chunk, the kernel on the previous one and the download of the one
 * before that overlapped (two internal streams of this context plus
 * `stream` for the kernels; up to three buffers carved from the workspace).
 *   x_host, y_host  host pointers, [rows, hidden] of `dtype`; y_host may
 *                   equal x_host
 *   weight          DEVICE pointer, [hidden] of `dtype`
 *   workspace       DEVICE pointer to workspace_bytes the caller owns; it
 *                   must hold at least one row (256-byte aligned slices)
 *   chunk_rows      rows per chunk; 0 = about rows / 16, within the buffers
 *   stream          cudaStream_t (as void*): work already on it is ordered
 *                   before the first upload, and it waits for the last
 *                   download, so synchronising it makes y_host readable
 * Asynchronous like rmsnorm_fwd: x_host must stay valid and unmodified, and
 * y_host and the workspace untouched, until `stream` has passed this call.
 * Calls on one device enqueue one at a time (a mutex); their pipelines
 * share the context's two streams.  Returns the statuses of rmsnorm_fwd, or
 * RMSNORM_ERR_INVALID_ARG when the workspace cannot hold a row. */
int rmsnorm_fwd_host(const void *x_host, const void *weight, void *y_host, int64_t rows,
                     int64_t hidden, float eps, int dtype, void *workspace,
                     size_t workspace_bytes, int64_t chunk_rows, void *stream);

/* The selector for rmsnorm_fwd_host's page-locked path, host only (as
 * rmsnorm_plan; x_host and y_host are used for their alignment only): the
 * plan rmsnorm_plan would choose, except that a block-per-row or persistent
 * grid of the register bodies with more than two blocks per SM becomes a
 * persistent grid of two blocks per SM.  Over the CPU-GPU link the link sets
 * the pace and the wide grid only adds requests in flight (measured on GB300,
 * 16384 x 4096 bf16 host to host: 337 against 322 GB/s).  Returns the
 * statuses of rmsnorm_plan. */
int rmsnorm_plan_host_mapped(const void *x_host, const void *weight, const void *y_host,
                             int64_t rows, int64_t hidden, int dtype, int sm_count,
                             int smem_optin, rmsnorm_plan_t *plan);

/* Per-head QK norm, in place ("CuTeDSL at Perplexity", section "QK Norm"):
 * every head of q and of k is RMS-normalised over its head_dim elements,
 *   x[d] <- (x[d] * rsqrt(sum_e x[e]^2 / head_dim + eps)) * (w[d] + weight_bias)
 * with q_weight for q heads and k_weight for k heads, fp32 inside, rounded to
 * the element type; q and k in one launch.
 *   q, k            DEVICE pointers; token t's q heads are the q_heads *
 *                   head_dim contiguous elements starting at element
 *                   t * q_token_stride (0 = q_heads * head_dim, i.e.
 *                   contiguous [tokens, q_heads, head_dim]); likewise k.
 *                   Strides let q and k be views into one fused QKV buffer.
 *   q_weight, k_weight  DEVICE pointers, [head_dim] each; may be equal
 *   q_heads, k_heads    >= 0 (either may be 0; its pointers may then be NULL)
 *   weight_bias     added to every weight element (0 for plain weights,
 *                   1 for "1 + w" parameterisations)
 *   eps             >= 0, finite
 * Heads whose bytes start on 16-byte boundaries (pointers, head_dim and
 * strides) take the vector kernel (a group of lanes per head); others a
 * scalar warp-per-head kernel.  Returns RMSNORM_OK, RMSNORM_ERR_INVALID_ARG
 * (bad sizes, a stride shorter than its heads, a missing pointer),
 * RMSNORM_ERR_UNSUPPORTED_DTYPE, RMSNORM_ERR_ALIASING (a q head and a k head
 * share bytes, or a weight lies inside a head), RMSNORM_ERR_NOT_INITIALIZED
 * or RMSNORM_ERR_CUDA.  Asynchronous on `stream`. */
int rmsnorm_qk_norm(void *q, void *k, const void *q_weight, const void *k_weight, int64_t tokens,
                    int64_t q_heads, int64_t k_heads, int64_t head_dim, int64_t q_token_stride,
                    int64_t k_token_stride, float weight_bias, float eps, int dtype, void *stream);

/* Launch shape of rmsnorm_qk_norm_ex: lanes_per_head lanes of a warp own a
 * head (-1: the scalar warp-per-head body), each with vecs_per_lane 16-byte
 * vectors; a lane group takes heads_per_group heads per iteration of a
 * grid-stride loop over grid blocks of 256 threads. */
typedef struct {
    int32_t lanes_per_head;
    int32_t vecs_per_lane;
    int32_t heads_per_group;
    int32_t grid;
} rmsnorm_qk_plan_t;

/* rmsnorm_qk_norm with a launch shape: plan == NULL or
 * plan->lanes_per_head == 0 chooses automatically (and, with a plan, writes
 * the choice back); otherwise the given shape is launched if a compiled body
 * matches it and its vectors cover the head (else RMSNORM_ERR_VARIANT). */
int rmsnorm_qk_norm_ex(void *q, void *k, const void *q_weight, const void *k_weight,
                       int64_t tokens, int64_t q_heads, int64_t k_heads, int64_t head_dim,
                       int64_t q_token_stride, int64_t k_token_stride, float weight_bias,
                       float eps, int dtype, void *stream, rmsnorm_qk_plan_t *plan);

/* The selector, host only (touches no memory behind the pointers and no
 * GPU): the plan rmsnorm_fwd_ex would launch for these arguments on a device
 * with `sm_count` SMs and `smem_optin` bytes of opt-in shared memory per
 * block.  Pointer values are used only for their alignment.  Returns
 * RMSNORM_OK, RMSNORM_ERR_INVALID_ARG, RMSNORM_ERR_UNSUPPORTED_DTYPE,
 * RMSNORM_ERR_MISALIGNED or RMSNORM_ERR_VARIANT. */
int rmsnorm_plan(const void *x, const void *weight, const void *y, int64_t rows, int64_t hidden,
                 int dtype, int sm_count, int smem_optin, int variant, rmsnorm_plan_t *out);

/* One compiled kernel instantiation, for building explicit plans (tuning
 * sweeps).  tpr / nv / block of 0 mean "chosen at launch". */
typedef struct {
    int32_t variant;   /* WARP_PER_ROW, CTA_PER_ROW (also used for PERSISTENT), STAGED, GENERIC */
    int32_t dtype;     /* rmsnorm_dtype_t */
    int32_t vec_bytes; /* 16 / 32; 0 = scalar */
    int32_t tpr;       /* threads per row fixed at compile time (warp-per-row) */
    int32_t nv;        /* vectors per thread fixed at compile time */
    int32_t block;     /* block size fixed at compile time, or the largest allowed */
    int32_t min_blocks;   /* resident blocks per SM the build was register-capped for; 0 = none */
    int32_t cache_policy; /* 0 plain, 1 L2 256-byte prefetch hint, 2 streaming (.cs) loads and
                           * stores, 3 staged rows written back by bulk copies */
    int32_t epilogue;     /* rmsnorm_epilogue_t the instantiation writes */
} rmsnorm_kernel_info_t;

/* SM count and opt-in shared memory per block of the current device, as
 * cached by rmsnorm_create (the values the selector uses).  Returns
 * RMSNORM_OK, RMSNORM_ERR_NOT_INITIALIZED or RMSNORM_ERR_INVALID_ARG. */
int rmsnorm_device_limits(int *sm_count, int *smem_optin);

/* Number of compiled kernel instantiations (host only, no GPU needed). */
int rmsnorm_kernel_count(void);

/* Describe instantiation `index` (0 <= index < rmsnorm_kernel_count()).
 * Returns RMSNORM_OK or RMSNORM_ERR_INVALID_ARG. */
int rmsnorm_kernel_info(int index, rmsnorm_kernel_info_t *out);

/* Host-only check of an explicit plan against a call's arguments on a device
 * with `sm_count` SMs and `smem_optin` bytes of opt-in shared memory per
 * block: the check rmsnorm_fwd_ex applies before launching a caller-supplied
 * plan.  Pointer values are used only for their alignment.  Returns
 * RMSNORM_OK or the status rmsnorm_fwd_ex would return. */
int rmsnorm_validate_plan(const rmsnorm_plan_t *plan, const void *x, const void *weight,
                          const void *y, int64_t rows, int64_t hidden, int dtype, int sm_count,
                          int smem_optin);

/* Variant of the last successful launch on the calling thread (0 if none). */
int rmsnorm_last_variant(void);

/* Copy the current device's status word to *status (RMSNORM_OK, or the
 * first device-side error recorded since the last read) and clear it.
 * Synchronises the device's legacy default stream.  Returns RMSNORM_OK,
 * RMSNORM_ERR_NOT_INITIALIZED, RMSNORM_ERR_INVALID_ARG or RMSNORM_ERR_CUDA. */
int rmsnorm_get_device_status(int *status);

/* Upper bound, in nanoseconds of %globaltimer, on every spin-wait inside the
 * staged kernel (default 1e9 = one second).  After it runs out the kernel
 * records RMSNORM_ERR_DEVICE_TIMEOUT, waits (again bounded) for its own
 * copies in flight, and returns.  0 restores the default. */
int rmsnorm_set_wait_limit_ns(uint64_t limit_ns);

/* Programmatic dependent launch ("CuTeDSL at Perplexity", section "Grid
 * synchronization", names it as the way to cut launch overhead between
 * kernels).  When on, every launch carries the programmatic stream
 * serialization attribute: the kernel may be scheduled while the previous
 * kernel on the stream is still finishing, and waits (griddepcontrol.wait)
 * for that kernel's completion and memory before its first global access,
 * so results are unchanged.  Process-wide; the initial value is on unless
 * the environment variable RMSNORM_PDL is "0".  rmsnorm_set_pdl returns
 * RMSNORM_OK or RMSNORM_ERR_INVALID_ARG (enable not 0 or 1);
 * rmsnorm_get_pdl returns the current setting (0 or 1). */
int rmsnorm_set_pdl(int enable);
int rmsnorm_get_pdl(void);

/* Failure-detection test hook: launch the staged kernel on a valid shape
 * with its row copies withheld, so every consumer wait runs out after
 * `limit_ns`; the kernel then records RMSNORM_ERR_DEVICE_TIMEOUT and returns
 * without touching y.  No fault, trap or hang is involved. */
int rmsnorm_test_staged_timeout(const void *x, const void *weight, void *y, int64_t rows,
                                int64_t hidden, int dtype, uint64_t limit_ns, void *stream);

/* Failure-detection test hook for the grid variant: the grid-barrier
 * arrival of block 0 is withheld, so every block's bounded wait runs out
 * after `limit_ns`; the kernel records RMSNORM_ERR_DEVICE_TIMEOUT, leaves y
 * untouched and clears its barrier counters.  rows in 1..64.  No fault,
 * trap or hang is involved. */
int rmsnorm_test_grid_timeout(const void *x, const void *weight, void *y, int64_t rows,
                              int64_t hidden, int dtype, uint64_t limit_ns, void *stream);

/* rmsnorm_fwd for callers that cannot allocate device memory.
 *
 * Some callers may not call cudaMalloc or anything that allocates: code
 * running inside a caller-managed memory pool or arena that must stay the
 * only owner of device memory, code that runs under a fixed memory budget
 * where an allocation mid-stream is not allowed, or a library embedded in a
 * host process whose allocator policy forbids it.  rmsnorm_create allocates
 * a device status word, so those callers cannot use rmsnorm_fwd.  This entry
 * point needs no rmsnorm_create and allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine): it runs the shared-memory-staged
 * kernel (RMSNORM_VARIANT_STAGED; same arithmetic as rmsnorm_fwd) and keeps
 * that kernel's status words in a static device array of 1024 ints (4 KiB,
 * one word per block of the launch), which every device that loads the
 * library holds until the process exits.  (The method's pages have no
 * counterpart of this entry point; it is a property of this library.)
 *
 * Arguments, layout, aliasing and asynchrony are those of rmsnorm_fwd; the
 * caller owns x, weight and y.  The first call on a device does a one-time
 * set-up with that device current (it looks up the static array's device
 * address and the device's limits); make that first call before any stream
 * capture.  Returns RMSNORM_OK, an argument error as rmsnorm_fwd does,
 * RMSNORM_ERR_UNSUPPORTED_DEVICE, RMSNORM_ERR_CUDA, RMSNORM_ERR_MISALIGNED
 * when x, weight or y is not 16-byte aligned or a row's byte length is not a
 * multiple of 16 (the staged kernel copies whole rows with bulk copies;
 * rmsnorm_fwd takes such shapes through its scalar body, this entry point
 * does not), or RMSNORM_ERR_TOO_LARGE when the row does not fit the staged
 * kernel's shared memory or the launch would need more than 1024 blocks.
 *
 * Every call shares the static array and it keeps the last call's contents;
 * each block clears its own word when it starts.  Calls that overlap on the
 * GPU (different streams, no ordering between them) race on the array.  A
 * bounded wait that runs out inside the kernel is not reported through
 * rmsnorm_get_device_status: the block's word records it and the rows that
 * block could not compute are written as NaN. */
int rmsnorm_fwd_staged_noalloc(const void *x, const void *weight, void *y, int64_t rows,
                               int64_t hidden, float eps, int dtype, void *stream);

/* Failure-detection test hook for rmsnorm_fwd_staged_noalloc (eps 1e-6):
 * the row copies are withheld, so every bounded wait runs out after
 * `limit_ns`; each block records RMSNORM_ERR_DEVICE_TIMEOUT in its word of
 * the static array and writes its rows as NaN.  No fault, trap or hang is
 * involved.  Allocates nothing. */
int rmsnorm_test_staged_noalloc_timeout(const void *x, const void *weight, void *y, int64_t rows,
                                        int64_t hidden, int dtype, uint64_t limit_ns,
                                        void *stream);

/* Copies the first n (<= 1024) words of rmsnorm_fwd_staged_noalloc's static
 * status array (one per block of the last launch: 0, or
 * RMSNORM_ERR_DEVICE_TIMEOUT) to host memory, after waiting for the device
 * (a blocking copy).  The same one-time set-up as that entry point; allocates
 * nothing.  Returns RMSNORM_OK, RMSNORM_ERR_INVALID_ARG, RMSNORM_ERR_CUDA or
 * RMSNORM_ERR_UNSUPPORTED_DEVICE. */
int rmsnorm_noalloc_block_status(int *host_out, int n);

/* Static text for a status code. */
const char *rmsnorm_status_string(int status);

/* Library version, (major << 16) | minor. */
int rmsnorm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_H */
