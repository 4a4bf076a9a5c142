// select.cpp -- host-side variant and launch-shape selector.
//
// Inputs: rows, hidden, element type, pointer alignment, SM count and opt-in
// shared memory.  Output: one rmsnorm_plan_t naming a compiled kernel
// instantiation and its launch shape.  Pure host logic (no CUDA calls), so it
// is testable without a GPU.
//
// The rules follow "CuTeDSL at Perplexity", section "Prefill and decode
// specialization": pick the per-thread vector first (16 bytes: 8 x bf16/f16,
// 4 x f32; 32 bytes on Blackwell), derive how many threads a row needs, and
// size the grid against the SM count: when there are fewer rows than SMs
// (decode) give every row its own block on its own SM -- or, for rows too
// long for one SM, several SMs through a thread-block cluster or a grid
// barrier (same page, section "Grid synchronization"); when there are many
// (prefill) use enough warps per SM to keep HBM busy.  The SM count is read
// from the device at context creation, not compiled in (same page, section
// "Blackwell support").  The epilogue (rmsnorm_epilogue_t) narrows the
// choice to the bodies compiled for it and, for the block-scaled outputs,
// has launch shapes of its own.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "host_link.h"
#include "internal.h"

namespace rmsnorm {
namespace {

constexpr int64_t kMaxHidden = int64_t(1) << 26; // 64 Mi elements per row
constexpr int kMaxThreadsPerSm = 2048;
constexpr int kSmemPerSm = 233472;               // 228 KiB per SM on sm_100-class parts
constexpr int kSmemReservedPerBlock = 1024;
constexpr int kStagedMaxStages = 32;
constexpr int kStagedMaxConsumers = 16;
constexpr int kStagedMaxNamedGroups = 15; // named barriers 1..15 (0 is __syncthreads)

int elem_size(int dtype)
{
    return dtype == RMSNORM_F32 ? 4 : 2;
}

// Elements per scale block of an epilogue (1: not block-scaled).
int epi_block(int epi)
{
    return epi == RMSNORM_EPI_MXFP8 || epi == RMSNORM_EPI_MXFP4 ? 32
           : epi == RMSNORM_EPI_NVFP4                          ? 16
                                                               : 1;
}

bool aligned(const void *p, int a)
{
    return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(a)) == 0;
}

int round_up(int v, int m)
{
    return (v + m - 1) / m * m;
}

// Finds the table entry for (variant, dtype, vec_bytes, tpr, nv, cache,
// epilogue) with no occupancy cap; -1 if none.
int find_kernel(int variant, int dtype, int vec_bytes, int tpr, int nv, int cache, int epi)
{
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    for (int i = 0; i < n; ++i) {
        const KernelDesc &d = t[i];
        if (d.variant == variant && d.dtype == dtype && d.vec_bytes == vec_bytes &&
            d.tpr == tpr && d.nv == nv && d.cache == cache && d.minb == 0 && d.epi == epi)
            return i;
    }
    return -1;
}

struct Shape {
    int64_t rows;
    int64_t hidden;
    int dtype;
    int esize;
    int64_t row_bytes;
    bool a16;
    bool a32;
    int sm_count;
    int smem_optin;
    int epi; // rmsnorm_epilogue_t
};

void clear(rmsnorm_plan_t *p)
{
    *p = rmsnorm_plan_t{};
    p->kernel_index = -1;
}

int grid_for(int64_t units, int64_t cap)
{
    int64_t g = std::min<int64_t>(units, cap);
    g = std::min<int64_t>(g, INT_MAX);
    return static_cast<int>(std::max<int64_t>(g, 1));
}

// ---- generic: any shape
int plan_generic(const Shape &s, rmsnorm_plan_t *p)
{
    clear(p);
    p->variant = RMSNORM_VARIANT_GENERIC;
    p->vec_bytes = 0;
    int64_t per = std::min<int64_t>(s.hidden, 4096);
    int block = round_up(static_cast<int>((per + 3) / 4), 32);
    block = std::max(32, std::min(block, 512));
    p->threads_per_row = block;
    p->vecs_per_thread = 0;
    p->block_threads = block;
    p->rows_per_block = 1;
    p->grid = grid_for(s.rows, int64_t(s.sm_count) * (kMaxThreadsPerSm / block));
    p->smem_bytes = 0;
    p->kernel_index = find_kernel(RMSNORM_VARIANT_GENERIC, s.dtype, 0, 0, 0, 0, s.epi);
    return p->kernel_index >= 0 ? RMSNORM_OK : RMSNORM_ERR_VARIANT;
}

// Exact lookup of a register-resident instantiation by its parameters.
int find_rowreg(int variant, int dtype, int vb, int tpr, int nv, int maxt, int minb, int cache,
                int epi)
{
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    for (int i = 0; i < n; ++i) {
        const KernelDesc &d = t[i];
        if (d.variant == variant && d.dtype == dtype && d.vec_bytes == vb && d.tpr == tpr &&
            d.nv == nv && d.block == maxt && d.minb == minb && d.cache == cache && d.epi == epi)
            return i;
    }
    return -1;
}

// Registers per thread the compiler may use under __launch_bounds__(maxt,
// minb): the 64 Ki register file shared by minb blocks, in steps of 8.
int reg_cap(int maxt, int minb)
{
    if (minb <= 0)
        return 128; // no cap asked for; the wide bodies use about this many
    int r = 65536 / (maxt * minb);
    r = r / 8 * 8;
    return std::min(255, std::max(16, r));
}

// Resident blocks of `tpr` threads per SM for an instantiation.
int blocks_per_sm(int tpr, int maxt, int minb)
{
    const int by_threads = kMaxThreadsPerSm / tpr;
    const int by_regs = 65536 / (tpr * reg_cap(maxt, minb));
    return std::max(1, std::min({by_threads, by_regs, 32}));
}

// ---- warp-per-row: a group of TPR lanes (<= 32) per row
int plan_warp_exact(const Shape &s, int tpr, int nv, int minb, int64_t grid_cap,
                    rmsnorm_plan_t *p, int vb = 16)
{
    clear(p);
    const int idx =
        find_rowreg(RMSNORM_VARIANT_WARP_PER_ROW, s.dtype, vb, tpr, nv, 256, minb, 0, s.epi);
    if (idx < 0)
        return RMSNORM_ERR_VARIANT;
    p->variant = RMSNORM_VARIANT_WARP_PER_ROW;
    p->vec_bytes = vb;
    p->threads_per_row = tpr;
    p->vecs_per_thread = nv;
    p->block_threads = 256;
    p->rows_per_block = 256 / tpr;
    const int64_t blocks = (s.rows + p->rows_per_block - 1) / p->rows_per_block;
    p->grid = grid_for(blocks, grid_cap);
    p->kernel_index = idx;
    return RMSNORM_OK;
}

// Forced warp-per-row: the narrowest group whose registers cover the row.
int plan_warp(const Shape &s, rmsnorm_plan_t *p)
{
    clear(p);
    if (!s.a16)
        return RMSNORM_ERR_MISALIGNED;
    const int64_t nvec = s.row_bytes / 16;
    static const int kOptions[][3] = {{4, 1, 0},  {8, 1, 0},  {8, 2, 0},  {16, 1, 0},
                                      {16, 2, 0}, {32, 1, 0}, {32, 2, 8}, {32, 4, 8}};
    for (const auto &o : kOptions) // the narrowest group compiled for this epilogue
        if (int64_t(o[0]) * o[1] >= nvec && plan_warp_exact(s, o[0], o[1], o[2], INT_MAX, p) ==
                                                RMSNORM_OK)
            return RMSNORM_OK;
    clear(p);
    return RMSNORM_ERR_VARIANT;
}

// ---- block-per-row with a given instantiation and block size
int plan_cta_exact(const Shape &s, int vb, int nv, int maxt, int minb, int cache, int tpr_fixed,
                   int tpr, int64_t grid_cap, int variant, rmsnorm_plan_t *p)
{
    clear(p);
    const int idx = find_rowreg(RMSNORM_VARIANT_CTA_PER_ROW, s.dtype, vb, tpr_fixed, nv, maxt,
                                minb, cache, s.epi);
    if (idx < 0 || tpr > maxt || tpr < 32)
        return RMSNORM_ERR_VARIANT;
    p->variant = variant;
    p->vec_bytes = vb;
    p->threads_per_row = tpr;
    p->vecs_per_thread = nv;
    p->block_threads = tpr;
    p->rows_per_block = 1;
    p->grid = grid_for(s.rows, grid_cap);
    p->kernel_index = idx;
    return RMSNORM_OK;
}

int tpr_for(int64_t nvec, int nv)
{
    const int64_t need = (nvec + nv - 1) / nv;
    return static_cast<int>(std::max<int64_t>(32, (need + 31) / 32 * 32));
}

// Decode (no more rows than SMs): one block per row on its own SM, as few
// vectors per thread as the block allows (latency: one round trip).
// 32-byte vectors once a row is 640 16-byte vectors or more.
int plan_decode(const Shape &s, int variant, rmsnorm_plan_t *p)
{
    const int64_t nvec16 = s.row_bytes / 16;
    // 2..8 KiB rows: the compile-time 512-thread body (idle threads beyond
    // the row), measured 3-13% faster than a block sized to the row.
    if (nvec16 > (s.rows >= 64 ? 256 : 128) && nvec16 <= 512)
        return plan_cta_exact(s, 16, 1, 512, 0, 0, 512, 512, INT_MAX, variant, p);
    // 32-byte vectors (half the threads) for 10..16 KiB rows, and for 2..4 KiB
    // rows when there are 64+ of them (row count close to the SM count).
    const bool vb32 = s.a32 && ((nvec16 >= 640 && nvec16 <= 1024) ||
                                (s.rows >= 64 && nvec16 > 128 && nvec16 <= 256));
    const int vb = vb32 ? 32 : 16;
    const int64_t nvec = s.row_bytes / vb;
    struct Opt { int nv, maxt, minb; };
    static const Opt k16[] = {{1, 1024, 2}, {2, 1024, 2}, {4, 1024, 0}, {8, 512, 0}};
    static const Opt k32[] = {{1, 1024, 1}, {2, 1024, 0}, {4, 512, 0}};
    const Opt *opts = vb32 ? k32 : k16;
    const int nopt = vb32 ? 3 : 4;
    for (int i = 0; i < nopt; ++i) {
        const int tpr = tpr_for(nvec, opts[i].nv);
        if (tpr > opts[i].maxt)
            continue;
        if (!vb32 && opts[i].nv == 1 && tpr == 512)
            return plan_cta_exact(s, 16, 1, 512, 0, 0, 512, 512, INT_MAX, variant, p);
        const int64_t cap = int64_t(s.sm_count) * blocks_per_sm(tpr, opts[i].maxt, opts[i].minb);
        return plan_cta_exact(s, vb, opts[i].nv, opts[i].maxt, opts[i].minb, 1, 0, tpr, cap,
                              variant, p);
    }
    return RMSNORM_ERR_VARIANT;
}

// Prefill, rows of 97..1024 16-byte vectors: lean blocks of <= 256 threads
// with 2, 3 or 4 vectors each (least idle lanes, then fewest vectors), the
// register cap keeping 6-8 blocks (rows) resident per SM.
int plan_prefill_mid(const Shape &s, int variant, bool persistent, rmsnorm_plan_t *p)
{
    const int64_t nvec = s.row_bytes / 16;
    struct Opt { int nv, maxt, minb; };
    static const Opt opts[] = {{2, 256, 8}, {3, 512, 3}, {4, 256, 6}};
    int best = -1, best_tpr = 0;
    int64_t best_waste = INT64_MAX;
    for (int i = 0; i < 3; ++i) {
        const int tpr = tpr_for(nvec, opts[i].nv);
        if (tpr > 256)
            continue;
        const int64_t waste = int64_t(tpr) * opts[i].nv - nvec;
        if (waste < best_waste) {
            best_waste = waste;
            best = i;
            best_tpr = tpr;
        }
    }
    if (best < 0)
        return RMSNORM_ERR_VARIANT;
    // Many rows on blocks of <= 96 threads: 64-thread blocks with 4 vectors
    // each on a capped grid (16 per SM, grid-stride) -- tens of thousands of
    // tiny blocks cost more to schedule than the rows they carry.
    int64_t cap = INT_MAX;
    Opt o = opts[best];
    if (!persistent && best_tpr <= 96 && s.rows > 32768 && tpr_for(nvec, 4) <= 64) {
        o = Opt{4, 512, 2}; // the 64-register body: measured faster here
        best_tpr = tpr_for(nvec, 4);
        cap = int64_t(s.sm_count) * 16;
    }
    if (persistent)
        cap = int64_t(s.sm_count) * blocks_per_sm(best_tpr, o.maxt, o.minb);
    return plan_cta_exact(s, 16, o.nv, o.maxt, o.minb, 1, 0, best_tpr, cap,
                          cap < s.rows ? RMSNORM_VARIANT_PERSISTENT : variant, p);
}

// Rows of any length: the looped two-pass body, 512 threads, two blocks per SM.
int plan_looped(const Shape &s, int variant, bool persistent, rmsnorm_plan_t *p)
{
    const int64_t cap = persistent ? int64_t(s.sm_count) * blocks_per_sm(512, 512, 2) : INT_MAX;
    return plan_cta_exact(s, 16, 0, 512, 2, 1, 0, 512, cap, variant, p);
}

// Prefill, rows of more than 1024 16-byte vectors: the fewest vectors per
// thread that keep the block at <= 640 threads, on a persistent grid sized
// to the blocks that fit on an SM.
int plan_prefill_wide(const Shape &s, int variant, bool persistent, rmsnorm_plan_t *p)
{
    const int64_t nvec = s.row_bytes / 16;
    struct Opt { int nv, maxt, minb; };
    static const Opt opts[] = {{2, 1024, 2}, {3, 512, 3}, {4, 512, 2}, {8, 512, 0}};
    for (const Opt &o : opts) {
        const int tpr = tpr_for(nvec, o.nv);
        if (tpr > std::min(640, o.maxt))
            continue;
        const int64_t cap =
            persistent ? int64_t(s.sm_count) * blocks_per_sm(tpr, o.maxt, o.minb) : INT_MAX;
        return plan_cta_exact(s, 16, o.nv, o.maxt, o.minb, 1, 0, tpr, cap, variant, p);
    }
    // Larger rows: the widest register body at its largest block.
    const int tpr = tpr_for(nvec, 8);
    if (tpr <= 512)
        return plan_cta_exact(s, 16, 8, 512, 0, 1, 0, tpr,
                              persistent ? int64_t(s.sm_count) : INT_MAX, variant, p);
    return plan_looped(s, variant, persistent, p);
}

// Forced block-per-row / persistent.
int plan_cta(const Shape &s, bool persistent, rmsnorm_plan_t *p)
{
    clear(p);
    if (!s.a16)
        return RMSNORM_ERR_MISALIGNED;
    const int variant = persistent ? RMSNORM_VARIANT_PERSISTENT : RMSNORM_VARIANT_CTA_PER_ROW;
    const int64_t nvec = s.row_bytes / 16;
    if (persistent && s.rows <= s.sm_count) {
        if (plan_decode(s, variant, p) == RMSNORM_OK)
            return RMSNORM_OK;
        return plan_looped(s, variant, false, p);
    }
    if (nvec <= 1024 && plan_prefill_mid(s, variant, persistent, p) == RMSNORM_OK)
        return RMSNORM_OK;
    if (nvec > 1024)
        return plan_prefill_wide(s, variant, persistent, p);
    return plan_decode(s, variant, p); // short rows: one block of >= 32 threads per row
}

// ---- staged: persistent blocks, rows streamed into shared-memory slots.
// `wpr` warps consume each row; `groups` rows are consumed at once per block.
int plan_staged(const Shape &s, int blocks_per_sm, int groups_wanted, int wpr, bool tma_store,
                rmsnorm_plan_t *p)
{
    clear(p);
    if (!s.a16)
        return RMSNORM_ERR_MISALIGNED;
    if (s.row_bytes > INT_MAX / 4 || wpr < 1 || wpr > kStagedMaxConsumers)
        return RMSNORM_ERR_VARIANT;
    const int row_bytes = static_cast<int>(s.row_bytes);
    const int budget = std::min(s.smem_optin, kSmemPerSm / blocks_per_sm - kSmemReservedPerBlock);
    // Largest stage count whose layout fits.
    int stages = 0;
    for (int st = kStagedMaxStages; st >= 1; --st) {
        if (staged_layout(row_bytes, st).smem_bytes <= budget) {
            stages = st;
            break;
        }
    }
    int groups = std::min({groups_wanted, kStagedMaxConsumers / wpr, tma_store ? stages / 2 : stages});
    if (wpr > 1)
        groups = std::min(groups, kStagedMaxNamedGroups);
    if (groups < 1 || stages < 2)
        return RMSNORM_ERR_VARIANT;
    stages = stages / groups * groups;
    p->variant = RMSNORM_VARIANT_STAGED;
    p->vec_bytes = 16;
    p->threads_per_row = 32 * wpr;
    p->vecs_per_thread = 0;
    p->block_threads = 32 * (groups * wpr + 1);
    p->rows_per_block = groups;
    p->stages = stages;
    p->grid = grid_for(s.rows, int64_t(s.sm_count) * blocks_per_sm);
    p->smem_bytes = staged_layout(row_bytes, stages).smem_bytes;
    p->kernel_index =
        find_kernel(RMSNORM_VARIANT_STAGED, s.dtype, 16, 32, 0, tma_store ? 3 : 0, s.epi);
    return p->kernel_index >= 0 ? RMSNORM_OK : RMSNORM_ERR_VARIANT;
}

// Rows of 32..72 KiB: the staged ring with 8 warps per row (one group) up to
// 48 KiB rows and 4 warps x 2 groups beyond; 4 slots up to 40 KiB rows, 2
// above (the sweep's best shapes for 40, 48 and 64 KiB rows).
int plan_staged_wide(const Shape &s, rmsnorm_plan_t *p)
{
    const bool small = s.row_bytes <= 48 * 1024;
    const int rc = plan_staged(s, 1, small ? 1 : 2, small ? 8 : 4, false, p);
    if (rc != RMSNORM_OK)
        return rc;
    // Ring depth: 4 slots up to 40 KiB rows, 3 up to 48 KiB (1.6 % ahead of 2
    // on 48 KiB rows), then 2.
    const int max_stages = s.row_bytes <= 40 * 1024 ? 4 : (s.row_bytes <= 48 * 1024 ? 3 : 2);
    const int groups = p->rows_per_block;
    int stages = std::min(p->stages, max_stages) / groups * groups;
    if (stages < groups || stages < 2)
        return RMSNORM_ERR_VARIANT;
    p->stages = stages;
    p->smem_bytes = staged_layout(static_cast<int>(s.row_bytes), stages).smem_bytes;
    return RMSNORM_OK;
}

// ---- cluster: a row over C blocks of one cluster (decode, long rows).
// Slice S = ceil(nvec / C) vectors per block; the fewest vectors per thread
// (at least `min_thread_bytes` per thread) that keep the block at <= 512
// threads (<= 1024 with 4 per thread).
int plan_cluster_exact(const Shape &s, int C, int vb, rmsnorm_plan_t *p,
                       int min_thread_bytes = 0)
{
    clear(p);
    if (s.epi != RMSNORM_EPI_PLAIN)
        return RMSNORM_ERR_VARIANT;
    if (!(vb == 32 ? s.a32 : s.a16))
        return RMSNORM_ERR_MISALIGNED;
    if ((C != 2 && C != 4 && C != 8) || s.rows > INT_MAX / C)
        return RMSNORM_ERR_VARIANT;
    const int64_t nvec = s.row_bytes / vb;
    const int64_t S = (nvec + C - 1) / C;
    for (int nv : {1, 2, 4}) {
        const int tpr = tpr_for(S, nv);
        if (tpr > (nv == 4 ? 1024 : 512) || nv * vb < min_thread_bytes)
            continue;
        const int idx = find_rowreg(RMSNORM_VARIANT_CLUSTER, s.dtype, vb, 0, nv, 1024, 0, 1, s.epi);
        if (idx < 0)
            continue;
        p->variant = RMSNORM_VARIANT_CLUSTER;
        p->vec_bytes = vb;
        p->threads_per_row = tpr * C;
        p->vecs_per_thread = nv;
        p->block_threads = tpr;
        p->rows_per_block = 1;
        p->stages = C;
        p->grid = static_cast<int>(s.rows * C);
        p->kernel_index = idx;
        return RMSNORM_OK;
    }
    return RMSNORM_ERR_VARIANT;
}

// ---- grid: rows spread over every SM with one grid barrier (a cooperative
// launch of kGridBlocksPerSm 512-thread blocks per SM); <= kGridMaxRows rows.
int plan_grid(const Shape &s, rmsnorm_plan_t *p)
{
    clear(p);
    if (s.epi != RMSNORM_EPI_PLAIN || s.rows > kGridMaxRows)
        return RMSNORM_ERR_VARIANT;
    if (!s.a16)
        return RMSNORM_ERR_MISALIGNED;
    const int idx = find_rowreg(RMSNORM_VARIANT_GRID, s.dtype, 16, 0, 0, 512, kGridBlocksPerSm, 1,
                                s.epi);
    if (idx < 0)
        return RMSNORM_ERR_VARIANT;
    p->variant = RMSNORM_VARIANT_GRID;
    p->vec_bytes = 16;
    // one row: one 256-thread block per SM (less barrier traffic; measured
    // 12.0 -> 10.4 us on a 2 MiB row); more rows: two 512-thread blocks
    p->block_threads = s.rows == 1 ? 256 : 512;
    p->grid = s.sm_count * (s.rows == 1 ? 1 : kGridBlocksPerSm);
    p->threads_per_row = p->block_threads * p->grid;
    p->vecs_per_thread = 0;
    p->rows_per_block = static_cast<int>(s.rows); // every block works on every row
    p->stages = 0;
    p->kernel_index = idx;
    return RMSNORM_OK;
}

// Forced cluster: the smallest cluster whose slices are <= 8 KiB (at most 8
// blocks), 16-byte vectors.
int plan_cluster(const Shape &s, rmsnorm_plan_t *p)
{
    int C = 2;
    while (C < 8 && s.row_bytes > int64_t(C) * 8192)
        C *= 2;
    return plan_cluster_exact(s, C, 16, p);
}

// Forced staged: one warp per row up to 8 KiB rows, wider groups beyond.
int plan_staged_auto(const Shape &s, rmsnorm_plan_t *p)
{
    int wpr = 1;
    while (wpr < 8 && int64_t(wpr) * 8192 < s.row_bytes)
        wpr *= 2;
    return plan_staged(s, 1, std::max(1, 8 / wpr), wpr, false, p);
}

int check_common(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                 int dtype, int sm_count, int smem_optin, int epi, Shape *s)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || hidden <= 0 || hidden > kMaxHidden || sm_count <= 0 || smem_optin < 0)
        return RMSNORM_ERR_INVALID_ARG;
    if (epi < RMSNORM_EPI_PLAIN || epi > RMSNORM_EPI_NVFP4)
        return RMSNORM_ERR_INVALID_ARG;
    if (hidden % epi_block(epi) != 0) // whole scale blocks
        return RMSNORM_ERR_INVALID_ARG;
    if (rows > 0 && rows > INT64_MAX / 4 / hidden)
        return RMSNORM_ERR_INVALID_ARG;
    s->rows = rows;
    s->hidden = hidden;
    s->dtype = dtype;
    s->esize = elem_size(dtype);
    s->row_bytes = hidden * s->esize;
    s->a16 = aligned(x, 16) && aligned(y, 16) && aligned(w, 16) && s->row_bytes % 16 == 0;
    s->a32 = aligned(x, 32) && aligned(y, 32) && aligned(w, 32) && s->row_bytes % 32 == 0;
    s->sm_count = sm_count;
    s->smem_optin = smem_optin;
    s->epi = epi;
    return RMSNORM_OK;
}

} // namespace

int plan_launch(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                int dtype, int sm_count, int smem_optin, int variant, rmsnorm_plan_t *out,
                int epi)
{
    if (!out)
        return RMSNORM_ERR_INVALID_ARG;
    Shape s;
    int rc = check_common(x, w, y, rows, hidden, dtype, sm_count, smem_optin, epi, &s);
    if (rc != RMSNORM_OK)
        return rc;
    switch (variant) {
    case RMSNORM_VARIANT_WARP_PER_ROW:
        return plan_warp(s, out);
    case RMSNORM_VARIANT_CTA_PER_ROW:
        return plan_cta(s, false, out);
    case RMSNORM_VARIANT_PERSISTENT:
        return plan_cta(s, true, out);
    case RMSNORM_VARIANT_STAGED:
        return plan_staged_auto(s, out);
    case RMSNORM_VARIANT_CLUSTER:
        return plan_cluster(s, out);
    case RMSNORM_VARIANT_GRID:
        return plan_grid(s, out);
    case RMSNORM_VARIANT_GENERIC:
        if (s.epi >= RMSNORM_EPI_MXFP8) { // no scalar body for the block-scaled outputs
            clear(out);
            return RMSNORM_ERR_VARIANT;
        }
        return plan_generic(s, out);
    case RMSNORM_VARIANT_AUTO:
        break;
    default:
        return RMSNORM_ERR_INVALID_ARG;
    }

    // ---- automatic choice (rules fitted to a sweep of every plan over row
    // sizes 128 B .. 64 KiB and 1 .. 2M rows on GB300; they depend on the
    // row's byte length, not on the element type)
    if (!s.a16) {
        if (s.epi >= RMSNORM_EPI_MXFP8) { // the block-scaled bodies need 16-byte vectors
            clear(out);
            return RMSNORM_ERR_MISALIGNED;
        }
        return plan_generic(s, out);
    }
    const int64_t nvec = s.row_bytes / 16;
    if (s.rows <= s.sm_count) {
        // Long decode rows over thread-block clusters or the whole GPU
        // (fitted to sweeps of rows 1..152 x rows of 32 KiB..2 MiB on GB300;
        // e.g. 1 x 64 Ki bf16 6.1 -> 2.6 us, 8 x 64 Ki 9.1 -> 3.3 us, 77 x
        // 64 Ki 10.7 -> 7.5 us, 1 x 1 Mi 117 -> 12.6 us):
        //  * rows above 32 KiB (up to 8 rows below 48 KiB): one wave of
        //    clusters, as large (<= 8) as keeps every block on its own SM --
        //    at least 4 blocks, or 2 for rows of 64 KiB and more;
        //  * rows above 64 KiB, up to 256 KiB, and up to 128 of them (more
        //    than one wave holds; exactly 64 KiB rows stay with the rule above):
        //    clusters over several waves, 64 bytes per thread, of 4 blocks
        //    below 128 KiB and 8 from there (96 and 128 rows of 80, 128 and
        //    256 KiB: 6-34 % faster than the looped body);
        //  * longer rows, up to 64 of them: every SM on every row, one grid
        //    barrier.
        // Other long-row decode shapes keep the block-per-row bodies below.
        if (s.epi == RMSNORM_EPI_PLAIN && s.row_bytes > 32 * 1024) {
            if (s.rows <= 8 || s.row_bytes >= 48 * 1024) {
                int C = 8;
                while (C > 2 && s.rows * C > s.sm_count)
                    C /= 2;
                if (s.rows * C <= s.sm_count && (C >= 4 || s.row_bytes >= 64 * 1024) &&
                    ((s.a32 && plan_cluster_exact(s, C, 32, out) == RMSNORM_OK) ||
                     plan_cluster_exact(s, C, 16, out) == RMSNORM_OK))
                    return RMSNORM_OK;
            }
            if (s.rows <= 128 && s.row_bytes > 64 * 1024 && s.row_bytes <= 256 * 1024 &&
                plan_cluster_exact(s, s.row_bytes >= 128 * 1024 ? 8 : 4, 16, out, 64) ==
                    RMSNORM_OK)
                return RMSNORM_OK;
            if (s.row_bytes > 256 * 1024 && plan_grid(s, out) == RMSNORM_OK)
                return RMSNORM_OK;
        }
        // Decode: a whole warp per row up to 1 KiB rows (idle lanes cost less
        // than shorter shuffle trees save); longer rows get a block.
        if (nvec <= 32)
            return plan_warp_exact(s, 32, 1, 0, INT_MAX, out);
        if (nvec <= 64)
            return plan_warp_exact(s, 32, 2, 0, INT_MAX, out);
        if (plan_decode(s, RMSNORM_VARIANT_PERSISTENT, out) == RMSNORM_OK)
            return RMSNORM_OK;
        // Rows too long for one block's registers: the looped body, one
        // 512-thread block per row.
        if (plan_looped(s, RMSNORM_VARIANT_PERSISTENT, false, out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    // Prefill with a block-scaled output (MXFP8 / MXFP4 / NVFP4): its body
    // issues about half again as many instructions per element as the plain
    // one, so it takes more elements per thread and, with 32-byte vectors,
    // persistent grids (the fastest plans of sweeps on GB300 over 2-32 KiB
    // bf16 rows for the three formats):
    //   1-2 KiB rows: a warp per row, 2 32-byte vectors per lane, 4 blocks
    //     of 256 threads per SM (16-byte vectors, 4 per lane, register-capped
    //     for 8 blocks, when unaligned for 32);
    //   2-3 KiB rows: one warp, a block of its own, 4 32-byte vectors per
    //     lane, 16 blocks per SM; 3-4 KiB rows: 32-byte vectors, 2 per
    //     thread, 16 blocks per SM;
    //   4-16 KiB rows: blocks of 64, 96 or 128 threads (a compile-time size)
    //     with 4 32-byte vectors per thread, one block per row (16-byte
    //     vectors, 4 per thread, when unaligned for 32);
    //   16-24 KiB rows: 32-byte vectors, 4 per thread, capped at 96
    //     registers, one block per row; 24-32 KiB rows: the same vectors
    //     uncapped, 2 per thread on 2 blocks per SM (MX) or 4 on 4 (NVFP4);
    //     32-40 KiB rows: the capped body on 6 blocks per SM; longer rows:
    //     the looped body.
    const bool blockq = s.epi >= RMSNORM_EPI_MXFP8;
    if (blockq && s.a32 && nvec > 64 && nvec <= 128 &&
        plan_warp_exact(s, 32, 2, 0, int64_t(s.sm_count) * 4, out, 32) == RMSNORM_OK)
        return RMSNORM_OK;
    if (blockq && nvec > 64 && nvec <= 128 &&
        plan_warp_exact(s, 32, 4, 8, int64_t(s.sm_count) * 16, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (blockq && s.a32 && nvec > 128 && nvec <= 192) {
        const int64_t cap = int64_t(s.sm_count) * 16;
        if (plan_cta_exact(s, 32, 4, 32, 16, 1, 32, 32, cap,
                           cap < s.rows ? RMSNORM_VARIANT_PERSISTENT : RMSNORM_VARIANT_CTA_PER_ROW,
                           out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    if (blockq && s.a32 && nvec > 128 && nvec <= 256) {
        const int tpr = tpr_for(nvec / 2, 2);
        const int64_t cap = int64_t(s.sm_count) * std::min(16, 2048 / tpr);
        if (plan_cta_exact(s, 32, 2, 1024, 0, 1, 0, tpr, cap,
                           cap < s.rows ? RMSNORM_VARIANT_PERSISTENT : RMSNORM_VARIANT_CTA_PER_ROW,
                           out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    if (blockq && s.a32 && nvec > 256 && nvec <= 1024) {
        // Blocks of a compile-time size with 4 vectors per thread, the
        // smallest that holds the row (faster than the 2-vector body sized to
        // the row even where the row fills only 70 % of their lanes).
        const int64_t n32 = nvec / 2;
        const int tprc = n32 <= 256 ? 64 : (n32 <= 384 ? 96 : 128);
        const int minb = tprc == 64 ? 16 : (tprc == 96 ? 10 : 8);
        if (plan_cta_exact(s, 32, 4, tprc, minb, 1, tprc, tprc, INT_MAX,
                           RMSNORM_VARIANT_CTA_PER_ROW, out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    if (blockq && s.a32 && nvec > 256 && nvec <= 1024 &&
        plan_cta_exact(s, 32, 2, 256, 6, 1, 0, tpr_for(nvec / 2, 2), INT_MAX,
                       RMSNORM_VARIANT_CTA_PER_ROW, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (blockq && nvec > 128 && nvec <= 1024 &&
        plan_cta_exact(s, 16, 4, 256, 6, 1, 0, tpr_for(nvec, 4), INT_MAX,
                       RMSNORM_VARIANT_CTA_PER_ROW, out) == RMSNORM_OK)
        return RMSNORM_OK;
    // 16-24 KiB and 32-40 KiB rows: the same vectors in the body capped at 96
    // registers, one block per row, and on a persistent grid of 6 blocks per
    // SM (interleaved timings on GB300, 20-40 KiB bf16 rows of the three
    // formats: 17-39 % faster than the uncapped body and the looped one; at
    // 24-32 KiB and 40-64 KiB those stay ahead or within 5 %).
    if (blockq && s.a32 && nvec > 1024 && nvec <= 1536 &&
        plan_cta_exact(s, 32, 4, 320, 2, 1, 0, tpr_for(nvec / 2, 4), INT_MAX,
                       RMSNORM_VARIANT_CTA_PER_ROW, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (blockq && s.a32 && nvec > 2048 && nvec <= 2560) {
        const int64_t cap = int64_t(s.sm_count) * 6;
        if (plan_cta_exact(s, 32, 4, 320, 2, 1, 0, tpr_for(nvec / 2, 4), cap,
                           cap < s.rows ? RMSNORM_VARIANT_PERSISTENT : RMSNORM_VARIANT_CTA_PER_ROW,
                           out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    // 24-32 KiB rows: MXFP8 / MXFP4 two 32-byte vectors per thread on 2
    // blocks per SM (1-4.5 % ahead there), NVFP4 four on 4 blocks per SM.
    if (blockq && s.a32 && nvec > 1536 && nvec <= 2048 && s.epi != RMSNORM_EPI_NVFP4 &&
        plan_cta_exact(s, 32, 2, 1024, 0, 1, 0, tpr_for(nvec / 2, 2), int64_t(s.sm_count) * 2,
                       RMSNORM_VARIANT_PERSISTENT, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (blockq && s.a32 && nvec > 1024 && nvec <= 2048 &&
        plan_cta_exact(s, 32, 4, 512, 0, 1, 0, tpr_for(nvec / 2, 4), int64_t(s.sm_count) * 4,
                       RMSNORM_VARIANT_PERSISTENT, out) == RMSNORM_OK)
        return RMSNORM_OK;
    // Prefill.  Short rows: lane groups of one warp, several rows per warp.
    if (nvec > 1024)
        goto wide;
    if (nvec <= 8)
        return plan_warp_exact(s, 8, 1, 0, int64_t(s.sm_count) * 16, out);
    if (nvec <= 16)
        return plan_warp_exact(s, 8, 2, 0, INT_MAX, out);
    if (nvec <= 32)
        return plan_warp_exact(s, 16, 2, 0, INT_MAX, out);
    if (nvec <= 64)
        return plan_warp_exact(s, 32, 2, 8, INT_MAX, out);
    if (nvec <= 128)
        return plan_warp_exact(s, 32, 4, 8, INT_MAX, out);
    if (plan_prefill_mid(s, RMSNORM_VARIANT_CTA_PER_ROW, false, out) == RMSNORM_OK)
        return RMSNORM_OK;
wide:
    // 16-24 KiB and 32-40 KiB rows: 32-byte vectors, 4 per thread, one block
    // per row (on the final sweep 2.6-6.8 % faster there than the persistent
    // and staged bodies below; at 32 KiB the persistent one stays ahead), two
    // blocks of <= 320 threads per SM.  The weight-offset output takes the
    // build capped at 96 registers, so that its two blocks always fit.
    if (s.epi <= RMSNORM_EPI_BIAS && s.a32 &&
        ((s.row_bytes > 16384 && s.row_bytes <= 24576) ||
         (s.row_bytes > 32768 && s.row_bytes <= 40960)) &&
        (s.epi == RMSNORM_EPI_PLAIN
             ? plan_cta_exact(s, 32, 4, 512, 0, 1, 0, tpr_for(nvec / 2, 4), INT_MAX,
                              RMSNORM_VARIANT_CTA_PER_ROW, out)
             : plan_cta_exact(s, 32, 4, 320, 2, 1, 0, tpr_for(nvec / 2, 4), INT_MAX,
                              RMSNORM_VARIANT_CTA_PER_ROW, out)) == RMSNORM_OK)
        return RMSNORM_OK;
    // 16..32 KiB rows: the register bodies on a persistent grid.
    if (nvec <= 2048 && plan_prefill_wide(s, RMSNORM_VARIANT_PERSISTENT, true, out) == RMSNORM_OK)
        return RMSNORM_OK;
    // 32..72 KiB rows: the shared-memory ring (plain and weight-bias outputs;
    // the block-scaled ones starve its 8-16 consumer warps of issue slots --
    // 2.8-3.0 TB/s against 4.3-4.9 on the looped body below -- and stay there).
    if (nvec <= 4608 && s.epi <= RMSNORM_EPI_BIAS && plan_staged_wide(s, out) == RMSNORM_OK)
        return RMSNORM_OK;
    // Longer rows: the looped body, one block per row -- 512 threads, or 256
    // for rows up to 80 KiB in batches of more than two rows per SM (with
    // fewer rows per SM, 256 x 80 KiB rows, the wider block is 17 % faster).
    {
        const bool narrow =
            nvec <= 5120 && (s.epi >= RMSNORM_EPI_MXFP8 || s.rows > 2 * int64_t(s.sm_count));
        if (plan_cta_exact(s, 16, 0, 512, 2, 1, 0, narrow ? 256 : 512, INT_MAX,
                           RMSNORM_VARIANT_CTA_PER_ROW, out) == RMSNORM_OK)
            return RMSNORM_OK;
    }
    return plan_generic(s, out);
}

int validate_plan(const rmsnorm_plan_t &p, const void *x, const void *w, const void *y,
                  int64_t rows, int64_t hidden, int dtype, int sm_count, int smem_optin, int epi)
{
    Shape s;
    int rc = check_common(x, w, y, rows, hidden, dtype, sm_count, smem_optin, epi, &s);
    if (rc != RMSNORM_OK)
        return rc;
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    if (p.kernel_index < 0 || p.kernel_index >= n)
        return RMSNORM_ERR_INVALID_ARG;
    const KernelDesc &d = t[p.kernel_index];
    if (d.dtype != dtype || d.epi != epi)
        return RMSNORM_ERR_INVALID_ARG;
    const int dv = d.variant;
    const bool cta_like = dv == RMSNORM_VARIANT_CTA_PER_ROW;
    if (!(p.variant == dv || (cta_like && p.variant == RMSNORM_VARIANT_PERSISTENT)))
        return RMSNORM_ERR_INVALID_ARG;
    if (p.grid < 1 || p.block_threads < 32 || p.block_threads > 1024 || p.block_threads % 32)
        return RMSNORM_ERR_INVALID_ARG;
    if (d.vec_bytes == 16 && !s.a16)
        return RMSNORM_ERR_MISALIGNED;
    if (d.vec_bytes == 32 && !s.a32)
        return RMSNORM_ERR_MISALIGNED;
    const int64_t nvec = d.vec_bytes ? s.row_bytes / d.vec_bytes : 0;
    switch (dv) {
    case RMSNORM_VARIANT_WARP_PER_ROW:
        if (p.block_threads != d.block || int64_t(d.tpr) * d.nv < nvec)
            return RMSNORM_ERR_VARIANT;
        break;
    case RMSNORM_VARIANT_CTA_PER_ROW:
        // nv == 0: the looped body takes any row length.
        if (p.block_threads > d.block || (d.nv > 0 && int64_t(p.block_threads) * d.nv < nvec))
            return RMSNORM_ERR_VARIANT;
        if (d.tpr != 0 && p.block_threads != d.tpr) // block size fixed at compile time
            return RMSNORM_ERR_VARIANT;
        break;
    case RMSNORM_VARIANT_STAGED: {
        const int consumers = p.block_threads / 32 - 1;
        const int wpr = p.threads_per_row / 32;
        if (consumers < 1 || consumers > kStagedMaxConsumers || wpr < 1 ||
            p.threads_per_row % 32 != 0 || consumers % wpr != 0 || s.row_bytes > INT_MAX / 4)
            return RMSNORM_ERR_VARIANT;
        const int groups = consumers / wpr;
        if (wpr > 1 && groups > kStagedMaxNamedGroups)
            return RMSNORM_ERR_VARIANT;
        if (p.stages < 1 || p.stages > kStagedMaxStages || p.stages % groups != 0)
            return RMSNORM_ERR_VARIANT;
        // Bulk-store mode releases a slot one row later: each group needs two.
        if (d.cache == 3 && p.stages < 2 * groups)
            return RMSNORM_ERR_VARIANT;
        const int need = staged_layout(static_cast<int>(s.row_bytes), p.stages).smem_bytes;
        if (p.smem_bytes != need || need > smem_optin || p.grid > rows)
            return RMSNORM_ERR_VARIANT;
        break;
    }
    case RMSNORM_VARIANT_GENERIC:
        break;
    case RMSNORM_VARIANT_GRID:
        // every block resident at once: at most the blocks the SMs hold
        if (p.grid > sm_count * kGridBlocksPerSm || p.block_threads > d.block ||
            rows > kGridMaxRows || p.rows_per_block != rows)
            return RMSNORM_ERR_VARIANT;
        break;
    case RMSNORM_VARIANT_CLUSTER: {
        const int C = p.stages;
        if (C != 2 && C != 4 && C != 8)
            return RMSNORM_ERR_VARIANT;
        const int64_t S = (nvec + C - 1) / C;
        if (p.block_threads > d.block || int64_t(p.block_threads) * d.nv < S)
            return RMSNORM_ERR_VARIANT;
        if (int64_t(p.grid) != rows * C) // one cluster per row, exactly
            return RMSNORM_ERR_VARIANT;
        break;
    }
    default:
        return RMSNORM_ERR_INVALID_ARG;
    }
    if (dv != RMSNORM_VARIANT_STAGED && dv != RMSNORM_VARIANT_CLUSTER && p.stages != 0)
        return RMSNORM_ERR_INVALID_ARG;
    if (dv != RMSNORM_VARIANT_STAGED && p.smem_bytes != 0)
        return RMSNORM_ERR_INVALID_ARG;
    return RMSNORM_OK;
}

// Over the CPU-GPU link the link, not the SMs, sets the pace: on GB300 every
// plan with enough rows in flight moves 16384 x 4096 bf16 host rows at about
// 337 GB/s (the copy engines with both directions busy reach 336), except
// the one-block-per-row grid of 16384 blocks, at 322 GB/s.  A persistent grid
// of two blocks per SM is at the plateau (337-338 GB/s), so block-per-row and
// wider persistent grids of the register bodies (which loop over rows at any
// grid size) are cut to it; other plans are kept.
int plan_host_link(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                   int dtype, int sm_count, int smem_optin, rmsnorm_plan_t *out)
{
    const int rc = plan_launch(x, w, y, rows, hidden, dtype, sm_count, smem_optin,
                               RMSNORM_VARIANT_AUTO, out);
    if (rc != RMSNORM_OK)
        return rc;
    const int cap = kHostLinkBlocksPerSm * sm_count;
    if ((out->variant == RMSNORM_VARIANT_CTA_PER_ROW ||
         out->variant == RMSNORM_VARIANT_PERSISTENT) &&
        out->grid > cap) {
        out->variant = RMSNORM_VARIANT_PERSISTENT;
        out->grid = cap;
    }
    return RMSNORM_OK;
}

} // namespace rmsnorm
