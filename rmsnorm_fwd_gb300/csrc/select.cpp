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
// (decode) give every row its own block on its own SM; when there are many
// (prefill) use enough warps per SM to keep HBM busy.  The SM count is read
// from the device at context creation, not compiled in (same page, section
// "Blackwell support").
#include <algorithm>
#include <climits>
#include <cstdint>

#include "internal.h"

namespace rmsnorm {
namespace {

constexpr int64_t kMaxHidden = int64_t(1) << 26; // 64 Mi elements per row
constexpr int kMaxThreadsPerSm = 2048;
constexpr int kSmemPerSm = 233472;               // 228 KiB per SM on sm_100-class parts
constexpr int kSmemReservedPerBlock = 1024;
constexpr int kStagedMaxStages = 32;
constexpr int kStagedMaxConsumers = 16;

int elem_size(int dtype)
{
    return dtype == RMSNORM_F32 ? 4 : 2;
}

bool aligned(const void *p, int a)
{
    return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(a)) == 0;
}

int round_up(int v, int m)
{
    return (v + m - 1) / m * m;
}

// Finds the table entry for (variant, dtype, vec_bytes, tpr, nv, cache) with
// no occupancy cap; -1 if none.
int find_kernel(int variant, int dtype, int vec_bytes, int tpr, int nv, int cache = 0)
{
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    for (int i = 0; i < n; ++i) {
        const KernelDesc &d = t[i];
        if (d.variant == variant && d.dtype == dtype && d.vec_bytes == vec_bytes &&
            d.tpr == tpr && d.nv == nv && d.cache == cache && d.minb == 0)
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
    p->kernel_index = find_kernel(RMSNORM_VARIANT_GENERIC, s.dtype, 0, 0, 0);
    return p->kernel_index >= 0 ? RMSNORM_OK : RMSNORM_ERR_VARIANT;
}

// ---- warp-per-row: TPR lanes x NV vectors of 16 (or 32) bytes per row
int plan_warp(const Shape &s, int vb, rmsnorm_plan_t *p)
{
    clear(p);
    if (vb == 16 ? !s.a16 : !s.a32)
        return RMSNORM_ERR_MISALIGNED;
    const int64_t nvec = s.row_bytes / vb;
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    int best = -1;
    int64_t best_cap = INT64_MAX;
    for (int i = 0; i < n; ++i) {
        const KernelDesc &d = t[i];
        if (d.variant != RMSNORM_VARIANT_WARP_PER_ROW || d.dtype != s.dtype || d.vec_bytes != vb ||
            d.minb != 0 || d.cache != 0)
            continue;
        const int64_t cap = int64_t(d.tpr) * d.nv;
        if (cap < nvec)
            continue;
        // Smallest capacity that covers the row; on ties the wider group
        // (fewer serial vectors per thread).
        if (cap < best_cap || (cap == best_cap && d.tpr > t[best].tpr)) {
            best = i;
            best_cap = cap;
        }
    }
    if (best < 0)
        return RMSNORM_ERR_VARIANT;
    const KernelDesc &d = t[best];
    p->variant = RMSNORM_VARIANT_WARP_PER_ROW;
    p->vec_bytes = vb;
    p->threads_per_row = d.tpr;
    p->vecs_per_thread = d.nv;
    p->block_threads = d.block;
    p->rows_per_block = d.block / d.tpr;
    const int64_t blocks = (s.rows + p->rows_per_block - 1) / p->rows_per_block;
    p->grid = grid_for(blocks, INT_MAX);
    p->smem_bytes = 0;
    p->kernel_index = best;
    return RMSNORM_OK;
}

// ---- block-per-row: blockDim = tpr threads x NV vectors per thread
int plan_cta(const Shape &s, int vb, bool persistent, rmsnorm_plan_t *p)
{
    clear(p);
    if (vb == 16 ? !s.a16 : !s.a32)
        return RMSNORM_ERR_MISALIGNED;
    const int64_t nvec = s.row_bytes / vb;
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    int best = -1, best_tpr = 0;
    double best_score = 1e30;
    for (int i = 0; i < n; ++i) {
        const KernelDesc &d = t[i];
        if (d.variant != RMSNORM_VARIANT_CTA_PER_ROW || d.dtype != s.dtype || d.vec_bytes != vb ||
            d.minb != 0 || d.cache != 0 || d.tpr != 0)
            continue;
        const int64_t need = (nvec + d.nv - 1) / d.nv;
        const int64_t tpr = std::max<int64_t>(32, (need + 31) / 32 * 32);
        if (tpr > d.block)
            continue;
        const double waste = double(tpr * d.nv - nvec) / double(tpr * d.nv);
        double score;
        if (persistent) {
            // Decode: fewest serial vectors per thread (latency), then waste.
            score = d.nv + waste;
        } else {
            // Prefill: little waste, and a block of 128..512 threads.
            const double dev = tpr < 128 ? (128.0 / tpr) : (tpr > 512 ? tpr / 512.0 : 1.0);
            score = waste * 4.0 + dev;
        }
        if (score < best_score) {
            best_score = score;
            best = i;
            best_tpr = static_cast<int>(tpr);
        }
    }
    if (best < 0)
        return RMSNORM_ERR_VARIANT;
    const KernelDesc &d = t[best];
    p->variant = persistent ? RMSNORM_VARIANT_PERSISTENT : RMSNORM_VARIANT_CTA_PER_ROW;
    p->vec_bytes = vb;
    p->threads_per_row = best_tpr;
    p->vecs_per_thread = d.nv;
    p->block_threads = best_tpr;
    p->rows_per_block = 1;
    if (persistent)
        p->grid = grid_for(s.rows, int64_t(s.sm_count) * std::max(1, kMaxThreadsPerSm / best_tpr));
    else
        p->grid = grid_for(s.rows, INT_MAX);
    p->smem_bytes = 0;
    p->kernel_index = best;
    return RMSNORM_OK;
}

// ---- staged: persistent blocks, rows streamed into shared-memory slots
int plan_staged(const Shape &s, int blocks_per_sm, int consumers_wanted, rmsnorm_plan_t *p)
{
    clear(p);
    if (!s.a16)
        return RMSNORM_ERR_MISALIGNED;
    if (s.row_bytes > INT_MAX / 4)
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
    if (stages < 2)
        return RMSNORM_ERR_VARIANT;
    int consumers = std::min({consumers_wanted, kStagedMaxConsumers, stages});
    stages = stages / consumers * consumers;
    p->variant = RMSNORM_VARIANT_STAGED;
    p->vec_bytes = 16;
    p->threads_per_row = 32;
    p->vecs_per_thread = 0;
    p->block_threads = 32 * (consumers + 1);
    p->rows_per_block = consumers;
    p->stages = stages;
    p->grid = grid_for(s.rows, int64_t(s.sm_count) * blocks_per_sm);
    p->smem_bytes = staged_layout(row_bytes, stages).smem_bytes;
    p->kernel_index = find_kernel(RMSNORM_VARIANT_STAGED, s.dtype, 16, 32, 0);
    return p->kernel_index >= 0 ? RMSNORM_OK : RMSNORM_ERR_VARIANT;
}

int check_common(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                 int dtype, int sm_count, int smem_optin, Shape *s)
{
    if (dtype != RMSNORM_F32 && dtype != RMSNORM_BF16 && dtype != RMSNORM_F16)
        return RMSNORM_ERR_UNSUPPORTED_DTYPE;
    if (rows < 0 || hidden <= 0 || hidden > kMaxHidden || sm_count <= 0 || smem_optin < 0)
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
    return RMSNORM_OK;
}

} // namespace

int plan_launch(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                int dtype, int sm_count, int smem_optin, int variant, rmsnorm_plan_t *out)
{
    if (!out)
        return RMSNORM_ERR_INVALID_ARG;
    Shape s;
    int rc = check_common(x, w, y, rows, hidden, dtype, sm_count, smem_optin, &s);
    if (rc != RMSNORM_OK)
        return rc;
    switch (variant) {
    case RMSNORM_VARIANT_WARP_PER_ROW:
        return plan_warp(s, 16, out);
    case RMSNORM_VARIANT_CTA_PER_ROW:
        return plan_cta(s, 16, false, out);
    case RMSNORM_VARIANT_PERSISTENT:
        return plan_cta(s, 16, true, out);
    case RMSNORM_VARIANT_STAGED:
        return plan_staged(s, 1, 8, out);
    case RMSNORM_VARIANT_GENERIC:
        return plan_generic(s, out);
    case RMSNORM_VARIANT_AUTO:
        break;
    default:
        return RMSNORM_ERR_INVALID_ARG;
    }

    // ---- automatic choice
    if (!s.a16)
        return plan_generic(s, out);
    const int64_t nvec = s.row_bytes / 16;
    // Decode: no more rows than SMs -> one block per row, one SM each.
    if (s.rows <= s.sm_count && nvec > 32 && plan_cta(s, 16, true, out) == RMSNORM_OK)
        return RMSNORM_OK;
    // Rows of at most 128 vectors (1024 x bf16, 512 x f32): a warp (or part
    // of one) per row, everything in registers.
    if (nvec <= 128 && plan_warp(s, 16, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (plan_cta(s, 16, false, out) == RMSNORM_OK)
        return RMSNORM_OK;
    if (plan_staged(s, 1, 8, out) == RMSNORM_OK)
        return RMSNORM_OK;
    return plan_generic(s, out);
}

int validate_plan(const rmsnorm_plan_t &p, const void *x, const void *w, const void *y,
                  int64_t rows, int64_t hidden, int dtype, int sm_count, int smem_optin)
{
    Shape s;
    int rc = check_common(x, w, y, rows, hidden, dtype, sm_count, smem_optin, &s);
    if (rc != RMSNORM_OK)
        return rc;
    int n = 0;
    const KernelDesc *t = kernel_table(&n);
    if (p.kernel_index < 0 || p.kernel_index >= n)
        return RMSNORM_ERR_INVALID_ARG;
    const KernelDesc &d = t[p.kernel_index];
    if (d.dtype != dtype)
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
        if (p.block_threads > d.block || int64_t(p.block_threads) * d.nv < nvec)
            return RMSNORM_ERR_VARIANT;
        if (d.tpr != 0 && p.block_threads != d.tpr) // block size fixed at compile time
            return RMSNORM_ERR_VARIANT;
        break;
    case RMSNORM_VARIANT_STAGED: {
        const int consumers = p.block_threads / 32 - 1;
        if (consumers < 1 || consumers > kStagedMaxConsumers || p.stages < 1 ||
            p.stages > kStagedMaxStages || p.stages % consumers != 0 || s.row_bytes > INT_MAX / 4)
            return RMSNORM_ERR_VARIANT;
        // Bulk-store mode releases a slot one row later: each consumer needs two.
        if (d.cache == 3 && p.stages < 2 * consumers)
            return RMSNORM_ERR_VARIANT;
        const int need = staged_layout(static_cast<int>(s.row_bytes), p.stages).smem_bytes;
        if (p.smem_bytes != need || need > smem_optin || p.grid > rows)
            return RMSNORM_ERR_VARIANT;
        break;
    }
    case RMSNORM_VARIANT_GENERIC:
        break;
    default:
        return RMSNORM_ERR_INVALID_ARG;
    }
    if (dv != RMSNORM_VARIANT_STAGED && p.smem_bytes != 0)
        return RMSNORM_ERR_INVALID_ARG;
    return RMSNORM_OK;
}

} // namespace rmsnorm
