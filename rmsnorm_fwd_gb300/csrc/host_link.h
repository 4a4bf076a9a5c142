// host_link.h -- the launch plan for rows in page-locked host memory.
#pragma once

#include <cstdint>

#include "rmsnorm.h"

namespace rmsnorm {

// The plan for rows the kernel reads and writes in page-locked host memory
// over the CPU-GPU link (rmsnorm_fwd_host): plan_launch's automatic choice,
// with block-per-row and persistent grids above kHostLinkBlocksPerSm blocks
// per SM cut to a persistent grid of that many (select.cpp).
constexpr int kHostLinkBlocksPerSm = 2;
int plan_host_link(const void *x, const void *w, const void *y, int64_t rows, int64_t hidden,
                   int dtype, int sm_count, int smem_optin, rmsnorm_plan_t *out);

} // namespace rmsnorm
