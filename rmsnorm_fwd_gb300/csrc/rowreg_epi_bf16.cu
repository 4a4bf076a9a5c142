// rowreg_epi_bf16.cu -- bf16 instantiations of the register-resident kernels
// with the weight-bias and MXFP8 epilogues (a translation unit of their own
// so they compile in parallel with the plain ones).
#include "rowreg.cuh"

namespace rmsnorm {
namespace rowreg {
namespace {
const KernelDesc kTable[] = {ROWREG_SET(RMSNORM_BF16, RMSNORM_EPI_BIAS),
                             ROWREG_SET_Q(RMSNORM_BF16, RMSNORM_EPI_MXFP8)};
} // namespace
} // namespace rowreg

const KernelDesc *rowreg_epi_kernels_bf16(int *n)
{
    *n = static_cast<int>(sizeof(rowreg::kTable) / sizeof(rowreg::kTable[0]));
    return rowreg::kTable;
}

} // namespace rmsnorm
