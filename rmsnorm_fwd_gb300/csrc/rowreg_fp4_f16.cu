// rowreg_fp4_f16.cu -- f16 instantiations of the register-resident kernels
// with the MXFP4 and NVFP4 epilogues (a translation unit of their own so
// they compile in parallel with the others).
#include "rowreg.cuh"

namespace rmsnorm {
namespace rowreg {
namespace {
const KernelDesc kTable[] = {ROWREG_SET_Q(RMSNORM_F16, RMSNORM_EPI_MXFP4),
                             ROWREG_SET_Q(RMSNORM_F16, RMSNORM_EPI_NVFP4)};
} // namespace
} // namespace rowreg

const KernelDesc *rowreg_fp4_kernels_f16(int *n)
{
    *n = static_cast<int>(sizeof(rowreg::kTable) / sizeof(rowreg::kTable[0]));
    return rowreg::kTable;
}

} // namespace rmsnorm
