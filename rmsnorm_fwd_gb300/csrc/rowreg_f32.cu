// rowreg_f32.cu -- f32 instantiations of the register-resident kernels
// (one translation unit per element type so they compile in parallel).
#include "rowreg.cuh"

namespace rmsnorm {
namespace rowreg {
namespace {
const KernelDesc kTable[] = {ROWREG_SET(RMSNORM_F32, RMSNORM_EPI_PLAIN)};
} // namespace
} // namespace rowreg

const KernelDesc *rowreg_kernels_f32(int *n)
{
    *n = static_cast<int>(sizeof(rowreg::kTable) / sizeof(rowreg::kTable[0]));
    return rowreg::kTable;
}

} // namespace rmsnorm
