// fp16 instantiations of the streaming GEMV kernels.
#include "gemv_kernels.cuh"

GEMV_DEFINE_KERNEL_TABLE(F16, f16)
