// fp16 instantiations of the streaming GEMV kernels.
#include "gemv_kernels.cuh"
#include "gemv_tiles.cuh"

GEMV_DEFINE_KERNEL_TABLE(F16, f16)
GEMV_DEFINE_TILES_TABLE(F16, f16)
