// bf16 instantiations of the streaming GEMV kernels.
#include "gemv_kernels.cuh"
#include "gemv_tiles.cuh"

GEMV_DEFINE_KERNEL_TABLE(BF16, bf16)
GEMV_DEFINE_TILES_TABLE(BF16, bf16)
