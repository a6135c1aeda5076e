// bf16 instantiations of the bulk GEMV kernel (B staged through shared
// memory by bulk asynchronous copies).
#include "gemv_bulk.cuh"

GEMV_DEFINE_BULK_TABLE(BF16, bf16)
