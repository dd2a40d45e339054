// Split-KV chunk kernel (mma.sync engine) for head_dim 256.
#include "split_kv_chunk_variants.cuh"

namespace kvd {
KVD_MMA_TABLE(256, 4, 34, 40, 46, 56)
}  // namespace kvd
