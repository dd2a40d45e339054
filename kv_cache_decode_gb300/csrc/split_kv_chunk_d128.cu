// Split-KV chunk kernel (mma.sync engine) for head_dim 128.
#include "split_kv_chunk_variants.cuh"

namespace kvd {
KVD_MMA_TABLE(128, 2, 32, 38, 44, 52)
}  // namespace kvd
