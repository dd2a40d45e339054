// Split-KV chunk kernel (mma.sync engine) for head_dim 64.
#include "split_kv_chunk_variants.cuh"

namespace kvd {
KVD_MMA_TABLE(64, 0, 30, 36, 42, 48)
}  // namespace kvd
