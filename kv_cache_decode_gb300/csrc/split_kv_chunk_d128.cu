// Split-KV chunk kernel variants for head_dim 128.
#include "split_kv_chunk_variants.cuh"

namespace kvd {
KVD_CHUNK_TABLE(128)
}  // namespace kvd
