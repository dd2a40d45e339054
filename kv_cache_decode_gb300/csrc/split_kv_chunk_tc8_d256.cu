// tcgen05 split-KV chunk kernel variants for 8-bit caches, head_dim 256
// (int8 and E4M3 codes; groups of up to 48 query heads).
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc8_table_d256(bool f32, bool fp8) {
    static const ChunkKernel table[2][2] = {
        {make_tc<256, false, 48, 64, true, false>(72), make_tc<256, true, 48, 64, true, false>(73)},
        {make_tc<256, false, 48, 64, true, true>(74), make_tc<256, true, 48, 64, true, true>(75)},
    };
    return &table[fp8 ? 1 : 0][f32 ? 1 : 0];
}

}  // namespace kvd
