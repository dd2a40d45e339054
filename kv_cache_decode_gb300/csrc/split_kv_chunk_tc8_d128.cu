// tcgen05 split-KV chunk kernel variants for 8-bit caches, head_dim 128
// (int8 and E4M3 codes; groups of up to 48 or 64 query heads).
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc8_table_d128(bool f32, int qr, bool fp8) {
    static const ChunkKernel table[2][2][2] = {
        {{make_tc<128, false, 48, 64, true, false>(64), make_tc<128, true, 48, 64, true, false>(65)},
         {make_tc<128, false, 48, 64, true, true>(66), make_tc<128, true, 48, 64, true, true>(67)}},
        {{make_tc<128, false, 64, 64, true, false>(68), make_tc<128, true, 64, 64, true, false>(69)},
         {make_tc<128, false, 64, 64, true, true>(70), make_tc<128, true, 64, 64, true, true>(71)}},
    };
    return &table[qr == 48 ? 0 : 1][fp8 ? 1 : 0][f32 ? 1 : 0];
}

}  // namespace kvd
