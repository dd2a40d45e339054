// tcgen05 split-KV chunk kernel variants for head_dim 64.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d64(bool f32, int qr) {
    static const ChunkKernel table[4][2] = {
        {make_tc<64, false, 8>(6), make_tc<64, true, 8>(7)},
        {make_tc<64, false, 16>(8), make_tc<64, true, 16>(9)},
        {make_tc<64, false, 48>(10), make_tc<64, true, 48>(11)},
        {make_tc<64, false, 64>(12), make_tc<64, true, 64>(13)},
    };
    const int r = qr == 8 ? 0 : (qr == 16 ? 1 : (qr == 48 ? 2 : 3));
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
