// tcgen05 split-KV chunk kernel variants for head_dim 64.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d64(bool f32, int qr) {
    static const ChunkKernel table[3][2] = {
        {make_tc<64, false, 48>(6), make_tc<64, true, 48>(7)},
        {make_tc<64, false, 64>(8), make_tc<64, true, 64>(9)},
        {make_tc<64, false, 128, 128>(10), make_tc<64, true, 128, 128>(11)},
    };
    const int r = qr == 48 ? 0 : (qr == 64 ? 1 : 2);
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
