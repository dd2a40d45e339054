// tcgen05 split-KV chunk kernel variants for head_dim 256.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d256(bool f32, int qr) {
    static const ChunkKernel table[3][2] = {
        {make_tc<256, false, 48>(22), make_tc<256, true, 48>(23)},
        {make_tc<256, false, 64>(24), make_tc<256, true, 64>(25)},
        {make_tc<256, false, 128, 128>(26), make_tc<256, true, 128, 128>(27)},
    };
    const int r = qr == 48 ? 0 : (qr == 64 ? 1 : 2);
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
