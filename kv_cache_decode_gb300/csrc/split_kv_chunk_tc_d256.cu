// tcgen05 split-KV chunk kernel variants for head_dim 256.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d256(bool f32, int qr) {
    static const ChunkKernel table[4][2] = {
        {make_tc<256, false, 8>(22), make_tc<256, true, 8>(23)},
        {make_tc<256, false, 16>(24), make_tc<256, true, 16>(25)},
        {make_tc<256, false, 48>(26), make_tc<256, true, 48>(27)},
        {make_tc<256, false, 64>(28), make_tc<256, true, 64>(29)},
    };
    const int r = qr == 8 ? 0 : (qr == 16 ? 1 : (qr == 48 ? 2 : 3));
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
