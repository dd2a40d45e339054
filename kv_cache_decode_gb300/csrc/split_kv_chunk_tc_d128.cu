// tcgen05 split-KV chunk kernel variants for head_dim 128.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d128(bool f32, int qr) {
    static const ChunkKernel table[4][2] = {
        {make_tc<128, false, 8>(14), make_tc<128, true, 8>(15)},
        {make_tc<128, false, 16>(16), make_tc<128, true, 16>(17)},
        {make_tc<128, false, 48>(18), make_tc<128, true, 48>(19)},
        {make_tc<128, false, 64>(20), make_tc<128, true, 64>(21)},
    };
    const int r = qr == 8 ? 0 : (qr == 16 ? 1 : (qr == 48 ? 2 : 3));
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
