// tcgen05 split-KV chunk kernel variants for head_dim 128.
#include "split_kv_chunk_tc_launch.cuh"

namespace kvd {

const ChunkKernel* tc_table_d128(bool f32, int qr) {
    static const ChunkKernel table[3][2] = {
        {make_tc<128, false, 48>(14), make_tc<128, true, 48>(15)},
        {make_tc<128, false, 64>(16), make_tc<128, true, 64>(17)},
        {make_tc<128, false, 128, 128>(18), make_tc<128, true, 128, 128>(19)},
    };
    const int r = qr == 48 ? 0 : (qr == 64 ? 1 : 2);
    return &table[r][f32 ? 1 : 0];
}

}  // namespace kvd
