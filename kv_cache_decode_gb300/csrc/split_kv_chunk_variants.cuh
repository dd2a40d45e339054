// Compiled variants of the split-KV chunk kernel for one head dimension.
// Per head-tile count HT (16 query heads each):
//   HT == 1: 4 token slices of 16 tokens over 64-token tiles;
//   HT >= 2: 2 token slices of 16 tokens over 32-token tiles (the K/V tile is
//            re-read from shared memory by each head tile).
#pragma once

#include "split_kv_chunk.cuh"

namespace kvd {

template <int D, int HT>
struct ChunkConfig {
    static constexpr int TS = (HT == 1) ? 4 : 2;
    static constexpr int TT = (HT == 1) ? 64 : 32;
    static constexpr int STAGES = (HT == 1 && D == 256) ? 2 : 4;
    // Two CTAs per SM when two fit in the SM's 228 KB of shared memory (1 KB
    // of it is reserved per CTA); __launch_bounds__ then caps registers to match.
    static constexpr int SMEM = ChunkShape<D, HT, TS, TT, STAGES>::SMEM_BYTES;
    static constexpr int MINB = (2 * (SMEM + 1024) <= 228 * 1024) ? 2 : 1;
};

template <int D, int HT, bool F32>
inline ChunkKernel make_chunk_kernel() {
    using C = ChunkConfig<D, HT>;
    using Sh = ChunkShape<D, HT, C::TS, C::TT, C::STAGES>;
    ChunkKernel k;
    k.fn = split_kv_chunk_kernel<D, HT, C::TS, C::TT, C::STAGES, F32, C::MINB>;
    k.head_dim = D;
    k.head_tiles = HT;
    k.threads = Sh::NT;
    k.smem_bytes = Sh::SMEM_BYTES;
    k.tile_tokens = C::TT;
    k.ctas_per_sm = C::MINB;
    k.f32_out = F32;
    return k;
}

#define KVD_CHUNK_TABLE(D)                                                                   \
    const ChunkKernel* chunk_table_d##D(int ht, bool f32) {                                 \
        static const ChunkKernel table[4][2] = {                                            \
            {make_chunk_kernel<D, 1, false>(), make_chunk_kernel<D, 1, true>()},            \
            {make_chunk_kernel<D, 2, false>(), make_chunk_kernel<D, 2, true>()},            \
            {make_chunk_kernel<D, 3, false>(), make_chunk_kernel<D, 3, true>()},            \
            {make_chunk_kernel<D, 4, false>(), make_chunk_kernel<D, 4, true>()},            \
        };                                                                                  \
        if (ht < 1 || ht > 4) return nullptr;                                               \
        return &table[ht - 1][f32 ? 1 : 0];                                                 \
    }

}  // namespace kvd
