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
    // Three stages at head_dim 128 (two CTAs, eight warps per SM), three at 256
    // (one CTA), four at 64.
    static constexpr int STAGES = (D == 64) ? 4 : 3;
    // Two CTAs per SM when two fit in the SM's 228 KB of shared memory (1 KB
    // of it is reserved per CTA); __launch_bounds__ then caps registers to match.
    static constexpr int SMEM = ChunkShape<D, HT, TS, TT, STAGES>::SMEM_BYTES;
    static constexpr int MINB = (2 * (SMEM + 1024) <= 228 * 1024) ? 2 : 1;
    // 8-bit cache: stages of 8-bit tiles (half the bytes, so more of them) and
    // the token slices' merge buffer, with the same CTAs per SM.
    static constexpr int STAGES8 = (D == 64) ? 8 : 5;
    static constexpr int SMEM8 = ChunkShape<D, HT, TS, TT, STAGES8, true>::SMEM_BYTES;
    static constexpr int MINB8 = (2 * (SMEM8 + 1024) <= 228 * 1024) ? 2 : 1;
};

template <int D, bool F32, bool PAGED, bool KV8, bool FP8>
cudaError_t launch_mma_chunk(const ChunkKernel& k, const DecodeParams& p, cudaStream_t stream) {
    using C = ChunkConfig<D, 1>;
    constexpr int ST = KV8 ? C::STAGES8 : C::STAGES, MB = KV8 ? C::MINB8 : C::MINB;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_split * p.row_blocks), 1, 1);  // row blocks of one run side by side
    cfg.blockDim = dim3((unsigned)k.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)k.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_chunk_kernel<D, 1, C::TS, C::TT, ST, F32, MB, PAGED, KV8, FP8>, p);
}

template <int D, bool F32, bool PAGED, bool KV8 = false, bool FP8 = false>
inline ChunkKernel make_mma_chunk_kernel(int index) {
    using C = ChunkConfig<D, 1>;
    constexpr int ST = KV8 ? C::STAGES8 : C::STAGES, MB = KV8 ? C::MINB8 : C::MINB;
    using Sh = ChunkShape<D, 1, C::TS, C::TT, ST, KV8>;
    ChunkKernel k;
    k.fn = reinterpret_cast<const void*>(split_kv_chunk_kernel<D, 1, C::TS, C::TT, ST, F32, MB, PAGED, KV8, FP8>);
    k.launch = launch_mma_chunk<D, F32, PAGED, KV8, FP8>;
    k.head_dim = D;
    k.threads = Sh::NT;
    k.smem_bytes = Sh::SMEM_BYTES;
    k.tile_tokens = C::TT;
    k.ctas_per_sm = MB;
    k.seg_unit = Sh::SEG_UNIT;
    k.seg_cost = Sh::SEG_COST;
    k.f32_out = F32;
    k.tensor_core = false;
    k.mma_rows = 0;
    k.index = index;
    return k;
}

// Variants of one head dimension: contiguous bf16 cache at indices IDX,
// IDX + 1, paged at PIDX, PIDX + 1, int8 at QIDX, QIDX + 1, paged int8 at
// PQIDX, PQIDX + 1, fp8 at FIDX, FIDX + 1 and paged fp8 at FIDX + 2, FIDX + 3
// (bf16 and fp32 output).
#define KVD_MMA_TABLE(D, IDX, PIDX, QIDX, PQIDX, FIDX)                                            \
    const ChunkKernel* mma_table_d##D(bool f32, bool paged, bool kv8, bool fp8) {                \
        static const ChunkKernel table[6][2] = {                                                 \
            {make_mma_chunk_kernel<D, false, false>(IDX), make_mma_chunk_kernel<D, true, false>(IDX + 1)}, \
            {make_mma_chunk_kernel<D, false, true>(PIDX), make_mma_chunk_kernel<D, true, true>(PIDX + 1)}, \
            {make_mma_chunk_kernel<D, false, false, true>(QIDX),                                 \
             make_mma_chunk_kernel<D, true, false, true>(QIDX + 1)},                             \
            {make_mma_chunk_kernel<D, false, true, true>(PQIDX),                                 \
             make_mma_chunk_kernel<D, true, true, true>(PQIDX + 1)},                             \
            {make_mma_chunk_kernel<D, false, false, true, true>(FIDX),                           \
             make_mma_chunk_kernel<D, true, false, true, true>(FIDX + 1)},                       \
            {make_mma_chunk_kernel<D, false, true, true, true>(FIDX + 2),                        \
             make_mma_chunk_kernel<D, true, true, true, true>(FIDX + 3)}};                       \
        return &table[(kv8 ? (fp8 ? 4 : 2) : 0) + (paged ? 1 : 0)][f32 ? 1 : 0];                 \
    }

}  // namespace kvd
