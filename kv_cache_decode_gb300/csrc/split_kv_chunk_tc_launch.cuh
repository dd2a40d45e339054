// tcgen05 split-KV chunk kernel: TMA tensor maps and launch (included by the
// per-head-dim instantiation files).
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "split_kv_chunk_tc.cuh"

namespace kvd {

// bf16 (or, u8, one-byte) tensor map with 128-byte swizzle; dims/strides
// innermost first (strides in bytes).
bool tc_encode_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, bool u8 = false);

template <int D, bool F32, int QR, int MR, bool KV8 = false, bool FP8 = false>
cudaError_t launch_tc_chunk(const ChunkKernel& k, const DecodeParams& p, cudaStream_t stream) {
    TcMaps maps;
    std::memset(&maps, 0, sizeof maps);
    {
        // q rows: B * Hq, times T query tokens when they are stacked in one tile.
        const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.B * p.T * p.Hq};
        const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)p.G};
        if (!tc_encode_map(&maps.q, p.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        // Cache rows: [B * S_max] for a contiguous cache, [num_pages * page]
        // for a pool of pages, whose boxes are one page (at most one tile) high.
        constexpr int T = TcShape<D, F32, QR, MR, KV8>::T;
        const bool paged = p.block_table != nullptr;
        const int cache_batch = p.vT > 1 ? p.B / p.vT : p.B;  // virtual sequences share their cache's rows
        const cuuint64_t rows = paged ? ((cuuint64_t)p.num_pages << p.page_shift) : (cuuint64_t)cache_batch * p.S_max;
        const int box_rows = paged ? std::min(1 << p.page_shift, T) : T;
        // (8-bit codes: one byte an element, boxes of 128 columns = 128 bytes)
        constexpr int ES = KV8 ? 1 : 2;
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, rows};
        const cuuint64_t strides[2] = {(cuuint64_t)D * ES, (cuuint64_t)p.Hkv * D * ES};
        const cuuint32_t box[3] = {(cuuint32_t)(128 / ES), 1, (cuuint32_t)box_rows};
        if (!tc_encode_map(&maps.k, p.k, 3, dims, strides, box, KV8)) return cudaErrorInvalidValue;
        if (!tc_encode_map(&maps.v, p.v, 3, dims, strides, box, KV8)) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_split, 1, 1);
    cfg.blockDim = dim3((unsigned)k.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)k.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_chunk_tc_kernel<D, F32, QR, MR, KV8, FP8>, p, maps);
}

template <int D, bool F32, int QR, int MR = 64, bool KV8 = false, bool FP8 = false>
static ChunkKernel make_tc(int index) {
    using Sh = TcShape<D, F32, QR, MR, KV8>;
    ChunkKernel k;
    k.fn = reinterpret_cast<const void*>(split_kv_chunk_tc_kernel<D, F32, QR, MR, KV8, FP8>);
    k.launch = launch_tc_chunk<D, F32, QR, MR, KV8, FP8>;
    k.head_dim = D;
    k.threads = Sh::THREADS;
    k.smem_bytes = Sh::SMEM_BYTES;
    k.tile_tokens = Sh::T;
    k.ctas_per_sm = 1;
    k.seg_unit = Sh::SEG_UNIT;
    k.seg_cost = Sh::SEG_COST;
    k.f32_out = F32;
    k.tensor_core = true;
    k.mma_rows = MR;
    k.index = index;
    return k;
}


}  // namespace kvd
