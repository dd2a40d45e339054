// KV append: the new token's key and value rows are copied into the cache at
// each sequence's current length (All About Transformer Inference,
// "Transformer inference basics", Generation: the new token's KV is appended
// to the KV cache). A bit copy in 16-byte vectors; no arithmetic. With a paged
// cache the row goes to its block's page (same page, "Tricks for improving
// generation throughput and latency", Paged Attention).
#include <algorithm>

#include "../../include/kvdecode.h"
#include "common.cuh"
#include "params.h"

namespace kvd {

__global__ void __launch_bounds__(256) kv_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       const int32_t* __restrict__ pos, int B,
                                                       int S_max, int Hkv, int vec_per_row,
                                                       int32_t* status, const PagedCache pg, int T,
                                                       const uint4* __restrict__ copy_src,
                                                       uint4* __restrict__ copy_dst, long long copy_n16) {
    // Let the attention kernel that follows start its launch; it waits for
    // this grid's writes before reading the cache (and the copied words).
    pdl_launch_dependents();
    const long long rows = (long long)B * T * Hkv;  // new rows: (b, i, h)
    const long long per_tensor = rows * vec_per_row;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < 2 * per_tensor;
         i += (long long)gridDim.x * blockDim.x) {
        const int which = (int)(i / per_tensor);
        const long long r = i - which * per_tensor;
        const long long row = r / vec_per_row;  // (b * T + i) * Hkv + h
        const int ch = (int)(r - row * vec_per_row);
        const long long bi = row / Hkv;
        const int h = (int)(row - bi * Hkv);
        const int b = (int)(bi / T), tk = (int)(bi - (long long)b * T);  // token tk of sequence b
        // Both loads are issued before either is used: one memory round trip.
        const uint4 val = __ldg((which == 0 ? k_new : v_new) + r);
        const int t = __ldg(pos + b) + tk;
        if (t < 0 || t >= S_max) {
            if (status && which == 0 && h == 0 && ch == 0) atomicOr(status, KVD_STATUS_POS_OUT_OF_RANGE);
            continue;
        }
        long long trow = (long long)b * S_max + t;  // cache row of the token
        if (pg.block_table) {
            const int page = __ldg(pg.block_table + (size_t)b * pg.max_blocks + (t >> pg.page_shift));
            if (page < 0 || page >= pg.num_pages) {
                if (status && which == 0 && h == 0 && ch == 0) atomicOr(status, KVD_STATUS_BAD_PAGE);
                continue;
            }
            trow = ((long long)page << pg.page_shift) + (t & ((1 << pg.page_shift) - 1));
        }
        const long long dst = (trow * Hkv + h) * vec_per_row + ch;
        (which == 0 ? k_cache : v_cache)[dst] = val;
    }
    // The host-input step: the queries, read from page-locked host memory,
    // go to the device staging buffer (four loads in flight per thread).
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < copy_n16; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (i + k * stride < copy_n16) v[k] = __ldcs(copy_src + i + k * stride);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (i + k * stride < copy_n16) copy_dst[i + k * stride] = v[k];
    }
}

cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, int B, int S_max, int Hkv, int D,
                          int32_t* status, const PagedCache& pg, cudaStream_t stream, int T,
                          const void* copy_src, void* copy_dst, size_t copy_bytes, int copy_blocks) {
    const int vec_per_row = D / 8;
    const long long work = 2LL * B * T * Hkv * vec_per_row;
    long long blocks = (work + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (copy_bytes > 0 && blocks < copy_blocks) blocks = copy_blocks;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    // The launch's own status (a stale error from earlier work is not picked up).
    return cudaLaunchKernelEx(&cfg, kv_append_kernel, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                              static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), pos, B, S_max,
                              Hkv, vec_per_row, status, pg, T, static_cast<const uint4*>(copy_src),
                              static_cast<uint4*>(copy_dst), (long long)(copy_bytes / 16));
}

}  // namespace kvd
