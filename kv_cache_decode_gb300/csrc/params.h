// Kernel parameter blocks and the host-side table of attention kernel variants.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvd {

struct DecodeParams {
    const void* q;        // bf16 [B, Hq, D]
    const void* k;        // bf16 [B, S_max, Hkv, D]
    const void* v;
    const int32_t* seq_lens;
    int B, S_max, len_cap, Hq, Hkv, G;
    float scale_log2;     // scale * log2(e): scores are kept in base-2 units
    int n_split;          // CTAs launched for the chunk kernel
    int tile_tokens, seg_unit, seg_cost;  // its schedule geometry (see schedule.cuh)
    // 1 when the launch directly follows this library's KV append on the stream
    // (kvd_decode_step): every input except the appended cache rows was then
    // complete when the launch began, so only the cache loads wait for the
    // preceding grid.
    int early;
    // Early mode after the host-input step's append, which also stages q: the
    // Q loads wait for the append's grid as well.
    int q_wait;
    const int32_t* pos;   // early mode: where the append put each sequence's new row
    void* out;            // bf16 or fp32 [B, Hq, D]
    float* lse;           // optional fp32 [B, Hq]
    int32_t* status;      // optional
    float* ws_o;          // [slots, G, D] partial unnormalised outputs
    float2* ws_ml;        // [slots, G] partial (max, sum), base-2 max
    // Paged cache (block_table non-null): k and v are pools [num_pages, page,
    // Hkv, D] of pages of 1 << page_shift tokens, and token t of sequence b is
    // row t & (page - 1) of page block_table[b * max_blocks + (t >> page_shift)]
    // (S_max is then max_blocks << page_shift). Entries outside [0, num_pages)
    // give zero rows and KVD_STATUS_BAD_PAGE.
    const int32_t* block_table;
    int max_blocks, page_shift, num_pages;
    // 8-bit cache (k_scale non-null): k and v hold int8 codes (kv_fp8 = 0) or
    // fp8 E4M3 codes (kv_fp8 = 1: the kernel's FP8 variant), and row (b, t, h) reads back as
    // k_scale[(b * S_max + t) * Hkv + h] * value(code) (v likewise).
    const float* k_scale;
    const float* v_scale;
    int kv_fp8;
    // Query tokens per sequence (1, or T > 1 for a speculative check step on
    // the mma.sync kernel or the tcgen05 kernel's 128-row variant): q, out
    // [B, T, Hq, D], lse [B, T, Hq]; query token i of sequence b attends to its
    // first seq_lens[b] - T + 1 + i tokens, and the workspace holds T * G rows
    // per slot.
    int T;
    // mma.sync kernel: blocks of 16 of a pair's T * G rows, one CTA each per
    // token run (n_split * row_blocks CTAs); 1 for the tcgen05 kernel.
    int row_blocks;
    // tcgen05 kernel with vT > 1 query tokens per sequence: B is then B * vT
    // virtual sequences (query token i of sequence s is sequence s * vT + i,
    // attending to its first L_s - vT + 1 + i tokens) and T is 1; the merge
    // reads the lengths the same way. 1 otherwise.
    int vT;
    // Unified-maximum softmax (bf16 caches): each segment's running maximum
    // starts at umax_phi2 = phi * log2(e) in the kernels' base-2 score units
    // and stays there while the row's scores allow (see the kernels).
    int umax;
    float umax_phi2;
};

// One compiled variant of the split-KV chunk kernel.
struct ChunkKernel {
    const void* fn;  // the __global__ function (for attributes)
    cudaError_t (*launch)(const struct ChunkKernel& k, const DecodeParams& p, cudaStream_t s);
    int head_dim, threads, smem_bytes, tile_tokens, ctas_per_sm;
    int seg_unit;    // tokens per schedule position (1 or tile_tokens, see schedule.cuh)
    int seg_cost;    // positions charged per pair by the schedule
    bool f32_out, tensor_core;
    int mma_rows;  // tcgen05 kernel: rows of its MMAs (128: several query tokens of a sequence in one tile)
    int index;  // position in the variant table (0..127), for the per-device attribute bitmask
};

// The kernel for a shape: bf16 groups of up to 16 query heads per KV head run
// on the mma.sync kernel (T query tokens as T * G rows, in blocks of 16),
// wider groups (17..64) on the tcgen05 kernel (T query tokens stacked in one
// 128-row tile when T times the group rounded up to 8 fits, else as T virtual
// sequences). 8-bit caches run on the tcgen05 kernel's converting variant
// for groups of 17..64 at head_dim 128 or 17..48 at 256 (T query tokens as
// virtual sequences), else on the mma.sync kernel.
const ChunkKernel* find_chunk_kernel(int head_dim, int group, bool f32_out, bool paged, bool kv8 = false,
                                     bool fp8 = false, int T = 1);
const ChunkKernel* mma_chunk_kernel(int head_dim, bool f32_out, bool paged, bool kv8, bool fp8);
const ChunkKernel* tc_chunk_kernel(int head_dim, bool f32_out, int group, int T = 1);
const ChunkKernel* tc8_chunk_kernel(int head_dim, bool f32_out, int group, bool fp8);

cudaError_t launch_merge(const DecodeParams& p, int head_dim, bool f32_out, int num_sms, cudaStream_t stream);
// Results of disjoint token shards combined by their normalisers (split_kv_merge.cu).
cudaError_t launch_merge_shards(const void* outs, const float* lses, int n, long long rows, int head_dim, bool in_f32,
                                void* out, bool out_f32, float* lse_out, cudaStream_t stream);
// A paged cache's table (block_table null: the cache is contiguous).
struct PagedCache {
    const int32_t* block_table;
    int max_blocks, page_shift, num_pages;
};

// T rows per sequence (k_new [B, T, Hkv, D]) go to pos[b] .. pos[b] + T - 1.
cudaError_t launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                          const int32_t* pos, int B, int S_max, int Hkv, int D,
                          int32_t* status, const PagedCache& pg, cudaStream_t stream, int T = 1,
                          const void* copy_src = nullptr, void* copy_dst = nullptr, size_t copy_bytes = 0,
                          int copy_blocks = 0);
// int8 cache (kv_quant.cu): the append quantizes the new rows (into pages
// when pg.block_table is set); the bulk conversion quantizes rows
// t < seq_lens[b] of a bf16 cache.
cudaError_t launch_append_q8(void* k_codes, void* v_codes, float* k_scale, float* v_scale, const void* k_new,
                             const void* v_new, const int32_t* pos, int B, int S_max, int Hkv, int D,
                             int32_t* status, const PagedCache& pg, cudaStream_t stream, int T = 1,
                             bool fp8 = false);
cudaError_t launch_quantize_q8(const void* src, void* codes, float* scales, const int32_t* seq_lens, int B,
                               int S_max, int len_cap, int Hkv, int D, cudaStream_t stream, bool fp8 = false);

}  // namespace kvd
