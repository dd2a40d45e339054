// C ABI of libkvdecode: argument validation, planning and launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>

#include "../../include/kvdecode.h"
#include "params.h"
#include "schedule.cuh"

namespace kvd {

const ChunkKernel* mma_table_d64(bool f32, bool paged, bool kv8, bool fp8);
const ChunkKernel* mma_table_d128(bool f32, bool paged, bool kv8, bool fp8);
const ChunkKernel* mma_table_d256(bool f32, bool paged, bool kv8, bool fp8);

const ChunkKernel* mma_chunk_kernel(int head_dim, bool f32_out, bool paged, bool kv8, bool fp8) {
    switch (head_dim) {
        case 64: return mma_table_d64(f32_out, paged, kv8, fp8);
        case 128: return mma_table_d128(f32_out, paged, kv8, fp8);
        case 256: return mma_table_d256(f32_out, paged, kv8, fp8);
        default: return nullptr;
    }
}

// The tcgen05 kernels take either cache form at run time (only their loads
// differ); the mma.sync kernel has a compiled variant per form. 8-bit caches
// run on the tcgen05 kernel's converting variant when the group is wide (see
// tc8_chunk_kernel), else on the mma.sync kernel, whose CTAs take 16 of a
// pair's rows each, for every group.
const ChunkKernel* find_chunk_kernel(int head_dim, int group, bool f32_out, bool paged, bool kv8, bool fp8, int T) {
    if (group < 1 || group > KVD_MAX_GROUP) return nullptr;
    if (kv8) {
        const ChunkKernel* k = tc8_chunk_kernel(head_dim, f32_out, group, fp8);
        return k ? k : mma_chunk_kernel(head_dim, f32_out, paged, true, fp8);
    }
    if (group <= 16) return mma_chunk_kernel(head_dim, f32_out, paged, false, false);
    return tc_chunk_kernel(head_dim, f32_out, group, T);
}

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_num_sms[kMaxDevices];
// Bit i % 64 of g_smem_ready[dev][i / 64] is set once kernel variant i may
// use its dynamic shared memory size on device dev.
std::atomic<uint64_t> g_smem_ready[kMaxDevices][2];

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A byte range [p, p + n) of device memory; empty when n == 0.
struct ByteRange {
    const void* p;
    size_t n;
    bool overlaps(const ByteRange& o) const {
        if (n == 0 || o.n == 0) return false;
        const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(o.p);
        return a < b + o.n && b < a + n;
    }
};

kvd_status check_shape(int batch, int Hq, int Hkv, int D, kvd_out_dtype dt) {
    if (batch < 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return KVD_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return KVD_ERR_INVALID_ARG;
    if (dt != KVD_OUT_BF16 && dt != KVD_OUT_F32) return KVD_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return KVD_ERR_UNSUPPORTED;
    if (Hq / Hkv > KVD_MAX_GROUP) return KVD_ERR_UNSUPPORTED;
    return KVD_OK;
}

// Both forms of a variant share their launch shape and schedule geometry, so
// planning and the host replica use the contiguous one. The split count is
// planned for the single-token bf16 kernel of the shape whatever the cache
// dtype and query tokens, so that one plan sizes every form's workspace.
const ChunkKernel* pick_kernel(int Hq, int Hkv, int D, kvd_out_dtype dt, bool paged = false, bool kv8 = false,
                               bool fp8 = false, int T = 1) {
    return find_chunk_kernel(D, Hq / Hkv, dt == KVD_OUT_F32, paged, kv8, fp8, T);
}

// int8 cache: the row scales of K and V.
struct QuantCache {
    float* k_scale;
    float* v_scale;
    bool fp8 = false;  // E4M3 codes rather than int8
};

// Paged cache arguments, checked; s_max of the contiguous calls becomes
// max_blocks * page_size.
kvd_status check_paged(const int32_t* block_table, int max_blocks, int page_size, int num_pages,
                       PagedCache* pg, int* s_max) {
    if (!block_table || !aligned(block_table, 4)) return KVD_ERR_INVALID_ARG;
    if (page_size < 16 || page_size > 4096 || (page_size & (page_size - 1)) != 0) return KVD_ERR_INVALID_ARG;
    if (max_blocks < 1 || num_pages < 1) return KVD_ERR_INVALID_ARG;
    // Token positions and pool rows (and one past the pool) stay 32-bit.
    if ((long long)max_blocks * page_size > 0x7fffffffLL || (long long)num_pages * page_size >= 0x7fffffffLL)
        return KVD_ERR_INVALID_ARG;
    int shift = 0;
    while ((1 << shift) < page_size) ++shift;
    *pg = PagedCache{block_table, max_blocks, shift, num_pages};
    *s_max = max_blocks * page_size;
    return KVD_OK;
}

kvd_status device_sms(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVD_ERR_CUDA;
    int v = g_num_sms[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            return KVD_ERR_CUDA;
        g_num_sms[dev].store(v, std::memory_order_relaxed);
    }
    *sms = v;
    return KVD_OK;
}

// Split count: one CTA per resident slot, but no fewer than two pipeline tiles
// of work per CTA for short or small batches.
int heuristic_split(const ChunkKernel* k, int batch, int Hkv, int max_len, int num_sms) {
    const long long upper = (long long)batch * Hkv * max_len;  // tokens, an upper bound
    const long long slots = (long long)num_sms * k->ctas_per_sm;
    const long long min_tokens = 2LL * k->tile_tokens;
    const long long by_work = std::max(1LL, (upper + min_tokens - 1) / min_tokens);
    return (int)std::max(1LL, std::min(slots, by_work));
}

size_t workspace_for(int n_split, int batch, int Hq, int Hkv, int D) {
    if (n_split <= 1 || batch == 0) return 0;
    const size_t P = (size_t)batch * Hkv, G = (size_t)(Hq / Hkv);
    const size_t slots = (size_t)n_split + P - 1;
    return align256(slots * G * D * sizeof(float)) + align256(slots * G * sizeof(float2));
}

kvd_status plan(int batch, int Hq, int Hkv, int D, int max_len, int num_sms, int n_split_req,
                kvd_out_dtype dt, int* n_split, size_t* ws, const ChunkKernel** kern, int T = 1) {
    kvd_status st = check_shape(batch, Hq, Hkv, D, dt);
    if (st != KVD_OK) return st;
    if (max_len < 0 || n_split_req < 0 || num_sms < 0) return KVD_ERR_INVALID_ARG;
    const ChunkKernel* k = pick_kernel(Hq, Hkv, D, dt);
    if (!k) return KVD_ERR_UNSUPPORTED;
    int n = n_split_req;
    if (n == 0) {
        int sms = num_sms;
        if (sms == 0) {
            st = device_sms(&sms);
            if (st != KVD_OK) return st;
        }
        n = heuristic_split(k, batch, Hkv, max_len, sms);
    }
    *n_split = n;
    *ws = workspace_for(n, batch, Hq * T, Hkv, D);  // T * G rows per slot
    if (kern) *kern = k;
    return KVD_OK;
}

enum Phase { kBoth = 3, kChunk = 1, kMerge = 2 };

// The KV append launched ahead of the attention by kvd_decode_step.
struct AppendArgs {
    void* k_cache;
    void* v_cache;
    const void* k_new;
    const void* v_new;
    const int32_t* pos;
    // The host-input step: the append also copies copy_bytes from copy_src
    // (page-locked host memory the device addresses) to copy_dst (the staged
    // queries), and the attention's Q loads wait for it.
    const void* copy_src = nullptr;
    void* copy_dst = nullptr;
    size_t copy_bytes = 0;
};

kvd_status check_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                        const int32_t* pos, int batch, int s_max, int Hkv, int D, const int32_t* status) {
    if (batch < 0 || s_max < 0 || Hkv <= 0 || D <= 0 || D % 8 != 0) return KVD_ERR_INVALID_ARG;
    if (!k_cache || !v_cache || !k_new || !v_new || !pos) return KVD_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(pos, 4) || (status && !aligned(status, 4)))
        return KVD_ERR_INVALID_ARG;
    return KVD_OK;
}

kvd_status decode(int phase, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* seq_lens, int batch, int s_max, int max_seq_len, int Hq, int Hkv,
                  int D, float scale, int n_split_req, void* workspace, size_t workspace_bytes,
                  void* out, kvd_out_dtype dt, float* lse, int32_t* status, kvd_stream_t stream,
                  const AppendArgs* app = nullptr, const PagedCache* pg = nullptr,
                  const QuantCache* q8 = nullptr, int T = 1, const float* umax_phi = nullptr) {
    kvd_status st = check_shape(batch, Hq, Hkv, D, dt);
    if (st != KVD_OK) return st;
    if (s_max <= 0 || max_seq_len < 0 || max_seq_len > s_max) return KVD_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || n_split_req < 0) return KVD_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return KVD_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(seq_lens, 4) || (lse && !aligned(lse, 4)) || (status && !aligned(status, 4)))
        return KVD_ERR_INVALID_ARG;
    // Cache rows: batch * s_max, or the pool's pages * page size.
    const long long cache_rows = pg ? ((long long)pg->num_pages << pg->page_shift) : (long long)batch * s_max;
    if ((size_t)cache_rows * Hkv * D > ((size_t)1 << 62)) return KVD_ERR_INVALID_ARG;

    int n_split = 0;
    size_t need = 0;
    const ChunkKernel* k = nullptr;
    if (T < 1) return KVD_ERR_INVALID_ARG;
    if (T > KVD_MAX_TOKENS) return KVD_ERR_UNSUPPORTED;
    // Unified maximum: phi in the logits' units (scale * q.k), bf16 caches.
    const float phi2 = umax_phi ? *umax_phi * 1.4426950408889634f : 0.f;
    if (umax_phi && !std::isfinite(phi2)) return KVD_ERR_INVALID_ARG;
    if (umax_phi && q8) return KVD_ERR_UNSUPPORTED;
    st = plan(batch, Hq, Hkv, D, max_seq_len, 0 /* query device if heuristic */, n_split_req, dt,
              &n_split, &need, &k, T);
    if (st != KVD_OK) return st;
    if (q8 && (!q8->k_scale || !q8->v_scale || !aligned(q8->k_scale, 4) || !aligned(q8->v_scale, 4)))
        return KVD_ERR_INVALID_ARG;
    k = pick_kernel(Hq, Hkv, D, dt, pg != nullptr, q8 != nullptr, q8 && q8->fp8, T);
    if (!k) return KVD_ERR_UNSUPPORTED;
    // The tensor-core path addresses cache rows and query rows with 32-bit TMA coordinates.
    if (k->tensor_core && (cache_rows > 0x7fffffffLL || (long long)batch * T * Hq > 0x7fffffffLL))
        return KVD_ERR_UNSUPPORTED;
    // mma.sync kernel: 16 of a pair's T * G rows per CTA. tcgen05 kernel: T
    // query tokens stacked in one 128-row tile, or (when they do not fit) as T
    // virtual sequences of one query token each.
    const int row_blocks = k->tensor_core ? 1 : (Hq / Hkv * T + 15) / 16;
    const int vT = (k->tensor_core && k->mma_rows != 128) ? T : 1;
    if (n_split_req == 0 && row_blocks > 1) {
        // The heuristic split fills the GPU with one CTA per resident slot; a
        // pair in row blocks launches row_blocks CTAs per token run, so the
        // run count is cut to keep the launch to one wave (a second, partial
        // wave measured up to a quarter slower). Fewer runs need less workspace.
        int sms = 0;
        st = device_sms(&sms);
        if (st != KVD_OK) return st;
        const int per_wave = (int)std::max(1LL, (long long)sms * k->ctas_per_sm / row_blocks);
        if (n_split > per_wave) {
            n_split = per_wave;
            need = workspace_for(n_split, batch, Hq * T, Hkv, D);
        }
    }
    if ((long long)n_split * row_blocks > 0x7fffffffLL) return KVD_ERR_INVALID_ARG;
    if ((long long)batch * vT > 0x7fffffffLL) return KVD_ERR_INVALID_ARG;
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return KVD_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(workspace, 256)) return KVD_ERR_INVALID_ARG;
    }
    if (batch == 0) return KVD_OK;

    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.seq_lens = seq_lens;
    p.B = batch * vT;
    p.S_max = s_max;
    p.len_cap = std::min(s_max, max_seq_len);
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.n_split = n_split;
    p.tile_tokens = k->tile_tokens;
    p.seg_unit = k->seg_unit;
    p.seg_cost = k->seg_cost;
    p.out = out;
    p.lse = lse;
    p.status = status;
    p.T = T / vT;
    p.row_blocks = row_blocks;
    p.vT = vT;
    p.umax = umax_phi ? 1 : 0;
    p.umax_phi2 = phi2;
    if (q8) {
        p.k_scale = q8->k_scale;
        p.v_scale = q8->v_scale;
        p.kv_fp8 = q8->fp8 ? 1 : 0;
    }
    if (pg) {
        p.block_table = pg->block_table;
        p.max_blocks = pg->max_blocks;
        p.page_shift = pg->page_shift;
        p.num_pages = pg->num_pages;
    }
    if (need > 0) {
        // T * G rows per slot (as workspace_for with T query tokens), or G
        // rows per virtual pair, which takes no more space.
        const size_t P = (size_t)p.B * Hkv, rows = (size_t)p.G * p.T, slots = (size_t)n_split + P - 1;
        uint8_t* w = static_cast<uint8_t*>(workspace);
        p.ws_o = reinterpret_cast<float*>(w);
        w += align256(slots * rows * D * sizeof(float));
        p.ws_ml = reinterpret_cast<float2*>(w);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (app) {
        int copy_sms = 0;
        if (app->copy_bytes > 0 && device_sms(&copy_sms) != KVD_OK) return KVD_ERR_CUDA;
        // The append, then the chunk kernel in early mode: it starts (and works
        // out its schedule) while the append runs, and only its cache loads
        // wait for the append's grid.
        const PagedCache none{nullptr, 0, 0, 0};
        const cudaError_t e =
            q8 ? launch_append_q8(app->k_cache, app->v_cache, q8->k_scale, q8->v_scale, app->k_new, app->v_new,
                                  app->pos, batch, s_max, Hkv, D, status, pg ? *pg : none, s, T, q8->fp8)
               : launch_append(app->k_cache, app->v_cache, app->k_new, app->v_new, app->pos, batch, s_max, Hkv,
                               D, status, pg ? *pg : none, s, T, app->copy_src, app->copy_dst, app->copy_bytes,
                               copy_sms);  // one CTA per SM: the attention's CTAs fit beside them
        if (e != cudaSuccess) return KVD_ERR_CUDA;
        p.early = 1;
        p.q_wait = app->copy_bytes > 0 ? 1 : 0;
        p.pos = app->pos;
    }
    if (phase & kChunk) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVD_ERR_CUDA;
        const uint64_t bit = 1ull << (k->index & 63);
        std::atomic<uint64_t>& ready = g_smem_ready[dev][(k->index >> 6) & 1];
        if (!(ready.load(std::memory_order_acquire) & bit)) {
            if (cudaFuncSetAttribute(k->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k->smem_bytes) !=
                cudaSuccess)
                return KVD_ERR_CUDA;
            ready.fetch_or(bit, std::memory_order_acq_rel);
        }
        if (k->launch(*k, p, s) != cudaSuccess) return KVD_ERR_CUDA;
    }
    if ((phase & kMerge) && n_split > 1) {
        int sms = 0;
        if (device_sms(&sms) != KVD_OK) return KVD_ERR_CUDA;
        if (launch_merge(p, D, dt == KVD_OUT_F32, sms, s) != cudaSuccess) return KVD_ERR_CUDA;
    }
    return KVD_OK;
}

}  // namespace
}  // namespace kvd

using namespace kvd;

extern "C" {

kvd_status kvd_decode_plan(int batch, int n_heads_q, int n_heads_kv, int head_dim, int max_seq_len,
                           int num_sms, int n_split_request, kvd_out_dtype out_dtype,
                           int* n_split_out, size_t* workspace_bytes_out) {
    if (!n_split_out || !workspace_bytes_out) return KVD_ERR_INVALID_ARG;
    return plan(batch, n_heads_q, n_heads_kv, head_dim, max_seq_len, num_sms, n_split_request,
                out_dtype, n_split_out, workspace_bytes_out, nullptr);
}

kvd_status kvd_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* pos, int batch, int s_max, int n_heads_kv, int head_dim,
                         int32_t* status_word, kvd_stream_t stream) {
    const kvd_status st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv,
                                       head_dim, status_word);
    if (st != KVD_OK) return st;
    if (batch == 0) return KVD_OK;
    const PagedCache none{nullptr, 0, 0, 0};
    return launch_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                         status_word, none, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

kvd_status kvd_decode_plan_multi(int batch, int n_tokens, int n_heads_q, int n_heads_kv, int head_dim,
                                 int max_seq_len, int num_sms, int n_split_request, kvd_out_dtype out_dtype,
                                 int* n_split_out, size_t* workspace_bytes_out) {
    if (!n_split_out || !workspace_bytes_out || n_tokens < 1) return KVD_ERR_INVALID_ARG;
    if (n_tokens > KVD_MAX_TOKENS) return KVD_ERR_UNSUPPORTED;
    return plan(batch, n_heads_q, n_heads_kv, head_dim, max_seq_len, num_sms, n_split_request, out_dtype,
                n_split_out, workspace_bytes_out, nullptr, n_tokens);
}

kvd_status kvd_kv_append_multi(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                               const int32_t* pos, int batch, int n_tokens, int s_max, int n_heads_kv,
                               int head_dim, int32_t* status_word, kvd_stream_t stream) {
    if (n_tokens < 1) return KVD_ERR_INVALID_ARG;
    const kvd_status st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                                       status_word);
    if (st != KVD_OK) return st;
    if (batch == 0) return KVD_OK;
    const PagedCache none{nullptr, 0, 0, 0};
    return launch_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim, status_word,
                         none, static_cast<cudaStream_t>(stream), n_tokens) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

kvd_status kvd_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* seq_lens, int batch, int n_tokens, int s_max,
                                      int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                      int n_split, void* workspace, size_t workspace_bytes, void* out,
                                      kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                      kvd_stream_t stream) {
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, nullptr, nullptr, nullptr, n_tokens);
}

kvd_status kvd_decode_step_multi(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                 const int32_t* pos, const void* q, const int32_t* seq_lens, int batch,
                                 int n_tokens, int s_max, int max_seq_len, int n_heads_q, int n_heads_kv,
                                 int head_dim, float scale, int n_split, void* workspace, size_t workspace_bytes,
                                 void* out, kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                 kvd_stream_t stream) {
    const kvd_status st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                                       status_word);
    if (st != KVD_OK) return st;
    const AppendArgs app{k_cache, v_cache, k_new, v_new, pos};
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, &app, nullptr, nullptr, n_tokens);
}

kvd_status kvd_merge_attention(const void* outs, const float* lses, int n_shards, long long rows, int head_dim,
                               kvd_out_dtype in_dtype, void* out, kvd_out_dtype out_dtype, float* lse_out,
                               kvd_stream_t stream) {
    if (!outs || !lses || !out || n_shards < 1 || rows < 0) return KVD_ERR_INVALID_ARG;
    if ((in_dtype != KVD_OUT_BF16 && in_dtype != KVD_OUT_F32) || (out_dtype != KVD_OUT_BF16 && out_dtype != KVD_OUT_F32))
        return KVD_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVD_ERR_UNSUPPORTED;
    if (!aligned(outs, 16) || !aligned(out, 16) || !aligned(lses, 4) || (lse_out && !aligned(lse_out, 4)))
        return KVD_ERR_INVALID_ARG;
    if ((unsigned long long)rows * (unsigned long long)(head_dim / 8) > 0x7fffffffULL * 256ULL) return KVD_ERR_INVALID_ARG;
    if (rows == 0) return KVD_OK;
    // The kernel reads outs and lses while it writes out and lse_out: the
    // written ranges may overlap neither the read ones nor each other.
    const size_t in_es = in_dtype == KVD_OUT_F32 ? 4 : 2, out_es = out_dtype == KVD_OUT_F32 ? 4 : 2;
    const size_t n_rows = (size_t)rows, n_sh = (size_t)n_shards, d = (size_t)head_dim;
    const ByteRange r_outs{outs, n_sh * n_rows * d * in_es}, r_lses{lses, n_sh * n_rows * 4},
        r_out{out, n_rows * d * out_es}, r_lse{lse_out, lse_out ? n_rows * 4 : 0};
    if (r_out.overlaps(r_outs) || r_out.overlaps(r_lses) || r_lse.overlaps(r_outs) || r_lse.overlaps(r_lses) ||
        r_lse.overlaps(r_out))
        return KVD_ERR_INVALID_ARG;
    return launch_merge_shards(outs, lses, n_shards, rows, head_dim, in_dtype == KVD_OUT_F32, out,
                               out_dtype == KVD_OUT_F32, lse_out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

size_t kvd_step_staging_bytes(int batch, int n_tokens, int n_heads_q, int n_heads_kv, int head_dim) {
    if (batch < 0 || n_tokens < 1 || n_heads_q < 1 || n_heads_kv < 1 || head_dim < 1) return 0;
    const size_t BT = (size_t)batch * n_tokens;
    return align256(BT * n_heads_q * head_dim * 2) + 2 * align256(BT * n_heads_kv * head_dim * 2) +
           2 * align256((size_t)batch * 4);
}

kvd_status kvd_decode_step_host(void* k_cache, void* v_cache, const void* q_host, const void* k_new_host,
                                const void* v_new_host, const int32_t* pos_host, const int32_t* seq_lens_host,
                                void* staging, size_t staging_bytes, int batch, int n_tokens, int s_max,
                                int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                int n_split, void* workspace, size_t workspace_bytes, void* out, void* out_host,
                                kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                kvd_stream_t stream) {
    if (!q_host || !k_new_host || !v_new_host || !pos_host || !seq_lens_host || !out_host || !staging)
        return KVD_ERR_INVALID_ARG;
    kvd_status st = check_shape(batch, n_heads_q, n_heads_kv, head_dim, out_dtype);
    if (st != KVD_OK) return st;
    if (n_tokens < 1) return KVD_ERR_INVALID_ARG;
    if (!aligned(staging, 256) || staging_bytes < kvd_step_staging_bytes(batch, n_tokens, n_heads_q, n_heads_kv,
                                                                         head_dim))
        return KVD_ERR_INVALID_ARG;
    // out == NULL: the kernels write the result straight into out_host, which
    // must then be page-locked host memory the device can address.
    void* out_dev = out;
    if (!out) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, out_host) != cudaSuccess || a.type != cudaMemoryTypeHost ||
            !a.devicePointer || !aligned(a.devicePointer, 16))
            return KVD_ERR_INVALID_ARG;
        out_dev = a.devicePointer;
    }
    if (batch == 0) return KVD_OK;
    // The staged inputs: q | k_new | v_new | pos | seq_lens, each 256-byte aligned.
    const size_t BT = (size_t)batch * n_tokens;
    const size_t qb = BT * n_heads_q * head_dim * 2, kb = BT * n_heads_kv * head_dim * 2, ib = (size_t)batch * 4;
    uint8_t* w = static_cast<uint8_t*>(staging);
    void* q = w;
    void* k_new = w + align256(qb);
    void* v_new = static_cast<uint8_t*>(k_new) + align256(kb);
    int32_t* pos = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(v_new) + align256(kb));
    int32_t* seq_lens = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(pos) + align256(ib));
    // Everything the step checks, before any copy is queued.
    st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim, status_word);
    if (st != KVD_OK) return st;
    int n = 0;
    size_t need = 0;
    st = plan(batch, n_heads_q, n_heads_kv, head_dim, max_seq_len, 0, n_split, out_dtype, &n, &need, nullptr,
              n_tokens);
    if (st != KVD_OK) return st;
    if (need > 0 && (!workspace || workspace_bytes < need)) return KVD_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Host inputs laid out like the staging buffer (one packet from q_host on)
    // go in one copy; otherwise one copy each.
    const uint8_t* hq = static_cast<const uint8_t*>(q_host);
    const uint8_t* stg = static_cast<const uint8_t*>(staging);
    auto at = [&](const void* dev) { return hq + (static_cast<const uint8_t*>(dev) - stg); };
    const bool packed = k_new_host == at(k_new) && v_new_host == at(v_new) &&
                        reinterpret_cast<const uint8_t*>(pos_host) == at(pos) &&
                        reinterpret_cast<const uint8_t*>(seq_lens_host) == at(seq_lens);
    // A packet the device can address (page-locked and mapped): the append
    // reads k_new, v_new and pos from it and copies q into the staging buffer,
    // and the attention reads pos and seq_lens from it, so that the host
    // link's transfer overlaps the attention's start (its cache loads run
    // meanwhile; its Q loads wait for the append). Otherwise the inputs are
    // copied in first (one cudaMemcpyAsync for a packet, else five).
    cudaPointerAttributes pa;
    const bool mapped = packed && cudaPointerGetAttributes(&pa, q_host) == cudaSuccess &&
                        pa.type == cudaMemoryTypeHost && pa.devicePointer && aligned(pa.devicePointer, 256);
    if (!mapped) (void)cudaGetLastError();
    AppendArgs app{k_cache, v_cache, k_new, v_new, pos};
    const int32_t* lens_dev = seq_lens;
    if (mapped) {
        const uint8_t* hd = static_cast<const uint8_t*>(pa.devicePointer);
        auto dev_at = [&](const void* staged) { return hd + (static_cast<const uint8_t*>(staged) - stg); };
        app.k_new = dev_at(k_new);
        app.v_new = dev_at(v_new);
        app.pos = reinterpret_cast<const int32_t*>(dev_at(pos));
        app.copy_src = hd;
        app.copy_dst = q;
        app.copy_bytes = qb;
        lens_dev = reinterpret_cast<const int32_t*>(dev_at(seq_lens));
    } else if (packed) {
        const size_t total = static_cast<const uint8_t*>(static_cast<const void*>(seq_lens)) + ib - stg;
        if (cudaMemcpyAsync(staging, q_host, total, cudaMemcpyHostToDevice, s) != cudaSuccess) return KVD_ERR_CUDA;
    } else {
        const struct { void* dst; const void* src; size_t n; } h2d[5] = {
            {q, q_host, qb}, {k_new, k_new_host, kb}, {v_new, v_new_host, kb}, {pos, pos_host, ib},
            {seq_lens, seq_lens_host, ib}};
        for (const auto& c : h2d)
            if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s) != cudaSuccess) return KVD_ERR_CUDA;
    }
    st = decode(kBoth, q, k_cache, v_cache, lens_dev, batch, s_max, max_seq_len, n_heads_q, n_heads_kv, head_dim,
                scale, n_split, workspace, workspace_bytes, out_dev, out_dtype, lse_out, status_word, stream, &app,
                nullptr, nullptr, n_tokens);
    if (st != KVD_OK) return st;
    if (!out) return KVD_OK;  // written in place over the host link
    const size_t ob = BT * n_heads_q * head_dim * (out_dtype == KVD_OUT_F32 ? 4 : 2);
    return cudaMemcpyAsync(out_host, out, ob, cudaMemcpyDeviceToHost, s) == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}

kvd_status kvd_decode_ex(const kvd_cache* cache, const void* q, const int32_t* seq_lens, int batch, int n_tokens,
                         int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale, int n_split,
                         void* workspace, size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                         float* lse_out, const void* k_new, const void* v_new, const int32_t* pos,
                         int32_t* status_word, kvd_stream_t stream) {
    if (!cache) return KVD_ERR_INVALID_ARG;
    const bool append = k_new || v_new || pos;
    if (append && !(k_new && v_new && pos)) return KVD_ERR_INVALID_ARG;
    if ((cache->k_scales != nullptr) != (cache->v_scales != nullptr)) return KVD_ERR_INVALID_ARG;
    PagedCache pg;
    int s_max = cache->s_max;
    const bool paged = cache->block_table != nullptr;
    if (paged) {
        const kvd_status st = check_paged(cache->block_table, cache->max_blocks, cache->page_size,
                                          cache->num_pages, &pg, &s_max);
        if (st != KVD_OK) return st;
    }
    if (cache->fp8 && !cache->k_scales) return KVD_ERR_INVALID_ARG;  // fp8 codes need their scales
    const QuantCache q8{cache->k_scales, cache->v_scales, cache->fp8 != 0};
    const bool quant = cache->k_scales != nullptr;
    AppendArgs app{cache->k, cache->v, k_new, v_new, pos};
    if (append) {
        const kvd_status st = check_append(cache->k, cache->v, k_new, v_new, pos, batch, s_max, n_heads_kv,
                                           head_dim, status_word);
        if (st != KVD_OK) return st;
    }
    return decode(kBoth, q, cache->k, cache->v, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, append ? &app : nullptr, paged ? &pg : nullptr, quant ? &q8 : nullptr, n_tokens);
}

// The 8-bit quantizer and appends (int8, or fp8 E4M3 when fp8 is set).
static kvd_status quantize8(const void* cache, void* codes, float* scales, const int32_t* seq_lens, int batch,
                            int s_max, int max_seq_len, int n_heads_kv, int head_dim, kvd_stream_t stream, bool fp8) {
    if (batch < 0 || s_max <= 0 || max_seq_len < 0 || max_seq_len > s_max || n_heads_kv <= 0) return KVD_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVD_ERR_UNSUPPORTED;
    if (!cache || !codes || !scales || !seq_lens || !aligned(cache, 16) || !aligned(codes, 16) ||
        !aligned(scales, 4) || !aligned(seq_lens, 4))
        return KVD_ERR_INVALID_ARG;
    if (batch == 0) return KVD_OK;
    return launch_quantize_q8(cache, codes, scales, seq_lens, batch, s_max, max_seq_len, n_heads_kv, head_dim,
                              static_cast<cudaStream_t>(stream), fp8) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

static kvd_status append8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                          const void* v_new, const int32_t* pos, int batch, int s_max, int n_heads_kv, int head_dim,
                          int32_t* status_word, kvd_stream_t stream, const PagedCache& pg, bool fp8) {
    kvd_status st = check_append(k_codes, v_codes, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                                 status_word);
    if (st != KVD_OK) return st;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVD_ERR_UNSUPPORTED;
    if (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4)) return KVD_ERR_INVALID_ARG;
    if (batch == 0) return KVD_OK;
    return launch_append_q8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, batch, s_max, n_heads_kv,
                            head_dim, status_word, pg, static_cast<cudaStream_t>(stream), 1, fp8) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

static kvd_status append8_paged(void* k_code_pages, void* v_code_pages, float* k_scale_pages, float* v_scale_pages,
                                const void* k_new, const void* v_new, const int32_t* block_table, const int32_t* pos,
                                int batch, int max_blocks, int page_size, int num_pages, int n_heads_kv,
                                int head_dim, int32_t* status_word, kvd_stream_t stream, bool fp8) {
    PagedCache pg;
    int s_max = 0;
    const kvd_status st = check_paged(block_table, max_blocks, page_size, num_pages, &pg, &s_max);
    if (st != KVD_OK) return st;
    return append8(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, pos, batch, s_max,
                   n_heads_kv, head_dim, status_word, stream, pg, fp8);
}

kvd_status kvd_kv_quantize_q8(const void* cache, void* codes, float* scales, const int32_t* seq_lens, int batch,
                              int s_max, int max_seq_len, int n_heads_kv, int head_dim, kvd_stream_t stream) {
    return quantize8(cache, codes, scales, seq_lens, batch, s_max, max_seq_len, n_heads_kv, head_dim, stream, false);
}

kvd_status kvd_kv_quantize_fp8(const void* cache, void* codes, float* scales, const int32_t* seq_lens, int batch,
                               int s_max, int max_seq_len, int n_heads_kv, int head_dim, kvd_stream_t stream) {
    return quantize8(cache, codes, scales, seq_lens, batch, s_max, max_seq_len, n_heads_kv, head_dim, stream, true);
}

kvd_status kvd_kv_append_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                            const void* v_new, const int32_t* pos, int batch, int s_max, int n_heads_kv,
                            int head_dim, int32_t* status_word, kvd_stream_t stream) {
    return append8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                   status_word, stream, PagedCache{nullptr, 0, 0, 0}, false);
}

kvd_status kvd_kv_append_fp8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                             const void* v_new, const int32_t* pos, int batch, int s_max, int n_heads_kv,
                             int head_dim, int32_t* status_word, kvd_stream_t stream) {
    return append8(k_codes, v_codes, k_scales, v_scales, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                   status_word, stream, PagedCache{nullptr, 0, 0, 0}, true);
}

kvd_status kvd_kv_append_q8_paged(void* k_code_pages, void* v_code_pages, float* k_scale_pages,
                                  float* v_scale_pages, const void* k_new, const void* v_new,
                                  const int32_t* block_table, const int32_t* pos, int batch, int max_blocks,
                                  int page_size, int num_pages, int n_heads_kv, int head_dim,
                                  int32_t* status_word, kvd_stream_t stream) {
    return append8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                         batch, max_blocks, page_size, num_pages, n_heads_kv, head_dim, status_word, stream, false);
}

kvd_status kvd_kv_append_fp8_paged(void* k_code_pages, void* v_code_pages, float* k_scale_pages,
                                   float* v_scale_pages, const void* k_new, const void* v_new,
                                   const int32_t* block_table, const int32_t* pos, int batch, int max_blocks,
                                   int page_size, int num_pages, int n_heads_kv, int head_dim,
                                   int32_t* status_word, kvd_stream_t stream) {
    return append8_paged(k_code_pages, v_code_pages, k_scale_pages, v_scale_pages, k_new, v_new, block_table, pos,
                         batch, max_blocks, page_size, num_pages, n_heads_kv, head_dim, status_word, stream, true);
}

kvd_status kvd_decode_attention_q8(const void* q, const void* k_codes, const void* v_codes, const float* k_scales,
                                   const float* v_scales, const int32_t* seq_lens, int batch, int s_max,
                                   int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                   int n_split, void* workspace, size_t workspace_bytes, void* out,
                                   kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                   kvd_stream_t stream) {
    const QuantCache q8{const_cast<float*>(k_scales), const_cast<float*>(v_scales)};
    return decode(kBoth, q, k_codes, v_codes, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, nullptr, nullptr, &q8);
}

kvd_status kvd_decode_step_q8(void* k_codes, void* v_codes, float* k_scales, float* v_scales, const void* k_new,
                              const void* v_new, const int32_t* pos, const void* q, const int32_t* seq_lens,
                              int batch, int s_max, int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                              float scale, int n_split, void* workspace, size_t workspace_bytes, void* out,
                              kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                              kvd_stream_t stream) {
    const kvd_status st = check_append(k_codes, v_codes, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                                       status_word);
    if (st != KVD_OK) return st;
    const AppendArgs app{k_codes, v_codes, k_new, v_new, pos};
    const QuantCache q8{k_scales, v_scales};
    return decode(kBoth, q, k_codes, v_codes, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, &app, nullptr, &q8);
}

kvd_status kvd_kv_append_paged(void* k_pages, void* v_pages, const void* k_new, const void* v_new,
                               const int32_t* block_table, const int32_t* pos, int batch,
                               int max_blocks, int page_size, int num_pages, int n_heads_kv,
                               int head_dim, int32_t* status_word, kvd_stream_t stream) {
    PagedCache pg;
    int s_max = 0;
    kvd_status st = check_paged(block_table, max_blocks, page_size, num_pages, &pg, &s_max);
    if (st != KVD_OK) return st;
    st = check_append(k_pages, v_pages, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim, status_word);
    if (st != KVD_OK) return st;
    if (batch == 0) return KVD_OK;
    return launch_append(k_pages, v_pages, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim,
                         status_word, pg, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVD_OK
               : KVD_ERR_CUDA;
}

kvd_status kvd_decode_attention_paged(const void* q, const void* k_pages, const void* v_pages,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      int batch, int max_blocks, int page_size, int num_pages,
                                      int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                                      float scale, int n_split, void* workspace,
                                      size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                                      float* lse_out, int32_t* status_word, kvd_stream_t stream) {
    PagedCache pg;
    int s_max = 0;
    const kvd_status st = check_paged(block_table, max_blocks, page_size, num_pages, &pg, &s_max);
    if (st != KVD_OK) return st;
    return decode(kBoth, q, k_pages, v_pages, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out,
                  status_word, stream, nullptr, &pg);
}

kvd_status kvd_decode_step_paged(void* k_pages, void* v_pages, const void* k_new, const void* v_new,
                                 const int32_t* pos, const void* q, const int32_t* block_table,
                                 const int32_t* seq_lens, int batch, int max_blocks, int page_size,
                                 int num_pages, int max_seq_len, int n_heads_q, int n_heads_kv,
                                 int head_dim, float scale, int n_split, void* workspace,
                                 size_t workspace_bytes, void* out, kvd_out_dtype out_dtype,
                                 float* lse_out, int32_t* status_word, kvd_stream_t stream) {
    PagedCache pg;
    int s_max = 0;
    kvd_status st = check_paged(block_table, max_blocks, page_size, num_pages, &pg, &s_max);
    if (st != KVD_OK) return st;
    st = check_append(k_pages, v_pages, k_new, v_new, pos, batch, s_max, n_heads_kv, head_dim, status_word);
    if (st != KVD_OK) return st;
    const AppendArgs app{k_pages, v_pages, k_new, v_new, pos};
    return decode(kBoth, q, k_pages, v_pages, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out,
                  status_word, stream, &app, &pg);
}

kvd_status kvd_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                                int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                int n_split, void* workspace, size_t workspace_bytes, void* out,
                                kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                kvd_stream_t stream) {
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q,
                  n_heads_kv, head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype,
                  lse_out, status_word, stream);
}

kvd_status kvd_decode_step(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                           const int32_t* pos, const void* q, const int32_t* seq_lens, int batch,
                           int s_max, int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                           float scale, int n_split, void* workspace, size_t workspace_bytes,
                           void* out, kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                           kvd_stream_t stream) {
    const kvd_status st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv,
                                       head_dim, status_word);
    if (st != KVD_OK) return st;
    const AppendArgs app{k_cache, v_cache, k_new, v_new, pos};
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q,
                  n_heads_kv, head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype,
                  lse_out, status_word, stream, &app);
}

kvd_status kvd_decode_attention_umax(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                                     int n_heads_q, int n_heads_kv, int head_dim, float scale, float phi,
                                     int n_split, void* workspace, size_t workspace_bytes, void* out,
                                     kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                     kvd_stream_t stream) {
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, nullptr, nullptr, nullptr, 1, &phi);
}

kvd_status kvd_decode_step_umax(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                const int32_t* pos, const void* q, const int32_t* seq_lens, int batch, int s_max,
                                int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim, float scale,
                                float phi, int n_split, void* workspace, size_t workspace_bytes, void* out,
                                kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                                kvd_stream_t stream) {
    const kvd_status st = check_append(k_cache, v_cache, k_new, v_new, pos, batch, s_max, n_heads_kv,
                                       head_dim, status_word);
    if (st != KVD_OK) return st;
    const AppendArgs app{k_cache, v_cache, k_new, v_new, pos};
    return decode(kBoth, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q, n_heads_kv,
                  head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype, lse_out, status_word,
                  stream, &app, nullptr, nullptr, 1, &phi);
}

kvd_status kvd_split_kv_chunk(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                              int n_heads_q, int n_heads_kv, int head_dim, float scale, int n_split,
                              void* workspace, size_t workspace_bytes, void* out,
                              kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                              kvd_stream_t stream) {
    return decode(kChunk, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q,
                  n_heads_kv, head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype,
                  lse_out, status_word, stream);
}

kvd_status kvd_split_kv_merge(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* seq_lens, int batch, int s_max, int max_seq_len,
                              int n_heads_q, int n_heads_kv, int head_dim, float scale, int n_split,
                              void* workspace, size_t workspace_bytes, void* out,
                              kvd_out_dtype out_dtype, float* lse_out, int32_t* status_word,
                              kvd_stream_t stream) {
    return decode(kMerge, q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q,
                  n_heads_kv, head_dim, scale, n_split, workspace, workspace_bytes, out, out_dtype,
                  lse_out, status_word, stream);
}

kvd_status kvd_schedule_describe(const int32_t* seq_lens_host, int batch, int s_max,
                                 int max_seq_len, int n_heads_q, int n_heads_kv, int head_dim,
                                 int n_split, kvd_out_dtype out_dtype, int32_t* rows_out,
                                 int max_rows, int* n_rows_out, int* n_split_eff_out) {
    kvd_status st = check_shape(batch, n_heads_q, n_heads_kv, head_dim, out_dtype);
    if (st != KVD_OK) return st;
    if (s_max <= 0 || max_seq_len < 0 || max_seq_len > s_max || n_split <= 0 || max_rows < 0)
        return KVD_ERR_INVALID_ARG;
    if ((batch > 0 && !seq_lens_host) || !n_rows_out || (max_rows > 0 && !rows_out))
        return KVD_ERR_INVALID_ARG;
    const ChunkKernel* k = pick_kernel(n_heads_q, n_heads_kv, head_dim, out_dtype);
    if (!k) return KVD_ERR_UNSUPPORTED;

    struct HostLen {
        const int32_t* lens;
        int cap;
        int operator()(int b) const { return clamp_len(lens[b], cap); }
    };
    const HostLen len{seq_lens_host, std::min(s_max, max_seq_len)};
    const RuntimeGeom geo{k->tile_tokens, k->seg_unit, k->seg_cost};
    long long total = 0;
    for (int b = 0; b < batch; ++b) total += pair_extent(len(b), geo);
    total *= n_heads_kv;
    const int C_eff = effective_ctas(n_split, total);
    int rows = 0;
    auto emit = [&](int c, int b, int h, int lo, int hi, int kind, int slot, int c_last) {
        if (rows < max_rows) {
            int32_t* r = rows_out + 8 * (size_t)rows;
            r[0] = c; r[1] = b; r[2] = h; r[3] = lo; r[4] = hi; r[5] = kind; r[6] = slot; r[7] = c_last;
        }
        ++rows;
    };
    for (int c = 0; c < C_eff; ++c) {
        Walker<HostLen, RuntimeGeom> w(len, geo, batch, n_heads_kv, c, C_eff, total);
        int b0 = batch;
        long long cum = 0, cum0 = total;
        for (int b = 0; b < batch; ++b) {
            const long long e = pair_extent(len(b), geo);
            if (is_first_seq_candidate(cum, e, n_heads_kv, w.S)) {
                b0 = b;
                cum0 = cum;
                break;
            }
            cum += (long long)n_heads_kv * e;
        }
        w.start(b0, cum0);
        auto on_empty = [&](int b, int h) { emit(c, b, h, 0, 0, 3, -1, c); };
        Tile t;
        int seg_lo = 0;
        while (w.next(t, on_empty)) {
            if (t.seg_start) seg_lo = t.tok_lo;
            if (t.seg_end) {
                const int pair = t.b * n_heads_kv + t.h;
                if (t.full)
                    emit(c, t.b, t.h, seg_lo, t.tok_hi, 0, -1, c);
                else
                    emit(c, t.b, t.h, seg_lo, t.tok_hi, t.owned ? 1 : 2, c + pair, t.c_last);
            }
        }
        w.finish(on_empty);
    }
    *n_rows_out = rows;
    if (n_split_eff_out) *n_split_eff_out = C_eff;
    return KVD_OK;
}

kvd_status kvd_kernel_info(int n_heads_q, int n_heads_kv, int head_dim, kvd_out_dtype out_dtype,
                           int* threads_out, int* smem_bytes_out, int* tile_tokens_out,
                           int* ctas_per_sm_out, int* seg_unit_out, int* seg_cost_out) {
    kvd_status st = check_shape(1, n_heads_q, n_heads_kv, head_dim, out_dtype);
    if (st != KVD_OK) return st;
    const ChunkKernel* k = pick_kernel(n_heads_q, n_heads_kv, head_dim, out_dtype);
    if (!k) return KVD_ERR_UNSUPPORTED;
    if (threads_out) *threads_out = k->threads;
    if (smem_bytes_out) *smem_bytes_out = k->smem_bytes;
    if (tile_tokens_out) *tile_tokens_out = k->tile_tokens;
    if (ctas_per_sm_out) *ctas_per_sm_out = k->ctas_per_sm;
    if (seg_unit_out) *seg_unit_out = k->seg_unit;
    if (seg_cost_out) *seg_cost_out = k->seg_cost;
    return KVD_OK;
}

const char* kvd_status_string(kvd_status s) {
    switch (s) {
        case KVD_OK: return "ok";
        case KVD_ERR_INVALID_ARG: return "invalid argument";
        case KVD_ERR_UNSUPPORTED: return "unsupported shape";
        case KVD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case KVD_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

const char* kvd_version(void) { return "kvdecode 0.1.0 (sm_103a)"; }

}  // extern "C"
