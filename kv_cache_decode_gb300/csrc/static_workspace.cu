// Decode attention for callers that cannot allocate device memory.
//
// Some callers may not allocate at decode time: a serving loop whose device
// memory is budgeted and frozen at start-up, a plugin that is handed only the
// tensors it works on, or a path that must not risk the device-wide
// synchronisation that cudaMalloc/cudaFree can cause. For them this entry point
// uses a scratch array that lives in the library itself: a file-scope
// __device__ array of KVD_STATIC_WORKSPACE_BYTES, present on every GPU that
// loads the library until the process exits. Inputs and outputs are still the
// caller's.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kvdecode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[KVD_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_static_workspace_addr[kMaxDevices];

// In host code g_static_workspace names a host-side stand-in, not device
// memory: its device address is looked up once per device, with that device
// current, and cached.
kvd_status static_workspace_address(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVD_ERR_CUDA;
    void* p = g_static_workspace_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return KVD_ERR_CUDA;
        g_static_workspace_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return KVD_OK;
}

}  // namespace

extern "C" kvd_status kvd_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* seq_lens, int batch, int s_max,
                                                  int max_seq_len, int n_heads_q, int n_heads_kv,
                                                  int head_dim, float scale, int n_split, void* out,
                                                  kvd_out_dtype out_dtype, float* lse_out,
                                                  int32_t* status_word, kvd_stream_t stream) {
    int n_split_eff = 0;
    size_t need = 0;
    kvd_status st = kvd_decode_plan(batch, n_heads_q, n_heads_kv, head_dim, max_seq_len, 0, n_split,
                                    out_dtype, &n_split_eff, &need);
    if (st != KVD_OK) return st;
    if (need > KVD_STATIC_WORKSPACE_BYTES) return KVD_ERR_WORKSPACE_TOO_SMALL;
    void* ws = nullptr;
    if (need > 0) {
        st = static_workspace_address(&ws);
        if (st != KVD_OK) return st;
    }
    // Nothing in the workspace needs to start at zero: every call writes the
    // partial states it reads.
    return kvd_decode_attention(q, k_cache, v_cache, seq_lens, batch, s_max, max_seq_len, n_heads_q,
                                n_heads_kv, head_dim, scale, n_split, ws, need > 0 ? KVD_STATIC_WORKSPACE_BYTES : 0,
                                out, out_dtype, lse_out, status_word, stream);
}
