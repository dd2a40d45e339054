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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvdecode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[KVD_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// The array's device address, per device, with the context it was looked up
// in: the module (and so the array) is loaded again, possibly elsewhere, when
// a device's primary context is destroyed and re-created (cudaDeviceReset), so
// the cached address is used only while the same context (by its unique id) is
// current.
struct CachedAddress {
    std::mutex m;
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};
CachedAddress g_static_workspace_addr[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(f);
}

// Unique id of the current context (0 if none is current or it cannot be read).
unsigned long long current_ctx_id() {
    static const CtxGetCurrentFn get = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get || !get_id || get(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// In host code g_static_workspace names a host-side stand-in, not device
// memory: its device address is looked up with the device current, once per
// device and context, and cached.
kvd_status static_workspace_address(void** addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVD_ERR_CUDA;
    CachedAddress& c = g_static_workspace_addr[dev];
    std::lock_guard<std::mutex> lock(c.m);
    const unsigned long long id = current_ctx_id();
    if (c.addr == nullptr || id == 0 || c.ctx_id != id) {
        // The lookup also makes the device's primary context current if none was.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return KVD_ERR_CUDA;
        c.addr = p;
        c.ctx_id = current_ctx_id();
    }
    *addr = c.addr;
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
