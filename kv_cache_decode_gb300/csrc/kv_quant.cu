// 8-bit KV cache: quantization of bf16 rows of D values into 8-bit codes and
// one float32 scale per row (one (token, KV head) row of K or V). The pages
// name int8 and fp8 quantization of the KV cache as a way to cut its memory
// traffic (All About Transformer Inference, "Tricks for improving generation
// throughput and latency", the quantization bullet) but give no scheme; this
// one is symmetric absmax: a = max_d |x_d|, then
//   int8: scale = a / 127, code_d = round-half-even(x_d / scale) clamped to
//         [-127, 127];
//   fp8 (OCP E4M3): scale = a / 448, code_d = x_d / scale rounded to the
//         nearest E4M3 value (ties to even, saturating at 448), a zero result
//         stored as +0;
// both divisions IEEE float32 (a = 0: scale 0, codes 0). Used by the appends
// (the new tokens' rows) and by the bulk conversion of an existing bf16 cache.
#include "../../include/kvdecode.h"
#include "common.cuh"
#include "params.h"

namespace kvd {

// One row per group of D / 8 threads, each holding 8 consecutive values (one
// 16-byte vector). Every thread of the warp takes part in the shuffles, with
// `live` false for rows past the end.
template <int D, bool FP8>
__device__ __forceinline__ void quantize_row(const uint4* src, uint2* dst_codes, float* dst_scale, bool live,
                                             int sub) {
    constexpr int VPR = D / 8;  // vectors per row: 8, 16 or 32 lanes
    uint4 v = live ? __ldg(src + sub) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
#pragma unroll
    for (int off = VPR / 2; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    const float sc = __fdiv_rn(a, FP8 ? 448.f : 127.f);
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int c = 0;
        if (a > 0.f) {
            if constexpr (FP8) {
                c = __nv_cvt_float_to_fp8(__fdiv_rn(f[i], sc), __NV_SATFINITE, __NV_E4M3);
                if ((c & 0x7f) == 0) c = 0;  // +0 for a zero result
            } else {
                c = max(-127, min(127, __float2int_rn(__fdiv_rn(f[i], sc))));
            }
        }
        packed[i >> 2] |= (uint32_t)(c & 0xff) << (8 * (i & 3));
    }
    if (live) {
        dst_codes[sub] = make_uint2(packed[0], packed[1]);
        if (sub == 0) *dst_scale = sc;
    }
}

// The new tokens' K and V rows, quantized and written at pos[b] + i; with a
// paged cache (pg.block_table non-null) at the row of the block's page, as
// the bf16 append.
template <int D, bool FP8>
__global__ void __launch_bounds__(256) kv_append_q8_kernel(int8_t* __restrict__ k_codes, int8_t* __restrict__ v_codes,
                                                          float* __restrict__ k_scale, float* __restrict__ v_scale,
                                                          const uint4* __restrict__ k_new,
                                                          const uint4* __restrict__ v_new,
                                                          const int32_t* __restrict__ pos, int B, int S_max,
                                                          int Hkv, int32_t* status, int T, const PagedCache pg) {
    // The attention kernel that follows may start; it waits for this grid
    // before reading the cache.
    pdl_launch_dependents();
    constexpr int VPR = D / 8;
    const long long per = (long long)B * T * Hkv;  // new rows of one tensor: (b, token i, h)
    const long long rows = 2 * per;
    const int sub = threadIdx.x % VPR;
    const long long groups = (long long)gridDim.x * (blockDim.x / VPR);
    for (long long g = (long long)blockIdx.x * (blockDim.x / VPR) + threadIdx.x / VPR;
         g - (threadIdx.x / VPR) < rows; g += groups) {
        const bool in = g < rows;
        const int which = in ? (int)(g / per) : 0;
        const long long r = in ? g - which * per : 0;  // (b * T + i) * Hkv + h
        const long long bi = r / Hkv;
        const int h = (int)(r - bi * Hkv);
        const int b = (int)(bi / T), i = (int)(bi - (long long)b * T);
        const int t = in ? __ldg(pos + b) + i : 0;
        bool ok = in && t >= 0 && t < S_max;
        if (in && !ok && status && which == 0 && h == 0 && sub == 0) atomicOr(status, KVD_STATUS_POS_OUT_OF_RANGE);
        long long trow = (long long)b * S_max + (ok ? t : 0);  // cache row of the token
        if (pg.block_table && ok) {
            const int page = __ldg(pg.block_table + (size_t)b * pg.max_blocks + (t >> pg.page_shift));
            if (page < 0 || page >= pg.num_pages) {
                if (status && which == 0 && h == 0 && sub == 0) atomicOr(status, KVD_STATUS_BAD_PAGE);
                ok = false;
                trow = 0;
            } else {
                trow = ((long long)page << pg.page_shift) + (t & ((1 << pg.page_shift) - 1));
            }
        }
        const long long dst_row = trow * Hkv + h;
        quantize_row<D, FP8>((which ? v_new : k_new) + r * VPR,
                        reinterpret_cast<uint2*>((which ? v_codes : k_codes) + dst_row * D),
                        (which ? v_scale : k_scale) + dst_row, ok, sub);
    }
}

// Rows t < seq_lens[b] (clamped to len_cap) of a bf16 cache [B, S_max, Hkv, D].
template <int D, bool FP8>
__global__ void __launch_bounds__(256) kv_quantize_q8_kernel(const uint4* __restrict__ src, int8_t* __restrict__ codes,
                                                            float* __restrict__ scales,
                                                            const int32_t* __restrict__ seq_lens, int B, int S_max,
                                                            int len_cap, int Hkv) {
    constexpr int VPR = D / 8;
    const long long rows = (long long)B * S_max * Hkv;
    const int sub = threadIdx.x % VPR;
    const long long groups = (long long)gridDim.x * (blockDim.x / VPR);
    for (long long g = (long long)blockIdx.x * (blockDim.x / VPR) + threadIdx.x / VPR;
         g - (threadIdx.x / VPR) < rows; g += groups) {
        const bool in = g < rows;
        const long long bt = in ? g / Hkv : 0;  // b * S_max + t
        const int b = (int)(bt / S_max), t = (int)(bt - (long long)b * S_max);
        int L = in ? __ldg(seq_lens + b) : 0;
        L = L < 0 ? 0 : (L > len_cap ? len_cap : L);
        const bool ok = in && t < L;
        quantize_row<D, FP8>(src + g * VPR, reinterpret_cast<uint2*>(codes + g * D), scales + g, ok, sub);
    }
}

cudaError_t launch_append_q8(void* k_codes, void* v_codes, float* k_scale, float* v_scale, const void* k_new,
                             const void* v_new, const int32_t* pos, int B, int S_max, int Hkv, int D,
                             int32_t* status, const PagedCache& pg, cudaStream_t stream, int T, bool fp8) {
    const long long rows = 2LL * B * T * Hkv;
    const int rows_per_block = 256 / (D / 8);
    long long blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    auto* kc = static_cast<int8_t*>(k_codes);
    auto* vc = static_cast<int8_t*>(v_codes);
    auto* kn = static_cast<const uint4*>(k_new);
    auto* vn = static_cast<const uint4*>(v_new);
#define KVD_APPEND8(DD, F) cudaLaunchKernelEx(&cfg, kv_append_q8_kernel<DD, F>, kc, vc, k_scale, v_scale, kn, vn, pos, B, S_max, Hkv, status, T, pg)
    switch (D) {
        case 64: return fp8 ? KVD_APPEND8(64, true) : KVD_APPEND8(64, false);
        case 128: return fp8 ? KVD_APPEND8(128, true) : KVD_APPEND8(128, false);
        case 256: return fp8 ? KVD_APPEND8(256, true) : KVD_APPEND8(256, false);
        default: return cudaErrorInvalidValue;
    }
#undef KVD_APPEND8
}

cudaError_t launch_quantize_q8(const void* src, void* codes, float* scales, const int32_t* seq_lens, int B,
                               int S_max, int len_cap, int Hkv, int D, cudaStream_t stream, bool fp8) {
    const long long rows = (long long)B * S_max * Hkv;
    const int rows_per_block = 256 / (D / 8);
    long long blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    auto* s = static_cast<const uint4*>(src);
    auto* c = static_cast<int8_t*>(codes);
#define KVD_QUANT8(DD, F) cudaLaunchKernelEx(&cfg, kv_quantize_q8_kernel<DD, F>, s, c, scales, seq_lens, B, S_max, len_cap, Hkv)
    switch (D) {
        case 64: return fp8 ? KVD_QUANT8(64, true) : KVD_QUANT8(64, false);
        case 128: return fp8 ? KVD_QUANT8(128, true) : KVD_QUANT8(128, false);
        case 256: return fp8 ? KVD_QUANT8(256, true) : KVD_QUANT8(256, false);
        default: return cudaErrorInvalidValue;
    }
#undef KVD_QUANT8
}

}  // namespace kvd
