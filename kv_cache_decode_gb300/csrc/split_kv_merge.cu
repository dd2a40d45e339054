// Merge kernel: combines the partial softmax states that several CTAs wrote
// for the same (sequence, KV head) pair. The pages say sequence-sharded KV is
// accumulated "like Flash Attention" (All About Transformer Inference,
// "Sharding the KV cache") but print no formula; this is the log-sum-exp
// identity in base 2: with partial maxima m_j, sums l_j and unnormalised
// outputs o_j, M = max_j m_j, w_j = 2^(m_j - M), out = sum_j w_j o_j /
// sum_j w_j l_j (partials with l_j = 0 are skipped).
//
// One CTA per (pair, query head of the group). The CTA first reduces M and
// L = sum_j w_j l_j over all partials, then splits the partials among thread
// groups that each accumulate a full output row with several independent
// loads in flight, and finally sums the groups through shared memory.
#include <math_constants.h>

#include "common.cuh"
#include "params.h"

namespace kvd {

constexpr int kMergeThreads = 128;
constexpr int kMergeChunk = 512;  // partial weights staged in shared memory per pass

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kMergeThreads) split_kv_merge_kernel(const DecodeParams p) {
    constexpr int COLS = D / 4;                     // float4 columns of one output row
    constexpr int GROUPS = kMergeThreads / COLS;    // thread groups splitting the partials
    static_assert(kMergeThreads % COLS == 0, "");
    __shared__ float s_w[kMergeChunk];
    __shared__ float s_red[kMergeThreads / 32];
    __shared__ float4 s_acc[GROUPS > 1 ? GROUPS - 1 : 1][COLS];

    pdl_wait();  // partials come from the chunk kernel just before on the stream

    const int pair = blockIdx.x;
    const int g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = p.G;
    const int2 rec = __ldcg(p.ws_rec + pair);
    // rec.x < 0: the chunk kernel wrote this pair in full. The range check
    // keeps every slot read inside the workspace whatever its contents.
    if (rec.x < 0 || rec.y < rec.x || rec.y >= p.n_split) return;
    const int n = rec.y - rec.x + 1;
    const size_t slot0 = (size_t)rec.x + pair;

    // Pass 1: M = max m_j over non-empty partials.
    float mx = -CUDART_INF_F;
    for (int j = tid; j < n; j += kMergeThreads) {
        const float2 ml = __ldcg(p.ws_ml + (slot0 + j) * G + g);
        if (ml.y > 0.f) mx = fmaxf(mx, ml.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    float M = s_red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, s_red[w]);
    __syncthreads();

    // Pass 2: weighted sums, kMergeChunk partials at a time.
    const int col = tid % COLS, grp = tid / COLS;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    for (int base = 0; base < n; base += kMergeChunk) {
        const int cnt = min(kMergeChunk, n - base);
        for (int j = tid; j < cnt; j += kMergeThreads) {
            const float2 ml = __ldcg(p.ws_ml + (slot0 + base + j) * G + g);
            const float w = (ml.y > 0.f) ? exp2f(ml.x - M) : 0.f;
            s_w[j] = w;
            lsum += w * ml.y;
        }
        __syncthreads();
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + ((slot0 + base) * G + g) * D) + col;
        const size_t jstride = (size_t)G * D / 4;  // float4 stride between consecutive slots
#pragma unroll 8
        for (int j = grp; j < cnt; j += GROUPS) {
            const float w = s_w[j];
            const float4 v = __ldcg(src + (size_t)j * jstride);
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        __syncthreads();
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane == 0) s_red[warp] = lsum;
    if (GROUPS > 1 && grp > 0) s_acc[grp - 1][col] = acc;
    __syncthreads();
    if (grp != 0) return;
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) L += s_red[w];
#pragma unroll
    for (int q = 1; q < GROUPS; ++q) {
        const float4 o = s_acc[q - 1][col];
        acc.x += o.x;
        acc.y += o.y;
        acc.z += o.z;
        acc.w += o.w;
    }

    const int b = pair / p.Hkv, h = pair % p.Hkv;
    const size_t row = (size_t)b * p.Hq + (size_t)h * G + g;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    if constexpr (F32OUT) {
        float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * D) + col;
        *out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
        uint2* out = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * D) + col;
        *out = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    }
    if (p.lse && col == 0)
        p.lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
}

template <int D, bool F32OUT>
static cudaError_t launch_merge_t(const DecodeParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.Hkv), (unsigned)p.G, 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_merge_kernel<D, F32OUT>, p);
}

cudaError_t launch_merge(const DecodeParams& p, int head_dim, bool f32_out, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return f32_out ? launch_merge_t<64, true>(p, stream) : launch_merge_t<64, false>(p, stream);
        case 128: return f32_out ? launch_merge_t<128, true>(p, stream) : launch_merge_t<128, false>(p, stream);
        case 256: return f32_out ? launch_merge_t<256, true>(p, stream) : launch_merge_t<256, false>(p, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvd
