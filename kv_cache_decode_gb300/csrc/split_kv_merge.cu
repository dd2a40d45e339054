// Merge kernel: combines the partial softmax states that several CTAs wrote
// for the same (sequence, KV head) pair. The pages say sequence-sharded KV is
// accumulated "like Flash Attention" (All About Transformer Inference,
// "Sharding the KV cache") but print no formula; this is the log-sum-exp
// identity in base 2: with partial maxima m_j, sums l_j and unnormalised
// outputs o_j, M = max_j m_j, w_j = 2^(m_j - M), out = sum_j w_j o_j /
// sum_j w_j l_j, evaluated as a running (online) merge over j.
#include <math_constants.h>

#include "common.cuh"
#include "params.h"

namespace kvd {

// One warp per query head of the group; lanes split the head dimension.
template <int D, bool F32OUT>
__global__ void __launch_bounds__(128) split_kv_merge_kernel(const DecodeParams p) {
    constexpr int PER_LANE = D / 32;
    pdl_wait();  // partials come from the chunk kernel just before on the stream

    const int pair = blockIdx.x;
    const int g = blockIdx.y * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int G = p.G;
    if (g >= G) return;
    const int2 rec = __ldcg(p.ws_rec + pair);
    // rec.x < 0: the chunk kernel wrote this pair in full. The range check
    // keeps every slot read inside the workspace whatever its contents.
    if (rec.x < 0 || rec.y < rec.x || rec.y >= p.n_split) return;

    float M = -CUDART_INF_F, L = 0.f;
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;

    for (int c = rec.x; c <= rec.y; ++c) {
        const size_t slot = (size_t)c + pair;
        const float2 ml = __ldcg(p.ws_ml + slot * G + g);
        if (!(ml.y > 0.f)) continue;
        const float Mn = fmaxf(M, ml.x);
        const float a = exp2f(M - Mn);  // 0 on the first partial (M = -inf)
        const float w = exp2f(ml.x - Mn);
        L = L * a + ml.y * w;
        const float* src = p.ws_o + (slot * G + g) * D + lane * PER_LANE;
        float v[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; i += 2) {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(src + i));
            v[i] = t.x;
            v[i + 1] = t.y;
        }
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) acc[i] = acc[i] * a + v[i] * w;
        M = Mn;
    }

    const int b = pair / p.Hkv, h = pair % p.Hkv;
    const size_t row = (size_t)b * p.Hq + (size_t)h * G + g;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    if constexpr (F32OUT) {
        float* out = reinterpret_cast<float*>(p.out) + row * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; i += 2)
            *reinterpret_cast<float2*>(out + i) = make_float2(acc[i] * inv, acc[i + 1] * inv);
    } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + row * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; i += 2)
            *reinterpret_cast<uint32_t*>(out + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    }
    if (p.lse && lane == 0)
        p.lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
}

template <int D, bool F32OUT>
static cudaError_t launch_merge_t(const DecodeParams& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.Hkv), (unsigned)((p.G + 3) / 4), 1);
    cfg.blockDim = dim3(128, 1, 1);
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
