// Merge kernel: combines the partial softmax states that several CTAs wrote
// for the same (sequence, KV head) pair. The pages say sequence-sharded KV is
// accumulated "like Flash Attention" (All About Transformer Inference,
// "Sharding the KV cache") but print no formula; this is the log-sum-exp
// identity in base 2: with partial maxima m_j, sums l_j and unnormalised
// outputs o_j, M = max_j m_j, w_j = 2^(m_j - M), out = sum_j w_j o_j /
// sum_j w_j l_j (partials with l_j = 0 are skipped).
//
// One thread per float4 column of one output row (pair, query head) and per
// one of S partial subsets: thread group s of a row takes partials s, s + S,
// s + 2S, ... The work is latency-bound (a few KB per row, read from L2), so
// each thread issues the loads of a whole batch of its partials before using
// any of them: one round trip for the pair's record, one per batch of kBatch
// partials. Batches after the first are folded in with the running maximum
// (rescaling the sums); the S subsets of a row are combined the same way
// through shared memory. The host picks S from the expected number of
// partials per pair, so that long split pairs need one or two batches.
// CTAs have 128 threads, or 256 when a row's subsets need them. Registers are
// capped so that merge CTAs fit on an SM beside a tcgen05 chunk CTA: launched early (programmatic dependent launch), they wait there for the
// chunk kernel to finish instead of being scheduled after it.
#include <math_constants.h>

#include "common.cuh"
#include "params.h"

namespace kvd {

constexpr int kBatch = 5;  // partials whose loads are in flight together

// NT threads: 128 (six CTAs' worth of registers per SM) or 256 (three).
template <int D, bool F32OUT, int NT>
__global__ void __launch_bounds__(NT, 768 / NT) split_kv_merge_kernel(const DecodeParams p, int S) {
    constexpr int COLS = D / 4;  // float4 columns of one output row
    static_assert(NT % COLS == 0, "");
    __shared__ float4 s_acc[NT];
    __shared__ float2 s_ml[NT / COLS];  // (M, L) per (row, subset)

    pdl_wait();  // partials come from the chunk kernel just before on the stream

    const int G = p.G;
    const int tid = threadIdx.x;
    const int col = tid % COLS, sub = (tid / COLS) % S, rloc = tid / (COLS * S);
    const long long rows = (long long)p.B * p.Hq;
    const long long row = (long long)blockIdx.x * (NT / (COLS * S)) + rloc;
    bool active = row < rows;
    int n = 0;
    size_t slot0 = 0;
    int g = 0;
    if (active) {
        const int pair = (int)(row / G);
        g = (int)(row % G);
        const int2 rec = __ldcg(p.ws_rec + pair);
        // rec.x < 0: the chunk kernel wrote this pair in full. The range check
        // keeps every slot read inside the workspace whatever its contents.
        if (rec.x < 0 || rec.y < rec.x || rec.y >= p.n_split) active = false;
        else {
            n = rec.y - rec.x + 1;
            slot0 = (size_t)rec.x + pair;
        }
    }
    const float2* mlp = p.ws_ml + slot0 * G + g;
    const float4* op = reinterpret_cast<const float4*>(p.ws_o + (slot0 * G + g) * D) + col;
    const size_t ml_stride = (size_t)G * S;         // float2 stride between this subset's slots
    const size_t o_stride = (size_t)G * D / 4 * S;  // float4 stride between this subset's slots
    mlp += (size_t)sub * G;
    op += (size_t)sub * G * D / 4;
    const int mine = active && sub < n ? (n - sub + S - 1) / S : 0;  // partials of this subset

    float M = -CUDART_INF_F, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < mine; base += kBatch) {
        const int cnt = min(kBatch, mine - base);
        float2 ml[kBatch];
        float4 o[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < cnt) {
                ml[j] = __ldcg(mlp + (size_t)(base + j) * ml_stride);
                o[j] = __ldcg(op + (size_t)(base + j) * o_stride);
            }
        }
        float mb = M;
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (j < cnt && ml[j].y > 0.f) mb = fmaxf(mb, ml[j].x);
        if (mb == -CUDART_INF_F) continue;  // every partial so far is empty
        const float r = exp2f(M - mb);      // 0 while M is still -inf
        L *= r;
        acc.x *= r;
        acc.y *= r;
        acc.z *= r;
        acc.w *= r;
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < cnt && ml[j].y > 0.f) {
                const float w = exp2f(ml[j].x - mb);
                L += w * ml[j].y;
                acc.x += w * o[j].x;
                acc.y += w * o[j].y;
                acc.z += w * o[j].z;
                acc.w += w * o[j].w;
            }
        }
        M = mb;
    }

    if (S > 1) {  // combine the subsets of each row (S is uniform over the CTA)
        s_acc[tid] = acc;
        if (col == 0) s_ml[tid / COLS] = make_float2(M, L);
        __syncthreads();
        if (sub != 0) return;
        float Mt = M;
        for (int q = 1; q < S; ++q) Mt = fmaxf(Mt, s_ml[tid / COLS + q].x);
        if (Mt != -CUDART_INF_F) {
            const float r0 = exp2f(M - Mt);
            L *= r0;
            acc.x *= r0;
            acc.y *= r0;
            acc.z *= r0;
            acc.w *= r0;
            for (int q = 1; q < S; ++q) {
                const float2 mq = s_ml[tid / COLS + q];
                const float4 aq = s_acc[tid + q * COLS];
                const float r = exp2f(mq.x - Mt);  // 0 for an empty subset
                L += r * mq.y;
                acc.x += r * aq.x;
                acc.y += r * aq.y;
                acc.z += r * aq.z;
                acc.w += r * aq.w;
            }
        }
        M = Mt;
    }
    if (!active) return;

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
    constexpr int COLS = D / 4;
    // Subsets per row: enough that the expected partials of a pair (runs of
    // about equal size, n_split of them over B * Hkv pairs, plus the partial
    // runs at both ends) fit in one batch per subset.
    const long long pairs = (long long)p.B * p.Hkv;
    const long long expect = (long long)p.n_split / (pairs > 0 ? pairs : 1) + 2;
    int S = 1;
    while (S * kBatch < expect && S * 2 * COLS <= 256) S *= 2;
    const int nt = (S * COLS <= 128) ? 128 : 256;
    const int rows_per_cta = nt / (COLS * S);
    const long long rows = (long long)p.B * p.Hq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((rows + rows_per_cta - 1) / rows_per_cta), 1, 1);
    cfg.blockDim = dim3(nt, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (nt == 128) return cudaLaunchKernelEx(&cfg, split_kv_merge_kernel<D, F32OUT, 128>, p, S);
    return cudaLaunchKernelEx(&cfg, split_kv_merge_kernel<D, F32OUT, 256>, p, S);
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
