// Merge kernel: combines the partial softmax states that several CTAs wrote
// for the same (sequence, KV head) pair. The pages say sequence-sharded KV is
// accumulated "like Flash Attention" (All About Transformer Inference,
// "Sharding the KV cache") but print no formula; this is the log-sum-exp
// identity in base 2: with partial maxima m_j, sums l_j and unnormalised
// outputs o_j, M = max_j m_j, w_j = 2^(m_j - M), out = sum_j w_j o_j /
// sum_j w_j l_j (partials with l_j = 0 are skipped).
//
// One thread per two float4 columns of one output row (pair, query head) and
// per one of S partial subsets: thread group s of a row takes partials s, s + S,
// s + 2S, ... The work is latency-bound (a few KB per row, read from L2), so:
//  * the contributing CTAs of each pair are recomputed from the lengths with
//    the chunk kernel's own schedule code, before the dependency wait (the
//    lengths are an input, not a chunk-kernel output), so no round trip is
//    spent reading it from the workspace;
//  * each thread issues the loads of a whole batch of its partials before
//    using any of them, one round trip per batch of kBatch partials. Batches
//    after the first are folded in with the running maximum (rescaling the
//    sums); the S subsets of a row are combined the same way through shared
//    memory. The host picks S from the expected partials per pair.
// CTAs have 128 threads, or 256 when a row's subsets need them. Registers are
// capped so that merge CTAs fit on an SM beside a tcgen05 chunk CTA: launched
// early (programmatic dependent launch), they do the schedule part there.
#include <math_constants.h>

#include "common.cuh"
#include "params.h"
#include "schedule.cuh"

namespace kvd {

constexpr int kBatch = 3;  // partials whose loads are in flight together
constexpr int kVec = 2;    // float4 columns per thread

// NT threads: 128 (six CTAs' worth of registers per SM) or 256 (three).
template <int D, bool F32OUT, int NT>
__global__ void __launch_bounds__(NT, 768 / NT) split_kv_merge_kernel(const DecodeParams p, int S) {
    constexpr int COLS = D / 4 / kVec;  // threads per output row (and subset)
    static_assert(NT % COLS == 0, "");
    __shared__ float4 s_acc[kVec][NT];
    __shared__ float2 s_ml[NT / COLS];  // (M, L) per (row, subset)
    __shared__ longlong2 s_sum[NT / 32];

    const int G = p.G;
    // Output rows: (b, i, query head) with T query tokens per sequence; a
    // pair's partial slot holds T * G rows, row i * G + g.
    const int T = p.T, TG = T * G;
    const long long rows_per_seq = (long long)T * p.Hq;
    const int tid = threadIdx.x;
    const int col = tid % COLS, sub = (tid / COLS) % S, rloc = tid / (COLS * S);
    const int rows_per_cta = NT / (COLS * S);
    const long long rows = (long long)p.B * rows_per_seq;
    const long long row = (long long)blockIdx.x * rows_per_cta + rloc;

    // ---- the schedule, from the lengths (before the dependency wait) ----
    const RuntimeGeom geo{p.tile_tokens, p.seg_unit, p.seg_cost};
    const DevLen len{p.seq_lens, p.len_cap, p.vT};
    auto ext = [&](int b) { return pair_extent(len(b), geo); };
    const long long row_lo = (long long)blockIdx.x * rows_per_cta;
    const int b_lo = (int)(row_lo / rows_per_seq);  // first sequence among this CTA's rows
    long long tot = 0, pre = 0;
    for (int b = tid; b < p.B; b += NT) {
        const long long e = ext(b);
        tot += e;
        if (b < b_lo) pre += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, off);
        pre += __shfl_xor_sync(0xffffffffu, pre, off);
    }
    if ((tid & 31) == 0) s_sum[tid >> 5] = make_longlong2(tot, pre);
    __syncthreads();
    tot = pre = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        tot += s_sum[w].x;
        pre += s_sum[w].y;
    }
    const long long total = tot * p.Hkv;
    const int C_eff = effective_ctas(p.n_split, total);
    bool active = false;
    int n = 0, g = 0;
    size_t slot0 = 0;
    if (row < rows) {
        const int b = (int)(row / rows_per_seq);
        const int rem = (int)(row - (long long)b * rows_per_seq);  // i * Hq + query head
        const int i = rem / p.Hq, hq = rem - i * p.Hq;
        const int h = hq / G;
        g = i * G + (hq - h * G);  // row within the pair's slot
        const int pair = b * p.Hkv + h;
        long long cum = pre * p.Hkv;
        for (int bb = b_lo; bb < b; ++bb) cum += ext(bb) * p.Hkv;
        const long long e = ext(b);
        if (e > 0) {
            const long long pstart = cum + (long long)h * e;
            const int c0 = cta_of_token(pstart + geo.x(), C_eff, total);
            const int c1 = cta_of_token(pstart + e - 1, C_eff, total);
            // c0 == c1: the one contributing CTA wrote the final row itself.
            if (c1 > c0) {
                active = true;
                n = c1 - c0 + 1;
                slot0 = (size_t)c0 + pair;
            }
        }
    }

    pdl_wait();  // partials come from the chunk kernel just before on the stream

    const size_t ml_stride = (size_t)TG * S;         // float2 stride between this subset's slots
    const size_t o_stride = (size_t)TG * D / 4 * S;  // float4 stride between this subset's slots
    const float2* mlp = p.ws_ml + (slot0 + sub) * TG + g;
    const float4* op = reinterpret_cast<const float4*>(p.ws_o + ((slot0 + sub) * TG + g) * D) + col * kVec;
    const int mine = active && sub < n ? (n - sub + S - 1) / S : 0;  // partials of this subset

    float M = -CUDART_INF_F, L = 0.f;
    float4 acc[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < mine; base += kBatch) {
        const int cnt = min(kBatch, mine - base);
        float2 ml[kBatch];
        float4 o[kBatch][kVec];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < cnt) {
                ml[j] = __ldcg(mlp + (size_t)(base + j) * ml_stride);
#pragma unroll
                for (int v = 0; v < kVec; ++v) o[j][v] = __ldcg(op + (size_t)(base + j) * o_stride + v);
            }
        }
        float mb = M;
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (j < cnt && ml[j].y > 0.f) mb = fmaxf(mb, ml[j].x);
        if (mb == -CUDART_INF_F) continue;  // every partial so far is empty
        const float r = exp2f(M - mb);      // 0 while M is still -inf
        L *= r;
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
            acc[v].x *= r;
            acc[v].y *= r;
            acc[v].z *= r;
            acc[v].w *= r;
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (j < cnt && ml[j].y > 0.f) {
                const float w = exp2f(ml[j].x - mb);
                L += w * ml[j].y;
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    acc[v].x += w * o[j][v].x;
                    acc[v].y += w * o[j][v].y;
                    acc[v].z += w * o[j][v].z;
                    acc[v].w += w * o[j][v].w;
                }
            }
        }
        M = mb;
    }

    if (S > 1) {  // combine the subsets of each row (S is uniform over the CTA)
#pragma unroll
        for (int v = 0; v < kVec; ++v) s_acc[v][tid] = acc[v];
        if (col == 0) s_ml[tid / COLS] = make_float2(M, L);
        __syncthreads();
        if (sub != 0) return;
        float Mt = M;
        for (int q = 1; q < S; ++q) Mt = fmaxf(Mt, s_ml[tid / COLS + q].x);
        if (Mt != -CUDART_INF_F) {
            const float r0 = exp2f(M - Mt);
            L *= r0;
#pragma unroll
            for (int v = 0; v < kVec; ++v) {
                acc[v].x *= r0;
                acc[v].y *= r0;
                acc[v].z *= r0;
                acc[v].w *= r0;
            }
            for (int q = 1; q < S; ++q) {
                const float2 mq = s_ml[tid / COLS + q];
                const float r = exp2f(mq.x - Mt);  // 0 for an empty subset
                L += r * mq.y;
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    const float4 aq = s_acc[v][tid + q * COLS];
                    acc[v].x += r * aq.x;
                    acc[v].y += r * aq.y;
                    acc[v].z += r * aq.z;
                    acc[v].w += r * aq.w;
                }
            }
        }
        M = Mt;
    }
    if (!active) return;

    const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
        const size_t c4 = (size_t)col * kVec + v;  // float4 column of the row
        if constexpr (F32OUT) {
            float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + row * D) + c4;
            *out = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
        } else {
            uint2* out = reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.out) + row * D) + c4;
            *out = make_uint2(pack_bf16x2(acc[v].x * inv, acc[v].y * inv),
                              pack_bf16x2(acc[v].z * inv, acc[v].w * inv));
        }
    }
    if (p.lse && col == 0)
        p.lse[row] = (L > 0.f) ? (M + log2f(L)) * 0.69314718055994531f : -CUDART_INF_F;
}

template <int D, bool F32OUT>
static cudaError_t launch_merge_t(const DecodeParams& p, int num_sms, cudaStream_t stream) {
    constexpr int COLS = D / 4 / kVec;
    // Subsets per row: enough that the expected partials of a pair (runs of
    // about equal size, n_split of them over B * Hkv pairs, plus the partial
    // runs at both ends) fit in one batch per subset, as long as all threads
    // stay resident at once (768 per SM at this register cap); past that,
    // more batches per thread cost less than a second wave of CTAs.
    const long long pairs = (long long)p.B * p.Hkv;
    const long long rows = (long long)p.B * p.T * p.Hq;
    const long long expect = (long long)p.n_split / (pairs > 0 ? pairs : 1) + 2;
    const long long resident = (long long)num_sms * 768;
    int S = 1;
    while (S * kBatch < expect && S * 2 * COLS <= 256 && rows * COLS * S * 2 <= resident) S *= 2;
    const int nt = (S * COLS <= 128) ? 128 : 256;
    const int rows_per_cta = nt / (COLS * S);
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

cudaError_t launch_merge(const DecodeParams& p, int head_dim, bool f32_out, int num_sms, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return f32_out ? launch_merge_t<64, true>(p, num_sms, stream) : launch_merge_t<64, false>(p, num_sms, stream);
        case 128: return f32_out ? launch_merge_t<128, true>(p, num_sms, stream) : launch_merge_t<128, false>(p, num_sms, stream);
        case 256: return f32_out ? launch_merge_t<256, true>(p, num_sms, stream) : launch_merge_t<256, false>(p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

// Shard merge: n attention results over disjoint shards of each sequence's
// tokens (each normalised, with its natural-log normaliser lse, as the
// attention calls return them) combined into the result over all shards:
// L = ln sum_j exp(lse_j), out = sum_j exp(lse_j - L) out_j, lse = L; shards
// with lse = -inf hold no token and add nothing (All About Transformer
// Inference, "Sharding the KV cache": sequence-sharded results accumulate as
// in Flash Attention). One thread per 8 columns of a row; each thread of a row
// forms the row's weights from the n lse values itself.
template <int D, bool IN_F32, bool OUT_F32>
__global__ void __launch_bounds__(256) merge_shards_kernel(const void* __restrict__ outs,
                                                           const float* __restrict__ lses, int n, long long rows,
                                                           void* __restrict__ out, float* __restrict__ lse_out) {
    constexpr int VPR = D / 8;
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = g / VPR;
    const int c8 = (int)(g - row * VPR);
    if (row >= rows) return;
    // A normaliser that is NaN or +inf is no shard's valid result: the row
    // is then NaN (out and lse), rather than a plausible-looking mix of the
    // other shards (fmaxf would skip a NaN, and +inf - +inf gives NaN weights).
    float M = -CUDART_INF_F;
    bool bad = false;
    for (int j = 0; j < n; ++j) {
        const float lj = __ldg(lses + (size_t)j * rows + row);
        bad |= !(lj < CUDART_INF_F) && !(lj == -CUDART_INF_F);
        M = fmaxf(M, lj);
    }
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = bad ? CUDART_NAN_F : 0.f;
    float tot = 0.f;
    if (!bad && M > -CUDART_INF_F) {
        for (int j = 0; j < n; ++j) {
            const float lj = __ldg(lses + (size_t)j * rows + row);
            if (!(lj > -CUDART_INF_F)) continue;
            const float w = expf(lj - M);
            tot += w;
            const size_t e = ((size_t)j * rows + row) * D + c8 * 8;
            if constexpr (IN_F32) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(outs) + e));
                const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(outs) + e) + 1);
                const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] += w * v[i];
            } else {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(outs) + e));
                const uint32_t u[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += w * bf16_lo(u[i]);
                    acc[2 * i + 1] += w * bf16_hi(u[i]);
                }
            }
        }
        const float inv = 1.f / tot;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] *= inv;
    }
    const size_t o = (size_t)row * D + c8 * 8;
    if constexpr (OUT_F32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
    }
    if (lse_out && c8 == 0) lse_out[row] = bad ? CUDART_NAN_F : (M > -CUDART_INF_F) ? M + logf(tot) : -CUDART_INF_F;
}

template <int D>
static cudaError_t launch_shards_t(const void* outs, const float* lses, int n, long long rows, bool in_f32,
                                   void* out, bool out_f32, float* lse_out, cudaStream_t s) {
    const long long threads = rows * (D / 8);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    if (in_f32 && out_f32) merge_shards_kernel<D, true, true><<<blocks, 256, 0, s>>>(outs, lses, n, rows, out, lse_out);
    else if (in_f32) merge_shards_kernel<D, true, false><<<blocks, 256, 0, s>>>(outs, lses, n, rows, out, lse_out);
    else if (out_f32) merge_shards_kernel<D, false, true><<<blocks, 256, 0, s>>>(outs, lses, n, rows, out, lse_out);
    else merge_shards_kernel<D, false, false><<<blocks, 256, 0, s>>>(outs, lses, n, rows, out, lse_out);
    return cudaGetLastError();
}

cudaError_t launch_merge_shards(const void* outs, const float* lses, int n, long long rows, int head_dim, bool in_f32,
                                void* out, bool out_f32, float* lse_out, cudaStream_t stream) {
    switch (head_dim) {
        case 64: return launch_shards_t<64>(outs, lses, n, rows, in_f32, out, out_f32, lse_out, stream);
        case 128: return launch_shards_t<128>(outs, lses, n, rows, in_f32, out, out_f32, lse_out, stream);
        case 256: return launch_shards_t<256>(outs, lses, n, rows, in_f32, out, out_f32, lse_out, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvd
