// Split-KV chunk kernel on the 5th-generation tensor cores (tcgen05), for wide
// query-head groups (17..64 query heads per KV head: multiquery and wide
// grouped-query attention).
//
// Same schedule, same outputs and same partial-state format as the mma.sync
// chunk kernel (split_kv_chunk.cuh); only the engine differs. Per 64-token
// tile of one (sequence, KV head) pair:
//   S  = Q K^T      tcgen05.mma, M = 64 query heads (group padded to 64),
//                   N = 64 tokens, K = head_dim; fp32 accumulator in TMEM
//   P  = 2^(S*scale*log2e - m)   four softmax warps, two threads per query head
//   O += P V        tcgen05.mma, M = 64, N = head_dim, K = 64 tokens, with P
//                   read from TMEM as the A operand; O in TMEM
// K, V and Q never pass through registers: TMA writes their tiles into
// 128-byte-swizzled shared memory, and the MMAs read them there, so each K/V
// byte crosses shared memory once (the mma.sync kernel re-reads it once per
// 16-head tile). P goes from the softmax registers to TMEM and from there into
// the P V product, without a shared-memory pass. The online softmax follows the log-sum-exp accumulation of
// sequence-sharded KV (All About Transformer Inference, "Sharding the KV
// cache") in base 2 (Efficiently Scaling Transformer Inference, section 3.5).
// The running maximum m used for the exponentials is only raised when a tile's
// maximum exceeds it by more than 2^8 (weights stay <= 256, exact in fp32), so
// rescaling O in TMEM is rare; the result is identical in exact arithmetic
// because O and l always share the same m.
//
// Warp roles (10 warps): 0 = TMA producer for K, 2 = TMA producer for V,
// 9 = TMA loader for Q at each new pair, 1 and 7 = S issuers (one thread
// each, one half of head_dim each; warp 1 also owns TMEM), 8 = O issuer,
// 3..6 = softmax / rescale / epilogue (one warp per TMEM lane quarter w % 4;
// within a warp, the two threads of a query head take one half of the tile's
// token columns each, and one half of O's columns in the epilogue).
// Pipelines: K ring of KST stages, V ring of VST stages, one S buffer (two
// partial sums) in TMEM, two P buffers in TMEM, Q slots in shared memory, O in
// TMEM. Every wait is bounded; a timeout flags KVD_STATUS_TIMEOUT and all
// roles wind down.
//
// 8-bit caches (KV8: int8 codes, or E4M3 codes with FP8, each row with a
// float32 scale): TMA fills 8-bit rings instead, and 8 more warps (4 per
// tensor) convert each tile exactly to f16 in the K and V rings (the layout
// TMA gives bf16 rows) and copy its row scales into a scale slot. The Q
// loader converts each pair's Q rows to f16 in place, the MMAs take f16
// operands, the softmax multiplies each score by its key row's scale and
// each weight by its value row's scale (E4M3 codes become their values / 256
// in f16: scores and output are scaled back by 256).
#pragma once

#include <math_constants.h>

#include "../../include/kvdecode.h"
#include "common.cuh"
#include "params.h"
#include "schedule.cuh"
#include "split_kv_chunk.cuh"  // DevLen, NoOp, block scans
#include "tc_common.cuh"

namespace kvd {

// MR: rows of the MMAs (64, or 128 for several query tokens of a sequence
// stacked in one tile); QR: Q rows stored per head_dim block. KV8: an 8-bit
// cache (int8 codes, or E4M3 codes with FP8) with a float32 scale per (token,
// KV head) row, converted to f16 tiles in shared memory by converter warps.
template <int D, bool F32OUT, int QR, int MR = 64, bool KV8 = false>
struct TcShape {
    static constexpr int T = 64;                 // tokens per tile
    static constexpr int NG = MR / 64;           // 16-row groups per softmax thread
    // Schedule: runs balanced in whole tiles (a tile's time is set by the
    // pipeline's latency, whatever its length), plus one tile's charge for
    // starting a pair inside a run (its Q load and first K tile).
    static constexpr int SEG_UNIT = T;
    static constexpr int SEG_COST = 1;
    static constexpr int KB = D / 64;            // 128-byte swizzle atoms across head_dim
    static constexpr int TILE_BYTES = T * D * 2; // one K (or V) tile (bf16, or f16 converted from 8-bit codes)
    static constexpr int KB_BYTES = T * 128;     // one 64-column block of a tile
    // Q is stored as KB blocks of QR rows (the group rounded up to 8, capped at
    // 64). The M = 64 MMA reads 64 rows from each block start; for QR < 64 the
    // extra rows alias the next block (or the K ring after Q): they only feed
    // accumulator rows of padded heads, which are never used.
    static constexpr int QB_BYTES = QR * 128;
    // Q slots: narrow groups keep a ring of four (a few KB each), so the
    // producer loads the next pairs' Q ahead of time; wide groups keep one.
    static constexpr int NQ = QR <= 16 ? 4 : 1;
    static constexpr int QS_BYTES = KB * QB_BYTES;  // one slot
    static constexpr int Q_BYTES = NQ * QS_BYTES;
    static constexpr int NP = F32OUT ? 2 : 1;    // hi (and lo) parts of P
    // 8-bit tiles as TMA writes them: KB8 blocks of 128 head-dim columns.
    static constexpr int TILE8_BYTES = KV8 ? T * D : 0;
    static constexpr int KB8 = D / 128;
    static constexpr int NSC = 4;                // row-scale slots (KV8)
    static constexpr int SC_BYTES = KV8 ? NSC * 2 * T * 4 : 0;
    // Stage counts: three V stages (a V stage is held until P V of its tile is
    // done, so the V ring needs the depth), K stages as the budget allows.
    // KV8: few f16 stages (a converted tile waits there only for its MMAs):
    // two for V, whose next tile is converted while the softmax runs; two
    // for K, or at head_dim 256 one (the next K tile is converted once S of
    // the current one is done, well within a tile's softmax), which leaves
    // the room for three 8-bit stages a tensor. The 8-bit rings hold the
    // loads in flight and are as deep as the rest allows.
    static constexpr int VST = KV8 ? 2 : (D == 256 ? 3 : (D == 128 ? 6 : 8));
    static constexpr int BUDGET = 224 * 1024 - Q_BYTES - VST * TILE_BYTES;
    static constexpr int KST_FIT = BUDGET / TILE_BYTES;
    static constexpr int KST = KV8 ? (D == 256 ? 1 : 2) : (KST_FIT > 8 ? 8 : KST_FIT);
    static constexpr int BUDGET8 = 224 * 1024 - Q_BYTES - (KST + VST) * TILE_BYTES - SC_BYTES;
    static constexpr int ST8_FIT = KV8 ? BUDGET8 / (2 * (TILE8_BYTES > 0 ? TILE8_BYTES : 1)) : 0;
    static constexpr int K8ST = ST8_FIT > 6 ? 6 : ST8_FIT, V8ST = K8ST;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + KST * TILE_BYTES;
    static constexpr int OFF_K8 = OFF_V + VST * TILE_BYTES;
    static constexpr int OFF_V8 = OFF_K8 + K8ST * TILE8_BYTES;
    static constexpr int OFF_SC = OFF_V8 + V8ST * TILE8_BYTES;
    static constexpr int OFF_BAR = OFF_SC + SC_BYTES;
    // barriers: k_full, k_empty [KST]; v_full, v_empty [VST]; q_full, q_empty [NQ];
    // s_full, s_free; p_full, o_fin [2]; mma_done; KV8: k8_full, k8_empty
    // [K8ST]; v8_full, v8_empty [V8ST]; q_conv [NQ]; sc_full, sc_empty [NSC]
    static constexpr int NBAR = 2 * KST + 2 * VST + 2 * NQ + 2 + 4 + 1 +
                                (KV8 ? 2 * K8ST + 2 * V8ST + NQ + 2 * NSC : 0);
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int STATIC_SMEM = 1024;  // block scans (checked by ptxas -v)
    // TMEM columns: S as two partial sums over the halves of head_dim, two P
    // buffers (bf16 pairs, 32 columns per part), O.
    static constexpr int TMEM_S = 0;             // S, first head_dim half: columns [0, T)
    static constexpr int TMEM_S2 = T;            // S, second half: columns [T, 2T)
    static constexpr int PCOLS = NP * T / 2;     // one P buffer
    static constexpr int TMEM_P = 2 * T;         // P buffers at [2T, 2T + 2 PCOLS)
    static constexpr int TMEM_O = 256;           // O at columns [256, 256 + D)
    static constexpr int TMEM_COLS = 512;
    // producers 0 (K) and 2 (V), S issuers 1 and 7, O issuer 8, Q loader 9, softmax 3..6
    // (and at MR = 128, 10..13 for the quarters' second group of 16 rows; KV8:
    // converters 10 .. 10 + NCW - 1 for K and the next NCW for V)
    static constexpr int NSW = 4 * NG;           // softmax warps
    static constexpr int NCW = KV8 ? 4 : 0;      // converter warps per tensor
    static constexpr int NWARPS = 6 + NSW + 2 * NCW;
    static constexpr int THREADS = NWARPS * 32;
    static_assert(KST >= 2 || KV8, "need at least two K stages");
    static_assert(!KV8 || (K8ST >= 3 && MR == 64 && D >= 128), "8-bit rings");
    static_assert(SMEM_BYTES + STATIC_SMEM <= 227 * 1024, "shared memory budget");
    static_assert(QR % 8 == 0 && QR <= MR && (MR == 64 || MR == 128), "Q rows per block");
    static_assert(TMEM_P + 2 * PCOLS <= TMEM_O && TMEM_O + D <= TMEM_COLS, "TMEM columns");
};

struct TcMaps {
    CUtensorMap q;  // 2D: [B*Hq rows, D] box (64, G), 128-byte swizzle
    CUtensorMap k;  // 3D: [B*S_max, Hkv, D] box (64, 1, 64), 128-byte swizzle
    CUtensorMap v;
};

// A paged tile's TMA loads: boxes of box_rows tokens (the page size, up to the
// tile), each from its block's page (entries e0..e3 of the block table, one
// per box). Tile rows are page-aligned (tiles start at multiples of T within a
// sequence, and a page is at least 16 tokens), so no box crosses a page. A
// box past the tile's tokens, or whose entry names no page, is read from past
// the pool's end: zeros (and flagged in *status when status is given). Kept
// out of line: a contiguous cache never calls it, so its code stays out of
// the kernel's instruction stream.
template <int NBOX, int BOXC, int KB_BYTES, int T>
__device__ __noinline__ void tma_paged_tile(uint32_t dst, const CUtensorMap* map, int h, int tok_lo, int tok_hi,
                                            int e0, int e1, int e2, int e3, int box_rows, int page_shift,
                                            int num_pages, uint32_t full, uint64_t pol, int32_t* status) {
    static_assert(T / 16 == 4, "four boxes at most");
    const int entry[4] = {e0, e1, e2, e3};
    const int oob = num_pages << page_shift;
#pragma unroll
    for (int q = 0; q < T / 16; ++q) {
        const int r0 = q * box_rows;
        if (r0 >= T) break;
        const int tok = tok_lo + r0;
        int row = oob;
        if (tok < tok_hi) {
            const int page = entry[q];
            if ((unsigned)page < (unsigned)num_pages)
                row = (page << page_shift) + (tok & ((1 << page_shift) - 1));
            else if (status)
                atomicOr(status, KVD_STATUS_BAD_PAGE);
        }
#pragma unroll
        for (int kb = 0; kb < NBOX; ++kb)
            tc::tma_load_3d(dst + kb * KB_BYTES + r0 * 128, map, kb * BOXC, h, row, full, pol);
    }
}

template <int D, bool F32OUT, int QR, int MR, bool KV8 = false, bool FP8 = false>
__global__ void __launch_bounds__(TcShape<D, F32OUT, QR, MR, KV8>::THREADS, 1)
    split_kv_chunk_tc_kernel(const DecodeParams p, const __grid_constant__ TcMaps maps) {
    using Sh = TcShape<D, F32OUT, QR, MR, KV8>;
    static_assert(!FP8 || KV8, "fp8 codes are an 8-bit cache");
    constexpr float OSC = FP8 ? 256.f : 1.f;  // output scale: E4M3 value rows arrive divided by 256
    constexpr int T = Sh::T, KB = Sh::KB, KST = Sh::KST, VST = Sh::VST, NW = Sh::NWARPS,
                  SEG_COST = Sh::SEG_COST;
    constexpr long long kBudget = 4000000000LL;  // ~2 s of clock cycles per wait

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ long long s_red[NW];
    __shared__ int s_redi[NW];
    __shared__ long long s_cum0;

    uint8_t* smem = smem_raw;  // 1024-byte aligned (128-byte swizzle atoms need it)
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + Sh::OFF_Q, sK = sbase + Sh::OFF_K, sV = sbase + Sh::OFF_V,
                   sK8 = sbase + Sh::OFF_K8, sV8 = sbase + Sh::OFF_V8, sBar = sbase + Sh::OFF_BAR;
    auto k_full = [&](int s) { return sBar + 8u * s; };
    auto k_empty = [&](int s) { return sBar + 8u * (KST + s); };
    auto v_full = [&](int s) { return sBar + 8u * (2 * KST + s); };
    auto v_empty = [&](int s) { return sBar + 8u * (2 * KST + VST + s); };
    constexpr int NQ = Sh::NQ;
    auto q_full = [&](int s) { return sBar + 8u * (2 * KST + 2 * VST + s); };
    auto q_empty = [&](int s) { return sBar + 8u * (2 * KST + 2 * VST + NQ + s); };
    const uint32_t sBar2 = sBar + 8u * (2 * KST + 2 * VST + 2 * NQ);  // base of the rest
    // One S buffer: s_full completes when both halves of S(i) are in TMEM,
    // s_free once the four softmax warps have read them.
    const uint32_t s_full = sBar2, s_free = sBar2 + 8u;
    auto p_full = [&](int b) { return sBar2 + 8u * (2 + b); };
    // o_fin[i & 1] completes when O += P(i) V(i) has finished (and P buffer
    // i & 1 may be written again). One barrier per P buffer (rather than one
    // for all tiles) keeps every waiter within one phase of the completion it
    // waits for, so parity waits are unambiguous.
    auto o_fin = [&](int b) { return sBar2 + 8u * (4 + b); };
    const uint32_t mma_done = sBar2 + 8u * 6;
    // KV8: the 8-bit rings (filled by TMA, emptied by the converters), the
    // f16 copy of each pair's Q, and the row-scale slots (filled by the
    // converters, read by the softmax).
    constexpr int K8ST = Sh::K8ST, V8ST = Sh::V8ST, NSC = Sh::NSC;
    const uint32_t sBar3 = sBar2 + 8u * 7;
    auto k8_full = [&](int s) { return sBar3 + 8u * s; };
    auto k8_empty = [&](int s) { return sBar3 + 8u * (K8ST + s); };
    auto v8_full = [&](int s) { return sBar3 + 8u * (2 * K8ST + s); };
    auto v8_empty = [&](int s) { return sBar3 + 8u * (2 * K8ST + V8ST + s); };
    auto q_conv = [&](int s) { return sBar3 + 8u * (2 * K8ST + 2 * V8ST + s); };
    auto sc_full = [&](int s) { return sBar3 + 8u * (2 * K8ST + 2 * V8ST + NQ + s); };
    auto sc_empty = [&](int s) { return sBar3 + 8u * (2 * K8ST + 2 * V8ST + NQ + NSC + s); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sh::OFF_MISC + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x;
    const int G = p.G;

    // ---- set-up (reads no inputs, so it overlaps the previous kernel's tail) ----
    if (tid == 32) {
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&maps.q)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&maps.k)) : "memory");
        asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(&maps.v)) : "memory");
    }
    if (tid == 0) {
        // (KV8: the converter warps of each tensor fill the f16 stages)
        for (int s = 0; s < KST; ++s) {
            tc::mbar_init(k_full(s), KV8 ? Sh::NCW : 1);
            tc::mbar_init(k_empty(s), 2);  // both S issuers
        }
        for (int s = 0; s < VST; ++s) {
            tc::mbar_init(v_full(s), KV8 ? Sh::NCW : 1);
            tc::mbar_init(v_empty(s), 1);
        }
        if constexpr (KV8) {
            for (int s = 0; s < K8ST; ++s) {
                tc::mbar_init(k8_full(s), 1);
                tc::mbar_init(k8_empty(s), Sh::NCW);
            }
            for (int s = 0; s < V8ST; ++s) {
                tc::mbar_init(v8_full(s), 1);
                tc::mbar_init(v8_empty(s), Sh::NCW);
            }
            for (int s = 0; s < NQ; ++s) tc::mbar_init(q_conv(s), 1);
            for (int s = 0; s < NSC; ++s) {
                tc::mbar_init(sc_full(s), 2 * Sh::NCW);  // the converter warps
                tc::mbar_init(sc_empty(s), Sh::NSW);  // the softmax warps
            }
        }
        for (int s = 0; s < NQ; ++s) {
            tc::mbar_init(q_full(s), 1);
            tc::mbar_init(q_empty(s), 2);
        }
        tc::mbar_init(s_full, 2);  // both S issuers
        tc::mbar_init(s_free, Sh::NSW);  // the softmax warps
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(p_full(b), Sh::NSW);
            tc::mbar_init(o_fin(b), 1);
        }
        tc::mbar_init(mma_done, 3);  // S issuers and O issuer
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    // Rows of Q past the group stay zero.
    for (int i = tid; i < Sh::Q_BYTES / 16; i += Sh::THREADS)
        reinterpret_cast<uint4*>(smem + Sh::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(tmem_slot), Sh::TMEM_COLS);
        tc::fence_before_sync();
    }

    // Inputs may be produced by the previous kernel on the stream. After this
    // library's append (p.early), only the cache loads need to wait for it.
    if (!p.early) pdl_wait();
    pdl_launch_dependents();

    // p.vT > 1 query tokens per sequence run as p.B = B * vT virtual
    // sequences (see DevLen): their q, out and lse rows are those of the
    // [B, vT, Hq] layouts, and virtual sequence b reads the cache rows (and
    // pos, and block-table row) of sequence b / vT.
    const int vt = p.vT > 1 ? p.vT : 1;
    const DevLen len{p.seq_lens, p.len_cap, vt};
    using Geo = FixedGeom<T, Sh::SEG_UNIT, SEG_COST>;
    // ---- total work, this CTA's run, first sequence ----
    // Warp 0 works the schedule out and leaves the walker, positioned at the
    // start of this CTA's run, in shared memory; each role takes a copy after
    // the set-up barrier. Up to 32 * WK sequences (the common case) it does so
    // with warp shuffles only, lane l taking sequences l, l + 32, ...; past
    // that, the whole block scans the lengths.
    using WalkerT = Walker<DevLen, Geo>;
    __shared__ __align__(16) unsigned char s_walker[sizeof(WalkerT)];
    __shared__ int s_has_work;
    constexpr int WK = 8;
    const bool by_warp = p.B <= 32 * WK;
    auto publish = [&](int C_eff, long long total, bool has_work, int b0, long long cum0) {
        WalkerT w(len, Geo{}, p.B, p.Hkv, c, has_work ? C_eff : c + 1, has_work ? total : 0);
        w.start(b0, cum0);
        memcpy(s_walker, &w, sizeof(WalkerT));
        s_has_work = has_work ? 1 : 0;
    };
    if (by_warp) {
        if (warp == 0) {
            int ext_r[WK];
            bool clamped = false;
#pragma unroll
            for (int k = 0; k < WK; ++k) {
                const int b = lane + 32 * k;
                ext_r[k] = 0;
                if (b < p.B) {
                    const int raw = __ldg(p.seq_lens + b / vt);
                    clamped |= (raw != clamp_len(raw, p.len_cap));
                    ext_r[k] = (int)pair_extent(len(b), Geo{});
                }
            }
            if (clamped && c == 0 && p.status) atomicOr(p.status, KVD_STATUS_SEQ_LEN_CLAMPED);
            int tot = 0;
#pragma unroll
            for (int k = 0; k < WK; ++k) tot += ext_r[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
            const long long total = (long long)tot * p.Hkv;
            const int C_eff = effective_ctas(p.n_split, total);
            const bool has_work = c < C_eff;
            const long long S = has_work ? run_begin(c, C_eff, total) : total;
            int b0 = p.B;
            long long cum0 = total;
            if (has_work) {
                // The first sequence touching the run: the first candidate in b
                // order (the condition, once true, stays true).
                long long carry = 0;
#pragma unroll
                for (int k = 0; k < WK; ++k) {
                    if (32 * k >= p.B) break;
                    const int x = ext_r[k];
                    int incl = x;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    const long long cs = carry + (long long)(incl - x) * p.Hkv;
                    const bool cand = (lane + 32 * k < p.B) && is_first_seq_candidate(cs, x, p.Hkv, S);
                    const unsigned m = __ballot_sync(0xffffffffu, cand);
                    if (m) {
                        const int f = __ffs(m) - 1;
                        b0 = 32 * k + f;
                        cum0 = __shfl_sync(0xffffffffu, cs, f);
                        break;
                    }
                    carry += (long long)__shfl_sync(0xffffffffu, incl, 31) * p.Hkv;
                }
            }
            if (lane == 0) publish(C_eff, total, has_work, b0, cum0);
        }
        __syncthreads();  // set-up done, walker published
    } else {
        __syncthreads();  // set-up done
        long long mine = 0;
        bool clamped = false;
        for (int b = tid; b < p.B; b += Sh::THREADS) {
            const int raw = __ldg(p.seq_lens + b / vt);
            clamped |= (raw != clamp_len(raw, p.len_cap));
            mine += pair_extent(len(b), Geo{});
        }
        if (clamped && c == 0 && p.status) atomicOr(p.status, KVD_STATUS_SEQ_LEN_CLAMPED);
        const long long total = block_sum_ll<NW>(mine, s_red) * p.Hkv;
        const int C_eff = effective_ctas(p.n_split, total);
        const bool has_work = c < C_eff;
        const long long S = has_work ? run_begin(c, C_eff, total) : total;
        int b0 = p.B;
        long long cum0 = total;
        for (long long base = 0, chunk = 0; has_work && chunk < p.B; chunk += Sh::THREADS) {
            const int b = (int)chunk + tid;
            const int L = (b < p.B) ? len(b) : 0;
            const long long e = pair_extent(L, Geo{});
            const long long v = e * p.Hkv;
            long long ctot;
            const long long cs = base + block_incl_scan_ll<NW>(v, s_red, &ctot) - v;
            const bool cand = (b < p.B) && is_first_seq_candidate(cs, e, p.Hkv, S);
            const int bmin = block_min_int<NW>(cand ? b : 0x7fffffff, s_redi);
            if (bmin != 0x7fffffff) {
                if (b == bmin) s_cum0 = cs;
                __syncthreads();
                b0 = bmin;
                cum0 = s_cum0;
                break;
            }
            base += ctot;
        }
        if (tid == 0) publish(C_eff, total, has_work, b0, cum0);
        __syncthreads();
    }
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    WalkerT walker;
    memcpy(&walker, s_walker, sizeof(WalkerT));
    const bool has_work = s_has_work != 0;

    if (!has_work) {
        // no tokens for this CTA: fall through to the common exit (TMEM release)
    } else if (warp == 0 || warp == 2) {
        // ===================== TMA producers =====================
        if (lane == 0) {
            const bool is_k = (warp == 0);
            const uint64_t pol_kv = l2_evict_first_policy();
            Tile t;
            int j = 0;
            // KV8: the 8-bit rings (128-column boxes of one-byte codes).
            const int NS = KV8 ? (is_k ? K8ST : V8ST) : (is_k ? KST : VST);
            const CUtensorMap* map = is_k ? &maps.k : &maps.v;
            constexpr int NBOX = KV8 ? Sh::KB8 : KB, BOXC = KV8 ? 128 : 64;
            constexpr uint32_t STAGE = KV8 ? Sh::TILE8_BYTES : Sh::TILE_BYTES;
            auto full_of = [&](int s2) { return KV8 ? (is_k ? k8_full(s2) : v8_full(s2)) : (is_k ? k_full(s2) : v_full(s2)); };
            auto empty_of = [&](int s2) {
                return KV8 ? (is_k ? k8_empty(s2) : v8_empty(s2)) : (is_k ? k_empty(s2) : v_empty(s2));
            };
            const uint32_t ring = KV8 ? (is_k ? sK8 : sV8) : (is_k ? sK : sV);
            // Early mode: only tiles holding a pair's appended rows (those from
            // pos on) wait for the append's grid; tiles before them stream
            // meanwhile. pos is an input (complete at launch), read once per
            // pair until the first wait.
            bool waited = !p.early;
            int pos_pair = -1, pos_b = -1;
            const bool paged = p.block_table != nullptr;
            const int box_rows = paged ? min(1 << p.page_shift, T) : T;
            if (!waited && walker.b < p.B) {  // issued now, first used at the first tile
                pos_pair = walker.b * p.Hkv + walker.h;
                pos_b = __ldg(p.pos + walker.b / vt);
            }
            while (walker.next(t, NoOp{})) {
                // Paged cache: the tile's block-table entries (one per box of
                // box_rows tokens, at most T / 16), loaded together before the
                // wait for the stage, so that their latency overlaps it.
                int entry[T / 16];
                if (paged) {
                    const int32_t* table = p.block_table + (size_t)(t.b / vt) * p.max_blocks;
#pragma unroll
                    for (int q = 0; q < T / 16; ++q) {
                        const int tok = t.tok_lo + q * box_rows;
                        entry[q] = (q * box_rows < T && tok < t.tok_hi) ? __ldg(table + (tok >> p.page_shift)) : -1;
                    }
                }
                if (!waited) {
                    const int pair = t.b * p.Hkv + t.h;
                    if (pair != pos_pair) {
                        pos_pair = pair;
                        pos_b = __ldg(p.pos + t.b / vt);
                    }
                    if (t.tok_hi > pos_b) {
                        pdl_wait();
                        waited = true;
                    }
                }
                const int s = j % NS;
                const uint32_t full = full_of(s);
                if (!tc::mbar_wait(empty_of(s), ((j / NS) & 1) ^ 1, abort_flag, kBudget)) break;
                tc::mbar_arrive_expect_tx(full, STAGE);
                const uint32_t dst = ring + (uint32_t)s * STAGE;
                if (!paged) {
                    const int row = (t.b / vt) * p.S_max + t.tok_lo;
#pragma unroll
                    for (int kb = 0; kb < NBOX; ++kb)
                        tc::tma_load_3d(dst + kb * Sh::KB_BYTES, map, kb * BOXC, t.h, row, full, pol_kv);
                } else {
                    tma_paged_tile<NBOX, BOXC, Sh::KB_BYTES, T>(dst, map, t.h, t.tok_lo, t.tok_hi, entry[0], entry[1],
                                                                entry[2], entry[3], box_rows, p.page_shift,
                                                                p.num_pages, full, pol_kv, is_k ? p.status : nullptr);
                }
                ++j;
            }
            // Do not leave with copies in flight: wait for the last loads to land.
            for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) {
                const int s = jj % NS;
                tc::mbar_wait(full_of(s), (jj / NS) & 1, abort_flag, kBudget / 4);
            }
        }
    } else if (warp == 9) {
        // ===================== Q loader =====================
        // Its own thread, so that waiting for the Q slot (free once the previous
        // pair's last S is done) never holds up the K stream. When the run goes
        // on into a next pair, that pair's Q rows are also prefetched into L2,
        // so its load is short when its turn comes.
        if constexpr (!KV8) {
            if (lane == 0) {
                const uint64_t pol_q = tc::l2_evict_last_policy();
                // q staged by the preceding append (host-input step): wait for it.
                if (p.early && p.q_wait) pdl_wait();
                Tile t;
                int qn = 0;
                while (walker.next(t, NoOp{})) {
                    if (!t.seg_start) continue;
                    const int qs = qn % NQ;
                    if (!tc::mbar_wait(q_empty(qs), ((qn / NQ) & 1) ^ 1, abort_flag, kBudget)) break;
                    // The pair's query rows: its G heads, or at M = 128 the G heads
                    // of each of the sequence's TQ query tokens, token i at rows
                    // i * G8 (8-row aligned, as the swizzled layout needs).
                    const int TQ = (MR == 128) ? p.T : 1, G8 = (G + 7) & ~7;
                    tc::mbar_arrive_expect_tx(q_full(qs), (uint32_t)(KB * 128 * G * TQ));
                    for (int i2 = 0; i2 < TQ; ++i2) {
                        const int qrow = (t.b * TQ + i2) * p.Hq + t.h * G;
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb)
                            tc::tma_load_2d(sQ + qs * Sh::QS_BYTES + kb * Sh::QB_BYTES + i2 * G8 * 128, &maps.q, kb * 64,
                                            qrow, q_full(qs), pol_q);
                    }
                    ++qn;
                    if (walker.pstart + walker.ext() < walker.E) {
                        const int nh = (t.h + 1 < p.Hkv) ? t.h + 1 : 0;
                        const int nb = (t.h + 1 < p.Hkv) ? t.b : t.b + 1;
                        if (nb < p.B)
                            for (int i2 = 0; i2 < TQ; ++i2)
                                tc::prefetch_l2(reinterpret_cast<const uint8_t*>(p.q) +
                                                    (((size_t)nb * TQ + i2) * p.Hq + (size_t)nh * G) * D * 2,
                                                (uint32_t)(G * D * 2));
                    }
                }
                if (qn > 0) tc::mbar_wait(q_full((qn - 1) % NQ), ((qn - 1) / NQ) & 1, abort_flag, kBudget / 4);
            }
        } else {
            // KV8: the whole warp then converts the pair's rows to f16 in place
            // (the MMAs take f16 operands against the f16 K and V tiles) and
            // signals q_conv, which the S issuers wait for.
            const uint64_t pol_q = tc::l2_evict_last_policy();
            if (p.early && p.q_wait) pdl_wait();
            Tile t;
            int qn = 0;
            bool ok = true;
            while (ok && walker.next(t, NoOp{})) {
                if (!t.seg_start) continue;
                const int qs = qn % NQ;
                if (lane == 0) {
                    ok = tc::mbar_wait(q_empty(qs), ((qn / NQ) & 1) ^ 1, abort_flag, kBudget);
                    if (ok) {
                        tc::mbar_arrive_expect_tx(q_full(qs), (uint32_t)(KB * 128 * G));
                        const int qrow = t.b * p.Hq + t.h * G;
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb)
                            tc::tma_load_2d(sQ + qs * Sh::QS_BYTES + kb * Sh::QB_BYTES, &maps.q, kb * 64, qrow,
                                            q_full(qs), pol_q);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                ok = __all_sync(0xffffffffu, tc::mbar_wait(q_full(qs), (qn / NQ) & 1, abort_flag, kBudget));
                if (!ok) break;
                // Each block's G rows are contiguous (128 bytes a row); the
                // conversion is elementwise, so the swizzle does not matter.
                const int n16 = G * 8;
#pragma unroll 1
                for (int kb = 0; kb < KB; ++kb) {
                    uint4* q4 = reinterpret_cast<uint4*>(smem + Sh::OFF_Q + qs * Sh::QS_BYTES + kb * Sh::QB_BYTES);
#pragma unroll 4
                    for (int idx = lane; idx < n16; idx += 32) {
                        uint4 v = q4[idx];
                        v.x = bf16x2_to_f16x2(v.x);
                        v.y = bf16x2_to_f16x2(v.y);
                        v.z = bf16x2_to_f16x2(v.z);
                        v.w = bf16x2_to_f16x2(v.w);
                        q4[idx] = v;
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(q_conv(qs));
                ++qn;
                if (lane == 0 && walker.pstart + walker.ext() < walker.E) {
                    const int nh = (t.h + 1 < p.Hkv) ? t.h + 1 : 0;
                    const int nb = (t.h + 1 < p.Hkv) ? t.b : t.b + 1;
                    if (nb < p.B)
                        tc::prefetch_l2(reinterpret_cast<const uint8_t*>(p.q) + ((size_t)nb * p.Hq + (size_t)nh * G) * D * 2,
                                        (uint32_t)(G * D * 2));
                }
            }
        }
    } else if (warp == 1 || warp == 7) {
        // ===================== S issuers (one thread each) =====================
        // S = Q K^T is issued as two independent accumulations over the two
        // halves of head_dim, by two threads into two TMEM column ranges that
        // the softmax adds: a tcgen05.mma of this shape costs its issuing
        // thread about as long as the tensor core needs for two of them, so
        // two issuers finish a tile's S in half the time and release its K
        // stage sooner. One S buffer: S(i) is issued once the softmax has read
        // S(i - 1) out of TMEM, early in that tile's softmax.
        if (lane == 0) {
            const int kh = (warp == 7) ? 1 : 0;
            constexpr int KH = D / 32;  // k-steps per half
            constexpr uint32_t idesc_s = tc::idesc_f32acc(MR, T, false, false, KV8);  // f16 operands for KV8
            const uint32_t s_base = tmem + (kh ? Sh::TMEM_S2 : Sh::TMEM_S);
            Tile t;
            int i = 0, qn = 0;
            while (walker.next(t, NoOp{})) {
                const int sk = i % KST;
                if (t.seg_start) {
                    if (!tc::mbar_wait(KV8 ? q_conv(qn % NQ) : q_full(qn % NQ), (qn / NQ) & 1, abort_flag, kBudget))
                        break;
                    ++qn;
                }
                const int qs = (qn - 1) % NQ;
                if (!tc::mbar_wait(k_full(sk), (i / KST) & 1, abort_flag, kBudget)) break;
                if (!tc::mbar_wait(s_free, (i & 1) ^ 1, abort_flag, kBudget)) break;
                tc::fence_after_sync();
                const uint32_t qt = sQ + (uint32_t)(qs * Sh::QS_BYTES);
                const uint32_t kt = sK + (uint32_t)(sk * Sh::TILE_BYTES);
#pragma unroll
                for (int k = 0; k < KH; ++k) {
                    const int kk = kh * KH + k;
                    const uint64_t a = tc::sdesc_sw128(qt + (kk >> 2) * Sh::QB_BYTES + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = tc::sdesc_sw128(kt + (kk >> 2) * Sh::KB_BYTES + (kk & 3) * 32, 16, 1024);
                    tc::mma_bf16(s_base, a, b, idesc_s, k > 0);
                }
                tc::mma_commit(s_full);
                tc::mma_commit(k_empty(sk));
                if (t.seg_end) tc::mma_commit(q_empty(qs));
                ++i;
            }
            // This thread's tensor-core work done before TMEM is released.
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, abort_flag, kBudget);
        }
    } else if (warp == 8) {
        // ===================== O issuer (one thread) =====================
        // O += P(i) V(i): A = P from TMEM buffer i & 1 (the hi part, then the
        // lo part for fp32 output), B = the V stage in MN-major layout.
        if (lane == 0) {
            constexpr uint32_t idesc_o = tc::idesc_f32acc(MR, D, false, true, KV8);
            Tile t;
            int i = 0;
            while (walker.next(t, NoOp{})) {
                const int sv = i % VST, pb = i & 1;
                if (!tc::mbar_wait(v_full(sv), (i / VST) & 1, abort_flag, kBudget)) break;
                if (!tc::mbar_wait(p_full(pb), (i >> 1) & 1, abort_flag, kBudget)) break;
                tc::fence_after_sync();
                const uint32_t vt = sV + (uint32_t)(sv * Sh::TILE_BYTES);
                const uint32_t pa = tmem + (uint32_t)(Sh::TMEM_P + pb * Sh::PCOLS);
#pragma unroll
                for (int k2 = 0; k2 < T / 16; ++k2) {
                    const uint64_t b = tc::sdesc_sw128(vt + k2 * 2048, Sh::KB_BYTES, 1024);
#pragma unroll
                    for (int part = 0; part < Sh::NP; ++part)
                        tc::mma_bf16_ts(tmem + Sh::TMEM_O, pa + (uint32_t)(part * (T / 2) + k2 * 8), b, idesc_o,
                                        (t.seg_start && k2 == 0 && part == 0) ? 0u : 1u);
                }
                tc::mma_commit(v_empty(sv));
                tc::mma_commit(o_fin(pb));
                ++i;
            }
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, abort_flag, kBudget);
        }
    } else if (KV8 && warp >= 10) {
        static_assert(!KV8 || Sh::NCW == 2 || Sh::NCW == 4, "converter warps per tensor");
        // ===================== converters (KV8: warps 10 .. 10 + NCW - 1 for K, the next NCW for V) =====================
        // Each tensor's NCW warps turn its 8-bit tiles into f16 tiles in the
        // layout TMA would have written for bf16 rows (128-byte swizzle,
        // 64-column blocks), and read the tile's row scales from global
        // memory into a scale slot for the softmax (zero past the tile's
        // last token, so those rows weigh nothing). Chunk g of the 4 D 16-byte
        // chunks of a tile goes to thread g % NCT of the tensor's NCT
        // threads; the low bits of g pick column chunk c = 4 h + (g & 3) of
        // row rho or rho ^ 5 of an 8-row group, so that the 8 threads of each
        // quarter-warp read 8 distinct 16-byte bank groups of the 8-bit tile
        // and write 8 distinct ones of the f16 tile; the higher bits pick the
        // 8-row group and the 128-column block.
        constexpr int NCW = Sh::NCW > 0 ? Sh::NCW : 1, NCT = NCW * 32;  // (NCW = 0 without KV8: unused)
        const bool is_k = warp < 10 + NCW;
        const int cth = (warp - 10 - (is_k ? 0 : NCW)) * 32 + lane;  // 0 .. NCT - 1 within the tensor
        const int N8 = is_k ? K8ST : V8ST, NF = is_k ? KST : VST;
        const uint32_t r8 = is_k ? sK8 : sV8, rf = is_k ? sK : sV;
        const float* gsc = is_k ? p.k_scale : p.v_scale;
        const float scmul = (FP8 && is_k) ? 256.f : 1.f;  // E4M3 key rows arrive divided by 256
        const int r = cth;                                 // the tile row whose scale this thread reads (r < T)
        // This thread's chunk: the bits of g % 64 give its row rlo within an
        // 8-row group and its column chunk c8; the swizzle depends on the row
        // only through rlo, so the offsets step evenly from chunk to chunk.
        const int clo = cth & 3, sel = (cth >> 2) & 1, h = (cth >> 3) & 1, rho = (cth >> 4) & 3;
        const int rlo = sel ? (rho ^ 5) : rho, c8 = 4 * h + clo;
        const uint32_t rg0 = (uint32_t)(cth >> 6);  // first 8-row group (NCT = 128: 0 or 1)
        const uint32_t src_off = rg0 * 1024 + rlo * 128 + ((c8 ^ rlo) * 16);
        const uint32_t dst_off = h * Sh::KB_BYTES + rg0 * 1024 + rlo * 128;
        const uint32_t d0 = ((2 * clo) ^ rlo) * 16, d1 = ((2 * clo + 1) ^ rlo) * 16;
        // The row scales are loaded two tiles ahead (a second walker runs in
        // front), so their latency hides behind the conversions in between.
        // Early mode: as the producers, the append is waited for before a
        // tile holding rows it writes.
        bool waited = !p.early;
        int pos_pair = -1, pos_b = -1;
        auto load_scale = [&](const Tile& ta) -> float {
            if (!waited) {
                const int pair = ta.b * p.Hkv + ta.h;
                if (pair != pos_pair) {
                    pos_pair = pair;
                    pos_b = __ldg(p.pos + ta.b / vt);
                }
                if (ta.tok_hi > pos_b) {
                    pdl_wait();
                    waited = true;
                }
            }
            // The row's scale: cache row b * S_max + token, or in a paged
            // cache its row in the pool (a table entry naming no page gives
            // zero codes, read past the pool's end, and a zero scale); zero
            // past the tile's last token.
            float v = 0.f;
            if (r < ta.tok_hi - ta.tok_lo && r < T) {
                const int tok = ta.tok_lo + r;
                long long row = (long long)(ta.b / vt) * p.S_max + tok;
                if (p.block_table) {
                    const int page = __ldg(p.block_table + (size_t)(ta.b / vt) * p.max_blocks + (tok >> p.page_shift));
                    row = ((unsigned)page < (unsigned)p.num_pages)
                              ? ((long long)page << p.page_shift) + (tok & ((1 << p.page_shift) - 1))
                              : -1;
                }
                if (row >= 0) v = __ldg(gsc + (size_t)row * p.Hkv + ta.h);  // (not used until two tiles on)
            }
            return v;
        };
        WalkerT ahead = walker;
        Tile t, ta;
        float sc_next[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) sc_next[k] = ahead.next(ta, NoOp{}) ? load_scale(ta) : 0.f;
        int j = 0;
        bool ok = true;
        while (ok && walker.next(t, NoOp{})) {
            const float sc = sc_next[0];
            sc_next[0] = sc_next[1];
            sc_next[1] = ahead.next(ta, NoOp{}) ? load_scale(ta) : 0.f;
            const int s8 = j % N8, sf = j % NF, ss = j % NSC;
            ok = __all_sync(0xffffffffu, tc::mbar_wait(is_k ? k8_full(s8) : v8_full(s8), (j / N8) & 1, abort_flag,
                                                       kBudget));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, tc::mbar_wait(is_k ? k_empty(sf) : v_empty(sf), ((j / NF) & 1) ^ 1,
                                                       abort_flag, kBudget));
            if (!ok) break;
            ok = __all_sync(0xffffffffu, tc::mbar_wait(sc_empty(ss), ((j / NSC) & 1) ^ 1, abort_flag, kBudget));
            if (!ok) break;
            const uint8_t* src = smem + (r8 - sbase) + (size_t)s8 * Sh::TILE8_BYTES + src_off;
            uint8_t* dst = smem + (rf - sbase) + (size_t)sf * Sh::TILE_BYTES + dst_off;
            // Each step moves this thread NCT / 64 8-row groups further down the
            // tile (1 KB of 8-bit rows a group); every 8 groups the 8-bit
            // tile's next 128-column block starts, which in f16 is the next
            // pair of 64-column blocks.
            constexpr int GPS = NCT / 64;  // 8-row groups a step
#pragma unroll 4
            for (int it = 0; it < D * 4 / NCT; ++it) {
                const uint4 w = *reinterpret_cast<const uint4*>(src + it * GPS * 1024);
                uint32_t f[8];
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t u = FP8 ? wv[q] : (wv[q] ^ 0x80808080u);
                    f[2 * q] = codes_to_f16x2<FP8, 0x4140, 0x9180>(u);
                    f[2 * q + 1] = codes_to_f16x2<FP8, 0x4342, 0xb3a2>(u);
                }
                const int grp = it * GPS;  // first 8-row group of the step (of 8 per 128-column block)
                uint8_t* drow = dst + (grp >> 3) * 2 * Sh::KB_BYTES + (grp & 7) * 1024;
                *reinterpret_cast<uint4*>(drow + d0) = make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4*>(drow + d1) = make_uint4(f[4], f[5], f[6], f[7]);
            }
            if (r < T) reinterpret_cast<float*>(smem + Sh::OFF_SC + ss * 2 * T * 4)[(is_k ? 0 : T) + r] = sc * scmul;
            tc::fence_proxy_async_smem();  // the f16 tile, for the tensor core
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(is_k ? k8_empty(s8) : v8_empty(s8));
                tc::mbar_arrive(is_k ? k_full(sf) : v_full(sf));
                tc::mbar_arrive(sc_full(ss));
            }
            ++j;
        }
    } else if ((warp >= 3 && warp <= 6) || warp >= 10) {
        // ===================== softmax / epilogue (warps 3..6, 10..13) =====================
        // One warp per TMEM lane quarter (a warp reaches the 32 lanes
        // 32 * (warp % 4) ...). At M = 64 its accumulator rows sit in lanes
        // 0-15 of the quarter (rows 16 q .. 16 q + 15); at M = 128 in all 32
        // lanes (rows 32 q .. 32 q + 31), two groups of 16, each with a warp of
        // its own (warps 3..6 the first, 10..13 the second). Through
        // the 16x32bx2 shape each row goes to two threads of the warp: thread
        // l takes row (16 lanes of the warp's group) + l % 16 and token columns
        // [32 (l / 16), 32 (l / 16) + 32) of every S tile (P columns
        // likewise), and output columns [(D / 2)(l / 16), ...) in the
        // epilogue. A row's maximum and sum need one shuffle between its two
        // threads; no other warp takes part.
        // Rows: at M = 64 the group's query heads; at M = 128 the T query
        // tokens of a sequence stacked (row = token * G8 + head, G8 = the group
        // rounded up to 8), token i seeing the first L - T + 1 + i tokens.
        constexpr int NG = 1;                        // row groups per warp
        constexpr int NST = Sh::NSW * 32;            // softmax threads
        constexpr int HT = T / 2;   // token columns per thread
        constexpr int HD = D / 2;   // output columns per thread
        const int quarter = warp & 3;
        const int rgw = warp >= 10 ? 1 : 0;          // this warp's group of 16 rows in its quarter
        const int hl = lane >> 4;
        const int st = (warp >= 10 ? warp - 6 : warp - 3) * 32 + lane;  // 0..NST-1 among the softmax threads
        const float scale_log2 = p.scale_log2;
        const int TQ = (MR == 128) ? p.T : 1;        // query tokens stacked in the rows
        const int G8 = (G + 7) & ~7;
        int tok_[NG], hd_[NG];
        bool act_[NG];
#pragma unroll
        for (int rg = 0; rg < NG; ++rg) {
            const int row = quarter * 16 * Sh::NG + 16 * (rg + rgw) + (lane & 15);
            tok_[rg] = (MR == 128) ? row / G8 : 0;
            hd_[rg] = (MR == 128) ? row - tok_[rg] * G8 : row;
            act_[rg] = tok_[rg] < TQ && hd_[rg] < G;
        }
        auto lanes = [&](int rg) { return (uint32_t)(quarter * 32 + 16 * (rg + rgw)) << 16; };
        // Output (or lse) row of (sequence b, KV head h, token i, head g); partial-state row within a slot.
        auto out_row = [&](int b, int h, int i2, int g) {
            return ((size_t)b * TQ + i2) * p.Hq + (size_t)h * G + g;
        };

        auto write_empty = [&](int b, int h) {
            for (int i2 = 0; i2 < TQ; ++i2) {
                const size_t r0 = out_row(b, h, i2, 0);
                if constexpr (F32OUT) {
                    float* o = reinterpret_cast<float*>(p.out) + r0 * D;
                    for (int k = st; k < G * D; k += NST) o[k] = 0.f;
                } else {
                    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + r0 * D;
                    for (int k = st; k < G * D; k += NST) o[k] = __float2bfloat16_rn(0.f);
                }
                if (p.lse)
                    for (int k = st; k < G; k += NST) p.lse[r0 + k] = -CUDART_INF_F;
            }
        };

        float m[NG], l[NG];  // running maximum of each row (the same in both of its threads); row-sum share
#pragma unroll
        for (int rg = 0; rg < NG; ++rg) m[rg] = l[rg] = 0.f;
        Tile t;
        int i = 0;
        bool ok = true;
        while (ok && walker.next(t, write_empty)) {
            ok = __all_sync(0xffffffffu, tc::mbar_wait(s_full, i & 1, abort_flag, kBudget));
            if (!ok) break;
            // KV8: the tile's key and value row scales (zero past its last token).
            const float* ksc = nullptr;
            const float* vsc = nullptr;
            if constexpr (KV8) {
                ok = __all_sync(0xffffffffu, tc::mbar_wait(sc_full(i % NSC), (i / NSC) & 1, abort_flag, kBudget));
                if (!ok) break;
                ksc = reinterpret_cast<const float*>(smem + Sh::OFF_SC + (i % NSC) * 2 * T * 4) + hl * HT;
                vsc = ksc + T;
            }
            tc::fence_after_sync();
            __syncwarp();
            const int nvalid = t.tok_hi - t.tok_lo;
            // P buffer i & 1 is free once O += P(i-2) V(i-2) has completed.
            const int pb = i & 1;
            if (i >= 2) {
                ok = __all_sync(0xffffffffu,
                                tc::mbar_wait(o_fin(pb), ((i >> 1) - 1) & 1, abort_flag, kBudget));
                if (!ok) break;
                tc::fence_after_sync();
            }
            float alpha[NG];
            bool need_any = false;
#pragma unroll
            for (int rg = 0; rg < NG; ++rg) {
                // S is held as two partial sums over the halves of head_dim.
                float s[HT];
                {
                    uint32_t sa[HT], sb[HT];
                    tc::tmem_ld_16x32bx2_x32<HT>(tmem + lanes(rg) + Sh::TMEM_S, sa);
                    tc::tmem_ld_16x32bx2_x32<HT>(tmem + lanes(rg) + Sh::TMEM_S2, sb);
                    tc::tmem_wait_ld();
                    if (rg == NG - 1) {
                        tc::fence_before_sync();
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(s_free);
                    }
                    // Scores in base-2 units; columns past the tile's last token
                    // (or, at M = 128, past the row's token's causal limit) masked.
                    int vis = nvalid;
                    if (MR == 128) vis = min(vis, t.L - (TQ - 1 - tok_[rg]) - t.tok_lo);
                    const int nv = vis - hl * HT;  // valid columns of this thread (may be <= 0)
#pragma unroll
                    for (int e = 0; e < HT; ++e) {
                        // (KV8: times the key row's scale; E4M3 key rows, which arrive
                        // divided by 256, have it times 256)
                        const float sc = KV8 ? scale_log2 * ksc[e] : scale_log2;
                        s[e] = (e < nv) ? (__uint_as_float(sa[e]) + __uint_as_float(sb[e])) * sc : -CUDART_INF_F;
                    }
                }
                float mx = s[0];
#pragma unroll
                for (int e = 1; e < HT; ++e) mx = fmaxf(mx, s[e]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const bool active = act_[rg];
                alpha[rg] = 1.f;
                if (t.seg_start) {
                    m[rg] = mx;
                    if (!KV8 && p.umax) {
                        // Unified maximum (FlashDecoding++'s asynchronized softmax):
                        // a row whose first tile's maximum lies within [phi - 64,
                        // phi + 8] (base 2) takes m = phi, shared by all partials of
                        // such rows, so the merge reduces to plain sums; otherwise
                        // it starts from its own maximum. The lazy rescale below
                        // moves m up past phi + 8 (exact either way).
                        const float phi2 = p.umax_phi2;
                        if (mx >= phi2 - 64.f && mx <= phi2 + 8.f) m[rg] = phi2;
                        if (active && m[rg] != phi2 && p.status) atomicOr(p.status, KVD_STATUS_UMAX_FALLBACK);
                    }
                    l[rg] = 0.f;
                } else if (mx > m[rg] + 8.f) {
                    // (a row with no visible column yet keeps m = -inf and takes its first maximum here)
                    need_any = true;
                    alpha[rg] = (m[rg] == -CUDART_INF_F) ? 0.f : exp2f(m[rg] - mx);
                    m[rg] = mx;
                    if (!KV8 && p.umax && active && p.status) atomicOr(p.status, KVD_STATUS_UMAX_FALLBACK);
                }
                // P = 2^(s - m), packed in pairs of adjacent tokens (bf16 hi part;
                // lo part for fp32 output). A row that has seen no column yet
                // (m = -inf, M = 128 only) gives zeros.
                const bool live = active && m[rg] != -CUDART_INF_F;
                uint32_t hi[HT / 2], lo[HT / 2];
                float ls = 0.f;
#pragma unroll
                for (int g = 0; g < HT / 2; ++g) {
                    const float e0 = live ? tc::ex2_approx(s[2 * g] - m[rg]) : 0.f;
                    const float e1 = live ? tc::ex2_approx(s[2 * g + 1] - m[rg]) : 0.f;
                    if constexpr (KV8) {
                        // Weights times the value rows' scales, in f16 (the V
                        // tiles hold the codes' values); the sums take the
                        // weights themselves.
                        const float w0 = e0 * vsc[2 * g], w1 = e1 * vsc[2 * g + 1];
                        hi[g] = pack_f16x2(w0, w1);
                        if constexpr (F32OUT) lo[g] = pack_f16x2(w0 - f16_lo(hi[g]), w1 - f16_hi(hi[g]));
                        ls += e0 + e1;
                        continue;
                    }
                    hi[g] = pack_bf16x2(e0, e1);
                    if constexpr (F32OUT) {
                        lo[g] = pack_bf16x2(e0 - bf16_lo(hi[g]), e1 - bf16_hi(hi[g]));
                        ls += e0 + e1;
                    } else {
                        // The weights actually multiplied into V are the rounded ones;
                        // summing those keeps the output an exact convex combination.
                        ls += bf16_lo(hi[g]) + bf16_hi(hi[g]);
                    }
                }
                l[rg] = l[rg] * alpha[rg] + ls;
                const uint32_t pt = tmem + lanes(rg) + (uint32_t)(Sh::TMEM_P + pb * Sh::PCOLS);
                tc::tmem_st_16x32bx2_x16<HT / 2>(pt, hi);
                if constexpr (F32OUT) tc::tmem_st_16x32bx2_x16<HT / 2>(pt + T / 2, lo);
            }
            if (__any_sync(0xffffffffu, need_any)) {
                // A running maximum moved: O (with P(i-1) V(i-1) in it) is
                // rescaled before P(i) V(i) joins it.
                ok = __all_sync(0xffffffffu,
                                tc::mbar_wait(o_fin((i - 1) & 1), ((i - 1) >> 1) & 1, abort_flag, kBudget));
                if (!ok) break;
                tc::fence_after_sync();
#pragma unroll
                for (int rg = 0; rg < NG; ++rg) {
                    if (!__any_sync(0xffffffffu, alpha[rg] != 1.f)) continue;
#pragma unroll 1
                    for (int cc = 0; cc < HD / 32; ++cc) {
                        uint32_t r[32];
                        const uint32_t ta = tmem + lanes(rg) + Sh::TMEM_O + cc * 32;
                        tc::tmem_ld_16x32bx2_x32<HD>(ta, r);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha[rg]);
                        tc::tmem_st_16x32bx2_x32<HD>(ta, r);
                    }
                }
            }
            tc::tmem_wait_st();
            if constexpr (KV8) {
                // This tile's scales are read: free their slot.
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(sc_empty(i % NSC));
            }
            // (KV8 tiles need no zeroing: every code converts to a finite value,
            // and the rows past the tile's end have zero scales.)
            if (!KV8 && nvalid < T) {
                // Rows past the sequence's end came from the cache's padding (or the
                // next sequence): zero them so that 0-weights never meet NaN.
                const int sv = i % VST;
                ok = __all_sync(0xffffffffu, tc::mbar_wait(v_full(sv), (i / VST) & 1, abort_flag, kBudget));
                if (!ok) break;
                uint8_t* vt = smem + Sh::OFF_V + sv * Sh::TILE_BYTES;
                const int n16 = (T - nvalid) * KB * 8;
                for (int idx = st; idx < n16; idx += NST) {
                    const int r = nvalid + idx / (KB * 8);
                    const int rem = idx % (KB * 8);
                    *reinterpret_cast<uint4*>(vt + (rem >> 3) * Sh::KB_BYTES + r * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                tc::fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(p_full(pb));

            if (t.seg_end) {
                ok = __all_sync(0xffffffffu, tc::mbar_wait(o_fin(pb), (i >> 1) & 1, abort_flag, kBudget));
                if (!ok) break;
                tc::fence_after_sync();
                const size_t pair = (size_t)t.b * p.Hkv + t.h;
                const size_t slot = (size_t)c + pair;
#pragma unroll
                for (int rg = 0; rg < NG; ++rg) {
                    const float ltot = l[rg] + __shfl_xor_sync(0xffffffffu, l[rg], 16);
                    const bool active = act_[rg];
                    const size_t qrow = out_row(t.b, t.h, tok_[rg], hd_[rg]);
                    // Partial slots hold the pair's T * G rows, token-major.
                    const size_t prow = slot * (size_t)(TQ * G) + (size_t)tok_[rg] * G + hd_[rg];
                    // Each thread writes 32 contiguous columns of its row per chunk;
                    // two chunks' TMEM loads share one wait.
                    const float inv = t.full ? ((ltot > 0.f) ? OSC / ltot : 0.f) : OSC;
                    const size_t grow = t.full ? qrow : prow;  // output (or partial) row
                    auto put = [&](int cc, const uint32_t (&r)[32]) {
                        const int col0 = hl * HD + cc * 32;
                        if (active && t.full && !F32OUT) {
                            uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + grow * D + col0);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                o[k] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * k]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                                                  pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                                                  pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                                                  pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
                        } else if (active) {
                            float4* o = reinterpret_cast<float4*>((t.full ? reinterpret_cast<float*>(p.out) : p.ws_o) + grow * D + col0);
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                o[k] = make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                                                   __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
                        }
                    };
                    constexpr int NCH = HD / 32;  // 32-column chunks per thread
                    // (the 14- and 18-warp variants have no registers for two chunks)
                    constexpr bool PAIRS = (MR == 64 && !KV8);
#pragma unroll 1
                    for (int cc = 0; PAIRS && cc + 1 < NCH; cc += 2) {
                        uint32_t r0[32], r1[32];
                        tc::tmem_ld_16x32bx2_x32<HD>(tmem + lanes(rg) + Sh::TMEM_O + cc * 32, r0);
                        tc::tmem_ld_16x32bx2_x32<HD>(tmem + lanes(rg) + Sh::TMEM_O + (cc + 1) * 32, r1);
                        tc::tmem_wait_ld();
                        put(cc, r0);
                        put(cc + 1, r1);
                    }
#pragma unroll 1
                    for (int cc = PAIRS ? NCH - NCH % 2 : 0; cc < NCH; ++cc) {
                        uint32_t r0[32];
                        tc::tmem_ld_16x32bx2_x32<HD>(tmem + lanes(rg) + Sh::TMEM_O + cc * 32, r0);
                        tc::tmem_wait_ld();
                        put(cc, r0);
                    }
                    if (active && hl == 0) {
                        if (t.full) {
                            if (p.lse) p.lse[qrow] = (ltot > 0.f) ? (m[rg] + log2f(ltot)) * 0.69314718055994531f : -CUDART_INF_F;
                        } else {
                            p.ws_ml[prow] = make_float2(m[rg], ltot);
                        }
                    }
                }
                tc::fence_before_sync();
            }
            ++i;
        }
        if (ok) walker.finish(write_empty);
    }

    __syncthreads();
    // No CTA finishes before the preceding grid (CTAs without loads included).
    if (p.early && tid == 0) pdl_wait();
    if (*abort_flag && tid == 0 && p.status) atomicOr(p.status, KVD_STATUS_TIMEOUT);
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Sh::TMEM_COLS);
    }
}

}  // namespace kvd
