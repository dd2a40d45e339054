// Split-KV chunk kernel on the 5th-generation tensor cores (tcgen05), for wide
// query-head groups (17..64 query heads per KV head: multiquery and wide
// grouped-query attention).
//
// Same schedule, same outputs and same partial-state format as the mma.sync
// chunk kernel (split_kv_chunk.cuh); only the engine differs. Per 64-token
// tile of one (sequence, KV head) pair:
//   S  = Q K^T      tcgen05.mma, M = 64 query heads (group padded to 64),
//                   N = 64 tokens, K = head_dim; fp32 accumulator in TMEM
//   P  = 2^(S*scale*log2e - m)   four softmax warps, one query head per thread
//   O += P V        tcgen05.mma, M = 64, N = head_dim, K = 64 tokens; O in TMEM
// Operands never pass through registers: TMA writes K, V and Q tiles into
// 128-byte-swizzled shared memory, and the MMAs read them there, so each K/V
// byte crosses shared memory once (the mma.sync kernel re-reads it once per
// 16-head tile). The online softmax follows the log-sum-exp accumulation of
// sequence-sharded KV (All About Transformer Inference, "Sharding the KV
// cache") in base 2 (Efficiently Scaling Transformer Inference, section 3.5).
// The running maximum m used for the exponentials is only raised when a tile's
// maximum exceeds it by more than 2^8 (weights stay <= 256, exact in fp32), so
// rescaling O in TMEM is rare; the result is identical in exact arithmetic
// because O and l always share the same m.
//
// Warp roles (14 warps): 0 = TMA producer for K, 2 = TMA producer for V,
// 13 = TMA loader for Q at each new pair, 1 and 11 = S issuers (one thread
// each, one half of head_dim each; warp 1 also owns TMEM), 12 = O issuer, 3..10 = softmax /
// rescale / epilogue (two warps per TMEM lane quarter w % 4, splitting the
// token columns of S and the output columns of O).
// Pipelines: K ring of KST stages, V ring of VST stages, two S buffers in
// TMEM, two P buffers in shared memory, one Q buffer, O in TMEM. Every wait is
// bounded; a timeout flags KVD_STATUS_TIMEOUT and all roles wind down.
#pragma once

#include <math_constants.h>

#include "../../include/kvdecode.h"
#include "common.cuh"
#include "params.h"
#include "schedule.cuh"
#include "split_kv_chunk.cuh"  // DevLen, NoOp, block scans
#include "tc_common.cuh"

namespace kvd {

template <int D, bool F32OUT, int QR>
struct TcShape {
    static constexpr int T = 64;                 // tokens per tile
    // Schedule: runs balanced in whole tiles (a tile's time is set by the
    // pipeline's latency, whatever its length), plus one tile's charge for
    // starting a pair inside a run (its Q load and first K tile).
    static constexpr int SEG_UNIT = T;
    static constexpr int SEG_COST = 1;
    static constexpr int KB = D / 64;            // 128-byte swizzle atoms across head_dim
    static constexpr int TILE_BYTES = T * D * 2; // one K (or V) tile
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
    static constexpr int P_BYTES = 64 * T * 2;   // one P buffer (64 rows x 64 tokens)
    static constexpr int NP = F32OUT ? 2 : 1;    // hi (and lo) parts of P
    // Stage counts: three V stages (a V stage is held until P V of its tile is
    // done, so the V ring needs the depth), K stages as the budget allows.
    static constexpr int VST = D == 256 ? 3 : (D == 128 ? 6 : 8);
    static constexpr int BUDGET = 224 * 1024 - Q_BYTES - NP * P_BYTES - VST * TILE_BYTES;
    static constexpr int KST_FIT = BUDGET / TILE_BYTES;
    static constexpr int KST = KST_FIT > 8 ? 8 : KST_FIT;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + KST * TILE_BYTES;
    static constexpr int OFF_P = OFF_V + VST * TILE_BYTES;
    static constexpr int OFF_BAR = OFF_P + NP * P_BYTES;
    // barriers: k_full, k_empty [KST]; v_full, v_empty [VST]; q_full, q_empty [NQ];
    // s_full, s_free, p_full, o_fin [2]; mma_done; xbar [4]
    static constexpr int NBAR = 2 * KST + 2 * VST + 2 * NQ + 8 + 1 + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // tmem base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int STATIC_SMEM = 2048;  // block scans and the exchange buffer (checked by ptxas -v)
    static constexpr int TMEM_S = 0;             // S, first head_dim half: columns 0 and T
    static constexpr int TMEM_S2 = 2 * T;        // S, second half: columns 2T and 3T
    static constexpr int TMEM_O = 4 * T;         // O at columns [4T, 4T + D)
    static constexpr int TMEM_COLS = (4 * T + D) <= 256 ? 256 : 512;
    // producers 0 (K) and 2 (V), S issuers 1 and 11, O issuer 12, Q loader 13, softmax 3..10
    static constexpr int NWARPS = 14;
    static constexpr int THREADS = NWARPS * 32;
    static_assert(KST >= 2, "need at least two K stages");
    static_assert(SMEM_BYTES + STATIC_SMEM <= 227 * 1024, "shared memory budget");
    static_assert(QR % 8 == 0 && QR <= 64, "Q rows per block");
    static_assert(4 * T + D <= 512, "TMEM columns");
};

struct TcMaps {
    CUtensorMap q;  // 2D: [B*Hq rows, D] box (64, G), 128-byte swizzle
    CUtensorMap k;  // 3D: [B*S_max, Hkv, D] box (64, 1, 64), 128-byte swizzle
    CUtensorMap v;
};

template <int D, bool F32OUT, int QR>
__global__ void __launch_bounds__(TcShape<D, F32OUT, QR>::THREADS, 1)
    split_kv_chunk_tc_kernel(const DecodeParams p, const __grid_constant__ TcMaps maps) {
    using Sh = TcShape<D, F32OUT, QR>;
    constexpr int T = Sh::T, KB = Sh::KB, KST = Sh::KST, VST = Sh::VST, NW = Sh::NWARPS,
                  SEG_COST = Sh::SEG_COST;
    constexpr long long kBudget = 4000000000LL;  // ~2 s of clock cycles per wait

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ long long s_red[NW];
    __shared__ int s_redi[NW];
    __shared__ long long s_cum0;
    __shared__ float xbuf[2 * 4 * 32];  // [exchange parity][quarter][half][16 rows]

    uint8_t* smem = smem_raw;  // 1024-byte aligned (128-byte swizzle atoms need it)
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + Sh::OFF_Q, sK = sbase + Sh::OFF_K, sV = sbase + Sh::OFF_V,
                   sP = sbase + Sh::OFF_P, sBar = sbase + Sh::OFF_BAR;
    auto k_full = [&](int s) { return sBar + 8u * s; };
    auto k_empty = [&](int s) { return sBar + 8u * (KST + s); };
    auto v_full = [&](int s) { return sBar + 8u * (2 * KST + s); };
    auto v_empty = [&](int s) { return sBar + 8u * (2 * KST + VST + s); };
    constexpr int NQ = Sh::NQ;
    auto q_full = [&](int s) { return sBar + 8u * (2 * KST + 2 * VST + s); };
    auto q_empty = [&](int s) { return sBar + 8u * (2 * KST + 2 * VST + NQ + s); };
    const uint32_t sBar2 = sBar + 8u * (2 * KST + 2 * VST + 2 * NQ - 1);  // base of the rest
    auto s_full = [&](int b) { return sBar2 + 8u * (1 + b); };
    auto s_free = [&](int b) { return sBar2 + 8u * (3 + b); };
    auto p_full = [&](int b) { return sBar2 + 8u * (5 + b); };
    // o_fin[i & 1] completes when O += P(i) V(i) has finished. One barrier per
    // P buffer (rather than one for all tiles) keeps every waiter within one
    // phase of the completion it waits for, so parity waits are unambiguous.
    auto o_fin = [&](int b) { return sBar2 + 8u * (7 + b); };
    const uint32_t mma_done = sBar2 + 8u * 9;
    auto xbar = [&](int q) { return sBar2 + 8u * (10 + q); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sh::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sh::OFF_MISC + 8);
    // The P buffer, part 0 = hi, 1 = lo. One buffer: P(i) is written only once
    // P(i-1) V(i-1) has completed.
    auto p_buf = [&](int /*tile parity*/, int part) { return sP + (uint32_t)(part * Sh::P_BYTES); };

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
        for (int s = 0; s < KST; ++s) {
            tc::mbar_init(k_full(s), 1);
            tc::mbar_init(k_empty(s), 2);  // both S issuers
        }
        for (int s = 0; s < VST; ++s) {
            tc::mbar_init(v_full(s), 1);
            tc::mbar_init(v_empty(s), 1);
        }
        for (int s = 0; s < NQ; ++s) {
            tc::mbar_init(q_full(s), 1);
            tc::mbar_init(q_empty(s), 2);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(s_full(b), 2);
            tc::mbar_init(s_free(b), 8);
            tc::mbar_init(p_full(b), 8);
            tc::mbar_init(o_fin(b), 1);
        }
        tc::mbar_init(mma_done, 3);  // S issuers and O issuer
        for (int q = 0; q < 4; ++q) tc::mbar_init(xbar(q), 2);
        *abort_flag = 0;
        tc::mbar_fence_init();
    }
    // Rows of Q past the group, and P rows of padded heads, stay zero.
    for (int i = tid; i < Sh::Q_BYTES / 16; i += Sh::THREADS)
        reinterpret_cast<uint4*>(smem + Sh::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < Sh::NP * Sh::P_BYTES / 16; i += Sh::THREADS)
        reinterpret_cast<uint4*>(smem + Sh::OFF_P)[i] = make_uint4(0, 0, 0, 0);
    tc::fence_proxy_async_smem();
    if (warp == 1) tc::tmem_alloc(smem_u32(tmem_slot), Sh::TMEM_COLS);

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
    // ---- total work, this CTA's run, first sequence (as in the mma.sync kernel) ----
    long long total;
    int C_eff, b0 = p.B;
    bool has_work;
    long long S, cum0;
    if (p.B <= Sh::THREADS) {
        // One pass (the common case), one sequence per thread: an inclusive
        // scan gives both the total and each sequence's start; the first
        // sequence touching the run is the first candidate, and its start is
        // the smallest candidate start (starts never decrease with b).
        const int b = tid;
        int L = 0;
        if (b < p.B) {
            const int raw = __ldg(p.seq_lens + b / vt);
            L = len(b);
            if (raw != clamp_len(raw, p.len_cap) && c == 0 && p.status) atomicOr(p.status, KVD_STATUS_SEQ_LEN_CLAMPED);
        }
        const long long e = pair_extent(L, Geo{});
        const long long v = e * p.Hkv;
        const long long cs = block_incl_scan_ll<NW>(v, s_red, &total) - v;  // also orders the set-up
        C_eff = effective_ctas(p.n_split, total);
        has_work = c < C_eff;
        S = has_work ? run_begin(c, C_eff, total) : total;
        cum0 = total;
        if (has_work) {
            const bool cand = (b < p.B) && is_first_seq_candidate(cs, e, p.Hkv, S);
            int bi = cand ? b : 0x7fffffff;
            long long ci = cand ? cs : 0x7fffffffffffffffLL;
            block_min_int_ll<NW>(bi, ci, s_redi, s_red);
            if (bi != 0x7fffffff) {
                b0 = bi;
                cum0 = ci;
            }
        }
    } else {
        long long mine = 0;
        bool clamped = false;
        for (int b = tid; b < p.B; b += Sh::THREADS) {
            const int raw = __ldg(p.seq_lens + b / vt);
            clamped |= (raw != clamp_len(raw, p.len_cap));
            mine += pair_extent(len(b), Geo{});
        }
        if (clamped && c == 0 && p.status) atomicOr(p.status, KVD_STATUS_SEQ_LEN_CLAMPED);
        total = block_sum_ll<NW>(mine, s_red) * p.Hkv;  // also orders the set-up
        C_eff = effective_ctas(p.n_split, total);
        has_work = c < C_eff;
        S = has_work ? run_begin(c, C_eff, total) : total;
        cum0 = total;
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
    }
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    Walker<DevLen, Geo> walker(len, Geo{}, p.B, p.Hkv, c, has_work ? C_eff : c + 1, has_work ? total : 0);
    walker.start(b0, cum0);

    if (!has_work) {
        // no tokens for this CTA: fall through to the common exit (TMEM release)
    } else if (warp == 0 || warp == 2) {
        // ===================== TMA producers =====================
        if (lane == 0) {
            const bool is_k = (warp == 0);
            const uint64_t pol_kv = l2_evict_first_policy();
            Tile t;
            int j = 0;
            const int NS = is_k ? KST : VST;
            const CUtensorMap* map = is_k ? &maps.k : &maps.v;
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
                const uint32_t full = is_k ? k_full(s) : v_full(s);
                const uint32_t empty = is_k ? k_empty(s) : v_empty(s);
                if (!tc::mbar_wait(empty, ((j / NS) & 1) ^ 1, abort_flag, kBudget)) break;
                tc::mbar_arrive_expect_tx(full, (uint32_t)Sh::TILE_BYTES);
                const uint32_t dst = (is_k ? sK : sV) + (uint32_t)(s * Sh::TILE_BYTES);
                if (!paged) {
                    const int row = (t.b / vt) * p.S_max + t.tok_lo;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tc::tma_load_3d(dst + kb * Sh::KB_BYTES, map, kb * 64, t.h, row, full, pol_kv);
                } else {
                    // Paged cache: the tile is fetched as boxes of box_rows
                    // tokens (the page size, up to the tile), each from its
                    // block's page. Tile rows are page-aligned (tiles start at
                    // multiples of T within a sequence, and a page is at least
                    // 16 tokens), so no box crosses a page. A box past the
                    // tile's tokens, or whose table entry names no page, is
                    // read from past the pool's end: zeros.
                    const int32_t* table = p.block_table + (size_t)(t.b / vt) * p.max_blocks;
                    const int oob = p.num_pages << p.page_shift;
                    for (int r0 = 0; r0 < T; r0 += box_rows) {
                        const int tok = t.tok_lo + r0;
                        int row = oob;
                        if (tok < t.tok_hi) {
                            const int page = __ldg(table + (tok >> p.page_shift));
                            if ((unsigned)page < (unsigned)p.num_pages)
                                row = (page << p.page_shift) + (tok & ((1 << p.page_shift) - 1));
                            else if (is_k && p.status)
                                atomicOr(p.status, KVD_STATUS_BAD_PAGE);
                        }
#pragma unroll
                        for (int kb = 0; kb < KB; ++kb)
                            tc::tma_load_3d(dst + kb * Sh::KB_BYTES + r0 * 128, map, kb * 64, t.h, row, full, pol_kv);
                    }
                }
                ++j;
            }
            // Do not leave with copies in flight: wait for the last loads to land.
            for (int jj = (j > NS ? j - NS : 0); jj < j; ++jj) {
                const int s = jj % NS;
                tc::mbar_wait(is_k ? k_full(s) : v_full(s), (jj / NS) & 1, abort_flag, kBudget / 4);
            }
        }
    } else if (warp == 13) {
        // ===================== Q loader =====================
        // Its own thread, so that waiting for the Q slot (free once the previous
        // pair's last S is done) never holds up the K stream. When the run goes
        // on into a next pair, that pair's Q rows are also prefetched into L2,
        // so its load is short when its turn comes.
        if (lane == 0) {
            const uint64_t pol_q = tc::l2_evict_last_policy();
            Tile t;
            int qn = 0;
            while (walker.next(t, NoOp{})) {
                if (!t.seg_start) continue;
                const int qs = qn % NQ;
                if (!tc::mbar_wait(q_empty(qs), ((qn / NQ) & 1) ^ 1, abort_flag, kBudget)) break;
                tc::mbar_arrive_expect_tx(q_full(qs), (uint32_t)(KB * 128 * G));
                const int qrow = t.b * p.Hq + t.h * G;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    tc::tma_load_2d(sQ + qs * Sh::QS_BYTES + kb * Sh::QB_BYTES, &maps.q, kb * 64, qrow, q_full(qs),
                                    pol_q);
                ++qn;
                if (walker.pstart + walker.ext() < walker.E) {
                    const int nh = (t.h + 1 < p.Hkv) ? t.h + 1 : 0;
                    const int nb = (t.h + 1 < p.Hkv) ? t.b : t.b + 1;
                    if (nb < p.B)
                        tc::prefetch_l2(reinterpret_cast<const uint8_t*>(p.q) + ((size_t)nb * p.Hq + (size_t)nh * G) * D * 2,
                                        (uint32_t)(G * D * 2));
                }
            }
            if (qn > 0) tc::mbar_wait(q_full((qn - 1) % NQ), ((qn - 1) / NQ) & 1, abort_flag, kBudget / 4);
        }
    } else if (warp == 1 || warp == 11) {
        // ===================== S issuers (one thread each) =====================
        // S = Q K^T is issued as two independent accumulations over the two
        // halves of head_dim, by two threads into two TMEM buffers that the
        // softmax adds: a tcgen05.mma of this shape costs its issuing thread
        // about as long as the tensor core needs for two of them, so two
        // issuers finish a tile's S in half the time and release its K stage
        // sooner.
        if (lane == 0) {
            const int kh = (warp == 11) ? 1 : 0;
            constexpr int KH = D / 32;  // k-steps per half
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(64, T, false, false);
            const uint32_t s_base = tmem + (kh ? Sh::TMEM_S2 : Sh::TMEM_S);
            Tile t;
            int i = 0, qn = 0;
            while (walker.next(t, NoOp{})) {
                const int sk = i % KST, sb = i & 1;
                if (t.seg_start) {
                    if (!tc::mbar_wait(q_full(qn % NQ), (qn / NQ) & 1, abort_flag, kBudget)) break;
                    ++qn;
                }
                const int qs = (qn - 1) % NQ;
                if (!tc::mbar_wait(k_full(sk), (i / KST) & 1, abort_flag, kBudget)) break;
                if (!tc::mbar_wait(s_free(sb), ((i >> 1) & 1) ^ 1, abort_flag, kBudget)) break;
                tc::fence_after_sync();
                const uint32_t qt = sQ + (uint32_t)(qs * Sh::QS_BYTES);
                const uint32_t kt = sK + (uint32_t)(sk * Sh::TILE_BYTES);
#pragma unroll
                for (int k = 0; k < KH; ++k) {
                    const int kk = kh * KH + k;
                    const uint64_t a = tc::sdesc_sw128(qt + (kk >> 2) * Sh::QB_BYTES + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = tc::sdesc_sw128(kt + (kk >> 2) * Sh::KB_BYTES + (kk & 3) * 32, 16, 1024);
                    tc::mma_bf16(s_base + sb * T, a, b, idesc_s, k > 0);
                }
                tc::mma_commit(s_full(sb));
                tc::mma_commit(k_empty(sk));
                if (t.seg_end) tc::mma_commit(q_empty(qs));
                ++i;
            }
            // This thread's tensor-core work done before TMEM is released.
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, abort_flag, kBudget);
        }
    } else if (warp == 12) {
        // ===================== O issuer (one thread) =====================
        if (lane == 0) {
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(64, D, false, true);
            Tile t;
            int i = 0;
            while (walker.next(t, NoOp{})) {
                const int sv = i % VST, sb = i & 1;
                if (!tc::mbar_wait(v_full(sv), (i / VST) & 1, abort_flag, kBudget)) break;
                if (!tc::mbar_wait(p_full(sb), (i >> 1) & 1, abort_flag, kBudget)) break;
                tc::fence_after_sync();
                const uint32_t vt = sV + (uint32_t)(sv * Sh::TILE_BYTES);
#pragma unroll
                for (int k2 = 0; k2 < T / 16; ++k2) {
                    const uint64_t b = tc::sdesc_sw128(vt + k2 * 2048, Sh::KB_BYTES, 1024);
#pragma unroll
                    for (int part = 0; part < Sh::NP; ++part) {
                        const uint64_t a = tc::sdesc_sw128(p_buf(sb, part) + k2 * 32, 16, 1024);
                        tc::mma_bf16(tmem + Sh::TMEM_O, a, b, idesc_o, (t.seg_start && k2 == 0 && part == 0) ? 0u : 1u);
                    }
                }
                tc::mma_commit(v_empty(sv));
                tc::mma_commit(o_fin(sb));
                ++i;
            }
            tc::mma_commit(mma_done);
            tc::mbar_wait(mma_done, 0, abort_flag, kBudget);
        }
    } else {
        // ===================== softmax / epilogue (warps 3..10) =====================
        // Two warps serve each TMEM lane quarter (a warp reaches the 32 lanes
        // 32 * (warp % 4) ...): the warp of half 0 takes token columns [0, 32)
        // of every S tile and output columns [0, D/2), the other the upper
        // halves. Row maxima and row sums are exchanged between the two through
        // shared memory, synchronised by a two-arrival mbarrier per quarter
        // (bounded waits, so an abort cannot strand the partner warp).
        constexpr int HT = T / 2;   // token columns per half
        constexpr int HD = D / 2;   // output columns per half
        const int sw = warp - 3;    // 0..7
        const int quarter = warp & 3;
        const int half = sw >> 2;
        // Lane layout of the epilogue (32x32b TMEM shape): lanes 0..15 hold rows.
        const int row = quarter * 16 + lane;   // group-local query head of this lane
        const bool has_row = lane < 16;
        const bool active = has_row && row < G;
        const int st = tid - 3 * 32;           // 0..255 among the softmax threads
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const float scale_log2 = p.scale_log2;
        int nx = 0;  // exchanges done with the partner warp

        auto write_empty = [&](int b, int h) {
            const size_t r0 = (size_t)b * p.Hq + (size_t)h * G;
            if constexpr (F32OUT) {
                float* o = reinterpret_cast<float*>(p.out) + r0 * D;
                for (int i2 = st; i2 < G * D; i2 += 256) o[i2] = 0.f;
            } else {
                __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + r0 * D;
                for (int i2 = st; i2 < G * D; i2 += 256) o[i2] = __float2bfloat16_rn(0.f);
            }
            if (p.lse)
                for (int i2 = st; i2 < G; i2 += 256) p.lse[r0 + i2] = -CUDART_INF_F;
        };

        // S is read with the 16x256b TMEM shape, which puts the quarter's 16
        // rows on all 32 threads in the mma accumulator layout: thread t holds
        // rows rA = t/4 and rB = t/4 + 8 of the quarter, columns 8g + 2(t%4) + 0..1
        // of each 8-column group g of its half. Row statistics are reduced over
        // the 4 threads of a quad, then with the partner warp (other half).
        const int rA = quarter * 16 + (lane >> 2), rB = rA + 8;
        const bool actA = rA < G, actB = rB < G;
        // Exchange two per-row floats (rows rA, rB) with the partner warp.
        auto exchange2 = [&](float va, float vb, float& oa, float& ob, bool& ok_) {
            float* buf = xbuf + ((nx & 1) * 4 + quarter) * 32;
            if ((lane & 3) == 0) {
                buf[half * 16 + (lane >> 2)] = va;
                buf[half * 16 + 8 + (lane >> 2)] = vb;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(xbar(quarter));
            ok_ = __all_sync(0xffffffffu, tc::mbar_wait(xbar(quarter), nx & 1, abort_flag, kBudget));
            oa = buf[(half ^ 1) * 16 + (lane >> 2)];
            ob = buf[(half ^ 1) * 16 + 8 + (lane >> 2)];
            ++nx;
        };
        // Per-row value of the quad layout moved to the lane layout (lane = row, lanes 0..15).
        auto to_lane = [&](float a, float b) {
            const float xa = __shfl_sync(0xffffffffu, a, (lane & 7) * 4);
            const float xb = __shfl_sync(0xffffffffu, b, (lane & 7) * 4);
            return (lane & 8) ? xb : xa;
        };

        float mA = 0.f, mB = 0.f;  // running maxima of rows rA, rB
        float lA = 0.f, lB = 0.f;  // this thread's share of the row sums
        Tile t;
        int i = 0;
        bool ok = true;
        while (ok && walker.next(t, write_empty)) {
            const int sb = i & 1;
            ok = __all_sync(0xffffffffu, tc::mbar_wait(s_full(sb), (i >> 1) & 1, abort_flag, kBudget));
            if (!ok) break;
            tc::fence_after_sync();
            __syncwarp();
            // S is held as two partial sums over the halves of head_dim.
            uint32_t sr[16], sr2[16];
            tc::tmem_ld_16x256b_x4(tmem + lane_base + Sh::TMEM_S + sb * T + half * HT, sr);
            tc::tmem_ld_16x256b_x4(tmem + lane_base + Sh::TMEM_S2 + sb * T + half * HT, sr2);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(s_free(sb));

            // Scores in base-2 units; columns past the tile's last token masked.
            const int nvalid = t.tok_hi - t.tok_lo;
            const int nv = nvalid - half * HT;  // valid columns of this half (may be <= 0)
            float s[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int col = 8 * (e >> 2) + 2 * (lane & 3) + (e & 1);
                s[e] = (col < nv) ? (__uint_as_float(sr[e]) + __uint_as_float(sr2[e])) * scale_log2 : -CUDART_INF_F;
            }
            float xA = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[4], s[5]));
            float xB = fmaxf(fmaxf(s[2], s[3]), fmaxf(s[6], s[7]));
            xA = fmaxf(xA, fmaxf(fmaxf(s[8], s[9]), fmaxf(s[12], s[13])));
            xB = fmaxf(xB, fmaxf(fmaxf(s[10], s[11]), fmaxf(s[14], s[15])));
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 1));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 1));
            xA = fmaxf(xA, __shfl_xor_sync(0xffffffffu, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(0xffffffffu, xB, 2));
            float oA, oB;
            exchange2(xA, xB, oA, oB, ok);
            if (!ok) break;
            const float mtA = fmaxf(xA, oA), mtB = fmaxf(xB, oB);

            bool needA = false, needB = false;
            float alphaA = 1.f, alphaB = 1.f;
            if (t.seg_start) {
                mA = mtA;
                mB = mtB;
                if (p.umax) {
                    // Unified maximum (FlashDecoding++'s asynchronized softmax):
                    // a row whose first tile's maximum lies within [phi - 64,
                    // phi + 8] (base 2) takes m = phi, shared by all partials of
                    // such rows, so the merge reduces to plain sums; otherwise
                    // it starts from its own maximum. The lazy rescale below
                    // moves m up past phi + 8 (exact either way).
                    const float phi2 = p.umax_phi2;
                    if (mtA >= phi2 - 64.f && mtA <= phi2 + 8.f) mA = phi2;
                    if (mtB >= phi2 - 64.f && mtB <= phi2 + 8.f) mB = phi2;
                    if (((actA && mA != phi2) || (actB && mB != phi2)) && p.status)
                        atomicOr(p.status, KVD_STATUS_UMAX_FALLBACK);
                }
                lA = lB = 0.f;
            } else {
                if (mtA > mA + 8.f) {
                    needA = true;
                    alphaA = exp2f(mA - mtA);
                    mA = mtA;
                }
                if (mtB > mB + 8.f) {
                    needB = true;
                    alphaB = exp2f(mB - mtB);
                    mB = mtB;
                }
                if (p.umax && ((actA && needA) || (actB && needB)) && p.status)
                    atomicOr(p.status, KVD_STATUS_UMAX_FALLBACK);
            }
            // P = 2^(s - m), packed per row and 8-column group (bf16 hi part; lo
            // part for fp32 output).
            uint32_t hiA[4], hiB[4], loA[4], loB[4];
            float lsA = 0.f, lsB = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float e0 = actA ? tc::ex2_approx(s[4 * g] - mA) : 0.f;
                const float e1 = actA ? tc::ex2_approx(s[4 * g + 1] - mA) : 0.f;
                const float e2 = actB ? tc::ex2_approx(s[4 * g + 2] - mB) : 0.f;
                const float e3 = actB ? tc::ex2_approx(s[4 * g + 3] - mB) : 0.f;
                hiA[g] = pack_bf16x2(e0, e1);
                hiB[g] = pack_bf16x2(e2, e3);
                if constexpr (F32OUT) {
                    loA[g] = pack_bf16x2(e0 - bf16_lo(hiA[g]), e1 - bf16_hi(hiA[g]));
                    loB[g] = pack_bf16x2(e2 - bf16_lo(hiB[g]), e3 - bf16_hi(hiB[g]));
                    lsA += e0 + e1;
                    lsB += e2 + e3;
                } else {
                    // The weights actually multiplied into V are the rounded ones;
                    // summing those keeps the output an exact convex combination.
                    lsA += bf16_lo(hiA[g]) + bf16_hi(hiA[g]);
                    lsB += bf16_lo(hiB[g]) + bf16_hi(hiB[g]);
                }
            }

            // O += P(i-1) V(i-1) must have completed: it reads the P buffer, and O
            // is rescaled below if the running maximum moved.
            if (i > 0) {
                ok = __all_sync(0xffffffffu, tc::mbar_wait(o_fin((i - 1) & 1), ((i - 1) >> 1) & 1, abort_flag, kBudget));
                if (!ok) break;
                tc::fence_after_sync();
            }
            if (__any_sync(0xffffffffu, needA || needB)) {
                // O rows sit one per TMEM lane (lanes 0..15 of the quarter).
                const float alpha = to_lane(alphaA, alphaB);
#pragma unroll 1
                for (int cc = 0; cc < HD / 32; ++cc) {
                    uint32_t r[32];
                    const uint32_t ta = tmem + lane_base + Sh::TMEM_O + half * HD + cc * 32;
                    __syncwarp();
                    tc::tmem_ld32(ta, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                    tc::tmem_st32(ta, r);
                }
                tc::tmem_wait_st();
            }
            lA = lA * alphaA + lsA;
            lB = lB * alphaB + lsB;
            {
                // Thread t addresses row t % 8 of matrix t / 8 (= 8-column group).
                const int rin = lane & 7, gq = lane >> 3;
                const uint32_t offA = (uint32_t)((quarter * 16 + rin) * 128 + (((half * 4 + gq) ^ rin) * 16));
                const uint32_t offB = offA + 8 * 128;
                stmatrix_x4(p_buf(sb, 0) + offA, hiA[0], hiA[1], hiA[2], hiA[3]);
                stmatrix_x4(p_buf(sb, 0) + offB, hiB[0], hiB[1], hiB[2], hiB[3]);
                if constexpr (F32OUT) {
                    stmatrix_x4(p_buf(sb, 1) + offA, loA[0], loA[1], loA[2], loA[3]);
                    stmatrix_x4(p_buf(sb, 1) + offB, loB[0], loB[1], loB[2], loB[3]);
                }
            }
            if (nvalid < T) {
                // Rows past the sequence's end came from the cache's padding (or the
                // next sequence): zero them so that 0-weights never meet NaN.
                const int sv = i % VST;
                ok = __all_sync(0xffffffffu, tc::mbar_wait(v_full(sv), (i / VST) & 1, abort_flag, kBudget));
                if (!ok) break;
                uint8_t* vt = smem + Sh::OFF_V + sv * Sh::TILE_BYTES;
                const int n16 = (T - nvalid) * KB * 8;
                for (int idx = st; idx < n16; idx += 256) {
                    const int r = nvalid + idx / (KB * 8);
                    const int rem = idx % (KB * 8);
                    *reinterpret_cast<uint4*>(vt + (rem >> 3) * Sh::KB_BYTES + r * 128 + (rem & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(p_full(sb));

            if (t.seg_end) {
                float qA = lA + __shfl_xor_sync(0xffffffffu, lA, 1);
                float qB = lB + __shfl_xor_sync(0xffffffffu, lB, 1);
                qA += __shfl_xor_sync(0xffffffffu, qA, 2);
                qB += __shfl_xor_sync(0xffffffffu, qB, 2);
                float pA, pB;
                exchange2(qA, qB, pA, pB, ok);
                if (!ok) break;
                // The epilogue works in the lane layout: this lane's row (lanes 0..15).
                const float ltot = to_lane(qA + pA, qB + pB);
                const float m_row = to_lane(mA, mB);
                ok = __all_sync(0xffffffffu, tc::mbar_wait(o_fin(sb), (i >> 1) & 1, abort_flag, kBudget));
                if (!ok) break;
                tc::fence_after_sync();
                const size_t pair = (size_t)t.b * p.Hkv + t.h;
                const size_t qrow = (size_t)t.b * p.Hq + (size_t)t.h * G + row;
                const size_t slot = (size_t)c + pair;
                // O is read with the 16x256b shape as well, so every thread holds
                // two rows (rA, rB) and 2 adjacent columns of each 8-column group:
                // a quad writes 32 contiguous bytes of a row (one full sector).
                const float totA = qA + pA, totB = qB + pB;
                const float invA = t.full ? ((totA > 0.f) ? 1.f / totA : 0.f) : 1.f;
                const float invB = t.full ? ((totB > 0.f) ? 1.f / totB : 0.f) : 1.f;
                const size_t grow = t.full ? (size_t)t.b * p.Hq + (size_t)t.h * G : slot * G;  // row of head 0
#pragma unroll 1
                for (int cc = 0; cc < HD / 32; ++cc) {
                    const int col0 = half * HD + cc * 32 + 2 * (lane & 3);
                    uint32_t r[16];
                    __syncwarp();
                    tc::tmem_ld_16x256b_x4(tmem + lane_base + Sh::TMEM_O + half * HD + cc * 32, r);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int col = col0 + 8 * g;
                        const float a0 = __uint_as_float(r[4 * g]) * invA, a1 = __uint_as_float(r[4 * g + 1]) * invA;
                        const float b0 = __uint_as_float(r[4 * g + 2]) * invB, b1 = __uint_as_float(r[4 * g + 3]) * invB;
                        if (t.full && !F32OUT) {
                            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out);
                            if (actA) *reinterpret_cast<uint32_t*>(o + (grow + rA) * D + col) = pack_bf16x2(a0, a1);
                            if (actB) *reinterpret_cast<uint32_t*>(o + (grow + rB) * D + col) = pack_bf16x2(b0, b1);
                        } else {
                            float* o = t.full ? reinterpret_cast<float*>(p.out) : p.ws_o;
                            if (actA) *reinterpret_cast<float2*>(o + (grow + rA) * D + col) = make_float2(a0, a1);
                            if (actB) *reinterpret_cast<float2*>(o + (grow + rB) * D + col) = make_float2(b0, b1);
                        }
                    }
                }
                tc::fence_before_sync();
                if (active && half == 0) {
                    if (t.full) {
                        if (p.lse) p.lse[qrow] = (m_row + log2f(ltot)) * 0.69314718055994531f;
                    } else {
                        p.ws_ml[slot * G + row] = make_float2(m_row, ltot);
                    }
                }
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
