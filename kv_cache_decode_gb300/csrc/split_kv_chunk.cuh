// Split-KV chunk kernel: each CTA streams its run of the KV cache once and
// computes, for the whole query-head group of every pair it touches, the
// partial softmax state (running max m, sum of exponentials l, unnormalised
// weighted sum of V rows o), writing either the final output (pairs it covers
// entirely) or the partial state for the merge kernel.
//
// The fused attention follows All About Transformer Inference, "What about
// attention?": read q, read the K and V rows once, q.K, softmax over the
// sequence, weights times V, write the output, with the score matrix never
// leaving the chip. The softmax is taken in base 2 with log2(e) folded into
// the scale (Efficiently Scaling Transformer Inference, section 3.5). The
// running-max update is the online form of the log-sum-exp merge used to
// accumulate sequence-sharded KV (All About Transformer Inference, "Sharding
// the KV cache"). K/V tiles are staged through a multi-buffered shared-memory
// pipeline so loads of later tiles overlap compute on the current one (the
// double-buffering idea of FlashDecoding++'s flat GEMM, here STAGES deep).
//
// Warp layout: HT head tiles of 16 query heads x TS token slices. Warp
// (ht, ts) keeps q rows [16 ht, 16 ht + 16) of the group as mma A fragments in
// registers, computes S = q K^T for tokens [ts*TW, (ts+1)*TW) of every tile
// with m16n8k16 bf16 MMAs (fp32 accumulate), takes the online softmax in
// registers and reuses P directly as the A operand of O += P V. At the end of
// a segment the TS token slices are merged through shared memory.
#pragma once

#include <math_constants.h>

#include "../../include/kvdecode.h"
#include "common.cuh"
#include "params.h"
#include "schedule.cuh"

namespace kvd {

struct NoOp {
    KVD_HD void operator()(int, int) const {}
};

template <int NW>
__device__ __forceinline__ long long block_sum_ll(long long v, long long* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) t += sh[w];
    __syncthreads();
    return t;
}

// Inclusive scan over the block; *total receives the block sum.
template <int NW>
__device__ __forceinline__ long long block_incl_scan_ll(long long v, long long* sh,
                                                        long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        long long n = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += n;
    }
    if (lane == 31) sh[warp] = v;
    __syncthreads();
    long long pre = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w < warp) pre += sh[w];
        tot += sh[w];
    }
    __syncthreads();
    *total = tot;
    return v + pre;
}

template <int NW>
__device__ __forceinline__ int block_min_int(int v, int* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, off));
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    int m = sh[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) m = min(m, sh[w]);
    __syncthreads();
    return m;
}

// Block-wide minimum of an (int, long long) pair, each taken independently.
template <int NW>
__device__ __forceinline__ void block_min_int_ll(int& vi, long long& vl, int* shi, long long* shl) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        vi = min(vi, __shfl_xor_sync(0xffffffffu, vi, off));
        vl = min(vl, __shfl_xor_sync(0xffffffffu, vl, off));
    }
    if (lane == 0) {
        shi[warp] = vi;
        shl[warp] = vl;
    }
    __syncthreads();
    vi = shi[0];
    vl = shl[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
        vi = min(vi, shi[w]);
        vl = min(vl, shl[w]);
    }
    __syncthreads();
}

template <int D, int HT, int TS, int TT, int STAGES, bool KV8 = false>
struct ChunkShape {
    static constexpr int NW = HT * TS;
    static constexpr int NT = NW * 32;
    static constexpr int TW = TT / TS;  // tokens per warp per tile
    static constexpr int NS = TW / 8;   // score n-tiles per warp
    static constexpr int KS = D / 16;   // k-steps over the head dimension
    static constexpr int ND = D / 8;    // output n-tiles (8 columns each)
    static constexpr int CH = D / 8;    // 16-byte chunks per K/V row
    static constexpr int TILE_ELEMS = TT * D;
    // A stage holds a tile's K and V rows: bf16, or (KV8) 8-bit codes followed
    // by the tile's float32 K and V row scales.
    static constexpr int STAGE_BYTES = KV8 ? 2 * TILE_ELEMS + 2 * TT * 4 : 2 * TILE_ELEMS * 2;
    static constexpr int MB_FLOATS_PER_WARP = (ND * 4 + 4) * 32;
    // The token slices are merged at the end of a segment through the stage of
    // the segment's last tile, which every warp has finished reading by then
    // (KV8: through a buffer of their own, an 8-bit stage being too small).
    static constexpr int MB_BYTES = (TS - 1) * HT * MB_FLOATS_PER_WARP * 4;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + (KV8 ? MB_BYTES : 0);
    // Schedule: runs balanced in tokens (the kernel is bandwidth-bound, so a
    // short tile costs less than a full one), no charge per pair (a new pair's
    // queries come from L2 while the previous tiles are still in flight).
    static constexpr int SEG_UNIT = 1;
    static constexpr int SEG_COST = 0;
    static_assert(KV8 || MB_BYTES <= STAGE_BYTES, "warp-merge data must fit in one stage");
    static_assert(!KV8 || TW == 16, "8-bit tiles: one 16-token k-step per warp");
    static_assert(STAGE_BYTES % 128 == 0, "stage alignment");
    static_assert(TW % 16 == 0, "each warp needs whole 16-token k-steps");
    static_assert(D % 16 == 0 && D >= 64, "head_dim");
};

// KV8: the cache holds 8-bit codes (int8, or fp8 E4M3 with FP8) with a
// float32 scale per (token, KV head) row. The codes are staged as they are
// and converted to f16 in registers, straight into the MMAs' B fragments
// (exactly: int8 codes are small integers, and E4M3 codes become their values
// / 256, which f16 holds exactly); q is taken to f16, the MMAs run in f16,
// each score is multiplied by its key row's scale and each weight by its
// value row's scale before P V (FP8: the scores by 256 more, and the output by
// 256 before it is written).
//
// Fragments from 8-bit rows: ldmatrix moves 16-byte rows of 8 threads' bytes
// as 8x8 matrices of 16-bit elements, so a thread receives 4 consecutive codes
// of one row (non-transposed) or 2 codes of each of 2 consecutive rows
// (transposed). The MMA's k index is then mapped to head-dim columns in a
// permuted order that matches those bytes, which a dot product allows as long
// as both operands use it:
// * S = q K^T: within each 16-column chunk, k = 2j, 2j + 1, 2j + 8, 2j + 9 of
//   thread j = lane % 4 are columns 4j .. 4j + 3 (q's A fragment is loaded in
//   the same order);
// * O += P V: the 8 columns of an n-tile are every other head-dim column of a
//   16-column chunk (even tile 2c: columns 16c + 2n, odd tile 2c + 1:
//   16c + 2n + 1), so thread j holds columns 16c + 4j .. 16c + 4j + 3 of its
//   rows across the two tiles, which the output writes put back in order.
// 8-bit rows are staged with 16-byte chunk c of row r at chunk position
// swz8<D>(r, c), so that the 8 rows of an ldmatrix matrix hit 8 distinct
// 16-byte bank groups.
template <int D>
__device__ __forceinline__ int swz8(int r, int c) {
    return D >= 128 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3));
}
// Two 8-bit codes of w (bytes selected by SEL_I8 / SEL_F8 as prmt selectors)
// as one f16x2: int8 codes biased to 0..255 (u = w ^ 0x80808080 given as w),
// placed in the low mantissa bits of 1024.0h and 1152 subtracted; E4M3 codes
// sign-extended to 16 bits, shifted so the exponent and mantissa bits sit at
// the top of an f16's exponent and mantissa (the bias difference of 8 makes
// the f16 equal to the code's value / 256; subnormals map the same way), and
// the sign's copy at bit 14 cleared.
template <bool FP8, uint32_t SEL_I8, uint32_t SEL_F8>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t w) {
    uint32_t a;
    if constexpr (FP8) {
        asm("prmt.b32 %0, %1, 0, %2;" : "=r"(a) : "r"(w), "n"(SEL_F8));
        return (a << 7) & 0xbf80bf80u;
    } else {
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(w), "r"(0x64646464u), "n"(SEL_I8));
        const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
        __half2 h = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int D, int HT, int TS, int TT, int STAGES, bool F32OUT, int MINB, bool PAGED, bool KV8 = false,
          bool FP8 = false>
__global__ void __launch_bounds__(HT* TS * 32, MINB) split_kv_chunk_kernel(const DecodeParams p) {
    static_assert(!FP8 || KV8, "fp8 codes are an 8-bit cache");
    constexpr float OSC = FP8 ? 256.f : 1.f;  // output scale: E4M3 value rows arrive divided by 256
    using Sh = ChunkShape<D, HT, TS, TT, STAGES, KV8>;
    constexpr int NW = Sh::NW, NT = Sh::NT, TW = Sh::TW, NS = Sh::NS, KS = Sh::KS,
                  ND = Sh::ND, CH = Sh::CH, TILE_ELEMS = Sh::TILE_ELEMS, SEG_COST = Sh::SEG_COST;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ long long s_red[NW];
    __shared__ int s_redi[NW];
    __shared__ long long s_cum0;

    __nv_bfloat16* stages = reinterpret_cast<__nv_bfloat16*>(smem);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ht = warp / TS, ts = warp % TS;
    const int G = p.G;
    // T query tokens per sequence (T > 1: a speculative check step): a pair
    // has T * G rows, row r being query token r / G of head r % G, and query
    // token i attends to the first L - T + 1 + i tokens.
    const int T = p.T, TG = T * G;
    // Pairs with more rows than one CTA holds (HT * 16) are split into
    // row_blocks blocks of rows: the CTAs of one token run are launched side by
    // side, one per block, and read the same K/V rows (the later reads mostly
    // from L2). Each writes the outputs or partial-state rows of its block.
    constexpr int ROWS = HT * 16;
    const int c = blockIdx.x / p.row_blocks;
    const int rbase = (blockIdx.x - c * p.row_blocks) * ROWS;
    const int rend = min(TG, rbase + ROWS);
    auto out_row = [&](int b, int h, int r) {  // row of out / lse ([B, T, Hq])
        const int i = r / G;
        return ((size_t)b * T + i) * p.Hq + (size_t)h * G + (r - i * G);
    };

    // Inputs may be produced by the previous kernel on the stream. After this
    // library's append (p.early), only the cache loads need to wait for it.
    if (!p.early) pdl_wait();
    pdl_launch_dependents();

    const DevLen len{p.seq_lens, p.len_cap, 1};  // T query tokens are rows of one pair here
    using Geo = FixedGeom<TT, Sh::SEG_UNIT, SEG_COST>;

    // ---- total work and this CTA's token run ----
    long long mine = 0;
    bool clamped = false;
    for (int b = tid; b < p.B; b += NT) {
        const int raw = __ldg(p.seq_lens + b);
        const int L = clamp_len(raw, p.len_cap);
        clamped |= (raw != L);
        mine += pair_extent(L, Geo{});
    }
    if (clamped && blockIdx.x == 0 && p.status) atomicOr(p.status, KVD_STATUS_SEQ_LEN_CLAMPED);
    const long long total = block_sum_ll<NW>(mine, s_red) * p.Hkv;
    const int C_eff = effective_ctas(p.n_split, total);
    if (c >= C_eff) {
        if (p.early) pdl_wait();  // no CTA finishes before the preceding grid
        return;
    }
    const long long S = run_begin(c, C_eff, total);

    // ---- first sequence touching the run ----
    int b0 = p.B;
    long long cum0 = total;
    {
        long long base = 0;
        for (int chunk = 0; chunk < p.B; chunk += NT) {
            const int b = chunk + tid;
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

    Walker<DevLen, Geo> lw(len, Geo{}, p.B, p.Hkv, c, C_eff, total);
    lw.start(b0, cum0);
    Walker<DevLen, Geo> cw = lw;

    const uint64_t policy = l2_evict_first_policy();
    const __nv_bfloat16* Kg = reinterpret_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* Vg = reinterpret_cast<const __nv_bfloat16*>(p.v);
    const size_t row_stride = (size_t)p.Hkv * D;  // elements between consecutive tokens

    // Issue the cp.async copies of one tile's K and V rows into a stage.
    // Row r of the stage holds token tok_lo + r; its 16-byte chunk ch is
    // stored at chunk position ch ^ (r & 7), so that ldmatrix reads of 8
    // consecutive rows hit 8 distinct bank groups.
    // A paged cache (PAGED) finds each token's row through the block table:
    // row t % page of page table[b][t / page]; a table entry that names no
    // page of the pool gives zero rows (the copy reads 0 bytes) and flags it.
    // The entries of a tile's pages (at most MAXP, pages being at least 16
    // tokens) are staged in shared memory one tile ahead (slot = tile index
    // & 1), so that the copies never wait on a table load.
    // Staged per page: the element offset of the page's first row (for the
    // tile's KV head), or -1 when the entry names no page of the pool.
    constexpr int MAXP = TT / 16 + 1;
    __shared__ long long s_pages[2][MAXP];
    auto page_offset = [&](int b, int blk) -> long long {  // block blk of sequence b
        const int page = __ldg(p.block_table + (size_t)b * p.max_blocks + blk);
        if ((unsigned)page >= (unsigned)p.num_pages) {
            if (p.status) atomicOr(p.status, KVD_STATUS_BAD_PAGE);
            return -1;
        }
        return (long long)(((size_t)page << p.page_shift) * row_stride);
    };
    auto stage_pages = [&](const Tile& t) -> long long {  // this thread's page of tile t (threads < MAXP)
        const int first = t.tok_lo >> p.page_shift, last = (t.tok_hi - 1) >> p.page_shift;
        return (first + tid <= last) ? page_offset(t.b, first + tid) : -1;
    };
    // Each thread copies the same 16-byte chunk ch of its RPT rows of K and
    // of V (a row's address is worked out once for both tensors).
    static_assert(NT % CH == 0 && TT % (NT / CH) == 0, "row split");
    constexpr int RSTEP = NT / CH, RPT = TT / RSTEP;
    constexpr int RUNROLL = RPT >= 16 ? 2 : RPT;  // rows per step (registers allow fewer at head_dim 256)
    auto issue = [&](const Tile& t, int stage, int ps) {
        const int nvalid = t.tok_hi - t.tok_lo;
        const uint32_t sbase = smem_u32(stages) + stage * Sh::STAGE_BYTES;
        const int ch = tid % CH, r0 = tid / CH;
        if constexpr (KV8 && PAGED) {
            // 8-bit rows from their pages (as the bf16 paged rows below), then
            // the row scales: a page's scales start at its first row's element
            // offset / D. An entry that names no page reads zero codes and a
            // zero scale.
            constexpr int CH8 = D / 16, RSTEP8 = NT / CH8, RPT8 = TT / RSTEP8;
            static_assert(NT % CH8 == 0 && TT % RSTEP8 == 0 && NT >= 2 * TT, "int8 row split");
            const int shift = p.page_shift, in_page = (1 << shift) - 1;
            const int first = t.tok_lo >> shift;
            // Each thread copies RPT8 consecutive rows (at most two pages), as
            // the bf16 paged rows below.
            static_assert(RPT8 <= 16, "a thread's rows span at most two pages");
            const int c8 = tid % CH8, rq = (tid / CH8) * RPT8;
            const int tok0 = t.tok_lo + rq;
            const int kb1 = min(RPT8, (((tok0 >> shift) + 1) << shift) - tok0);  // rows on the first page
            const long long po0 = (rq < nvalid) ? s_pages[ps][(tok0 >> shift) - first] : -1;
            const long long po1 = (kb1 < RPT8 && rq + kb1 < nvalid) ? s_pages[ps][(tok0 >> shift) + 1 - first] : -1;
            const long long base0 = po0 + (long long)(tok0 & in_page) * (long long)row_stride;
            const long long base1 = po1 - (long long)kb1 * (long long)row_stride;
            const int8_t* kb = reinterpret_cast<const int8_t*>(p.k) + (size_t)t.h * D + c8 * 16;
            const int8_t* vb = reinterpret_cast<const int8_t*>(p.v) + (size_t)t.h * D + c8 * 16;
#pragma unroll
            for (int k = 0; k < RPT8; ++k) {
                const int r = rq + k;
                const bool second = k >= kb1;
                const bool ok = r < nvalid && (second ? po1 : po0) >= 0;
                const size_t off = ok ? (size_t)((second ? base1 : base0) + (long long)k * (long long)row_stride) : 0;
                const uint32_t dst = sbase + (uint32_t)(r * D + swz8<D>(r, c8) * 16);
                cp_async_16(dst, kb + off, ok ? 16 : 0, policy);
                cp_async_16(dst + TILE_ELEMS, vb + off, ok ? 16 : 0, policy);
            }
            if (tid < 2 * TT) {
                const int r = tid % TT, tok = t.tok_lo + r;
                const long long po = (r < nvalid) ? s_pages[ps][(tok >> shift) - first] : -1;
                const bool ok = po >= 0;
                const float* base = tid < TT ? p.k_scale : p.v_scale;
                const size_t so = ok ? (size_t)po / D + (size_t)(tok & in_page) * p.Hkv + t.h : 0;
                cp_async_4(sbase + 2 * TILE_ELEMS + tid * 4, base + so, ok ? 4 : 0);
            }
        } else if constexpr (KV8) {
            // 8-bit rows: D / 16 chunks of 16 bytes each (chunk c of row r at
            // swz8(r, c)); then the tile's row scales, one 4-byte copy per row
            // and tensor.
            constexpr int CH8 = D / 16, RSTEP8 = NT / CH8, RPT8 = TT / RSTEP8;
            static_assert(NT % CH8 == 0 && TT % RSTEP8 == 0 && NT >= 2 * TT, "int8 row split");
            const size_t row0 = ((size_t)t.b * p.S_max + t.tok_lo) * p.Hkv + t.h;
            const int c8 = tid % CH8, q0 = tid / CH8;
            const int8_t* kb = reinterpret_cast<const int8_t*>(p.k) + row0 * D + c8 * 16;
            const int8_t* vb = reinterpret_cast<const int8_t*>(p.v) + row0 * D + c8 * 16;
#pragma unroll
            for (int k = 0; k < RPT8; ++k) {
                const int r = q0 + k * RSTEP8;
                const bool ok = r < nvalid;
                const size_t off = ok ? (size_t)r * row_stride : 0;
                const uint32_t dst = sbase + (uint32_t)(r * D + swz8<D>(r, c8) * 16);
                cp_async_16(dst, kb + off, ok ? 16 : 0, policy);
                cp_async_16(dst + TILE_ELEMS, vb + off, ok ? 16 : 0, policy);
            }
            if (tid < 2 * TT) {
                const int r = tid % TT;
                const float* sc = (tid < TT ? p.k_scale : p.v_scale) + row0 + (size_t)r * p.Hkv;
                const bool ok = r < nvalid;
                cp_async_4(sbase + 2 * TILE_ELEMS + tid * 4, ok ? sc : p.k_scale, ok ? 4 : 0);
            }
        } else if constexpr (!PAGED) {
            const size_t row0 = ((size_t)t.b * p.S_max + t.tok_lo) * p.Hkv + t.h;
            const __nv_bfloat16* kb = Kg + row0 * D + ch * 8;
            const __nv_bfloat16* vb = Vg + row0 * D + ch * 8;
#pragma unroll(RUNROLL)
            for (int k = 0; k < RPT; ++k) {
                const int r = r0 + k * RSTEP;
                const bool ok = r < nvalid;
                const size_t off = ok ? (size_t)r * row_stride : 0;
                const uint32_t dst = sbase + (uint32_t)((r * D + ((ch ^ (r & 7)) * 8)) * 2);
                cp_async_16(dst, kb + off, ok ? 16 : 0, policy);
                cp_async_16(dst + TILE_ELEMS * 2, vb + off, ok ? 16 : 0, policy);
            }
        } else {
            // Paged: each thread copies RPT consecutive rows, which lie on at
            // most two pages (a page holds at least 16 tokens, RPT <= 16): a
            // row's offset is its page's base plus a multiple of the row
            // stride, with the two page entries read once per tile.
            static_assert(RPT <= 16, "a thread's rows span at most two pages");
            const int shift = p.page_shift, in_page = (1 << shift) - 1;
            const int first = t.tok_lo >> shift;
            const int rq = r0 * RPT;        // this thread's first row
            const int tok0 = t.tok_lo + rq;
            const int kb1 = min(RPT, (((tok0 >> shift) + 1) << shift) - tok0);  // rows on the first page
            const long long po0 = (rq < nvalid) ? s_pages[ps][(tok0 >> shift) - first] : -1;
            const long long po1 = (kb1 < RPT && rq + kb1 < nvalid) ? s_pages[ps][(tok0 >> shift) + 1 - first] : -1;
            // row k: base + k * row_stride, base chosen by page
            const long long base0 = po0 + (long long)(tok0 & in_page) * (long long)row_stride;
            const long long base1 = po1 - (long long)kb1 * (long long)row_stride;
            const __nv_bfloat16* kb = Kg + (size_t)t.h * D + ch * 8;
            const __nv_bfloat16* vb = Vg + (size_t)t.h * D + ch * 8;
#pragma unroll(RUNROLL)
            for (int k = 0; k < RPT; ++k) {
                const int r = rq + k;
                const bool second = k >= kb1;
                const bool ok = r < nvalid && (second ? po1 : po0) >= 0;
                const size_t off = ok ? (size_t)((second ? base1 : base0) + (long long)k * (long long)row_stride) : 0;
                const uint32_t dst = sbase + (uint32_t)((r * D + ((ch ^ (r & 7)) * 8)) * 2);
                cp_async_16(dst, kb + off, ok ? 16 : 0, policy);
                cp_async_16(dst + TILE_ELEMS * 2, vb + off, ok ? 16 : 0, policy);
            }
        }
    };

    // Zero output for an empty pair this CTA owns (its block of rows).
    auto write_empty = [&](int b, int h) {
        for (int i = rbase * D + tid; i < rend * D; i += NT) {
            const size_t e = out_row(b, h, i / D) * D + (i % D);
            if constexpr (F32OUT)
                reinterpret_cast<float*>(p.out)[e] = 0.f;
            else
                reinterpret_cast<__nv_bfloat16*>(p.out)[e] = __float2bfloat16_rn(0.f);
        }
        if (p.lse)
            for (int i = rbase + tid; i < rend; i += NT) p.lse[out_row(b, h, i)] = -CUDART_INF_F;
    };

    // ---- per-warp state ----
    uint32_t qf[KS][4];
    float o[ND][4];
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    // Unified-maximum softmax (bf16 caches): m starts each segment at phi, and
    // an0/an1 record that a row has had a score in it since.
    const bool umax = !KV8 && p.umax;
    const float phi2 = p.umax_phi2;
    bool an0 = false, an1 = false;
#pragma unroll
    for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) qf[kk][0] = qf[kk][1] = qf[kk][2] = qf[kk][3] = 0u;

    const int r0 = rbase + ht * 16 + (lane >> 2);  // pair-local rows of this thread
    const int r1 = r0 + 8;
    const int cq0 = T - 1 - r0 / G, cq1 = T - 1 - r1 / G;  // tokens a row sees fewer than the last
    const float scale_log2 = p.scale_log2;

    // ---- prologue ----
    if (p.early) pdl_wait();  // the appended rows
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        Tile t;
        const bool has = lw.next(t, NoOp{});
        if constexpr (PAGED) {
            if (has && tid < MAXP) s_pages[s & 1][tid] = stage_pages(t);
            __syncthreads();
        }
        if (has) issue(t, s, s & 1);
        cp_async_commit();
    }
    // Paged: the entries of the next tile to issue, loaded a tile ahead.
    long long pg_next = -1;
    auto peek_pages = [&]() {
        if (tid < MAXP) {
            Walker<DevLen, Geo> pk = lw;
            Tile tn;
            pg_next = pk.next(tn, NoOp{}) ? stage_pages(tn) : -1;
        }
    };
    if constexpr (PAGED) {
        peek_pages();
        if (tid < MAXP) s_pages[(STAGES - 1) & 1][tid] = pg_next;
    }

    int it = 0;
    Tile ct;
    while (cw.next(ct, write_empty)) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            Tile t;
            const bool has = lw.next(t, NoOp{});
            if (has) issue(t, (it + STAGES - 1) % STAGES, (it + STAGES - 1) & 1);
            cp_async_commit();
            if constexpr (PAGED) {
                // Inside a segment the next tile starts where this one ends, in
                // the same sequence: its blocks follow directly (read only
                // while they hold tokens of the sequence). Otherwise walk ahead.
                if (has && !t.seg_end) {
                    if (tid < MAXP) {
                        const int blk = (t.tok_hi >> p.page_shift) + tid;
                        pg_next = (((long long)blk << p.page_shift) < t.L) ? page_offset(t.b, blk) : -1;
                    }
                } else {
                    peek_pages();
                }
            }
        }
        const int stage = it % STAGES;
        ++it;

        if (ct.seg_start) {
            const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
            // When the run goes on into another pair, that pair's query rows are
            // brought into L2 now, so that its first loads are short.
            if (tid == 0 && cw.pstart + cw.ext() < cw.E) {
                const int nh = (ct.h + 1 < p.Hkv) ? ct.h + 1 : 0;
                const int nb = (ct.h + 1 < p.Hkv) ? ct.b : ct.b + 1;
                if (nb < p.B)
                    for (int i = 0; i < T; ++i)
                        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(
                                         reinterpret_cast<uint64_t>(qb + (((size_t)nb * T + i) * p.Hq + (size_t)nh * G) * D)),
                                     "r"((uint32_t)(G * D * 2))
                                     : "memory");
            }
            const bool v0 = r0 < TG, v1 = r1 < TG;
            const uint32_t* q0 = reinterpret_cast<const uint32_t*>(qb + (v0 ? out_row(ct.b, ct.h, r0) : 0) * D);
            const uint32_t* q1 = reinterpret_cast<const uint32_t*>(qb + (v1 ? out_row(ct.b, ct.h, r1) : 0) * D);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                if constexpr (KV8) {
                    // k = 2j, 2j + 1 | 2j + 8, 2j + 9 are columns 4j .. 4j + 3 of the chunk
                    const int w = kk * 8 + 2 * (lane & 3);
                    const uint2 a = v0 ? __ldg(reinterpret_cast<const uint2*>(q0 + w)) : make_uint2(0u, 0u);
                    const uint2 b = v1 ? __ldg(reinterpret_cast<const uint2*>(q1 + w)) : make_uint2(0u, 0u);
                    qf[kk][0] = bf16x2_to_f16x2(a.x);
                    qf[kk][1] = bf16x2_to_f16x2(b.x);
                    qf[kk][2] = bf16x2_to_f16x2(a.y);
                    qf[kk][3] = bf16x2_to_f16x2(b.y);
                } else {
                    const int w = kk * 8 + (lane & 3);  // 32-bit word index of column kk*16 + 2*(lane&3)
                    qf[kk][0] = v0 ? __ldg(q0 + w) : 0u;
                    qf[kk][1] = v1 ? __ldg(q1 + w) : 0u;
                    qf[kk][2] = v0 ? __ldg(q0 + w + 4) : 0u;
                    qf[kk][3] = v1 ? __ldg(q1 + w + 4) : 0u;
                }
            }
            m0 = m1 = umax ? phi2 : -CUDART_INF_F;
            an0 = an1 = false;
            l0 = l1 = 0.f;
#pragma unroll
            for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        }

        const int nvalid = ct.tok_hi - ct.tok_lo;
        const int wbase = ts * TW;
        // Causal limits of this thread's rows, relative to the tile (T = 1: the tile's end or beyond).
        const int lim0 = ct.L - cq0 - ct.tok_lo, lim1 = ct.L - cq1 - ct.tok_lo;
        if (wbase < nvalid) {
            const uint32_t kbase = smem_u32(stages) + stage * Sh::STAGE_BYTES;
            const uint32_t vbase = kbase + (KV8 ? TILE_ELEMS : TILE_ELEMS * 2);
            const float* kscale = nullptr;
            const float* vscale = nullptr;
            if constexpr (KV8) {
                kscale = reinterpret_cast<const float*>(smem + stage * Sh::STAGE_BYTES + 2 * TILE_ELEMS);
                vscale = kscale + TT;
            }

            // S = q K^T over this warp's TW tokens, as two independent accumulation
            // chains (even and odd k-steps) to halve the MMA dependency chain.
            float s[NS][4], s2[NS][4];
#pragma unroll
            for (int j = 0; j < NS; ++j)
                s[j][0] = s[j][1] = s[j][2] = s[j][3] = s2[j][0] = s2[j][1] = s2[j][2] = s2[j][3] = 0.f;
            if constexpr (KV8) {
                // Matrix mi of an ldmatrix: tokens 8 (mi & 1) .. + 7 of the
                // warp's 16, head-dim chunk 2 kc + (mi >> 1).
#pragma unroll
                for (int kc = 0; kc < KS / 2; ++kc) {
                    const int row = wbase + ((lane >> 3) & 1) * 8 + (lane & 7);
                    const int ch = 2 * kc + (lane >> 4);
                    uint32_t r[4];
                    ldmatrix_x4(kbase + (uint32_t)(row * D + swz8<D>(row, ch) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int mi = 0; mi < 4; ++mi) {
                        const uint32_t w = FP8 ? r[mi] : (r[mi] ^ 0x80808080u);
                        const uint32_t b0 = codes_to_f16x2<FP8, 0x4140, 0x9180>(w);
                        const uint32_t b1 = codes_to_f16x2<FP8, 0x4342, 0xb3a2>(w);
                        if (mi >> 1)
                            mma_16816<true>(s2[mi & 1], qf[2 * kc + 1], b0, b1);
                        else
                            mma_16816<true>(s[mi & 1], qf[2 * kc], b0, b1);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                    for (int n2 = 0; n2 < NS / 2; ++n2) {
                        const int row = wbase + n2 * 16 + ((lane >> 4) & 1) * 8 + (lane & 7);
                        const int ch = kk * 2 + ((lane >> 3) & 1);
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kbase + (uint32_t)((row * D + ((ch ^ (row & 7)) * 8)) * 2), b0, b1, b2, b3);
                        if (kk & 1) {
                            mma_16816<false>(s2[2 * n2], qf[kk], b0, b1);
                            mma_16816<false>(s2[2 * n2 + 1], qf[kk], b2, b3);
                        } else {
                            mma_16816<false>(s[2 * n2], qf[kk], b0, b1);
                            mma_16816<false>(s[2 * n2 + 1], qf[kk], b2, b3);
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NS; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) s[j][e] += s2[j][e];

            // Scale to base-2 units, mask tokens past the tile's end, row maxima.
            float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = wbase + j * 8 + (lane & 3) * 2 + (e & 1);
                    float sc = scale_log2;
                    if constexpr (KV8) sc *= kscale[tok] * (FP8 ? 256.f : 1.f);
                    s[j][e] = (tok < nvalid && tok < (e < 2 ? lim0 : lim1)) ? s[j][e] * sc : -CUDART_INF_F;
                }
                mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
                mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
            }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            float mu0, mu1, a0, a1;
            if (umax) {
                // Unified maximum (FlashDecoding++'s asynchronized softmax): m
                // stays at phi while the row's scores lie within [phi - 64,
                // phi + 8] (base 2), so every partial of such a row shares it
                // and the merges reduce to plain sums. A larger score moves m
                // up with the usual rescale, and a row whose first scores lie
                // below the window starts from its own maximum (nothing is
                // accumulated yet, so no rescale): the result stays exact.
                const float n0 = (mx0 > m0 + 8.f || (!an0 && mx0 < m0 - 64.f && mx0 > -CUDART_INF_F)) ? mx0 : m0;
                const float n1 = (mx1 > m1 + 8.f || (!an1 && mx1 < m1 - 64.f && mx1 > -CUDART_INF_F)) ? mx1 : m1;
                a0 = (an0 && n0 != m0) ? exp2f(m0 - n0) : 1.f;
                a1 = (an1 && n1 != m1) ? exp2f(m1 - n1) : 1.f;
                if ((n0 != m0 || n1 != m1) && (lane & 3) == 0 && p.status)
                    atomicOr(p.status, KVD_STATUS_UMAX_FALLBACK);
                an0 |= mx0 > -CUDART_INF_F;
                an1 |= mx1 > -CUDART_INF_F;
                mu0 = m0 = n0;
                mu1 = m1 = n1;
            } else {
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                mu0 = (mn0 == -CUDART_INF_F) ? 0.f : mn0;
                mu1 = (mn1 == -CUDART_INF_F) ? 0.f : mn1;
                a0 = exp2f(m0 - mu0);
                a1 = exp2f(m1 - mu1);
                m0 = mn0;
                m1 = mn1;
            }

            // P = 2^(s - m) as bf16 A fragments (hi part; lo part for fp32 output).
            uint32_t pa[NS / 2][4];
            uint32_t pl[F32OUT ? NS / 2 : 1][4];
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const float e0 = exp2f(s[j][0] - mu0), e1 = exp2f(s[j][1] - mu0);
                const float e2 = exp2f(s[j][2] - mu1), e3 = exp2f(s[j][3] - mu1);
                if constexpr (KV8) {
                    // Weights times the value rows' scales, in f16; the sums
                    // take the weights themselves.
                    const int tok = wbase + j * 8 + (lane & 3) * 2;
                    const float w0 = vscale[tok], w1 = vscale[tok + 1];
                    const uint32_t h01 = pack_f16x2(e0 * w0, e1 * w1), h23 = pack_f16x2(e2 * w0, e3 * w1);
                    pa[j >> 1][(j & 1) * 2 + 0] = h01;
                    pa[j >> 1][(j & 1) * 2 + 1] = h23;
                    if constexpr (F32OUT) {
                        pl[j >> 1][(j & 1) * 2 + 0] = pack_f16x2(e0 * w0 - f16_lo(h01), e1 * w1 - f16_hi(h01));
                        pl[j >> 1][(j & 1) * 2 + 1] = pack_f16x2(e2 * w0 - f16_lo(h23), e3 * w1 - f16_hi(h23));
                    }
                    ls0 += e0 + e1;
                    ls1 += e2 + e3;
                    continue;
                }
                const uint32_t h01 = pack_bf16x2(e0, e1), h23 = pack_bf16x2(e2, e3);
                pa[j >> 1][(j & 1) * 2 + 0] = h01;
                pa[j >> 1][(j & 1) * 2 + 1] = h23;
                if constexpr (F32OUT) {
                    pl[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(e0 - bf16_lo(h01), e1 - bf16_hi(h01));
                    pl[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(e2 - bf16_lo(h23), e3 - bf16_hi(h23));
                    ls0 += e0 + e1;
                    ls1 += e2 + e3;
                } else {
                    // The weights actually multiplied into V are the rounded ones;
                    // summing those keeps the output an exact convex combination.
                    ls0 += bf16_lo(h01) + bf16_hi(h01);
                    ls1 += bf16_lo(h23) + bf16_hi(h23);
                }
            }
            l0 = l0 * a0 + ls0;
            l1 = l1 * a1 + ls1;
            if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
                for (int n = 0; n < ND; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
            }

            // O += P V.
            if constexpr (KV8) {
                // Matrix mi of a transposed ldmatrix: tokens 8 (mi & 1) .. + 7,
                // head-dim chunk 2 qq + (mi >> 1); a thread holds columns 2g,
                // 2g + 1 of the chunk for tokens 2j, 2j + 1 (or + 8).
#pragma unroll
                for (int qq = 0; qq < KS / 2; ++qq) {
                    const int row = wbase + ((lane >> 3) & 1) * 8 + (lane & 7);
                    const int ch = 2 * qq + (lane >> 4);
                    uint32_t r[4];
                    ldmatrix_x4_trans(vbase + (uint32_t)(row * D + swz8<D>(row, ch) * 16), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t lo = FP8 ? r[2 * c] : (r[2 * c] ^ 0x80808080u);
                        const uint32_t hi = FP8 ? r[2 * c + 1] : (r[2 * c + 1] ^ 0x80808080u);
                        const int q = 2 * qq + c;
                        const uint32_t e0 = codes_to_f16x2<FP8, 0x4240, 0xa280>(lo);
                        const uint32_t e1 = codes_to_f16x2<FP8, 0x4240, 0xa280>(hi);
                        const uint32_t d0 = codes_to_f16x2<FP8, 0x4341, 0xb391>(lo);
                        const uint32_t d1 = codes_to_f16x2<FP8, 0x4341, 0xb391>(hi);
                        mma_16816<true>(o[2 * q], pa[0], e0, e1);
                        mma_16816<true>(o[2 * q + 1], pa[0], d0, d1);
                        if constexpr (F32OUT) {
                            mma_16816<true>(o[2 * q], pl[0], e0, e1);
                            mma_16816<true>(o[2 * q + 1], pl[0], d0, d1);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int k2 = 0; k2 < NS / 2; ++k2) {
#pragma unroll
                    for (int n2 = 0; n2 < ND / 2; ++n2) {
                        const int row = wbase + k2 * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                        const int ch = n2 * 2 + ((lane >> 4) & 1);
                        uint32_t v0, v1, v2, v3;
                        ldmatrix_x4_trans(vbase + (uint32_t)((row * D + ((ch ^ (row & 7)) * 8)) * 2), v0, v1, v2, v3);
                        mma_16816<false>(o[2 * n2], pa[k2], v0, v1);
                        mma_16816<false>(o[2 * n2 + 1], pa[k2], v2, v3);
                        if constexpr (F32OUT) {
                            mma_16816<false>(o[2 * n2], pl[k2], v0, v1);
                            mma_16816<false>(o[2 * n2 + 1], pl[k2], v2, v3);
                        }
                    }
                }
            }
        }

        if (ct.seg_end) {
            // Row sums are spread over the 4 lanes of a quad.
            l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
            l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
            l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

            if constexpr (TS > 1) {
                float* mbuf = reinterpret_cast<float*>(smem + (KV8 ? STAGES * Sh::STAGE_BYTES : stage * Sh::STAGE_BYTES));
                __syncthreads();  // every warp is done with this stage's K/V rows
                if (ts > 0) {
                    float* mb = mbuf + ((ts - 1) * HT + ht) * Sh::MB_FLOATS_PER_WARP;
#pragma unroll
                    for (int n = 0; n < ND; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) mb[(n * 4 + e) * 32 + lane] = o[n][e];
                    mb[(ND * 4 + 0) * 32 + lane] = m0;
                    mb[(ND * 4 + 1) * 32 + lane] = m1;
                    mb[(ND * 4 + 2) * 32 + lane] = l0;
                    mb[(ND * 4 + 3) * 32 + lane] = l1;
                }
                __syncthreads();
                if (ts == 0) {
#pragma unroll
                    for (int t2 = 1; t2 < TS; ++t2) {
                        const float* mb = mbuf + ((t2 - 1) * HT + ht) * Sh::MB_FLOATS_PER_WARP;
                        const float om0 = mb[(ND * 4 + 0) * 32 + lane];
                        const float om1 = mb[(ND * 4 + 1) * 32 + lane];
                        const float ol0 = mb[(ND * 4 + 2) * 32 + lane];
                        const float ol1 = mb[(ND * 4 + 3) * 32 + lane];
                        // A slice with nothing summed (l = 0) takes no part: its
                        // maximum may be -inf or, with the unified maximum, the
                        // phi it started from. A row no slice has seen a token
                        // of (causal rows) stays empty.
                        const float e0 = l0 > 0.f ? m0 : -CUDART_INF_F, f0 = ol0 > 0.f ? om0 : -CUDART_INF_F;
                        const float e1 = l1 > 0.f ? m1 : -CUDART_INF_F, f1 = ol1 > 0.f ? om1 : -CUDART_INF_F;
                        const float M0 = fmaxf(e0, f0), M1 = fmaxf(e1, f1);
                        const float U0 = (M0 == -CUDART_INF_F) ? 0.f : M0, U1 = (M1 == -CUDART_INF_F) ? 0.f : M1;
                        const float A0 = exp2f(e0 - U0), B0 = exp2f(f0 - U0);
                        const float A1 = exp2f(e1 - U1), B1 = exp2f(f1 - U1);
                        l0 = A0 * l0 + B0 * ol0;
                        l1 = A1 * l1 + B1 * ol1;
                        m0 = M0;
                        m1 = M1;
#pragma unroll
                        for (int n = 0; n < ND; ++n) {
                            o[n][0] = A0 * o[n][0] + B0 * mb[(n * 4 + 0) * 32 + lane];
                            o[n][1] = A0 * o[n][1] + B0 * mb[(n * 4 + 1) * 32 + lane];
                            o[n][2] = A1 * o[n][2] + B1 * mb[(n * 4 + 2) * 32 + lane];
                            o[n][3] = A1 * o[n][3] + B1 * mb[(n * 4 + 3) * 32 + lane];
                        }
                    }
                }
            }

            if (ts == 0) {
                // Output column pair n of this thread: columns col_of(n), + 1
                // of rows r0 (acc(n, 0), acc(n, 1)) and r1 (acc(n, 2), acc(n, 3)).
                // KV8: pairs 2c and 2c + 1 are columns 16c + 4j .. + 3, from
                // the even and odd n-tiles of chunk c alternately.
                auto col_of = [&](int n) {
                    return KV8 ? (n >> 1) * 16 + (lane & 3) * 4 + (n & 1) * 2 : n * 8 + (lane & 3) * 2;
                };
                auto acc = [&](int n, int e) -> float {
                    if constexpr (KV8)
                        return o[(n & ~1) + (e & 1)][(e & 2) + (n & 1)];
                    else
                        return o[n][e];
                };
                const size_t pair = (size_t)ct.b * p.Hkv + ct.h;
                const bool v0 = r0 < TG, v1 = r1 < TG;
                const size_t or0 = v0 ? out_row(ct.b, ct.h, r0) : 0, or1 = v1 ? out_row(ct.b, ct.h, r1) : 0;
                if (ct.full) {
                    // (a row that sees no token, possible only when L < T, is zero)
                    const float i0 = l0 > 0.f ? OSC / l0 : 0.f, i1 = l1 > 0.f ? OSC / l1 : 0.f;
#pragma unroll
                    for (int n = 0; n < ND; ++n) {
                        const int d = col_of(n);
                        if constexpr (F32OUT) {
                            float* out = reinterpret_cast<float*>(p.out);
                            if (v0) *reinterpret_cast<float2*>(out + or0 * D + d) = make_float2(acc(n, 0) * i0, acc(n, 1) * i0);
                            if (v1) *reinterpret_cast<float2*>(out + or1 * D + d) = make_float2(acc(n, 2) * i1, acc(n, 3) * i1);
                        } else {
                            __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
                            if (v0) *reinterpret_cast<uint32_t*>(out + or0 * D + d) = pack_bf16x2(acc(n, 0) * i0, acc(n, 1) * i0);
                            if (v1) *reinterpret_cast<uint32_t*>(out + or1 * D + d) = pack_bf16x2(acc(n, 2) * i1, acc(n, 3) * i1);
                        }
                    }
                    if (p.lse && (lane & 3) == 0) {
                        if (v0) p.lse[or0] = l0 > 0.f ? (m0 + log2f(l0)) * 0.69314718055994531f : -CUDART_INF_F;
                        if (v1) p.lse[or1] = l1 > 0.f ? (m1 + log2f(l1)) * 0.69314718055994531f : -CUDART_INF_F;
                    }
                } else {
                    const size_t slot = (size_t)c + pair;
                    float* wo = p.ws_o + slot * TG * D;
#pragma unroll
                    for (int n = 0; n < ND; ++n) {
                        const int d = col_of(n);
                        if (v0) *reinterpret_cast<float2*>(wo + (size_t)r0 * D + d) = make_float2(acc(n, 0) * OSC, acc(n, 1) * OSC);
                        if (v1) *reinterpret_cast<float2*>(wo + (size_t)r1 * D + d) = make_float2(acc(n, 2) * OSC, acc(n, 3) * OSC);
                    }
                    if ((lane & 3) == 0) {
                        if (v0) p.ws_ml[slot * TG + r0] = make_float2(m0, l0);
                        if (v1) p.ws_ml[slot * TG + r1] = make_float2(m1, l1);
                    }
                }
            }
            if constexpr (TS > 1) __syncthreads();
        }
        // The next tile's page entries, for its issue after the barrier at the
        // top of the next iteration (its slot was last read two issues ago).
        if constexpr (PAGED) {
            if (tid < MAXP) s_pages[(it + STAGES - 1) & 1][tid] = pg_next;
        }
    }
    cw.finish(write_empty);
    cp_async_wait<0>();
}

}  // namespace kvd
