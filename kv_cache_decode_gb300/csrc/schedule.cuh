// Work schedule of the split-KV decode: shared by the device kernels and by the
// host-side replica used for planning and tests, so both walk the same path.
//
// The (sequence b, KV head h) pairs are laid end to end in b-major order on a
// line of positions, each position standing for U consecutive tokens of a pair
// (U = 1, or U = TT, the kernel's pipeline tile). A pair of L_b > 0 tokens
// occupies X + ceil(L_b / U) positions: a prefix of X positions that stands
// for the fixed cost of starting a pair inside a CTA's run (loading its
// queries, filling the pipeline), then its tokens. Empty pairs occupy nothing.
// CTA c of the C_eff working CTAs gets the contiguous run
// [c*total/C_eff, (c+1)*total/C_eff) of positions, so runs are balanced to one
// position of estimated time. Within a run a CTA walks pairs and cuts each
// pair's tokens inside the run (a "segment") into tiles of at most TT tokens.
// A kernel whose time per tile is fixed (latency-bound) takes U = TT, so that
// its runs are balanced in tiles; a bandwidth-bound one takes U = 1.
//
// Every pair has one owner: for a non-empty pair, the CTA whose run contains
// its first token; for an empty pair, the CTA whose run contains its position
// (the last CTA for empty pairs at the very end). If the owner covers the pair
// entirely it writes the final output; otherwise each contributing CTA c writes
// a partial (m, l, o) into slot c + p, and the merge kernel, which recomputes
// the range of contributing CTAs from the same walk, combines them. Slots are
// unique because walking segments in order, each step increments c, p or both.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define KVD_HD __host__ __device__ __forceinline__
// The walker's callbacks are device lambdas in kernels and plain functors on
// the host; each instantiation is only ever called from its own side.
#define KVD_HD_TEMPLATE _Pragma("nv_exec_check_disable")
#else
#define KVD_HD inline
#define KVD_HD_TEMPLATE
#endif

namespace kvd {

KVD_HD int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

// Attended length of sequence b. With vt > 1 (the tcgen05 kernel's form of
// vt query tokens per sequence) b is a virtual sequence s * vt + i: query
// token i of cache sequence s, which attends to the first L_s - vt + 1 + i
// tokens (none when that is not positive).
struct DevLen {
    const int32_t* lens;
    int cap;
    int vt;
    KVD_HD int operator()(int b) const {
        if (vt <= 1) return clamp_len(load(b), cap);
        const int s = b / vt;
        const int L = clamp_len(load(s), cap) - vt + 1 + (b - s * vt);
        return L > 0 ? L : 0;
    }
    KVD_HD int load(int s) const {
#ifdef __CUDA_ARCH__
        return __ldg(lens + s);
#else
        return lens[s];
#endif
    }
};

// Geometry of the walk: tokens per tile TT, tokens per position U (1 or TT)
// and start-up cost X (positions). Compile-time constants in kernels, so that
// the divisions become shifts and a zero cost compiles away; run-time values
// in the host replica.
template <int TT_, int U_, int X_>
struct FixedGeom {
    static_assert(U_ == 1 || U_ == TT_, "a position is one token or one tile");
    KVD_HD constexpr int tt() const { return TT_; }
    KVD_HD constexpr int unit() const { return U_; }
    KVD_HD constexpr int x() const { return X_; }
};
struct RuntimeGeom {
    int tt_, unit_, x_;
    KVD_HD int tt() const { return tt_; }
    KVD_HD int unit() const { return unit_; }
    KVD_HD int x() const { return x_; }
};

// Positions occupied by a pair of L >= 0 tokens.
template <class Geom>
KVD_HD long long pair_extent(int L, Geom g) {
    const int n = (L + g.unit() - 1) / g.unit();
    return (long long)n + (n > 0 ? g.x() : 0);
}

// Number of CTAs that receive work: at most one per position, at least one
// (the last CTA also owns trailing empty pairs, so one is needed even for no work).
KVD_HD int effective_ctas(int n_split, long long total) {
    if (total <= 0) return 1;
    return (long long)n_split < total ? n_split : (int)total;
}

// a / b for a >= 0, b > 0, with 32-bit arithmetic when both fit (a 64-bit
// division is a long software sequence on the GPU, and these sit on the
// kernels' start-up path).
KVD_HD long long div_nonneg(long long a, long long b) {
    if (((unsigned long long)a | (unsigned long long)b) < (1ull << 32))
        return (long long)((unsigned)a / (unsigned)b);
    return a / b;
}

KVD_HD long long run_begin(int c, int C_eff, long long total) {
    return div_nonneg((long long)c * total, C_eff);
}

// The CTA whose run [run_begin(c), run_begin(c + 1)) contains position t < total.
KVD_HD int cta_of_token(long long t, int C_eff, long long total) {
    return (int)div_nonneg((t + 1) * (long long)C_eff - 1, total);
}

struct Tile {
    int b, h;          // pair
    int L;             // its (clamped) length
    int tok_lo, tok_hi;  // pair-relative token range of this tile
    bool seg_start, seg_end;
    bool owned;        // this CTA owns the pair
    bool full;         // ... and covers all of it (final write)
    int c_last;        // last contributing CTA (owned && !full)
};

// Walks one CTA's run. LenFn: int(int b) returning the clamped length;
// Geom: FixedGeom<TT, U, X> or RuntimeGeom.
template <class LenFn, class Geom>
struct Walker {
    LenFn len;
    Geom g;
    int B, Hkv;
    int c, C_eff;
    long long total, S, E;  // this CTA's run [S, E) of positions
    // state
    int b, h, L;
    long long pstart, pos;  // position of the current pair, position reached

    Walker() = default;
    KVD_HD_TEMPLATE
    KVD_HD Walker(LenFn f, Geom g_, int B_, int Hkv_, int c_, int C_eff_, long long total_)
        : len(f), g(g_), B(B_), Hkv(Hkv_), c(c_), C_eff(C_eff_), total(total_) {
        S = run_begin(c, C_eff, total);
        E = run_begin(c + 1, C_eff, total);
        b = B; h = 0; L = 0; pstart = total; pos = S;
    }

    KVD_HD long long ext() const { return pair_extent(L, g); }

    // b0 = first sequence whose pairs end after S or start at or after S;
    // cum0 = position of pair (b0, 0).
    KVD_HD_TEMPLATE
    KVD_HD void start(int b0, long long cum0) {
        b = b0;
        h = 0;
        pstart = cum0;
        L = (b < B) ? len(b) : 0;
        if (b < B && L > 0 && pstart < S) {
            h = (int)div_nonneg(S - pstart, ext());
            pstart += (long long)h * ext();
        }
        pos = S;
    }

    KVD_HD_TEMPLATE
    KVD_HD void advance_pair() {
        pstart += ext();
        if (++h == Hkv) {
            h = 0;
            ++b;
            L = (b < B) ? len(b) : 0;
        }
    }

    // Next tile of the run; calls on_empty(b, h) for each empty pair passed
    // on the way (those pairs lie inside this run, so this CTA owns them).
    KVD_HD_TEMPLATE
    template <class F>
    KVD_HD bool next(Tile& t, F&& on_empty) {
        if (pos >= E) return false;
        while (pos >= pstart + ext()) {
            if (L == 0) on_empty(b, h);
            advance_pair();
        }
        const long long real0 = pstart + g.x();  // position of the pair's first token
        if (g.x() > 0 && pos < real0) {
            pos = real0;                         // skip the pair's start-up prefix
            if (pos >= E) return false;
        }
        const long long pend = pstart + ext();
        const long long seg_lo = real0 > S ? real0 : S;
        const long long seg_hi = pend < E ? pend : E;
        long long te = pos + g.tt() / g.unit();
        if (te > seg_hi) te = seg_hi;
        t.b = b;
        t.h = h;
        t.L = L;
        t.tok_lo = (int)(pos - real0) * g.unit();
        t.tok_hi = (int)(te - real0) * g.unit();
        if (t.tok_hi > L) t.tok_hi = L;
        t.seg_start = (pos == seg_lo);
        t.seg_end = (te == seg_hi);
        t.owned = (real0 >= S);
        t.full = t.owned && (pend <= E);
        t.c_last = (t.owned && !t.full) ? cta_of_token(pend - 1, C_eff, total) : c;
        pos = te;
        return true;
    }

    // After the last tile: the last CTA also owns the empty pairs that sit at
    // the very end of the line.
    KVD_HD_TEMPLATE
    template <class F>
    KVD_HD void finish(F&& on_empty) {
        if (c != C_eff - 1) return;
        if (pos < E) pos = E;  // the run may end inside a prefix
        while (b < B) {
            if (pos < pstart + ext()) break;  // cannot happen once pos == total
            if (L == 0) on_empty(b, h);
            advance_pair();
        }
    }
};

// Condition selecting b0 in Walker::start, given sequence b's cumulative
// position (counting all its Hkv pairs) and the extent of one of its pairs.
KVD_HD bool is_first_seq_candidate(long long cum_start_b, long long ext_b, int Hkv, long long S) {
    return (cum_start_b + (long long)Hkv * ext_b > S) || (cum_start_b >= S);
}

}  // namespace kvd
