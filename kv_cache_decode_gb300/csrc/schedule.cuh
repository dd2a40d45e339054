// Work schedule of the split-KV decode: shared by the device kernels and by the
// host-side replica used for planning and tests, so both walk the same path.
//
// The (sequence b, KV head h) pairs are laid end to end in b-major order, pair
// p = b * Hkv + h holding L_b tokens; total = Hkv * sum_b L_b. CTA c of the
// C_eff working CTAs gets the contiguous token run [c*total/C_eff,
// (c+1)*total/C_eff). Within a run the CTA walks pairs and cuts each pair's
// part (a "segment") into pipeline tiles of at most TT tokens.
//
// Every pair has one owner: the CTA whose run contains the pair's first token
// (or the last CTA for empty pairs at the very end). If the owner covers the
// pair entirely it writes the final output; otherwise each contributing CTA c
// writes a partial (m, l, o) into slot c + p, and the owner records the range
// of contributing CTAs for the merge kernel. Slots are unique because walking
// segments in order, each step increments c, p or both.
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

// Number of CTAs that receive work: at most one per token, at least one (the
// last CTA also owns trailing empty pairs, so one is needed even for no work).
KVD_HD int effective_ctas(int n_split, long long total) {
    if (total <= 0) return 1;
    return (long long)n_split < total ? n_split : (int)total;
}

KVD_HD long long run_begin(int c, int C_eff, long long total) {
    return (long long)c * total / C_eff;
}

// The CTA whose run [run_begin(c), run_begin(c + 1)) contains token t < total.
KVD_HD int cta_of_token(long long t, int C_eff, long long total) {
    return (int)(((t + 1) * (long long)C_eff - 1) / total);
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

// Walks one CTA's token run. LenFn: int(int b) returning the clamped length.
template <class LenFn>
struct Walker {
    LenFn len;
    int B, Hkv, TT;
    int c, C_eff;
    long long total, S, E;  // this CTA's run [S, E)
    // state
    int b, h, L;
    long long pstart, pos;

    KVD_HD_TEMPLATE
    KVD_HD Walker(LenFn f, int B_, int Hkv_, int TT_, int c_, int C_eff_, long long total_)
        : len(f), B(B_), Hkv(Hkv_), TT(TT_), c(c_), C_eff(C_eff_), total(total_) {
        S = run_begin(c, C_eff, total);
        E = run_begin(c + 1, C_eff, total);
        b = B; h = 0; L = 0; pstart = total; pos = S;
    }

    // b0 = first sequence whose pairs end after S or start at or after S;
    // cum0 = token offset of pair (b0, 0).
    KVD_HD_TEMPLATE
    KVD_HD void start(int b0, long long cum0) {
        b = b0;
        h = 0;
        pstart = cum0;
        L = (b < B) ? len(b) : 0;
        if (b < B && L > 0 && pstart < S) {
            h = (int)((S - pstart) / L);
            pstart += (long long)h * L;
        }
        pos = S;
    }

    KVD_HD_TEMPLATE
    KVD_HD void advance_pair() {
        pstart += L;
        if (++h == Hkv) {
            h = 0;
            ++b;
            L = (b < B) ? len(b) : 0;
        }
    }

    // Next tile of the run; calls on_empty(b, h) for each empty pair passed
    // on the way (those pairs start inside this run, so this CTA owns them).
    KVD_HD_TEMPLATE
    template <class F>
    KVD_HD bool next(Tile& t, F&& on_empty) {
        if (pos >= E) return false;
        while (pos >= pstart + L) {
            if (L == 0) on_empty(b, h);
            advance_pair();
        }
        const long long pend = pstart + L;
        const long long seg_lo = pstart > S ? pstart : S;
        const long long seg_hi = pend < E ? pend : E;
        long long te = pos + TT;
        if (te > seg_hi) te = seg_hi;
        t.b = b;
        t.h = h;
        t.L = L;
        t.tok_lo = (int)(pos - pstart);
        t.tok_hi = (int)(te - pstart);
        t.seg_start = (pos == seg_lo);
        t.seg_end = (te == seg_hi);
        t.owned = (pstart >= S);
        t.full = t.owned && (pend <= E);
        t.c_last = (t.owned && !t.full) ? cta_of_token(pend - 1, C_eff, total) : c;
        pos = te;
        return true;
    }

    // After the last tile: the last CTA also owns the empty pairs that start at
    // the very end of the token order.
    KVD_HD_TEMPLATE
    template <class F>
    KVD_HD void finish(F&& on_empty) {
        if (c != C_eff - 1) return;
        while (b < B) {
            if (pos < pstart + L) break;  // cannot happen once pos == total
            if (L == 0) on_empty(b, h);
            advance_pair();
        }
    }
};

// Condition selecting b0 in Walker::start, given sequence b's cumulative start
// (in tokens, counting all its Hkv pairs) and its clamped length.
KVD_HD bool is_first_seq_candidate(long long cum_start_b, int L_b, int Hkv, long long S) {
    return (cum_start_b + (long long)Hkv * L_b > S) || (cum_start_b >= S);
}

}  // namespace kvd
