// Device helpers shared by the gate (hspz_gate.cu) and the materializer
// (hspz_materialize.cu): packed-sequence access, the table scoring of an
// 8-base step and the walk state of one X-drop side walk ("D. Score gate",
// D.2; "E. X-drop materialization", E.2/E.3).
#pragma once
#include "hspz_internal.cuh"

namespace hspz {
namespace {

struct Seqs {
    const uint32_t *__restrict__ ref;
    const uint32_t *__restrict__ qry;
    uint64_t Lr, Lq;
};

__device__ __forceinline__ uint32_t nib_at(const uint32_t *__restrict__ p, uint64_t i) {
    const uint64_t j = i + kPadBases;
    return (__ldg(p + (j >> 3)) >> ((uint32_t)(j & 7u) * 4u)) & 0xFu;
}
__device__ __forceinline__ uint32_t code_of(uint32_t nib) { return (nib & kNibN) ? 4u : (nib & 3u); }
__device__ __forceinline__ int pair_score(const int *__restrict__ tab, const Seqs &s, uint64_t r, uint64_t q) {
    return tab[code_of(nib_at(s.ref, r)) * 5u + code_of(nib_at(s.qry, q))];
}

// ------------------------------------------------------------------ fast gate
// For matrices that are complement symmetric on A/C/G/T (score(r, q) =
// score(r ^ 3, q ^ 3) with A0 C1 G2 T3) and fit int8, the score of a base pair
// depends only on x = r ^ q and the reference base's strong/weak class
// (bit 2 of the reference nibble), so eight pairs are scored by two byte
// permutes of one 8-entry table.  A walk advances eight bases per step:
// the eight running sums come from byte dot products, a step that cannot hold
// the stop (its lowest running sum is not more than X below the highest
// maximum it could reach) just takes the new maximum, and only a step that
// might hold the stop is replayed base by base.  N anywhere in a step's
// sixteen nibbles sends that step to the 5 x 5 matrix.

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Scores of one 8-base step, in walk order, as 8 int32 running sums from S.
// RIGHT: walk order = nibbles 0..7 of the aligned words; left: 7..0.
template <bool RIGHT, bool HAS_N = true>
__device__ __forceinline__ void step_sums(uint32_t R, uint32_t Q, uint32_t keep, uint32_t tlo, uint32_t thi,
                                          const int *__restrict__ tab25, int S, int (&Sv)[8]) {
    // without N in either sequence only the padding is N, and keep masks it
    const uint32_t nmask = HAS_N ? ((R | Q) & 0x88888888u & keep) : 0u;
    if (__builtin_expect(nmask == 0, 1)) {
        // masked-off nibbles select entry 0 in sign mode: score 0
        const uint32_t idx = (((R ^ Q) & 0x77777777u) & keep) | (0x88888888u & ~keep);
        const uint32_t w0 = prmt(tlo, thi, idx), w1 = prmt(tlo, thi, idx >> 16);
        const uint32_t a = RIGHT ? w0 : w1, b = RIGHT ? w1 : w0;
        const int c1 = RIGHT ? 0x00000001 : 0x01000000, c2 = RIGHT ? 0x00000101 : 0x01010000;
        const int c3 = RIGHT ? 0x00010101 : 0x01010100, c4 = 0x01010101;
        Sv[0] = __dp4a((int)a, c1, S);
        Sv[1] = __dp4a((int)a, c2, S);
        Sv[2] = __dp4a((int)a, c3, S);
        Sv[3] = __dp4a((int)a, c4, S);
        Sv[4] = __dp4a((int)b, c1, Sv[3]);
        Sv[5] = __dp4a((int)b, c2, Sv[3]);
        Sv[6] = __dp4a((int)b, c3, Sv[3]);
        Sv[7] = __dp4a((int)b, c4, Sv[3]);
    } else {
        int run = S;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int nib = RIGHT ? k : 7 - k;
            const uint32_t kb = (keep >> (4 * nib)) & 0xFu;
            const uint32_t rn = (R >> (4 * nib)) & 0xFu, qn = (Q >> (4 * nib)) & 0xFu;
            const uint32_t rc = (rn & 8u) ? 4u : (rn & 3u), qc = (qn & 8u) ? 4u : (qn & 3u);
            run += kb ? tab25[rc * 5 + qc] : 0;
            Sv[k] = run;
        }
    }
}

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Mask of the low min(n, 8) nibbles (the bases of a step inside the walk).
__device__ __forceinline__ uint32_t low_nibbles(uint32_t n) {
    const uint32_t s = min(n, 8u) * 4u;
    uint32_t d;
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(0xFFFFFFFFu), "r"(s));  // shifts of 32 give 0
    return ~d;
}

// Mask of the high min(n, 8) nibbles: the bases of a step of a walk that
// reads the packed words downwards (walk order = nibbles 7..0).
__device__ __forceinline__ uint32_t high_nibbles(uint32_t n) {
    const uint32_t s = 32u - min(n, 8u) * 4u;
    uint32_t d;
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(0xFFFFFFFFu), "r"(s));  // shifts of 32 give 0
    return d;
}

// The bases of the step at the front of a walk of `rem` bases left.
template <bool BACK>
__device__ __forceinline__ uint32_t step_keep(uint32_t rem) {
    return BACK ? high_nibbles(rem) : low_nibbles(rem);
}

struct WalkState {
    const uint32_t *pr, *pq;
    uint32_t shr, shq, r0, r1, q0, q1, rem;
    int S, M;
};

// Where one side of anchor (ar, aq) starts: word pointers, shifts and length.
__device__ __forceinline__ void walk_place(WalkState &w, const Seqs &sq, const uint32_t *ref_rev,
                                           const uint32_t *qry_rev, uint32_t ar, uint32_t aq, int side) {
    const uint32_t Lr = (uint32_t)sq.Lr, Lq = (uint32_t)sq.Lq;
    const uint32_t rb = side ? ar : Lr - ar;
    const uint32_t qb = side ? aq : Lq - aq;
    w.rem = side ? min(Lr - ar, Lq - aq) : min(ar, aq);
    const uint32_t jr = rb + (uint32_t)kPadBases, jq = qb + (uint32_t)kPadBases;
    w.pr = (side ? sq.ref : ref_rev) + (jr >> 3);
    w.pq = (side ? sq.qry : qry_rev) + (jq >> 3);
    w.shr = (jr & 7u) * 4u;
    w.shq = (jq & 7u) * 4u;
    w.S = 0;
    w.M = 0;
}

// Where one side of anchor (ar, aq) starts on the forward packed copies.
// The right side (side 1) reads upwards from the anchor base.  The left side
// (side 0) scores ar-1, ar-2, ... : its step window is the 8 bases just below
// the current position, read from the same words downwards (BACK walks), so
// the left and right walks of an anchor share the cache lines around it.
__device__ __forceinline__ void walk_place_fwd(WalkState &w, const Seqs &sq, uint32_t ar, uint32_t aq, int side) {
    const uint32_t Lr = (uint32_t)sq.Lr, Lq = (uint32_t)sq.Lq;
    w.rem = side ? min(Lr - ar, Lq - aq) : min(ar, aq);
    // unsigned wrap of ar - 8 for ar < 8 is undone by the padding offset
    const uint32_t jr = (side ? ar : ar - 8u) + (uint32_t)kPadBases;
    const uint32_t jq = (side ? aq : aq - 8u) + (uint32_t)kPadBases;
    w.pr = sq.ref + (jr >> 3);
    w.pq = sq.qry + (jq >> 3);
    w.shr = (jr & 7u) * 4u;
    w.shq = (jq & 7u) * 4u;
    w.S = 0;
    w.M = 0;
}

// Moves a walk one step on: the window words slide up (or down for BACK) by
// one word and the newly needed word of each sequence is loaded.
template <bool BACK = false>
__device__ __forceinline__ void walk_advance(WalkState &w, int S_next) {
    w.rem -= 8;
    w.S = S_next;
    if (BACK) {
        w.r1 = w.r0;
        w.q1 = w.q0;
        w.pr--;
        w.pq--;
        w.r0 = __ldg(w.pr);
        w.q0 = __ldg(w.pq);
    } else {
        w.r0 = w.r1;
        w.q0 = w.q1;
        w.pr++;
        w.pq++;
        w.r1 = __ldg(w.pr + 1);
        w.q1 = __ldg(w.pq + 1);
    }
}

// The common 8-base step.  It advances the walk and returns false unless the
// step may hold the stop, reaches `need` or ends at the edge; then it leaves
// the walk untouched and returns true for walk_resolve.
template <bool HAS_N, bool BACK = false>
__device__ __forceinline__ bool walk_step(WalkState &w, uint32_t tlo, uint32_t thi, const int *__restrict__ tab25,
                                          int X, int need, int (&Sv)[8], int &Mb, bool &maybe_stop) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    step_sums<!BACK, HAS_N>(R, Q, step_keep<BACK>(w.rem), tlo, thi, tab25, w.S, Sv);
    const int hi = max(max(max(Sv[0], Sv[1]), max(Sv[2], Sv[3])), max(max(Sv[4], Sv[5]), max(Sv[6], Sv[7])));
    const int lo = min(min(min(Sv[0], Sv[1]), min(Sv[2], Sv[3])), min(min(Sv[4], Sv[5]), min(Sv[6], Sv[7])));
    Mb = max(w.M, hi);
    // sign bits: lo - Mb + X < 0 when the step may hold the stop, need - 1 - Mb < 0 when it reaches need
    const int gap = lo - Mb + X;
    maybe_stop = gap < 0;
    if (!(((gap | (need - 1 - Mb)) < 0) | (w.rem <= 8))) {
        w.M = Mb;
        walk_advance<BACK>(w, Sv[7]);
        return false;
    }
    return true;
}

// Settles a flagged step.  Returns true when the side is over, with *acc
// telling whether its maximum reached `need`; else the walk has advanced.
template <bool BACK = false>
__device__ __forceinline__ bool walk_resolve(WalkState &w, const int (&Sv)[8], int Mb, bool maybe_stop, int X,
                                             int need, bool *acc) {
    if (maybe_stop) {
        int M = w.M;
#pragma unroll
        for (int k = 0; k < 8; k++) {
            if (M - Sv[k] > X) {
                w.M = M;
                *acc = M >= need;
                return true;
            }
            M = max(M, Sv[k]);
        }
    }
    w.M = Mb;
    if (Mb >= need) {
        *acc = true;
        return true;
    }
    if (w.rem <= 8) {
        *acc = false;
        return true;
    }
    walk_advance<BACK>(w, Sv[7]);
    return false;
}

// hi = max(M, the eight sums of a step), lo = the lowest of the eight.
__device__ __forceinline__ void step_range(const int (&Sv)[8], int M, int &hi, int &lo) {
    hi = max(max(max(Sv[0], Sv[1]), max(Sv[2], Sv[3])), max(max(Sv[4], Sv[5]), max(Sv[6], Sv[7])));
    hi = max(hi, M);
    lo = min(min(min(Sv[0], Sv[1]), min(Sv[2], Sv[3])), min(min(Sv[4], Sv[5]), min(Sv[6], Sv[7])));
}

// The 8-base step with an exact stop test, for scoring where X >= 7 * the
// largest single-pair score (and X >= 0).  Base k of the step stops the walk
// when it falls more than X below the running maximum m(k-1) of the bases
// before it.  After such a stop the remaining (at most 7) sums of the step
// cannot climb back above m(k-1), so the step's final running maximum is the
// side maximum at the stop: the step never has to be replayed base by base.
// Nor does the stop test need the running maxima: with hi = max(M, sums of
// the step) and lo = the lowest sum of the step, some base stops the walk
// exactly when lo + X < hi.  (A stop at k gives lo <= S(k) < m(k-1) - X <=
// hi - X.  Conversely, if lo + X < hi and hi is M or a sum before lo's base,
// lo's base itself stops the walk; hi cannot come after lo's base, since
// at most 7 pairs lie between them and they cannot rise by more than X.)
// The step has no branches or selects, so every lane of a round runs it
// together.  A lane whose side is over (stop, `need` reached or edge) gets
// rem = 0: its keep mask is then empty, so its later steps score nothing and
// leave S and M as they are (S <= M holds throughout).  The window words and
// pointers move every step; only the loads are skipped once rem = 0, so fully
// unrolled steps address their words with immediate offsets.  rem = 0
// afterwards means the side is over with w.M its maximum.
template <bool HAS_N, bool BACK>
__device__ __forceinline__ void walk_step_lead(WalkState &w, uint32_t tlo, uint32_t thi,
                                               const int *__restrict__ tab25, int X, int need) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    int Sv[8];
    step_sums<!BACK, HAS_N>(R, Q, step_keep<BACK>(w.rem), tlo, thi, tab25, w.S, Sv);
    int hi, lo;
    step_range(Sv, w.M, hi, lo);
    const bool over = (((lo + X - hi) | (need - 1 - hi)) < 0) | (w.rem <= 8);
    w.M = hi;
    w.S = Sv[7];
    w.rem = over ? 0u : w.rem - 8u;
    if (BACK) {
        w.r1 = w.r0;
        w.q1 = w.q0;
        w.pr--;
        w.pq--;
        if (w.rem) {
            w.r0 = __ldg(w.pr);
            w.q0 = __ldg(w.pq);
        }
    } else {
        w.r0 = w.r1;
        w.q0 = w.q1;
        w.pr++;
        w.pq++;
        if (w.rem) {
            w.r1 = __ldg(w.pr + 1);
            w.q1 = __ldg(w.pq + 1);
        }
    }
}

// walk_step_lead for a walk that cannot reach its sequence edge during the
// step: the step's bases are all inside, so the keep mask is all or nothing
// (`keep`: ~0 while the side walks, 0 once it is over) and rem is neither
// read nor changed.
template <bool HAS_N, bool BACK>
__device__ __forceinline__ void walk_step_inner(WalkState &w, uint32_t &keep, uint32_t tlo, uint32_t thi,
                                                const int *__restrict__ tab25, int X, int need) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    int Sv[8];
    step_sums<!BACK, HAS_N>(R, Q, keep, tlo, thi, tab25, w.S, Sv);
    int hi, lo;
    step_range(Sv, w.M, hi, lo);
    w.M = hi;
    w.S = Sv[7];
    keep = (((lo + X - hi) | (need - 1 - hi)) < 0) ? 0u : keep;
    if (BACK) {
        w.r1 = w.r0;
        w.q1 = w.q0;
        w.pr--;
        w.pq--;
        if (keep) {
            w.r0 = __ldg(w.pr);
            w.q0 = __ldg(w.pq);
        }
    } else {
        w.r0 = w.r1;
        w.q0 = w.q1;
        w.pr++;
        w.pq++;
        if (keep) {
            w.r1 = __ldg(w.pr + 1);
            w.q1 = __ldg(w.pq + 1);
        }
    }
}

// Exact side walk with the earliest maximum (E.2/E.3).  64-bit sums.
__device__ __forceinline__ void side_exact(const Seqs &s, const int *__restrict__ tab, int64_t X, uint32_t ar,
                                           uint32_t aq, bool right, int64_t &best, uint64_t &best_n) {
    int64_t S = 0, M = 0;
    uint64_t nb = 0;
    const uint64_t lim = right ? min(s.Lr - ar, s.Lq - aq) : (uint64_t)min(ar, aq);
    for (uint64_t n = 1; n <= lim; ++n) {
        S += right ? pair_score(tab, s, ar + n - 1, aq + n - 1) : pair_score(tab, s, ar - n, aq - n);
        if (M - S > X) break;
        if (S > M) {
            M = S;
            nb = n;
        }
    }
    best = M;
    best_n = nb;
}

unsigned grid_cap(uint64_t n, int threads) {
    uint64_t g = (n + threads - 1) / threads;
    const uint64_t cap = 152ull * 64;
    return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

Seqs seqs(SeqView r, SeqView q) { return Seqs{r.packed, q.packed, r.len, q.len}; }

}  // namespace
}  // namespace hspz
