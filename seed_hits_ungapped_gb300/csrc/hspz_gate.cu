// Score-only X-drop gate ("D. Score gate", D.1-D.3), the fused expansion +
// gate of one MAX_HITS chunk ("C. Hit discovery" C.5 feeding D.2), and the
// exact materializer ("E. X-drop materialization", E.1-E.5).
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

// Gate decision for one anchor (D.2).  Left side first: bases before the
// anchor, stepping outward; then the right side from the anchor base.  A side
// stops before the step whose score falls more than X below the running
// maximum, or at a sequence edge.  The keep test total >= T is monotone in
// either side's running maximum, so the walk accepts as soon as the maxima
// reached so far already meet T; a rejection needs both sides walked to
// their stop.  All values stay inside int32 under the library's limits.
__device__ __forceinline__ int gate_one(const Seqs &s, const int *__restrict__ tab, int X, int T, uint32_t ar,
                                        uint32_t aq) {
    if (ar >= s.Lr || aq >= s.Lq) return 0;
    int S = 0, M = 0;
    const uint32_t nl = min(ar, aq);
    for (uint32_t n = 1; n <= nl; ++n) {
        S += pair_score(tab, s, ar - n, aq - n);
        if (M - S > X) break;
        if (S > M) {
            M = S;
            if (M >= T) return 1;
        }
    }
    const int ML = M;
    S = 0;
    M = 0;
    const uint64_t nr = min(s.Lr - ar, s.Lq - aq);
    for (uint64_t n = 0; n < nr; ++n) {
        S += pair_score(tab, s, ar + n, aq + n);
        if (M - S > X) break;
        if (S > M) {
            M = S;
            if (ML + M >= T) return 1;
        }
    }
    return 0;
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

// One side of the X-drop walk.  Returns the side maximum before the stop
// (or the maximum at which the walk already reached `need`, with *accepted).
template <bool RIGHT>
__device__ __forceinline__ int walk_fast(const uint32_t *__restrict__ ref, const uint32_t *__restrict__ qry,
                                         uint32_t ar, uint32_t aq, uint32_t limit, uint32_t tlo, uint32_t thi,
                                         const int *__restrict__ tab25, int X, int need, bool *accepted) {
    int S = 0, M = 0;
    if (limit == 0) return 0;
    // nibble index (with padding) of the lowest base of the first step
    const uint32_t jr = (RIGHT ? ar : ar - 8u) + (uint32_t)kPadBases;
    const uint32_t jq = (RIGHT ? aq : aq - 8u) + (uint32_t)kPadBases;
    const uint32_t shr = (jr & 7u) * 4u, shq = (jq & 7u) * 4u;
    const uint32_t *pr = ref + (jr >> 3), *pq = qry + (jq >> 3);
    uint32_t r0 = __ldg(pr), r1 = __ldg(pr + 1), q0 = __ldg(pq), q1 = __ldg(pq + 1);
    uint32_t rem = limit;
    for (;;) {
        const uint32_t R = __funnelshift_r(r0, r1, shr);
        const uint32_t Q = __funnelshift_r(q0, q1, shq);
        uint32_t keep = 0xFFFFFFFFu;
        if (rem < 8) keep = RIGHT ? ((1u << (4 * rem)) - 1u) : ~((1u << (4 * (8 - rem))) - 1u);
        int Sv[8];
        step_sums<RIGHT>(R, Q, keep, tlo, thi, tab25, S, Sv);
        const int hi = max(max(max(Sv[0], Sv[1]), max(Sv[2], Sv[3])), max(max(Sv[4], Sv[5]), max(Sv[6], Sv[7])));
        const int lo = min(min(min(Sv[0], Sv[1]), min(Sv[2], Sv[3])), min(min(Sv[4], Sv[5]), min(Sv[6], Sv[7])));
        const int Mb = max(M, hi);
        if (lo < Mb - X) {  // the stop may lie in this step: replay it base by base
#pragma unroll
            for (int k = 0; k < 8; k++) {
                if (M - Sv[k] > X) {
                    *accepted = M >= need;
                    return M;
                }
                M = max(M, Sv[k]);
            }
        }
        M = Mb;
        if (M >= need) {
            *accepted = true;
            return M;
        }
        if (rem <= 8) return M;
        rem -= 8;
        S = Sv[7];
        if (RIGHT) {
            r0 = r1;
            q0 = q1;
            pr++;
            pq++;
            r1 = __ldg(pr + 1);
            q1 = __ldg(pq + 1);
        } else {
            r1 = r0;
            q1 = q0;
            pr--;
            pq--;
            r0 = __ldg(pr);
            q0 = __ldg(pq);
        }
    }
}

__device__ __forceinline__ int gate_fast(const Seqs &s, const int *__restrict__ tab25, uint32_t tlo, uint32_t thi,
                                         int X, int T, uint32_t ar, uint32_t aq) {
    if (ar >= s.Lr || aq >= s.Lq) return 0;
    bool acc = false;
    const int ML = walk_fast<false>(s.ref, s.qry, ar, aq, min(ar, aq), tlo, thi, tab25, X, T, &acc);
    if (acc) return 1;
    const uint32_t nr = (uint32_t)min(s.Lr - ar, s.Lq - aq);
    walk_fast<true>(s.ref, s.qry, ar, aq, nr, tlo, thi, tab25, X, T - ML, &acc);
    return acc ? 1 : 0;
}

__device__ __forceinline__ uint32_t upper_bound_g(const uint32_t *__restrict__ P, uint32_t lo, uint32_t hi,
                                                  uint32_t key) {
    while (lo < hi) {
        uint32_t mid = lo + ((hi - lo) >> 1);
        if (__ldg(P + mid) <= key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

constexpr int kFuseThreads = 256;
constexpr int kFuseItems = 4;
constexpr int kFuseTile = kFuseThreads * kFuseItems;
constexpr int kFuseSeeds = 2048;

// Fused C.5 + D.2/D.3: the CTA owns kFuseTile consecutive anchor slots of the
// chunk.  Each slot's seed is the first seed whose inclusive prefix exceeds
// the slot's global id; its occurrence index follows from the backward slot
// rule j = P[s] - 1 - id.  The anchor is written, then gated.
template <bool GATE>
__global__ void __launch_bounds__(kFuseThreads) k_expand_gate(const uint32_t *__restrict__ P,
                                                              const uint32_t *__restrict__ lo,
                                                              const uint32_t *__restrict__ pos, uint32_t sb,
                                                              uint32_t se, uint32_t hb, uint64_t n_hits,
                                                              uint32_t span, Seqs sq, ScoreArgs sa,
                                                              uint2 *__restrict__ out, uint8_t *__restrict__ flags) {
    __shared__ int tab[25];
    __shared__ uint32_t sP[kFuseSeeds];
    __shared__ uint32_t s_first, s_count;
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    const uint64_t t0 = (uint64_t)blockIdx.x * kFuseTile;
    const uint64_t t1 = min(n_hits, t0 + kFuseTile);
    if (threadIdx.x == 0) {
        uint32_t a = upper_bound_g(P, sb, se, hb + (uint32_t)t0);
        uint32_t b = upper_bound_g(P, a, se, hb + (uint32_t)(t1 - 1));
        s_first = a;
        s_count = b - a + 1;
    }
    __syncthreads();
    const uint32_t first = s_first, count = s_count;
    const bool cached = count <= (uint32_t)kFuseSeeds;
    if (cached)
        for (uint32_t i = threadIdx.x; i < count; i += kFuseThreads) sP[i] = __ldg(P + first + i);
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < kFuseItems; ++k) {
        const uint64_t t = t0 + (uint64_t)k * kFuseThreads + threadIdx.x;
        if (t >= t1) break;
        const uint32_t gid = hb + (uint32_t)t;
        uint32_t s, pend;
        if (cached) {
            uint32_t l = 0, h = count;
            while (l < h) {
                uint32_t mid = (l + h) >> 1;
                if (sP[mid] <= gid) l = mid + 1; else h = mid;
            }
            s = first + l;
            pend = sP[l];
        } else {
            s = upper_bound_g(P, first, first + count, gid);
            pend = __ldg(P + s);
        }
        const uint32_t j = pend - 1 - gid;
        const uint32_t re = __ldg(pos + __ldg(lo + s) + j), qe = s + span - 1;
        out[t] = make_uint2(re, qe);
        if (GATE) flags[t] = (uint8_t)gate_one(sq, tab, sa.xdrop, sa.T, re, qe);
    }
}

// ------------------------------------------------------------------ warp helpers for the fused fast kernel
constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Mask of the low min(n, 8) nibbles (the bases of a step inside the walk).
__device__ __forceinline__ uint32_t low_nibbles(uint32_t n) {
    const uint32_t s = min(n, 8u) * 4u;
    uint32_t d;
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(0xFFFFFFFFu), "r"(s));  // shifts of 32 give 0
    return ~d;
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

__device__ __forceinline__ void walk_advance(WalkState &w, int S_next) {
    w.rem -= 8;
    w.S = S_next;
    w.r0 = w.r1;
    w.q0 = w.q1;
    w.pr++;
    w.pq++;
    w.r1 = __ldg(w.pr + 1);
    w.q1 = __ldg(w.pq + 1);
}

// The common 8-base step.  It advances the walk and returns false unless the
// step may hold the stop, reaches `need` or ends at the edge; then it leaves
// the walk untouched and returns true for walk_resolve.
template <bool HAS_N>
__device__ __forceinline__ bool walk_step(WalkState &w, uint32_t tlo, uint32_t thi, const int *__restrict__ tab25,
                                          int X, int need, int (&Sv)[8], int &Mb, bool &maybe_stop) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab25, w.S, Sv);
    const int hi = max(max(max(Sv[0], Sv[1]), max(Sv[2], Sv[3])), max(max(Sv[4], Sv[5]), max(Sv[6], Sv[7])));
    const int lo = min(min(min(Sv[0], Sv[1]), min(Sv[2], Sv[3])), min(min(Sv[4], Sv[5]), min(Sv[6], Sv[7])));
    Mb = max(w.M, hi);
    // sign bits: lo - Mb + X < 0 when the step may hold the stop, need - 1 - Mb < 0 when it reaches need
    const int gap = lo - Mb + X;
    maybe_stop = gap < 0;
    if (!(((gap | (need - 1 - Mb)) < 0) | (w.rem <= 8))) {
        w.M = Mb;
        walk_advance(w, Sv[7]);
        return false;
    }
    return true;
}

// Settles a flagged step.  Returns true when the side is over, with *acc
// telling whether its maximum reached `need`; else the walk has advanced.
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
    walk_advance(w, Sv[7]);
    return false;
}

// The 8-base step with an exact stop test, for scoring where X >= 7 * the
// largest single-pair score (and X >= 0).  Base k of the step stops the walk
// when it falls more than X below the running maximum m(k-1) of the bases
// before it.  After such a stop the remaining (at most 7) sums of the step
// cannot climb back above m(k-1), so the step's final running maximum is the
// side maximum at the stop: the step never has to be replayed base by base.
// Returns true when the side is over (stop, `need` reached or edge) with
// w.M = the side maximum; otherwise the walk has advanced.
template <bool HAS_N>
__device__ __forceinline__ bool walk_step_exact(WalkState &w, uint32_t tlo, uint32_t thi,
                                                const int *__restrict__ tab25, int X, int need) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    int Sv[8];
    step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab25, w.S, Sv);
    // d collects the sign of S(k) + X - m(k-1) for every base k
    int m = w.M, d = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        d |= Sv[k] + X - m;
        m = max(m, Sv[k]);
    }
    w.M = m;
    if (((d | (need - 1 - m)) < 0) | (w.rem <= 8)) return true;
    walk_advance(w, Sv[7]);
    return false;
}

// walk_step_exact without branches, for the steps every lane of a round runs
// together: a lane whose side is over (or that has no walk) keeps its state,
// and only its loads are skipped.
template <bool HAS_N>
__device__ __forceinline__ void walk_step_exact_sel(WalkState &w, bool &stepping, uint32_t tlo, uint32_t thi,
                                                    const int *__restrict__ tab25, int X, int need) {
    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
    int Sv[8];
    step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab25, w.S, Sv);
    int m = w.M, d = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) {
        d |= Sv[k] + X - m;
        m = max(m, Sv[k]);
    }
    const bool over = ((d | (need - 1 - m)) < 0) | (w.rem <= 8);
    const bool adv = stepping && !over;
    w.M = stepping ? m : w.M;
    stepping = adv;
    w.rem = adv ? w.rem - 8u : w.rem;
    w.S = adv ? Sv[7] : w.S;
    w.r0 = adv ? w.r1 : w.r0;
    w.q0 = adv ? w.q1 : w.q0;
    w.pr += adv ? 1 : 0;
    w.pq += adv ? 1 : 0;
    if (adv) {
        w.r1 = __ldg(w.pr + 1);
        w.q1 = __ldg(w.pq + 1);
    }
}

// Steps of each side that a round runs without votes before its vote loop.
// A round lasts the longest walk of its 32 lanes (for random anchors ~8 steps
// on the left, ~6 on the right), so these steps are rarely extra, and a
// branch-free step costs fewer instructions than a step of the vote loop and
// lets consecutive steps overlap.  Measured on workload_a: (7, 5) beat
// shorter and longer leads.
constexpr int kLeadLeft = 7, kLeadRight = 5;

// One synchronous round of 32 anchors, one per lane (`walk0` false for an
// empty slot): all lanes start their left side together, step until every
// lane's side is over, then do the right side the same way.  The right
// side's first words are loaded with the left side's.  EXACT selects
// walk_step_exact; otherwise flagged steps are settled by walk_resolve,
// together, after every lane has flagged.  Returns the keep decision.
template <bool HAS_N, bool EXACT>
__device__ __forceinline__ bool gate_round(uint2 a, bool walk0, const Seqs &sq, const uint32_t *__restrict__ ref_rev,
                                           const uint32_t *__restrict__ qry_rev, uint32_t tlo, uint32_t thi,
                                           const int *__restrict__ tab, int X, int T) {
    bool accepted = false;
    int need = T;
    uint32_t nr0 = 0, nr1 = 0, nq0 = 0, nq1 = 0;  // the right side's first words
#pragma unroll 1
    for (int side = 0; side < 2; side++) {
        const bool walk = walk0 && !accepted;
        WalkState w;
        if (walk) {
            walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, side);
            if (side == 0) {  // the left side's first words, and the right side's, in one go
                w.r0 = __ldg(w.pr);
                w.r1 = __ldg(w.pr + 1);
                w.q0 = __ldg(w.pq);
                w.q1 = __ldg(w.pq + 1);
                const uint32_t jr = a.x + (uint32_t)kPadBases, jq = a.y + (uint32_t)kPadBases;
                nr0 = __ldg(sq.ref + (jr >> 3));
                nr1 = __ldg(sq.ref + (jr >> 3) + 1);
                nq0 = __ldg(sq.qry + (jq >> 3));
                nq1 = __ldg(sq.qry + (jq >> 3) + 1);
            } else {
                w.r0 = nr0;
                w.r1 = nr1;
                w.q0 = nq0;
                w.q1 = nq1;
            }
        }
        bool stepping = walk;
        if (EXACT) {
            if (!walk) w = WalkState{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
            if (side == 0) {
#pragma unroll
                for (int i = 0; i < kLeadLeft; i++) walk_step_exact_sel<HAS_N>(w, stepping, tlo, thi, tab, X, need);
            } else {
#pragma unroll
                for (int i = 0; i < kLeadRight; i++) walk_step_exact_sel<HAS_N>(w, stepping, tlo, thi, tab, X, need);
            }
            while (__any_sync(kFullMask, stepping)) {
                if (stepping && walk_step_exact<HAS_N>(w, tlo, thi, tab, X, need)) stepping = false;
            }
            if (walk) {
                accepted = w.M >= need;
                need = T - w.M;
            }
        } else {
            bool ended = !walk;
            int Sv[8], Mb = 0;
            bool maybe_stop = false;
            while (__any_sync(kFullMask, !ended)) {
                while (__any_sync(kFullMask, stepping)) {
                    if (stepping && walk_step<HAS_N>(w, tlo, thi, tab, X, need, Sv, Mb, maybe_stop)) stepping = false;
                }
                if (!ended) {
                    bool acc = false;
                    if (walk_resolve(w, Sv, Mb, maybe_stop, X, need, &acc)) {
                        ended = true;
                        accepted = acc;
                        need = T - w.M;
                    } else {
                        stepping = true;
                    }
                }
            }
        }
    }
    return accepted;
}

constexpr int kWWarps = 8;             // warps per CTA
constexpr int kWUnit = 256;            // anchor slots per warp
constexpr int kWTile = kWWarps * kWUnit;
constexpr int kWSeeds = 2048;          // cached seed prefixes per CTA

// The seeds of the first and last anchor slot of every tile (thread per tile).
__global__ void k_tile_seeds(const uint32_t *__restrict__ P, uint32_t sb, uint32_t se, uint32_t hb, uint64_t n_hits,
                             uint64_t n_tiles, uint32_t *__restrict__ tiles) {
    for (uint64_t t = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; t < n_tiles;
         t += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t s0 = t * kWTile, s1 = min(n_hits, s0 + kWTile) - 1;
        const uint32_t a = upper_bound_g(P, sb, se, hb + (uint32_t)s0);
        tiles[2 * t] = a;
        tiles[2 * t + 1] = upper_bound_g(P, a, se, hb + (uint32_t)s1);
    }
}

// Fused expansion + gate.  The CTA owns kWTile consecutive anchor slots and
// caches the prefixes of the seeds they come from; after that one barrier
// every warp works alone on its own 256 slots:
//   1. lane l expands slots 8l..8l+7 of the warp's share into shared memory
//      (search for the first slot's seed, then walk forward);
//   2. the gate runs in 8 synchronous rounds of 32 anchors (one per lane):
//      all lanes start their left side together, step until every lane has
//      flagged a step that may hold its stop, reaches `need` or ends at the
//      edge, settle together, then the same for the right side;
//   3. the warp stores its anchors and flags with coalesced writes.
template <bool HAS_N, bool EXACT>
__global__ void __launch_bounds__(kWWarps * 32, 5)
    k_expand_gate_w(const uint32_t *__restrict__ P, const uint32_t *__restrict__ lo,
                    const uint32_t *__restrict__ pos, uint32_t sb, uint32_t se, uint32_t hb, uint64_t n_hits,
                    uint32_t span, Seqs sq, const uint32_t *__restrict__ ref_rev,
                    const uint32_t *__restrict__ qry_rev, const uint32_t *__restrict__ tiles, ScoreArgs sa,
                    uint2 *__restrict__ out, uint8_t *__restrict__ flags) {
    __shared__ uint2 sA_all[kWTile];
    __shared__ uint32_t sP[kWSeeds];
    __shared__ int tab[25];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t tile0 = (uint64_t)blockIdx.x * kWTile;
    const uint32_t tile_count = (uint32_t)min((uint64_t)kWTile, n_hits - tile0);
    if (tid < 25) tab[tid] = sa.m[tid];
    const uint32_t first = __ldg(tiles + 2 * (uint64_t)blockIdx.x), ns = __ldg(tiles + 2 * (uint64_t)blockIdx.x + 1) - first + 1;
    const bool cached = ns <= (uint32_t)kWSeeds;
    if (cached)
        for (uint32_t i = tid; i < ns; i += kWWarps * 32) sP[i] = __ldg(P + first + i);
    __syncthreads();
    const uint32_t wbase = (uint32_t)warp * kWUnit;  // this warp's slots within the tile
    if (wbase >= tile_count) return;
    const uint32_t count = min((uint32_t)kWUnit, tile_count - wbase);
    const uint64_t t0 = tile0 + wbase;
    uint2 *sA = sA_all + wbase;

    // 1. expansion
    const uint32_t i0 = (uint32_t)lane * 8u;
    if (i0 < count) {
        const uint32_t g0 = hb + (uint32_t)t0 + i0;
        uint32_t l;
        if (cached) {
            uint32_t x = 0, y = ns;
            while (x < y) {
                const uint32_t mid = (x + y) >> 1;
                if (sP[mid] <= g0) x = mid + 1; else y = mid;
            }
            l = x;
        } else {
            l = upper_bound_g(P, first, first + ns, g0) - first;
        }
        uint32_t pend = cached ? sP[l] : __ldg(P + first + l);
        uint32_t base = __ldg(lo + first + l);
        const uint32_t kmax = min(8u, count - i0);
        for (uint32_t k = 0; k < kmax; k++) {
            const uint32_t g = g0 + k;
            while (pend <= g) {
                l++;
                pend = cached ? sP[l] : __ldg(P + first + l);
                base = __ldg(lo + first + l);
            }
            sA[i0 + k] = make_uint2(__ldg(pos + base + (pend - 1 - g)), first + l + span - 1);
        }
    }
    __syncwarp();

    // 2. gate rounds
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop, T = sa.T;
    for (uint32_t round = 0; round * 32 < count; round++) {
        const uint32_t ai = round * 32u + (uint32_t)lane;
        const bool valid = ai < count;
        uint2 a = make_uint2(0, 0);
        if (valid) a = sA[ai];
        const bool accepted = gate_round<HAS_N, EXACT>(a, valid, sq, ref_rev, qry_rev, tlo, thi, tab, X, T);
        if (valid) flags[t0 + ai] = accepted ? 1 : 0;
    }
    // 3. anchors
    for (uint32_t i = lane; i < count; i += 32) out[t0 + i] = sA[i];
}

// Round-based fast gate over an anchor array in global memory (the standalone
// gate, and the gate of the reference-bucketed mode, whose anchors arrive
// sorted by reference window with their raw ids).  One warp per unit of 256
// anchors, 8 synchronous rounds of 32 as in k_expand_gate_w; the flag of
// anchor i goes to flags[raw ? raw[i] : i].
template <bool HAS_N, bool EXACT>
__global__ void __launch_bounds__(kWWarps * 32, 5)
    k_gate_rounds(const uint2 *__restrict__ anchors, const uint32_t *__restrict__ raw, uint64_t n, Seqs sq,
                  const uint32_t *__restrict__ ref_rev, const uint32_t *__restrict__ qry_rev, ScoreArgs sa,
                  uint8_t *__restrict__ flags) {
    __shared__ int tab[25];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 25) tab[tid] = sa.m[tid];
    __syncthreads();
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop, T = sa.T;
    const uint64_t n_units = (n + kWUnit - 1) / kWUnit;
    for (uint64_t u = (uint64_t)blockIdx.x * kWWarps + warp; u < n_units; u += (uint64_t)gridDim.x * kWWarps) {
        const uint64_t t0 = u * kWUnit;
        const uint32_t count = (uint32_t)min((uint64_t)kWUnit, n - t0);
        for (uint32_t round = 0; round * 32 < count; round++) {
            const uint32_t ai = round * 32u + (uint32_t)lane;
            const bool valid = ai < count;
            uint2 a = make_uint2(0, 0);
            if (valid) a = anchors[t0 + ai];
            const bool inside = valid && a.x < sq.Lr && a.y < sq.Lq;
            const bool accepted = gate_round<HAS_N, EXACT>(a, inside, sq, ref_rev, qry_rev, tlo, thi, tab, X, T);
            if (valid) flags[raw ? raw[t0 + ai] : t0 + ai] = accepted ? 1 : 0;
        }
    }
}

template <bool FAST>
__global__ void __launch_bounds__(256) k_gate(const uint2 *__restrict__ anchors, uint64_t n, Seqs sq, ScoreArgs sa,
                                              uint8_t *__restrict__ flags) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint2 a = anchors[i];
        flags[i] = (uint8_t)(FAST ? gate_fast(sq, tab, sa.tab_lo, sa.tab_hi, sa.xdrop, sa.T, a.x, a.y)
                                  : gate_one(sq, tab, sa.xdrop, sa.T, a.x, a.y));
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

// One lane per survivor (E.1-E.5).  The lane walks its left side, then its
// right side, in one loop (both over forward-running copies), so lanes do not
// wait for one another between the sides; consecutive survivors come from the
// same homology and take similar total walks.  The earliest maximum is kept
// lazily: the step in which the maximum last rose and the running sum at that
// step's start; when the side ends that one step is scored again to find the
// exact base (E.2 invariant).  A side that passes 2^20 steps (|S| could then
// approach 2^31) sends the survivor to the 64-bit base-by-base walk.
template <bool HAS_N>
__global__ void __launch_bounds__(256) k_materialize_lane(const uint2 *__restrict__ anchors, uint64_t n_anchors,
                                                          uint32_t id_base, const uint32_t *__restrict__ ids,
                                                          uint64_t n_ids, const uint64_t *__restrict__ d_n, Seqs sq,
                                                          const uint32_t *__restrict__ ref_rev,
                                                          const uint32_t *__restrict__ qry_rev, ScoreArgs sa,
                                                          uint4 *__restrict__ out, uint8_t *__restrict__ done) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    if (d_n) n_ids = *d_n <= n_ids ? *d_n : 0;
    for (uint64_t k = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; k < n_ids; k += stride) {
        const uint32_t id = ids[k];
        const uint64_t slot = (uint64_t)id - id_base;
        const uint2 a = (id >= id_base && slot < n_anchors) ? anchors[slot] : make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        uint4 rec = make_uint4(0, 0, 0, 0);
        uint8_t ok = 0;
        if (a.x < sq.Lr && a.y < sq.Lq) {
            int64_t ML = 0, MR = 0;
            uint32_t nL = 0, nR = 0;
            bool long_walk = false;
            {
                int side = 0;
                WalkState w;
                walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 0);
                w.r0 = __ldg(w.pr);
                w.r1 = __ldg(w.pr + 1);
                w.q0 = __ldg(w.pq);
                w.q1 = __ldg(w.pq + 1);
                int mstep = -1, mS = 0;
                uint32_t steps = 0;
                for (;;) {
                    const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
                    const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
                    int Sv[8];
                    step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab, w.S, Sv);
                    const int hi = max(max(max(Sv[0], Sv[1]), max(Sv[2], Sv[3])),
                                       max(max(Sv[4], Sv[5]), max(Sv[6], Sv[7])));
                    const int lo = min(min(min(Sv[0], Sv[1]), min(Sv[2], Sv[3])),
                                       min(min(Sv[4], Sv[5]), min(Sv[6], Sv[7])));
                    const int Mb = max(w.M, hi);
                    const bool maybe_stop = lo < Mb - X;
                    if (!(maybe_stop | (w.rem <= 8))) {
                        if (hi > w.M) {
                            mstep = (int)steps;
                            mS = w.S;
                        }
                        w.M = Mb;
                        walk_advance(w, Sv[7]);
                        if (++steps >= (1u << 20)) {
                            long_walk = true;
                            break;
                        }
                        continue;
                    }
                    // a step that may hold the stop, or the edge: settle it base by base
                    int Mf = w.M, kset = -1;
                    bool dropped = false;
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        if (Mf - Sv[j] > X) {
                            dropped = true;
                            break;
                        }
                        if (Sv[j] > Mf) {
                            Mf = Sv[j];
                            kset = j;
                        }
                    }
                    if (!dropped && w.rem > 8) {  // no stop after all: walk on
                        if (kset >= 0) {
                            mstep = (int)steps;
                            mS = w.S;
                        }
                        w.M = Mf;
                        walk_advance(w, Sv[7]);
                        if (++steps >= (1u << 20)) {
                            long_walk = true;
                            break;
                        }
                        continue;
                    }
                    uint32_t nbest = 0;
                    if (kset >= 0) {
                        nbest = steps * 8u + (uint32_t)kset + 1u;
                    } else if (mstep >= 0) {  // score the step of the maximum again
                        const uint32_t back = steps - (uint32_t)mstep;
                        const uint32_t *pr = w.pr - back, *pq = w.pq - back;
                        int Sm[8];
                        step_sums<true, HAS_N>(__funnelshift_r(__ldg(pr), __ldg(pr + 1), w.shr),
                                        __funnelshift_r(__ldg(pq), __ldg(pq + 1), w.shq), 0xFFFFFFFFu, tlo, thi,
                                        tab, mS, Sm);
                        int kk = 7;
#pragma unroll
                        for (int j = 6; j >= 0; j--)
                            if (Sm[j] == Mf) kk = j;
                        nbest = (uint32_t)mstep * 8u + (uint32_t)kk + 1u;
                    }
                    if (side == 1) {
                        MR = Mf;
                        nR = nbest;
                        break;
                    }
                    ML = Mf;
                    nL = nbest;
                    side = 1;
                    walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 1);
                    w.r0 = __ldg(w.pr);
                    w.r1 = __ldg(w.pr + 1);
                    w.q0 = __ldg(w.pq);
                    w.q1 = __ldg(w.pq + 1);
                    mstep = -1;
                    mS = 0;
                    steps = 0;
                }
            }
            if (long_walk) {
                uint64_t n0, n1;
                side_exact(sq, tab, sa.xdrop, a.x, a.y, false, ML, n0);
                side_exact(sq, tab, sa.xdrop, a.x, a.y, true, MR, n1);
                nL = (uint32_t)n0;
                nR = (uint32_t)n1;
            }
            int64_t score = ML + MR;
            if (score > 2147483647LL) score = 2147483647LL;
            if (score >= sa.T) {
                rec = make_uint4(a.x - nL, a.y - nL, nL + nR - 1u, (uint32_t)(int32_t)score);
                ok = 1;
            }
        }
        out[k] = rec;
        done[k] = ok;
    }
}

// k_materialize_lane for scoring where the 8-base stop test is exact
// (X >= 7 x the largest pair score, see walk_step_exact).  Lanes step in
// blocks of kMatBlock branch-free steps between checks: a lane whose side
// ended keeps its state until the block is over, then, in a short divergent
// settle, places the side's earliest maximum by scoring the step of its last
// rise again and starts its right side or finishes.  Same records as
// k_materialize_lane.
constexpr int kMatBlock = 8;

template <bool HAS_N>
__global__ void __launch_bounds__(256) k_materialize_blocks(const uint2 *__restrict__ anchors, uint64_t n_anchors,
                                                            uint32_t id_base, const uint32_t *__restrict__ ids,
                                                            uint64_t n_ids, const uint64_t *__restrict__ d_n, Seqs sq,
                                                            const uint32_t *__restrict__ ref_rev,
                                                            const uint32_t *__restrict__ qry_rev, ScoreArgs sa,
                                                            uint4 *__restrict__ out, uint8_t *__restrict__ done) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    if (d_n) n_ids = *d_n <= n_ids ? *d_n : 0;
    // the grid-stride loop runs the same number of trips in every lane of a warp
    const uint64_t first = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    const uint64_t trips = (n_ids + stride - 1) / stride;
    for (uint64_t t = 0; t < trips; t++) {
        const uint64_t k = first + t * stride;
        uint2 a = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        if (k < n_ids) {
            const uint32_t id = ids[k];
            const uint64_t slot = (uint64_t)id - id_base;
            if (id >= id_base && slot < n_anchors) a = anchors[slot];
        }
        const bool inside = a.x < sq.Lr && a.y < sq.Lq;
        WalkState w{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        if (inside) {
            walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 0);
            w.r0 = __ldg(w.pr);
            w.r1 = __ldg(w.pr + 1);
            w.q0 = __ldg(w.pq);
            w.q1 = __ldg(w.pq + 1);
        }
        bool active = inside, stepping = inside, long_walk = false;
        int side = 0, ML = 0, MR = 0;
        uint32_t nL = 0, nR = 0, steps = 0;
        int mstep = -1, mS = 0;  // the step in which the maximum last rose, and the sum at its start
        while (__any_sync(kFullMask, active)) {
#pragma unroll
            for (int u = 0; u < kMatBlock; u++) {
                const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
                const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
                int Sv[8];
                step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab, w.S, Sv);
                int m = w.M, d = 0;
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    d |= Sv[j] + X - m;
                    m = max(m, Sv[j]);
                }
                const bool over = (d < 0) | (w.rem <= 8);
                const bool rose = stepping && m > w.M;
                mstep = rose ? (int)steps : mstep;
                mS = rose ? w.S : mS;
                const bool adv = stepping && !over;
                w.M = stepping ? m : w.M;
                stepping = adv;
                steps += adv ? 1u : 0u;
                w.rem = adv ? w.rem - 8u : w.rem;
                w.S = adv ? Sv[7] : w.S;
                w.r0 = adv ? w.r1 : w.r0;
                w.q0 = adv ? w.q1 : w.q0;
                w.pr += adv ? 1 : 0;
                w.pq += adv ? 1 : 0;
                if (adv) {
                    w.r1 = __ldg(w.pr + 1);
                    w.q1 = __ldg(w.pq + 1);
                }
            }
            if (stepping && steps >= (1u << 20)) {  // |S| must stay far from 2^31
                long_walk = true;
                stepping = false;
                active = false;
            }
            if (active && !stepping) {
                // the side is over: its maximum w.M, first reached in step mstep
                uint32_t nbest = 0;
                if (mstep >= 0) {
                    const uint32_t back = steps - (uint32_t)mstep;
                    const uint32_t *pr = w.pr - back, *pq = w.pq - back;
                    const uint32_t keep = low_nibbles(w.rem + 8u * back);
                    int Sm[8];
                    step_sums<true, HAS_N>(__funnelshift_r(__ldg(pr), __ldg(pr + 1), w.shr),
                                           __funnelshift_r(__ldg(pq), __ldg(pq + 1), w.shq), keep, tlo, thi, tab, mS,
                                           Sm);
                    int kk = 7;
#pragma unroll
                    for (int j = 6; j >= 0; j--)
                        if (Sm[j] == w.M) kk = j;
                    nbest = (uint32_t)mstep * 8u + (uint32_t)kk + 1u;
                }
                if (side == 0) {
                    ML = w.M;
                    nL = nbest;
                    side = 1;
                    walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 1);
                    w.r0 = __ldg(w.pr);
                    w.r1 = __ldg(w.pr + 1);
                    w.q0 = __ldg(w.pq);
                    w.q1 = __ldg(w.pq + 1);
                    mstep = -1;
                    mS = 0;
                    steps = 0;
                    stepping = true;
                } else {
                    MR = w.M;
                    nR = nbest;
                    active = false;
                }
            }
        }
        if (k >= n_ids) continue;
        uint4 rec = make_uint4(0, 0, 0, 0);
        uint8_t ok = 0;
        if (inside) {
            int64_t L = ML, Rt = MR;
            if (long_walk) {
                uint64_t n0, n1;
                side_exact(sq, tab, sa.xdrop, a.x, a.y, false, L, n0);
                side_exact(sq, tab, sa.xdrop, a.x, a.y, true, Rt, n1);
                nL = (uint32_t)n0;
                nR = (uint32_t)n1;
            }
            int64_t score = L + Rt;
            if (score > 2147483647LL) score = 2147483647LL;
            if (score >= sa.T) {
                rec = make_uint4(a.x - nL, a.y - nL, nL + nR - 1u, (uint32_t)(int32_t)score);
                ok = 1;
            }
        }
        out[k] = rec;
        done[k] = ok;
    }
}

// One thread per survivor (E.1-E.5), any matrix: 64-bit base-by-base walks.
__global__ void __launch_bounds__(128) k_materialize(const uint2 *__restrict__ anchors, uint64_t n_anchors, uint32_t id_base,
                                                     const uint32_t *__restrict__ ids, uint64_t n_ids,
                                                     const uint64_t *__restrict__ d_n, Seqs sq, ScoreArgs sa,
                                                     uint4 *__restrict__ out, uint8_t *__restrict__ done) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    if (d_n) n_ids = *d_n <= n_ids ? *d_n : 0;
    for (uint64_t k = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; k < n_ids;
         k += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t id = ids[k];
        const uint64_t slot = (uint64_t)id - id_base;  // wraps above n_anchors when id < id_base
        const uint2 a = (id >= id_base && slot < n_anchors) ? anchors[slot] : make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        uint4 rec = make_uint4(0, 0, 0, 0);
        uint8_t ok = 0;
        if (a.x < sq.Lr && a.y < sq.Lq) {
            int64_t ML, MR;
            uint64_t nL, nR;
            side_exact(sq, tab, sa.xdrop, a.x, a.y, false, ML, nL);
            side_exact(sq, tab, sa.xdrop, a.x, a.y, true, MR, nR);
            int64_t score = ML + MR;
            if (score > 2147483647LL) score = 2147483647LL;
            if (score >= sa.T) {
                rec = make_uint4(a.x - (uint32_t)nL, a.y - (uint32_t)nL, (uint32_t)(nL + nR - 1), (uint32_t)(int32_t)score);
                ok = 1;
            }
        }
        out[k] = rec;
        done[k] = ok;
    }
}

unsigned grid_cap(uint64_t n, int threads) {
    uint64_t g = (n + threads - 1) / threads;
    const uint64_t cap = 152ull * 64;
    return (unsigned)(g < 1 ? 1 : (g > cap ? cap : g));
}

Seqs seqs(SeqView r, SeqView q) { return Seqs{r.packed, q.packed, r.len, q.len}; }

}  // namespace

uint64_t expand_gate_tile_words(uint64_t max_chunk_hits) { return 2 * ((max_chunk_hits + kWTile - 1) / kWTile) + 2; }

cudaError_t launch_expand_gate(const uint32_t *d_P, const uint32_t *d_lo, const uint32_t *d_pos, const hspz_chunk &c,
                               int span, SeqView ref, SeqView qry, const ScoreArgs &sa, hspz_anchor *d_out,
                               uint8_t *d_flags, uint32_t *d_tiles, cudaStream_t st) {
    const uint64_t n = (uint64_t)c.hit_end - c.hit_begin;
    if (!n) return cudaSuccess;
    const uint64_t blocks = (n + kFuseTile - 1) / kFuseTile;
    uint2 *out = reinterpret_cast<uint2 *>(d_out);
    const unsigned g = (unsigned)blocks;
    const uint32_t sb = c.seed_begin, se = c.seed_end, hb = c.hit_begin;
    if (!d_flags) {
        k_expand_gate<false><<<g, kFuseThreads, 0, st>>>(d_P, d_lo, d_pos, sb, se, hb, n, span, seqs(ref, qry), sa, out, d_flags); count_launch();
    } else if (sa.fast) {
        const uint64_t n_tiles = (n + kWTile - 1) / kWTile;
        k_tile_seeds<<<(unsigned)((n_tiles + 255) / 256), 256, 0, st>>>(d_P, sb, se, hb, n, n_tiles, d_tiles); count_launch();
        auto kern = sa.exact ? (ref.has_n || qry.has_n ? k_expand_gate_w<true, true> : k_expand_gate_w<false, true>)
                             : (ref.has_n || qry.has_n ? k_expand_gate_w<true, false> : k_expand_gate_w<false, false>);
        kern<<<(unsigned)n_tiles, kWWarps * 32, 0, st>>>(d_P, d_lo, d_pos, sb, se, hb, n, span, seqs(ref, qry), ref.rev,
                                                         qry.rev, d_tiles, sa, out, d_flags); count_launch();
    } else {
        k_expand_gate<true><<<g, kFuseThreads, 0, st>>>(d_P, d_lo, d_pos, sb, se, hb, n, span, seqs(ref, qry), sa, out, d_flags); count_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_gate(const hspz_anchor *d_anchors, const uint32_t *d_raw, uint64_t n, SeqView ref, SeqView qry,
                        const ScoreArgs &sa, uint8_t *d_flags, cudaStream_t st) {
    if (!n) return cudaSuccess;
    if (sa.fast) {
        const uint64_t units = (n + kWUnit - 1) / kWUnit, want = (units + kWWarps - 1) / kWWarps;
        const unsigned g = (unsigned)(want < 152ull * 40 ? want : 152ull * 40);
        auto kern = sa.exact ? (ref.has_n || qry.has_n ? k_gate_rounds<true, true> : k_gate_rounds<false, true>)
                             : (ref.has_n || qry.has_n ? k_gate_rounds<true, false> : k_gate_rounds<false, false>);
        kern<<<g, kWWarps * 32, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), d_raw, n, seqs(ref, qry), ref.rev,
                                         qry.rev, sa, d_flags); count_launch();
    } else if (!d_raw) {
        k_gate<false><<<grid_cap(n, 256), 256, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), n, seqs(ref, qry), sa,
                                                         d_flags); count_launch();
    } else {
        return cudaErrorInvalidValue;  // raw ids come only with the fast gate
    }
    return cudaGetLastError();
}

cudaError_t launch_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                               uint64_t n_ids,
                               SeqView ref, SeqView qry, const ScoreArgs &sa, hspz_segment_pair *d_out,
                               uint8_t *d_done, cudaStream_t st, const uint64_t *d_n) {
    if (!n_ids) return cudaSuccess;
    const uint2 *an = reinterpret_cast<const uint2 *>(d_anchors);
    uint4 *out = reinterpret_cast<uint4 *>(d_out);
    if (sa.fast) {
        const uint64_t blocks = (n_ids + 255) / 256;
        const unsigned g = (unsigned)(blocks < 152ull * 64 ? blocks : 152ull * 64);
        const bool has_n = ref.has_n || qry.has_n;
        auto kern = sa.exact ? (has_n ? k_materialize_blocks<true> : k_materialize_blocks<false>)
                             : (has_n ? k_materialize_lane<true> : k_materialize_lane<false>);
        kern<<<g, 256, 0, st>>>(an, n_anchors, id_base, d_ids, n_ids, d_n, seqs(ref, qry), ref.rev, qry.rev, sa, out,
                                d_done); count_launch();
    } else {
        k_materialize<<<grid_cap(n_ids, 128), 128, 0, st>>>(an, n_anchors, id_base, d_ids, n_ids, d_n, seqs(ref, qry),
                                                                    sa, out, d_done); count_launch();
    }
    return cudaGetLastError();
}

}  // namespace hspz
