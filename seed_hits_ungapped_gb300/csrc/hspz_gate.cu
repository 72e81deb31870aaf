// Score-only X-drop gate ("D. Score gate", D.1-D.3) and the fused expansion +
// gate of one MAX_HITS chunk ("C. Hit discovery" C.5 feeding D.2).
#include "hspz_walk.cuh"

namespace hspz {
namespace {

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

// Steps of each side that a round runs without votes before its vote loop.
// A round lasts the longest walk of its 32 lanes (for random anchors ~8 steps
// on the left, ~6 on the right), so these steps are rarely extra, and
// unrolled steps without votes overlap and address their words with
// immediate offsets.  Measured on workload_a with 4-warp CTAs: (8, 6) beat
// (8, 5), (7, 6), (7, 5) and shorter leads.
#ifndef HSPZ_LEAD_LEFT
#define HSPZ_LEAD_LEFT 8
#endif
#ifndef HSPZ_LEAD_RIGHT
#define HSPZ_LEAD_RIGHT 6
#endif
constexpr int kLeadLeft = HSPZ_LEAD_LEFT, kLeadRight = HSPZ_LEAD_RIGHT;

// One side of a synchronous round.  Lanes with `walk` start together and step
// until every lane's side is over (BACK: the left side, read downwards from
// the anchor on the forward copies).  EXACT selects walk_step_lead;
// otherwise flagged steps are settled by walk_resolve, together, after every
// lane has flagged.  Leaves the side maximum in w.M and returns whether it
// reached `need`.
// The LEAD branch-free steps of one side (exact stop test), for the lanes
// with `walk`.  Afterwards w.rem = 0 for a lane whose side is over (stop,
// `need` reached, edge or no walk); otherwise the lane's side goes on from
// LEAD words past its start with w.rem bases left.
template <bool HAS_N, bool BACK, int LEAD>
__device__ __forceinline__ void side_lead(WalkState &w, bool walk, uint32_t tlo, uint32_t thi,
                                          const int *__restrict__ tab, int X, int need) {
    if (!walk) w.rem = 0;
    if (__all_sync(kFullMask, w.rem == 0u || w.rem > 8u * LEAD)) {
        // no walk of the round can reach its edge during the lead steps
        uint32_t keep = w.rem ? 0xFFFFFFFFu : 0u;
        if constexpr (HAS_N) {
            // the steps that test for N are longer: a partly rolled loop keeps
            // the code within the instruction cache
#pragma unroll 4
            for (int i = 0; i < LEAD; i++) walk_step_inner<HAS_N, BACK>(w, keep, tlo, thi, tab, X, need);
        } else {
#pragma unroll
            for (int i = 0; i < LEAD; i++) walk_step_inner<HAS_N, BACK>(w, keep, tlo, thi, tab, X, need);
        }
        w.rem = keep ? w.rem - 8u * LEAD : 0u;
    } else {
        // rounds near a sequence edge are rare: a rolled loop keeps the code small
#pragma unroll 1
        for (int i = 0; i < LEAD; i++) walk_step_lead<HAS_N, BACK>(w, tlo, thi, tab, X, need);
    }
}

template <bool HAS_N, bool EXACT, bool BACK>
__device__ __forceinline__ bool gate_side(WalkState &w, bool walk, uint32_t tlo, uint32_t thi,
                                          const int *__restrict__ tab, int X, int need) {
    if (EXACT) {
        side_lead<HAS_N, BACK, BACK ? kLeadLeft : kLeadRight>(w, walk, tlo, thi, tab, X, need);
        // the tail: the same steps under a warp vote, while any lane walks
        while (__any_sync(kFullMask, w.rem != 0)) walk_step_lead<HAS_N, BACK>(w, tlo, thi, tab, X, need);
        return walk && w.M >= need;
    }
    bool stepping = walk, ended = !walk, accepted = false;
    int Sv[8], Mb = 0;
    bool maybe_stop = false;
    while (__any_sync(kFullMask, !ended)) {
        while (__any_sync(kFullMask, stepping)) {
            if (stepping && walk_step<HAS_N, BACK>(w, tlo, thi, tab, X, need, Sv, Mb, maybe_stop)) stepping = false;
        }
        if (!ended) {
            bool acc = false;
            if (walk_resolve<BACK>(w, Sv, Mb, maybe_stop, X, need, &acc)) {
                ended = true;
                accepted = acc;
            } else {
                stepping = true;
            }
        }
    }
    return accepted;
}

// One synchronous round of 32 anchors, one per lane (`walk0` false for an
// empty slot): all lanes walk their left side, then their right side, both
// on the forward packed copies.  The left side's first window ends at the
// anchor, so its upper words are the right side's first word; only one more
// word per sequence is loaded for the right side, with the left side's.
// Returns the keep decision.
template <bool HAS_N, bool EXACT>
__device__ __forceinline__ bool gate_round(uint2 a, bool walk0, const Seqs &sq, uint32_t tlo, uint32_t thi,
                                           const int *__restrict__ tab, int X, int T) {
    WalkState w{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t nr1 = 0, nq1 = 0;  // the right side's second words
    if (walk0) {
        walk_place_fwd(w, sq, a.x, a.y, 0);
        w.r0 = __ldg(w.pr);
        w.r1 = __ldg(w.pr + 1);
        w.q0 = __ldg(w.pq);
        w.q1 = __ldg(w.pq + 1);
        nr1 = __ldg(w.pr + 2);
        nq1 = __ldg(w.pq + 2);
    }
    // the right side's first words: the left side's upper words before it moves
    const uint32_t nr0 = w.r1, nq0 = w.q1;
    bool accepted = gate_side<HAS_N, EXACT, true>(w, walk0, tlo, thi, tab, X, T);
    const int need = T - w.M;
    const bool walk1 = walk0 && !accepted;
    if (walk1) {
        walk_place_fwd(w, sq, a.x, a.y, 1);
        w.r0 = nr0;
        w.r1 = nr1;
        w.q0 = nq0;
        w.q1 = nq1;
    }
    accepted |= gate_side<HAS_N, EXACT, false>(w, walk1, tlo, thi, tab, X, need);
    return accepted;
}

// Right-side lead steps of a round whose long right walks are deferred.
#ifndef HSPZ_DEFER_RIGHT
#define HSPZ_DEFER_RIGHT 4
#endif
constexpr int kDeferRight = HSPZ_DEFER_RIGHT;
constexpr int kQueue = 64;  // deferred right walks a warp can hold (one round adds at most 32)

// gate_round for the exact step test, except that a right walk still going
// after kDeferRight steps is not finished here: *pending is set and the
// walk's running sum and maximum (w.S, w.M) and the maximum it still needs
// (*need) are left for gate_deferred.  A round lasts its slowest walk, and
// right walks mostly end within 2-4 steps while a few run much longer, so
// finishing those few together, 32 at a time, keeps the other lanes busy.
template <bool HAS_N>
__device__ __forceinline__ bool gate_round_defer(uint2 a, bool walk0, const Seqs &sq, uint32_t tlo, uint32_t thi,
                                                 const int *__restrict__ tab, int X, int T, WalkState &w,
                                                 int &need, bool &pending) {
    w = WalkState{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t nr1 = 0, nq1 = 0;
    if (walk0) {
        walk_place_fwd(w, sq, a.x, a.y, 0);
        w.r0 = __ldg(w.pr);
        w.r1 = __ldg(w.pr + 1);
        w.q0 = __ldg(w.pq);
        w.q1 = __ldg(w.pq + 1);
        nr1 = __ldg(w.pr + 2);
        nq1 = __ldg(w.pq + 2);
    }
    const uint32_t nr0 = w.r1, nq0 = w.q1;
    bool accepted = gate_side<HAS_N, true, true>(w, walk0, tlo, thi, tab, X, T);
    need = T - w.M;
    const bool walk1 = walk0 && !accepted;
    if (walk1) {
        walk_place_fwd(w, sq, a.x, a.y, 1);
        w.r0 = nr0;
        w.r1 = nr1;
        w.q0 = nq0;
        w.q1 = nq1;
    }
    side_lead<HAS_N, false, kDeferRight>(w, walk1, tlo, thi, tab, X, need);
    pending = w.rem != 0;
    return accepted | (walk1 && w.M >= need);
}

// Finishes `cnt` deferred right walks (queue entries first .. first+cnt-1,
// one per lane) and writes their flags: each walk is placed again
// kDeferRight words past the anchor with its saved sum and maximum, then all
// step together under a warp vote.
template <bool HAS_N>
__device__ __forceinline__ void gate_deferred(const uint32_t *qslot, const int *qS, const int *qM, const int *qN,
                                              uint32_t first, uint32_t cnt, const uint2 *sA, const Seqs &sq,
                                              uint32_t tlo, uint32_t thi, const int *__restrict__ tab, int X,
                                              uint8_t *__restrict__ flags) {
    const int lane = threadIdx.x & 31;
    const bool mine = (uint32_t)lane < cnt;
    WalkState w{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t ai = 0;
    int need = 0;
    if (mine) {
        const uint32_t e = first + (uint32_t)lane;
        ai = qslot[e];
        need = qN[e];
        const uint2 a = sA[ai];
        walk_place_fwd(w, sq, a.x, a.y, 1);
        w.pr += kDeferRight;
        w.pq += kDeferRight;
        w.rem -= 8u * kDeferRight;
        w.S = qS[e];
        w.M = qM[e];
        w.r0 = __ldg(w.pr);
        w.r1 = __ldg(w.pr + 1);
        w.q0 = __ldg(w.pq);
        w.q1 = __ldg(w.pq + 1);
    }
    __syncwarp();  // every entry is read before the queue is written again
    while (__any_sync(kFullMask, w.rem != 0)) walk_step_lead<HAS_N, false>(w, tlo, thi, tab, X, need);
    if (mine) __stcs(flags + ai, (uint8_t)(w.M >= need ? 1 : 0));
}

#ifndef HSPZ_GATE_MIN_BLOCKS
#define HSPZ_GATE_MIN_BLOCKS 10  // resident CTAs per SM the register budget allows
#endif
constexpr int kWWarps = 4;             // warps per CTA
constexpr int kWUnit = 256;            // anchor slots per warp
constexpr int kWTile = kWWarps * kWUnit;
constexpr int kWSeeds = 1024;          // cached seed prefixes per CTA

// The seeds of the first and last anchor slot of every tile, one thread per
// tile boundary b (anchor a = min(n, 1024 b) of the chunk): the last seed of
// tile b - 1 is the first seed whose prefix reaches hb + a, and the first seed
// of tile b the first whose prefix passes it, which is the same seed unless a
// seed ends exactly at the boundary.  So one binary search serves both.
__global__ void k_tile_seeds(const uint32_t *__restrict__ P, uint32_t sb, uint32_t se, uint32_t hb, uint64_t n_hits,
                             uint64_t n_tiles, uint32_t *__restrict__ tiles) {
    for (uint64_t b = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; b <= n_tiles;
         b += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t key = hb + (uint32_t)min(n_hits, b * (uint64_t)kWTile);
        uint32_t first;
        if (b == 0) {
            first = upper_bound_g(P, sb, se, key);
        } else {
            const uint32_t last = upper_bound_g(P, sb, se, key - 1);
            tiles[2 * b - 1] = last;
            if (b == n_tiles) continue;
            first = __ldg(P + last) > key ? last : upper_bound_g(P, last, se, key);
        }
        tiles[2 * b] = first;
    }
}

// Fused expansion + gate.  The CTA owns kWTile consecutive anchor slots and
// caches the prefixes of the seeds they come from (and their bucket starts,
// when the tile spans at most kWSeeds / 2 seeds); after that one barrier
// every warp works alone on its own 256 slots:
//   1. lane l finds the seed and occurrence of slots 8l..8l+7 of the warp's
//      share (search for the first slot's seed, then walk forward), then the
//      positions of slots l + 32k are loaded into shared memory;
//   2. the gate runs in 8 synchronous rounds of 32 anchors (one per lane):
//      all lanes walk their left sides together, first a fixed number of
//      branch-free steps, then single steps under a warp vote while any lane
//      still walks; then their right sides the same way (EXACT: a few lead
//      steps, with the longer right walks deferred and finished 32 at a time);
//   3. the warp stores its flags (per round) and anchors with coalesced,
//      cache-streaming writes.
template <bool HAS_N, bool EXACT>
__global__ void __launch_bounds__(kWWarps * 32, HSPZ_GATE_MIN_BLOCKS)
    k_expand_gate_w(const uint32_t *__restrict__ P, const uint32_t *__restrict__ lo,
                    const uint32_t *__restrict__ pos, uint32_t sb, uint32_t se, uint32_t hb, uint64_t n_hits,
                    uint32_t span, Seqs sq, const uint32_t *__restrict__ tiles, ScoreArgs sa,
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
    // a tile of at most kWSeeds / 2 seeds (the usual case) caches their bucket
    // starts too, in the upper half, loaded together with the prefixes
    const bool lo_cached = ns <= (uint32_t)kWSeeds / 2;
    const uint32_t *sL = sP + kWSeeds / 2;
    if (lo_cached) {
        for (uint32_t i = tid; i < ns; i += kWWarps * 32) {
            sP[i] = __ldg(P + first + i);
            sP[kWSeeds / 2 + i] = __ldg(lo + first + i);
        }
    } else if (cached) {
        for (uint32_t i = tid; i < ns; i += kWWarps * 32) sP[i] = __ldg(P + first + i);
    }
    __syncthreads();
    const uint32_t wbase = (uint32_t)warp * kWUnit;  // this warp's slots within the tile
    // with EXACT every warp reaches the barrier after the expansion, even one without slots
    if (!EXACT && wbase >= tile_count) return;
    const uint32_t count = wbase < tile_count ? min((uint32_t)kWUnit, tile_count - wbase) : 0u;
    const uint64_t t0 = tile0 + wbase;
    uint2 *sA = sA_all + wbase;

    // 1. expansion.  The lane first finds the seed and occurrence of each of
    // its 8 consecutive slots (from the cached prefixes) and takes their 8
    // bucket starts from the cache, or issues their 8 loads together when the
    // tile's bucket starts are not cached; the position indices then pass through
    // shared memory, so that lane l loads the positions of slots l + 32k:
    // each load instruction covers 32 consecutive anchors (a few buckets)
    // rather than 32 buckets.  The staging words sit in the warp's anchor
    // slots, XOR-swizzled so that both passes are free of bank conflicts.
    uint32_t *sW = reinterpret_cast<uint32_t *>(sA);  // 2 x 256 staging words
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
        const uint32_t kmax = min(8u, count - i0);
        uint32_t sk[8], jk[8];
#pragma unroll
        for (uint32_t k = 0; k < 8; k++) {
            const uint32_t g = g0 + min(k, kmax - 1);  // slots past the unit repeat its last one
            while (pend <= g) {
                l++;
                pend = cached ? sP[l] : __ldg(P + first + l);
            }
            sk[k] = l;
            jk[k] = pend - 1 - g;
        }
        uint32_t base[8];
#pragma unroll
        for (uint32_t k = 0; k < 8; k++) base[k] = sk[k];
        if (lo_cached) {
#pragma unroll
            for (uint32_t k = 0; k < 8; k++) base[k] = sL[base[k]];
        } else {
#pragma unroll
            for (uint32_t k = 0; k < 8; k++) base[k] = __ldg(lo + first + base[k]);
        }

        const uint32_t swz = (uint32_t)(lane >> 2);  // (slot >> 5) & 7 for slots 8l..8l+7
#pragma unroll
        for (uint32_t k = 0; k < 8; k++)
            if (k < kmax) {
                sW[(i0 + k) ^ swz] = base[k] + jk[k];
                sW[256 + ((i0 + k) ^ swz)] = sk[k];
            }
    }
    __syncwarp();
    {
        uint32_t pi[8], sv[8];
#pragma unroll
        for (uint32_t k = 0; k < 8; k++) {
            const uint32_t s = (uint32_t)lane + 32u * k;
            if (s < count) {
                pi[k] = sW[s ^ k];
                sv[k] = sW[256 + (s ^ k)];
            }
        }
        __syncwarp();  // every staging word is read before the slots are written
#pragma unroll
        for (uint32_t k = 0; k < 8; k++)
            if ((uint32_t)lane + 32u * k < count) pi[k] = __ldcs(pos + pi[k]);
#pragma unroll
        for (uint32_t k = 0; k < 8; k++)
            if ((uint32_t)lane + 32u * k < count) sA[lane + 32u * k] = make_uint2(pi[k], first + sv[k] + span - 1);
    }
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop, T = sa.T;
    if (EXACT) {
        // 2. gate rounds with deferred right walks.  After this barrier no warp
        // reads the seed prefixes again, so each warp's quarter of sP becomes its
        // queue of deferred walks (slot, running sum, maximum, needed maximum).
        __syncthreads();
        if (!count) return;
        uint32_t *qslot = sP + (uint32_t)warp * (kWSeeds / kWWarps);
        int *qS = reinterpret_cast<int *>(qslot + kQueue), *qM = qS + kQueue, *qN = qM + kQueue;
        const uint32_t lane_lt = (1u << lane) - 1u;
        uint32_t qn = 0;  // warp-uniform queue length
        for (uint32_t round = 0; round * 32 < count; round++) {
            const uint32_t ai = round * 32u + (uint32_t)lane;
            const bool valid = ai < count;
            uint2 a = make_uint2(0, 0);
            if (valid) a = sA[ai];
            WalkState w;
            int need;
            bool pending;
            const bool accepted = gate_round_defer<HAS_N>(a, valid, sq, tlo, thi, tab, X, T, w, need, pending);
            if (valid && !pending) __stcs(flags + t0 + ai, (uint8_t)(accepted ? 1 : 0));
            const uint32_t pb = __ballot_sync(kFullMask, pending);
            if (pending) {
                const uint32_t e = qn + __popc(pb & lane_lt);
                qslot[e] = ai;
                qS[e] = w.S;
                qM[e] = w.M;
                qN[e] = need;
            }
            qn += __popc(pb);
            if (qn >= 32) {
                __syncwarp();
                gate_deferred<HAS_N>(qslot, qS, qM, qN, qn - 32, 32, sA, sq, tlo, thi, tab, X, flags + t0);
                qn -= 32;
            }
        }
        if (qn) {
            __syncwarp();
            gate_deferred<HAS_N>(qslot, qS, qM, qN, 0, qn, sA, sq, tlo, thi, tab, X, flags + t0);
        }
    } else {
        __syncwarp();
        // 2. gate rounds
        for (uint32_t round = 0; round * 32 < count; round++) {
            const uint32_t ai = round * 32u + (uint32_t)lane;
            const bool valid = ai < count;
            uint2 a = make_uint2(0, 0);
            if (valid) a = sA[ai];
            const bool accepted = gate_round<HAS_N, EXACT>(a, valid, sq, tlo, thi, tab, X, T);
            if (valid) __stcs(flags + t0 + ai, (uint8_t)(accepted ? 1 : 0));
        }
    }
    // 3. anchors
    // positions, flags and anchors stream through once (cache-streaming loads and stores),
    // so the packed sequences the walks read stay in L2
    for (uint32_t i = lane; i < count; i += 32) __stcs(out + t0 + i, sA[i]);
}

// Round-based fast gate over an anchor array in global memory (the standalone
// gate, and the gate of the reference-bucketed mode, whose anchors arrive
// sorted by reference window with their raw ids).  One warp per unit of 256
// anchors, 8 synchronous rounds of 32 as in k_expand_gate_w; the flag of
// anchor i goes to flags[raw ? raw[i] : i].
template <bool HAS_N, bool EXACT>
__global__ void __launch_bounds__(kWWarps * 32, HSPZ_GATE_MIN_BLOCKS)
    k_gate_rounds(const uint2 *__restrict__ anchors, const uint32_t *__restrict__ raw, uint64_t n, Seqs sq, ScoreArgs sa,
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
            const bool accepted = gate_round<HAS_N, EXACT>(a, inside, sq, tlo, thi, tab, X, T);
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
        k_tile_seeds<<<(unsigned)((n_tiles + 256) / 256), 256, 0, st>>>(d_P, sb, se, hb, n, n_tiles, d_tiles); count_launch();
        auto kern = sa.exact ? (ref.has_n || qry.has_n ? k_expand_gate_w<true, true> : k_expand_gate_w<false, true>)
                             : (ref.has_n || qry.has_n ? k_expand_gate_w<true, false> : k_expand_gate_w<false, false>);
        kern<<<(unsigned)n_tiles, kWWarps * 32, 0, st>>>(d_P, d_lo, d_pos, sb, se, hb, n, span, seqs(ref, qry), d_tiles, sa,
                                                         out, d_flags); count_launch();
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
        kern<<<g, kWWarps * 32, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), d_raw, n, seqs(ref, qry), sa,
                                         d_flags); count_launch();
    } else if (!d_raw) {
        k_gate<false><<<grid_cap(n, 256), 256, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), n, seqs(ref, qry), sa,
                                                         d_flags); count_launch();
    } else {
        return cudaErrorInvalidValue;  // raw ids come only with the fast gate
    }
    return cudaGetLastError();
}

}  // namespace hspz
