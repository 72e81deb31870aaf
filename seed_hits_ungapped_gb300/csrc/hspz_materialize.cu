// Exact X-drop materialization ("E. X-drop materialization", E.1-E.5): one
// lane per survivor, the earliest maximum of each side, 16-byte SegmentPairs.
#include "hspz_walk.cuh"

namespace hspz {
namespace {

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

// Survivors on one diagonal share their walks.  Take survivor a and the next
// survivor b on a's diagonal, d bases further on (the next entry of the id
// list, when it lies on the same diagonal).  After its first d pairs a's right
// walk scores exactly b's pairs, its running sum differs from b's by a
// constant C (a's sum after d pairs), and as soon as a's walk stands at its
// running maximum at a step count n0 >= d, b's running maximum at the same
// base is b's running sum there too.  From then on a's maximum is C plus b's
// maximum, a's drop test is b's drop test, and b cannot have stopped before
// (its drops up to there were no larger than a's).  So a's side ends where
// b's ends, with maximum C + M_b, first reached d + n_b pairs out if
// C + M_b > S_a(n0), else at a's own earliest maximum so far.  Left walks
// join the previous survivor's left walk the same way.  With CHAIN, a walk
// stops at such a join (checked at step ends) and records (S_a(n0), its
// earliest maximum, C); k_chain_resolve then settles the linked
// survivors.  Every kChainSeg-th entry of the id list (a breaker) never
// joins, so every segment of kChainSeg entries settles on its own; the
// breakers' lanes come first, packed into warps of their own, since their
// walks run the whole length of their homologies.
#ifndef HSPZ_MATERIALIZE_CHAIN
#define HSPZ_MATERIALIZE_CHAIN 1
#endif
constexpr bool kMaterializeChain = HSPZ_MATERIALIZE_CHAIN != 0;
constexpr uint32_t kLinkR = 1, kLinkL = 2, kJoinR = 4, kJoinL = 8;
constexpr uint64_t kChainSeg = 32;  // one warp settles a segment
constexpr uint64_t kChainSlice = 1ull << 25;  // ids per launch pair: 1.3 GB of scratch at most

// Entries of a slice [n_off, n_off + cap) of an id list of capacity n_total
// whose live length (*d_n) is known on the device only; a live length above
// the capacity means nothing is materialized (the caller reports it).
__device__ __forceinline__ uint64_t live_count(uint64_t live, uint64_t n_off, uint64_t cap, uint64_t n_total) {
    if (live > n_total || live <= n_off) return 0;
    return live - n_off < cap ? live - n_off : cap;
}
struct ChainSide {
    long long M;  // the side maximum, or the running sum (and maximum) at the join
    uint32_t n;   // pairs out to the earliest base of that maximum
    int32_t C;    // joined: the running sum after the first d pairs
};
struct ChainInfo {
    uint32_t flags;  // kLinkR / kLinkL: the next / previous entry is the neighbour on this diagonal; kJoinR, kJoinL
    uint32_t dR;     // linked: bases along the diagonal to the next survivor
};

__device__ __forceinline__ uint2 survivor_anchor(const uint2 *__restrict__ anchors, uint64_t n_anchors,
                                                 uint32_t id_base, const uint32_t *__restrict__ ids, uint64_t k) {
    const uint32_t id = ids[k];
    const uint64_t slot = (uint64_t)id - id_base;  // wraps above n_anchors when id < id_base
    return (id >= id_base && slot < n_anchors) ? anchors[slot] : make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
}

// k_materialize_lane for scoring where the 8-base stop test is exact
// (X >= 7 x the largest pair score, see walk_step_lead).  Lanes step in
// blocks of kMatBlock branch-free steps between checks: a lane whose side
// ended keeps its state until the block is over, then, in a short divergent
// settle, places the side's earliest maximum by scoring the step of its last
// rise again and starts its right side or finishes.  Same records as
// k_materialize_lane.  With CHAIN, walks also end at joins (see ChainSide);
// a survivor linked to a neighbour leaves its two sides in sR / sL and its
// links in info for k_chain_resolve, every other survivor gets its record.
constexpr int kMatBlock = 8;

#ifndef HSPZ_MAT_MIN_BLOCKS
#define HSPZ_MAT_MIN_BLOCKS 4
#endif
template <bool HAS_N, bool CHAIN>
__global__ void __launch_bounds__(256, HSPZ_MAT_MIN_BLOCKS) k_materialize_blocks(const uint2 *__restrict__ anchors, uint64_t n_anchors,
                                                            uint32_t id_base, const uint32_t *__restrict__ ids,
                                                            uint64_t n_ids, const uint64_t *__restrict__ d_n,
                                                            uint64_t n_off, uint64_t n_total, Seqs sq,
                                                            const uint32_t *__restrict__ ref_rev,
                                                            const uint32_t *__restrict__ qry_rev, ScoreArgs sa,
                                                            uint4 *__restrict__ out, uint8_t *__restrict__ done,
                                                            ChainSide *__restrict__ sR, ChainSide *__restrict__ sL,
                                                            ChainInfo *__restrict__ info,
                                                            const uint32_t *__restrict__ out_pos) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    const uint32_t tlo = sa.tab_lo, thi = sa.tab_hi;
    const int X = sa.xdrop;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    if (d_n) n_ids = live_count(*d_n, n_off, n_ids, n_total);
    // the grid-stride loop runs the same number of trips in every lane of a warp
    const uint64_t first = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    const uint64_t trips = (n_ids + stride - 1) / stride;
    const uint64_t n_break = (n_ids + kChainSeg - 1) / kChainSeg;
    for (uint64_t t = 0; t < trips; t++) {
        // CHAIN: lanes 0 .. n_break-1 take the breakers (entries 0, kChainSeg, ...), the rest the other entries
        const uint64_t g = first + t * stride;
        const bool breaker = CHAIN && g < n_break;
        const uint64_t k = !CHAIN ? g : breaker ? g * kChainSeg : (g - n_break) + (g - n_break) / (kChainSeg - 1) + 1;
        uint2 a = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
        if (k < n_ids) a = survivor_anchor(anchors, n_anchors, id_base, ids, k);
        const bool inside = a.x < sq.Lr && a.y < sq.Lq;
        uint32_t dL = 0, dR = 0;  // bases to the previous / next survivor on this diagonal (0: none)
        if (CHAIN && inside) {
            if (k > 0) {
                const uint2 p = survivor_anchor(anchors, n_anchors, id_base, ids, k - 1);
                if (p.x < sq.Lr && p.y < sq.Lq && p.x - p.y == a.x - a.y && p.y < a.y) dL = a.y - p.y;
            }
            if (k + 1 < n_ids) {
                const uint2 q = survivor_anchor(anchors, n_anchors, id_base, ids, k + 1);
                if (q.x < sq.Lr && q.y < sq.Lq && q.x - q.y == a.x - a.y && q.y > a.y) dR = q.y - a.y;
            }
        }
        WalkState w{sq.ref, sq.qry, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        if (inside) {
            walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 0);
            w.r0 = __ldg(w.pr);
            w.r1 = __ldg(w.pr + 1);
            w.q0 = __ldg(w.pq);
            w.q1 = __ldg(w.pq + 1);
        }
        bool active = inside, stepping = inside, long_walk = false, joined = false, jL = false;
        int side = 0, ML = 0, MR = 0, CL = 0, CR = 0;
        uint32_t nL = 0, nR = 0, steps = 0;
        // the first step whose end lies at least d pairs out (CHAIN joins are checked from there on)
        uint32_t tjoin = (dL && !breaker) ? (dL - 1u) >> 3 : 0xFFFFFFFFu;
        int mstep = -1, mS = 0;  // the step in which the maximum last rose, and the sum at its start
        while (__any_sync(kFullMask, active)) {
#pragma unroll
            for (int u = 0; u < kMatBlock; u++) {
                const uint32_t R = __funnelshift_r(w.r0, w.r1, w.shr);
                const uint32_t Q = __funnelshift_r(w.q0, w.q1, w.shq);
                int Sv[8];
                step_sums<true, HAS_N>(R, Q, low_nibbles(w.rem), tlo, thi, tab, w.S, Sv);
                // exact stop test from the step's range (X >= 7 x the largest pair score; see
                // walk_step_lead): m is also the running maximum at the step's end
                int m, lo;
                step_range(Sv, w.M, m, lo);
                const bool over = (lo + X - m < 0) | (w.rem <= 8);
                // a join: past the neighbour and standing at the running maximum
                const bool join = CHAIN && stepping && !over && steps >= tjoin && m == Sv[7];
                joined |= join;
                const bool rose = stepping && m > w.M;
                mstep = rose ? (int)steps : mstep;
                mS = rose ? w.S : mS;
                const bool adv = stepping && !over && !join;
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
                // the side is over (or joined): its maximum w.M, first reached in step mstep
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
                int Cs = 0;
                if (CHAIN && joined) {  // the running sum after the first d pairs, scored again
                    WalkState w0;
                    walk_place(w0, sq, ref_rev, qry_rev, a.x, a.y, side);
                    const uint32_t *pr = w0.pr, *pq = w0.pq;
                    for (uint32_t left = side ? dR : dL; left;) {
                        const uint32_t kk = min(left, 8u);
                        int Sc[8];
                        step_sums<true, HAS_N>(__funnelshift_r(__ldg(pr), __ldg(pr + 1), w0.shr),
                                               __funnelshift_r(__ldg(pq), __ldg(pq + 1), w0.shq), low_nibbles(kk),
                                               tlo, thi, tab, Cs, Sc);
                        Cs = Sc[7];
                        left -= kk;
                        pr++;
                        pq++;
                    }
                }
                if (side == 0) {
                    ML = w.M;
                    nL = nbest;
                    CL = Cs;
                    jL = joined;
                    joined = false;
                    side = 1;
                    walk_place(w, sq, ref_rev, qry_rev, a.x, a.y, 1);
                    w.r0 = __ldg(w.pr);
                    w.r1 = __ldg(w.pr + 1);
                    w.q0 = __ldg(w.pq);
                    w.q1 = __ldg(w.pq + 1);
                    mstep = -1;
                    mS = 0;
                    steps = 0;
                    tjoin = (dR && !breaker) ? (dR - 1u) >> 3 : 0xFFFFFFFFu;
                    stepping = true;
                } else {
                    MR = w.M;
                    nR = nbest;
                    CR = Cs;
                    active = false;
                }
            }
        }
        if (k >= n_ids) continue;
        int64_t L = ML, Rt = MR;
        if (inside && long_walk) {
            uint64_t n0, n1;
            side_exact(sq, tab, sa.xdrop, a.x, a.y, false, L, n0);
            side_exact(sq, tab, sa.xdrop, a.x, a.y, true, Rt, n1);
            nL = (uint32_t)n0;
            nR = (uint32_t)n1;
            joined = jL = false;
        }
        if (CHAIN && (dL | dR)) {  // a run member: k_chain_resolve settles it
            info[k] = ChainInfo{(dR ? kLinkR : 0u) | (dL ? kLinkL : 0u) | (joined ? kJoinR : 0u) | (jL ? kJoinL : 0u),
                                dR};
            sR[k] = ChainSide{(long long)Rt, nR, CR};
            sL[k] = ChainSide{(long long)L, nL, CL};
            continue;
        }
        if (CHAIN) info[k] = ChainInfo{0u, 0u};
        uint4 rec = make_uint4(0, 0, 0, 0);
        uint8_t ok = 0;
        if (inside) {
            int64_t score = L + Rt;
            if (score > 2147483647LL) score = 2147483647LL;
            if (score >= sa.T) {
                rec = make_uint4(a.x - nL, a.y - nL, nL + nR - 1u, (uint32_t)(int32_t)score);
                ok = 1;
            }
        }
        const uint64_t ko = out_pos ? (uint64_t)out_pos[k] : k;  // grouped order: back to the list's
        out[ko] = rec;
        done[ko] = ok;
    }
}

// Settles the linked survivors left by k_materialize_blocks<.., true>, one
// warp per segment of kChainSeg = 32 entries, a lane per entry.  Right
// sides: a joined side's maximum is C plus the next entry's maximum, so the
// maxima are suffix sums of C, each closed by a side that did not join (past
// the segment's end, the next breaker's right side closes them); a joined
// side's position is d plus the next entry's position where C + that maximum
// exceeds its own maximum at the join, else its own: suffix sums again.  Left
// sides the same way as prefix sums (the segment's first entry is a breaker).
// Each linked entry's record is written.
template <typename V>
__device__ __forceinline__ V seg_suffix_sum(V v, bool open, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const V v2 = __shfl_down_sync(kFullMask, v, off);
        const bool o2 = __shfl_down_sync(kFullMask, open, off);
        if (open && lane + off < 32) {
            v += v2;
            open = o2;
        }
    }
    return v;
}

template <typename V>
__device__ __forceinline__ V seg_prefix_sum(V v, bool open, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const V v2 = __shfl_up_sync(kFullMask, v, off);
        const bool o2 = __shfl_up_sync(kFullMask, open, off);
        if (open && lane >= off) {
            v += v2;
            open = o2;
        }
    }
    return v;
}

// Whether an entry's suffix sum runs past the segment's end: every entry from
// it to the last lane is open.
__device__ __forceinline__ bool open_to_end(bool open, int lane) {
    const unsigned closed = __ballot_sync(kFullMask, !open);
    return (closed >> lane) == 0u;
}

__global__ void __launch_bounds__(256) k_chain_resolve(const uint2 *__restrict__ anchors, uint64_t n_anchors,
                                                       uint32_t id_base, const uint32_t *__restrict__ ids,
                                                       uint64_t n_ids, const uint64_t *__restrict__ d_n,
                                                       uint64_t n_off, uint64_t n_total, int32_t T,
                                                       const ChainSide *__restrict__ sR,
                                                       const ChainSide *__restrict__ sL,
                                                       const ChainInfo *__restrict__ info, uint4 *__restrict__ out,
                                                       uint8_t *__restrict__ done, const uint32_t *__restrict__ out_pos) {
    if (d_n) n_ids = live_count(*d_n, n_off, n_ids, n_total);
    const int lane = threadIdx.x & 31;
    const uint64_t n_seg = (n_ids + kChainSeg - 1) / kChainSeg;
    const uint64_t n_warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    for (uint64_t sg = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; sg < n_seg; sg += n_warps) {
        const uint64_t j = sg * kChainSeg + lane;
        const uint64_t last = min(sg * kChainSeg + kChainSeg, n_ids) - 1;
        const ChainInfo f = j < n_ids ? info[j] : ChainInfo{0u, 0u};
        const bool member = (f.flags & (kLinkR | kLinkL)) != 0;
        const ChainSide zero{0, 0u, 0};
        const ChainSide r = member ? sR[j] : zero, l = member ? sL[j] : zero;
        // the side after the segment: the next breaker's, when the last entry links to it
        long long Mc = 0;
        uint32_t nc = 0;
        if (last + 1 < n_ids && (info[last].flags & kLinkR)) {
            Mc = sR[last + 1].M;
            nc = sR[last + 1].n;
        }
        // right maxima and positions
        const bool jr = (f.flags & kJoinR) != 0;
        long long MR = seg_suffix_sum<long long>(jr ? (long long)r.C : r.M, jr, lane);
        if (open_to_end(jr, lane)) MR += Mc;
        const bool cr = jr && MR > r.M;
        uint32_t nR = seg_suffix_sum<uint32_t>(cr ? f.dR : r.n, cr, lane);
        if (open_to_end(cr, lane)) nR += nc;
        // left maxima and positions (an entry's left distance is the previous entry's dR)
        const bool jl = (f.flags & kJoinL) != 0;
        const long long ML = seg_prefix_sum<long long>(jl ? (long long)l.C : l.M, jl, lane);
        const uint32_t dL = __shfl_up_sync(kFullMask, f.dR, 1);
        const bool cl = jl && ML > l.M;
        const uint32_t nL = seg_prefix_sum<uint32_t>(cl ? dL : l.n, cl, lane);
        if (!member) continue;
        const uint2 a = survivor_anchor(anchors, n_anchors, id_base, ids, j);
        long long score = ML + MR;
        if (score > 2147483647LL) score = 2147483647LL;
        uint4 rec = make_uint4(0, 0, 0, 0);
        uint8_t ok = 0;
        if (score >= T) {
            rec = make_uint4(a.x - nL, a.y - nL, nL + nR - 1u, (uint32_t)(int32_t)score);
            ok = 1;
        }
        const uint64_t jo = out_pos ? (uint64_t)out_pos[j] : j;
        out[jo] = rec;
        done[jo] = ok;
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

// Grouped order: key = the diagonal (ref end - query end) of entry j's anchor,
// all ones for an entry outside the sequences; value = j.
__global__ void k_diag_keys(const uint2 *__restrict__ anchors, uint64_t n_anchors, uint32_t id_base,
                            const uint32_t *__restrict__ ids, uint64_t n, uint64_t Lr, uint64_t Lq,
                            uint32_t *__restrict__ keys, uint32_t *__restrict__ vals) {
    for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n; j += (uint64_t)gridDim.x * blockDim.x) {
        const uint2 a = survivor_anchor(anchors, n_anchors, id_base, ids, j);
        keys[j] = (a.x < Lr && a.y < Lq) ? a.x - a.y : 0xFFFFFFFFu;
        vals[j] = (uint32_t)j;
    }
}

__global__ void k_gather_ids(const uint32_t *__restrict__ ids, const uint32_t *__restrict__ perm, uint64_t n,
                             uint32_t *__restrict__ out) {
    for (uint64_t j = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; j < n; j += (uint64_t)gridDim.x * blockDim.x)
        out[j] = ids[perm[j]];
}

}  // namespace

cudaError_t launch_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                               uint64_t n_ids,
                               SeqView ref, SeqView qry, const ScoreArgs &sa, hspz_segment_pair *d_out,
                               uint8_t *d_done, cudaStream_t st, const uint64_t *d_n, bool grouped) {
    if (!n_ids) return cudaSuccess;
    const uint2 *an = reinterpret_cast<const uint2 *>(d_anchors);
    uint4 *out = reinterpret_cast<uint4 *>(d_out);
    if (sa.fast) {
        const uint64_t blocks = (n_ids + 255) / 256;
        const unsigned g = (unsigned)(blocks < 152ull * 64 ? blocks : 152ull * 64);
        const bool has_n = ref.has_n || qry.has_n;
        if (sa.exact && kMaterializeChain) {
            // walks join their diagonal neighbours' walks and the joins are settled after;
            // slices of at most kChainSlice ids bound the scratch (no link crosses a slice)
            // grouped (host-known count only): each slice's entries are first sorted by
            // diagonal (stable, so each diagonal keeps the list's order), walked in that
            // order, and every record goes back to its entry's place
            grouped = grouped && !d_n;
            const uint64_t slice = n_ids < kChainSlice ? n_ids : kChainSlice;
            const uint64_t gwords = grouped ? 3 * slice + radix_sort_scratch_words(slice) : 0;
            void *scratch = nullptr;
            cudaError_t e = pool_alloc(&scratch, slice * (2 * sizeof(ChainSide) + sizeof(ChainInfo)) + gwords * 4, st);
            if (e != cudaSuccess) return e;
            ChainSide *sR = reinterpret_cast<ChainSide *>(scratch), *sL = sR + slice;
            ChainInfo *info = reinterpret_cast<ChainInfo *>(sL + slice);
            uint32_t *keys = reinterpret_cast<uint32_t *>(info + slice), *perm = keys + slice, *ids2 = perm + slice,
                     *rscratch = ids2 + slice;
            auto kern = has_n ? k_materialize_blocks<true, true> : k_materialize_blocks<false, true>;
            const uint64_t segs = (slice + kChainSeg - 1) / kChainSeg, sb = (segs + 7) / 8;  // a warp per segment
            const unsigned gs = (unsigned)((slice + 255) / 256 < 152ull * 64 ? (slice + 255) / 256 : 152ull * 64);
            const unsigned gr = (unsigned)(sb < 152ull * 64 ? sb : 152ull * 64);
            for (uint64_t off = 0; off < n_ids && e == cudaSuccess; off += slice) {
                const uint64_t len = n_ids - off < slice ? n_ids - off : slice;
                const uint32_t *ids = d_ids + off, *pos = nullptr;
                if (grouped) {
                    k_diag_keys<<<grid_cap(len, 256), 256, 0, st>>>(an, n_anchors, id_base, ids, len, ref.len, qry.len,
                                                                    keys, perm); count_launch();
                    e = cudaGetLastError();
                    if (e == cudaSuccess) e = launch_radix_sort_pairs(keys, perm, len, 32, rscratch, st);
                    if (e != cudaSuccess) break;
                    k_gather_ids<<<grid_cap(len, 256), 256, 0, st>>>(ids, perm, len, ids2); count_launch();
                    ids = ids2;
                    pos = perm;
                }
                kern<<<gs, 256, 0, st>>>(an, n_anchors, id_base, ids, len, d_n, off, n_ids, seqs(ref, qry), ref.rev,
                                         qry.rev, sa, out + off, d_done + off, sR, sL, info, pos); count_launch();
                k_chain_resolve<<<gr, 256, 0, st>>>(an, n_anchors, id_base, ids, len, d_n, off, n_ids, sa.T, sR, sL,
                                                    info, out + off, d_done + off, pos); count_launch();
                e = cudaGetLastError();
            }
            const cudaError_t ef = pool_free(scratch, st);
            return e != cudaSuccess ? e : ef;
        }
        if (sa.exact) {
            auto kern = has_n ? k_materialize_blocks<true, false> : k_materialize_blocks<false, false>;
            kern<<<g, 256, 0, st>>>(an, n_anchors, id_base, d_ids, n_ids, d_n, 0, n_ids, seqs(ref, qry), ref.rev, qry.rev,
                                    sa, out, d_done, nullptr, nullptr, nullptr, nullptr); count_launch();
        } else {
            auto kern = has_n ? k_materialize_lane<true> : k_materialize_lane<false>;
            kern<<<g, 256, 0, st>>>(an, n_anchors, id_base, d_ids, n_ids, d_n, seqs(ref, qry), ref.rev, qry.rev, sa,
                                    out, d_done); count_launch();
        }
    } else {
        k_materialize<<<grid_cap(n_ids, 128), 128, 0, st>>>(an, n_anchors, id_base, d_ids, n_ids, d_n, seqs(ref, qry),
                                                                    sa, out, d_done); count_launch();
    }
    return cudaGetLastError();
}

}  // namespace hspz
