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

// k_materialize_lane for scoring where the 8-base stop test is exact
// (X >= 7 x the largest pair score, see walk_step_lead).  Lanes step in
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

}  // namespace

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
