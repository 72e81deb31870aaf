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

__global__ void __launch_bounds__(256) k_gate(const uint2 *__restrict__ anchors, uint64_t n, Seqs sq, ScoreArgs sa,
                                              uint8_t *__restrict__ flags) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint2 a = anchors[i];
        flags[i] = (uint8_t)gate_one(sq, tab, sa.xdrop, sa.T, a.x, a.y);
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

// One thread per survivor (E.1-E.5).
__global__ void __launch_bounds__(128) k_materialize(const uint2 *__restrict__ anchors, uint64_t n_anchors, uint32_t id_base,
                                                     const uint32_t *__restrict__ ids, uint64_t n_ids, Seqs sq,
                                                     ScoreArgs sa, uint4 *__restrict__ out,
                                                     uint8_t *__restrict__ done) {
    __shared__ int tab[25];
    if (threadIdx.x < 25) tab[threadIdx.x] = sa.m[threadIdx.x];
    __syncthreads();
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

cudaError_t launch_expand_gate(const uint32_t *d_P, const uint32_t *d_lo, const uint32_t *d_pos, const hspz_chunk &c,
                               int span, SeqView ref, SeqView qry, const ScoreArgs &sa, hspz_anchor *d_out,
                               uint8_t *d_flags, cudaStream_t st) {
    const uint64_t n = (uint64_t)c.hit_end - c.hit_begin;
    if (!n) return cudaSuccess;
    const uint64_t blocks = (n + kFuseTile - 1) / kFuseTile;
    uint2 *out = reinterpret_cast<uint2 *>(d_out);
    if (d_flags) {
        k_expand_gate<true><<<(unsigned)blocks, kFuseThreads, 0, st>>>(d_P, d_lo, d_pos, c.seed_begin, c.seed_end,
                                                                       c.hit_begin, n, span, seqs(ref, qry), sa, out,
                                                                       d_flags); count_launch();
    } else {
        k_expand_gate<false><<<(unsigned)blocks, kFuseThreads, 0, st>>>(d_P, d_lo, d_pos, c.seed_begin, c.seed_end,
                                                                        c.hit_begin, n, span, seqs(ref, qry), sa, out,
                                                                        d_flags); count_launch();
    }
    return cudaGetLastError();
}

cudaError_t launch_gate(const hspz_anchor *d_anchors, uint64_t n, SeqView ref, SeqView qry, const ScoreArgs &sa,
                        uint8_t *d_flags, cudaStream_t st) {
    if (!n) return cudaSuccess;
    k_gate<<<grid_cap(n, 256), 256, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), n, seqs(ref, qry), sa,
                                              d_flags); count_launch();
    return cudaGetLastError();
}

cudaError_t launch_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                               uint64_t n_ids,
                               SeqView ref, SeqView qry, const ScoreArgs &sa, hspz_segment_pair *d_out,
                               uint8_t *d_done, cudaStream_t st) {
    if (!n_ids) return cudaSuccess;
    k_materialize<<<grid_cap(n_ids, 128), 128, 0, st>>>(reinterpret_cast<const uint2 *>(d_anchors), n_anchors, id_base, d_ids,
                                                         n_ids, seqs(ref, qry), sa, reinterpret_cast<uint4 *>(d_out),
                                                         d_done); count_launch();
    return cudaGetLastError();
}

}  // namespace hspz
