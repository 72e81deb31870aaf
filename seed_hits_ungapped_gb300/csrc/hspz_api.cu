// Host side of libhspz: argument checks, handles, the keep threshold, hit
// discovery orchestration and the MAX_HITS chunk walk ("C. Hit discovery",
// C.2-C.3), and the C ABI entry points declared in include/hspz.h.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <mutex>

#include "hspz_internal.cuh"

namespace hspz {

cudaError_t build_index_tables(const uint8_t *d_ref, uint64_t ref_len, const SeedShape &sh, uint32_t *d_idx,
                               uint32_t **d_pos_out, uint64_t *n_pos_out, cudaStream_t st);

namespace {
thread_local std::string g_last_error;
constexpr uint64_t kMaxSeqLen = (1ull << 32) - 1024;
constexpr int64_t kMaxK = 1ll << 30;
constexpr int64_t kMaxX = 1ll << 30;
constexpr int64_t kMaxAbsScore = 1ll << 16;
}  // namespace

// ------------------------------------------------------------------ memory pool
// Stream-ordered allocations of the library (plans, per-call scratch, index
// build temporaries) come from one pool per device that keeps freed memory
// cached (release threshold = unlimited), so a plan or scratch buffer of the
// same size as before is handed out again without mapping new memory.
// hspz_release_cached_memory trims the pools back.
namespace {
constexpr int kMaxPoolDevices = 64;
std::mutex g_pool_mutex;
cudaMemPool_t g_pools[kMaxPoolDevices] = {};

cudaError_t device_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxPoolDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t pool_alloc(void **p, size_t bytes, cudaStream_t st) {
    cudaMemPool_t pool;
    cudaError_t e = device_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(p, bytes ? bytes : 1, pool, st);
}

cudaError_t pool_free(void *p, cudaStream_t st) { return p ? cudaFreeAsync(p, st) : cudaSuccess; }

namespace {
// Small results (totals, counts) come back to the host through pinned,
// device-mapped host memory that a one-thread kernel writes, not through a
// device-to-host copy: on the copy engine such a copy waits behind the large
// downloads queued before it on other streams (a streamed batch's results,
// tens of GB on dense), which held the next batch's planning for ~0.3 s.
__global__ void k_read_back(const uint64_t *__restrict__ src, volatile uint64_t *dst, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
    __threadfence_system();
}

// One staging area per host thread (a call launches and collects on the same
// thread); kept for the thread's lifetime.
thread_local uint64_t *tl_read_back = nullptr;
}  // namespace

cudaError_t read_back_launch(const uint64_t *d_src, int n, cudaStream_t st) {
    if (n < 1 || n > 8) return cudaErrorInvalidValue;
    if (!tl_read_back) {
        uint64_t *h = nullptr;
        cudaError_t e = cudaHostAlloc(reinterpret_cast<void **>(&h), 64, cudaHostAllocMapped | cudaHostAllocPortable);
        if (e != cudaSuccess) return e;
        tl_read_back = h;
    }
    uint64_t *d = nullptr;
    cudaError_t e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&d), tl_read_back, 0);
    if (e != cudaSuccess) return e;
    k_read_back<<<1, 32, 0, st>>>(d_src, d, n); count_launch();
    return cudaGetLastError();
}

cudaError_t read_back_finish(uint64_t *host, int n, cudaStream_t st) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    const volatile uint64_t *h = tl_read_back;
    for (int i = 0; i < n; i++) host[i] = h[i];
    return cudaSuccess;
}

static std::atomic<uint64_t> g_launches{0};
void count_launch(uint64_t k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

void set_error(const std::string &msg) { g_last_error = msg; }

int cuda_fail(cudaError_t e, const char *what) {
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return e == cudaErrorMemoryAllocation ? HSPZ_E_NOMEM : HSPZ_E_CUDA;
}

int parse_pattern(const char *pat, SeedShape *sh) {
    if (!pat) pat = "1110100110010101111";
    int n = 0, w = 0;
    for (; pat[n]; n++) {
        if (n >= kMaxSpan) return HSPZ_E_INVAL;
        if (pat[n] == '1') {
            if (w >= kMaxWeight) return HSPZ_E_INVAL;
            sh->care[w++] = n;
        } else if (pat[n] != '0') {
            return HSPZ_E_INVAL;
        }
    }
    if (w < 1 || pat[0] != '1' || pat[n - 1] != '1') return HSPZ_E_INVAL;
    sh->span = n;
    sh->weight = w;
    for (int i = w; i < kMaxSpan; i++) sh->care[i] = 0;
    return HSPZ_OK;
}

// Keep threshold: the f32 rounding of integers is monotone, so the totals the
// f32 comparison keeps are exactly those at or above the rounding boundary
// between (float)K and its float predecessor.  Start from that boundary and
// settle the tie with the compiler's own int -> float conversion.
static int keep_threshold(int32_t K, int32_t *T) {
    if (K < 1 || K > kMaxK) return HSPZ_E_INVAL;
    const float f = (float)K;
    const float prev = nextafterf(f, 0.0f);
    const double mid = 0.5 * ((double)prev + (double)f);
    int64_t c = (int64_t)ceil(mid);
    while (c > 1 && (float)(c - 1) >= f) c--;
    while ((float)c < f) c++;
    *T = (int32_t)c;
    return HSPZ_OK;
}

int make_score_args(const hspz_score_params *p, ScoreArgs *out) {
    if (!p) return HSPZ_E_INVAL;
    if (p->xdrop < 0 || p->xdrop > kMaxX) return HSPZ_E_INVAL;
    for (int i = 0; i < 25; i++)
        if (p->matrix[i] > kMaxAbsScore || p->matrix[i] < -kMaxAbsScore) return HSPZ_E_INVAL;
    int32_t T;
    if (keep_threshold(p->K, &T)) return HSPZ_E_INVAL;
    memcpy(out->m, p->matrix, sizeof(out->m));
    out->xdrop = p->xdrop;
    out->T = T;
    // complement-symmetric 8-entry table (see the gate kernels): entry
    // x | parity(r) << 2 with x = r ^ q over codes A0 C1 G2 T3.
    int8_t tab[8];
    bool fast = true;
    for (int r = 0; r < 4; r++)
        for (int q = 0; q < 4; q++) {
            int e = (r ^ q) | (((r ^ (r >> 1)) & 1) << 2);
            int v = p->matrix[5 * r + q];
            int vc = p->matrix[5 * (r ^ 3) + (q ^ 3)];
            if (v != vc || v < -128 || v > 127) fast = false;
            tab[e] = (int8_t)v;
        }
    if (fast && tab[0] < 0) fast = false;
    out->tab_lo = (uint8_t)tab[0] | ((uint32_t)(uint8_t)tab[1] << 8) | ((uint32_t)(uint8_t)tab[2] << 16) |
                  ((uint32_t)(uint8_t)tab[3] << 24);
    out->tab_hi = (uint8_t)tab[4] | ((uint32_t)(uint8_t)tab[5] << 8) | ((uint32_t)(uint8_t)tab[6] << 16) |
                  ((uint32_t)(uint8_t)tab[7] << 24);
    out->fast = fast ? 1 : 0;
    // After a stop inside an 8-base step, at most 7 more pair scores follow in
    // that step; they cannot lift the running sum back above the maximum
    // before the stop when X is at least 7 times the largest pair score.
    int smax = 0;
    for (int i = 0; i < 25; i++) smax = p->matrix[i] > smax ? p->matrix[i] : smax;
    out->exact = (fast && (int64_t)p->xdrop >= 7 * (int64_t)smax) ? 1 : 0;
    return HSPZ_OK;
}

// ------------------------------------------------------------------ chunk walk
// "C.3": one chunk if the hits left fit the cap, else the lower bound over the
// seed prefixes for hit_begin + cap, located through the inclusive block sums
// (256 seeds per block) and then inside the one block that holds it; the seed
// found there is kept whole.  fetch(b, out) copies prefix block b.
using FetchBlock = std::function<int(uint64_t block, uint32_t *out, uint64_t *n)>;

static int chunk_walk(uint64_t S, uint64_t total, uint64_t max_hits, const uint64_t *blk_incl, uint64_t nb,
                      const uint32_t *full_P, const FetchBlock &fetch, std::vector<hspz_chunk> &out) {
    out.clear();
    uint64_t sb = 0, hb = 0;
    std::vector<uint32_t> blk(kCountBlock);
    while (sb < S) {
        uint64_t se, he;
        if (max_hits == 0 || total - hb <= max_hits) {
            se = S;
            he = total;
        } else {
            const uint64_t target = hb + max_hits;
            uint64_t e;
            if (full_P) {
                e = (uint64_t)(std::lower_bound(full_P, full_P + S, target,
                                                [](uint32_t a, uint64_t t) { return (uint64_t)a < t; }) -
                               full_P);
                he = full_P[e];
            } else {
                const uint64_t b = (uint64_t)(std::lower_bound(blk_incl, blk_incl + nb, target) - blk_incl);
                if (b >= nb) return HSPZ_E_INVAL;
                uint64_t got = 0;
                int rc = fetch(b, blk.data(), &got);
                if (rc) return rc;
                const uint64_t k = (uint64_t)(std::lower_bound(blk.data(), blk.data() + got, target,
                                                               [](uint32_t a, uint64_t t) { return (uint64_t)a < t; }) -
                                              blk.data());
                if (k >= got) return HSPZ_E_INVAL;
                e = b * kCountBlock + k;
                he = blk[k];
            }
            se = e + 1;
        }
        out.push_back(hspz_chunk{(uint32_t)sb, (uint32_t)se, (uint32_t)hb, (uint32_t)he});
        sb = se;
        hb = he;
    }
    return HSPZ_OK;
}

}  // namespace hspz

using namespace hspz;

// ---------------------------------------------------------------- C ABI
extern "C" {

const char *hspz_strerror(int status) {
    switch (status) {
        case HSPZ_OK: return "ok";
        case HSPZ_E_INVAL: return "invalid argument";
        case HSPZ_E_HIT_OVERFLOW: return "total hits exceed the 32-bit hit index";
        case HSPZ_E_CAPACITY: return "output capacity too small";
        case HSPZ_E_CUDA: return "CUDA error";
        case HSPZ_E_NOMEM: return "out of memory";
        case HSPZ_E_UNSUPPORTED: return "unsupported";
        default: return "unknown status";
    }
}

const char *hspz_last_error(void) { return g_last_error.c_str(); }

int hspz_abi_version(void) { return HSPZ_ABI_VERSION; }

int hspz_release_cached_memory(void) {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    for (int d = 0; d < kMaxPoolDevices; d++) {
        if (!g_pools[d]) continue;
        cudaError_t e = cudaMemPoolTrimTo(g_pools[d], 0);
        if (e != cudaSuccess) return cuda_fail(e, "hspz_release_cached_memory");
    }
    return HSPZ_OK;
}

uint64_t hspz_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int hspz_keep_threshold(int32_t K, int32_t *T_out) {
    if (!T_out) return HSPZ_E_INVAL;
    return keep_threshold(K, T_out);
}

int hspz_build_index(const uint8_t *d_ref, uint64_t ref_len, const char *seed_pattern, hspz_index **index_out,
                     void *stream) {
    if (!index_out || (!d_ref && ref_len) || ref_len > kMaxSeqLen) return HSPZ_E_INVAL;
    *index_out = nullptr;
    SeedShape sh;
    if (parse_pattern(seed_pattern, &sh)) {
        set_error("bad seed pattern");
        return HSPZ_E_INVAL;
    }
    cudaStream_t st = (cudaStream_t)stream;
    hspz_index *ix = new (std::nothrow) hspz_index();
    if (!ix) return HSPZ_E_NOMEM;
    ix->shape = sh;
    ix->ref_len = ref_len;
    cudaGetDevice(&ix->device);
    const uint64_t nb = 1ull << (2 * sh.weight);
    ix->ref_words = packed_words(ref_len);
    cudaError_t e = cudaMalloc((void **)&ix->d_idx, nb * 4);
    if (e == cudaSuccess) e = cudaMalloc((void **)&ix->d_ref, ix->ref_words * 4);
    if (e == cudaSuccess) e = cudaMalloc((void **)&ix->d_ref_rev, ix->ref_words * 4);
    unsigned long long *d_ncount = nullptr, ncount = 0;
    if (e == cudaSuccess) e = pool_alloc(&d_ncount, 8, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_ncount, 0, 8, st);
    if (e == cudaSuccess) e = launch_pack(d_ref, ref_len, 1, 0, ix->d_ref, ix->ref_words, st, d_ncount);
    if (e == cudaSuccess) e = launch_pack(d_ref, ref_len, 1, 1, ix->d_ref_rev, ix->ref_words, st);
    if (e == cudaSuccess) e = build_index_tables(d_ref, ref_len, sh, ix->d_idx, &ix->d_pos, &ix->n_pos, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&ncount, d_ncount, 8, cudaMemcpyDeviceToHost, st);
    if (d_ncount) pool_free(d_ncount, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    ix->has_n = ncount != 0;
    if (e != cudaSuccess) {
        int rc = cuda_fail(e, "hspz_build_index");
        hspz_index_free(ix);
        return rc;
    }
    *index_out = ix;
    return HSPZ_OK;
}

void hspz_index_free(hspz_index *ix) {
    if (!ix) return;
    if (ix->d_idx) cudaFree(ix->d_idx);
    if (ix->d_pos) cudaFree(ix->d_pos);
    if (ix->d_ref) cudaFree(ix->d_ref);
    if (ix->d_ref_rev) cudaFree(ix->d_ref_rev);
    delete ix;
}

int hspz_index_info(const hspz_index *ix, uint64_t *n_positions, uint32_t *span, uint32_t *weight) {
    if (!ix) return HSPZ_E_INVAL;
    if (n_positions) *n_positions = ix->n_pos;
    if (span) *span = (uint32_t)ix->shape.span;
    if (weight) *weight = (uint32_t)ix->shape.weight;
    return HSPZ_OK;
}

int hspz_index_tables(const hspz_index *ix, const uint32_t **d_idx, const uint32_t **d_pos) {
    if (!ix) return HSPZ_E_INVAL;
    if (d_idx) *d_idx = ix->d_idx;
    if (d_pos) *d_pos = ix->d_pos;
    return HSPZ_OK;
}

void hspz_plan_free(hspz_plan *p) {
    if (!p) return;
    // stream-ordered: the buffers go back to the device pool once the work
    // queued on the plan's stream so far has finished
    for (void *q : {(void *)p->d_P, (void *)p->d_lo, (void *)p->d_cnt, (void *)p->d_blk, (void *)p->d_qry,
                    (void *)p->d_qry_rev, (void *)p->d_tiles})
        if (q) pool_free(q, p->stream);
    delete p;
}

int hspz_find_hits(const hspz_index *ix, const uint8_t *d_query, uint64_t query_len, uint64_t max_hits,
                   uint32_t flags, hspz_plan **plan_out, uint64_t *total_hits, void *stream) {
    if (!ix || !plan_out || (!d_query && query_len) || query_len > kMaxSeqLen || (flags & ~1u)) return HSPZ_E_INVAL;
    *plan_out = nullptr;
    cudaStream_t st = (cudaStream_t)stream;
    hspz_plan *p = new (std::nothrow) hspz_plan();
    if (!p) return HSPZ_E_NOMEM;
    p->index = ix;
    p->query_len = query_len;
    const int span = ix->shape.span;
    const uint64_t S = query_len >= (uint64_t)span ? query_len - span + 1 : 0;
    p->n_seeds = S;
    const uint64_t nb = (S + kCountBlock - 1) / kCountBlock;
    p->n_blocks = nb;
    p->qry_words = packed_words(query_len);
    cudaError_t e = cudaSuccess;
    const uint64_t sa = S ? S : 1;
    p->stream = st;
    e = pool_alloc(&p->d_P, sa * 4, st);
    if (e == cudaSuccess) e = pool_alloc(&p->d_lo, sa * 4, st);
    if (e == cudaSuccess) e = pool_alloc(&p->d_cnt, sa * 4, st);
    if (e == cudaSuccess) e = pool_alloc(&p->d_blk, (3 * nb + 2) * 8, st);
    if (e == cudaSuccess) e = pool_alloc(&p->d_qry, p->qry_words * 4, st);
    if (e == cudaSuccess) e = pool_alloc(&p->d_qry_rev, p->qry_words * 4, st);
    // the total and the query's N count sit side by side after the block sums
    uint64_t *bsum = p->d_blk, *bexcl = p->d_blk + nb, *bincl = p->d_blk + 2 * nb, *dtot = p->d_blk + 3 * nb;
    if (e == cudaSuccess) e = cudaMemsetAsync(dtot, 0, 16, st);
    if (e == cudaSuccess)
        e = launch_pack(d_query, query_len, 0, 0, p->d_qry, p->qry_words, st, (unsigned long long *)(dtot + 1));
    if (e == cudaSuccess) e = launch_pack(d_query, query_len, 0, 1, p->d_qry_rev, p->qry_words, st);
    if (e == cudaSuccess && S) e = launch_count(d_query, S, ix->shape, ix->d_idx, p->d_cnt, p->d_lo, bsum, st);
    if (e == cudaSuccess && S) e = launch_scan_u64(bsum, nb, bexcl, bincl, dtot, st);
    if (e == cudaSuccess && S) e = launch_prefix(p->d_cnt, S, bexcl, p->d_P, st);
    uint64_t tot_n[2] = {0, 0};
    if (e == cudaSuccess) e = read_back_launch(dtot, 2, st);
    if (e == cudaSuccess) e = read_back_finish(tot_n, 2, st);
    const uint64_t total = tot_n[0];
    p->has_n = tot_n[1] != 0;
    if (e != cudaSuccess) {
        int rc = cuda_fail(e, "hspz_find_hits");
        hspz_plan_free(p);
        return rc;
    }
    if (total_hits) *total_hits = total;
    if (total > 0xFFFFFFFFull) {  // C.2: refused, never wrapped
        set_error("total hits exceed the 32-bit hit index");
        hspz_plan_free(p);
        return HSPZ_E_HIT_OVERFLOW;
    }
    p->total = total;
    // C.3 chunk walk
    std::vector<uint64_t> blk_incl;
    std::vector<uint32_t> full;
    const bool cut = max_hits != 0 && total > max_hits;
    int rc = HSPZ_OK;
    if (cut && (flags & HSPZ_WALK_FULL)) {
        full.resize(S);
        e = cudaMemcpyAsync(full.data(), p->d_P, S * 4, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    } else if (cut) {
        blk_incl.resize(nb);
        e = cudaMemcpyAsync(blk_incl.data(), bincl, nb * 8, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) {
        rc = cuda_fail(e, "hspz_find_hits chunk walk");
        hspz_plan_free(p);
        return rc;
    }
    FetchBlock fetch = [&](uint64_t b, uint32_t *out, uint64_t *n) -> int {
        const uint64_t s0 = b * kCountBlock;
        const uint64_t cnt = std::min<uint64_t>(kCountBlock, S - s0);
        cudaError_t e2 = cudaMemcpyAsync(out, p->d_P + s0, cnt * 4, cudaMemcpyDeviceToHost, st);
        if (e2 == cudaSuccess) e2 = cudaStreamSynchronize(st);
        if (e2 != cudaSuccess) return cuda_fail(e2, "chunk walk block copy");
        *n = cnt;
        return HSPZ_OK;
    };
    rc = chunk_walk(S, total, max_hits, blk_incl.empty() ? nullptr : blk_incl.data(), nb,
                    full.empty() ? nullptr : full.data(), fetch, p->chunks);
    if (rc) {
        hspz_plan_free(p);
        return rc;
    }
    p->max_chunk_hits = 0;
    for (const auto &c : p->chunks)
        p->max_chunk_hits = std::max<uint64_t>(p->max_chunk_hits, (uint64_t)c.hit_end - c.hit_begin);
    e = pool_alloc(&p->d_tiles, expand_gate_tile_words(p->max_chunk_hits) * 4, st);
    if (e != cudaSuccess) {
        rc = cuda_fail(e, "hspz_find_hits tile scratch");
        hspz_plan_free(p);
        return rc;
    }
    *plan_out = p;
    return HSPZ_OK;
}

int hspz_plan_info(const hspz_plan *p, uint64_t *n_seeds, uint64_t *total_hits, uint32_t *n_chunks,
                   uint64_t *max_chunk_hits) {
    if (!p) return HSPZ_E_INVAL;
    if (n_seeds) *n_seeds = p->n_seeds;
    if (total_hits) *total_hits = p->total;
    if (n_chunks) *n_chunks = (uint32_t)p->chunks.size();
    if (max_chunk_hits) *max_chunk_hits = p->max_chunk_hits;
    return HSPZ_OK;
}

int hspz_plan_chunks(const hspz_plan *p, hspz_chunk *chunks, uint32_t cap, uint32_t *n_chunks) {
    if (!p || !n_chunks) return HSPZ_E_INVAL;
    *n_chunks = (uint32_t)p->chunks.size();
    if (cap < p->chunks.size()) return HSPZ_E_CAPACITY;
    if (!p->chunks.empty()) {
        if (!chunks) return HSPZ_E_INVAL;
        memcpy(chunks, p->chunks.data(), p->chunks.size() * sizeof(hspz_chunk));
    }
    return HSPZ_OK;
}

int hspz_plan_prefix(const hspz_plan *p, const uint32_t **d_prefix) {
    if (!p || !d_prefix) return HSPZ_E_INVAL;
    *d_prefix = p->d_P;
    return HSPZ_OK;
}

int hspz_expand(const hspz_plan *p, uint32_t chunk, int mode, hspz_anchor *d_anchors, uint64_t cap, void *stream) {
    if (!p || chunk >= p->chunks.size() || mode < 0 || mode > 2) return HSPZ_E_INVAL;
    const hspz_chunk &c = p->chunks[chunk];
    const uint64_t hits = (uint64_t)c.hit_end - c.hit_begin;
    if (cap < hits) return HSPZ_E_CAPACITY;
    if (hits && !d_anchors) return HSPZ_E_INVAL;
    const uint64_t seeds = (uint64_t)c.seed_end - c.seed_begin;
    // C.4: warp-per-seed when the chunk averages at least 16 hits per seed
    const int dense = mode == HSPZ_EXPAND_DENSE || (mode == HSPZ_EXPAND_AUTO && hits >= 16 * seeds);
    cudaError_t e = launch_expand(p->d_P, p->d_cnt, p->d_lo, p->index->d_pos, c, p->index->shape.span, dense,
                                  d_anchors, (cudaStream_t)stream);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_expand");
}

int hspz_expand_gate(const hspz_plan *p, uint32_t chunk, const hspz_score_params *params, hspz_anchor *d_anchors,
                     uint8_t *d_flags, uint64_t cap, void *stream) {
    if (!p || chunk >= p->chunks.size()) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    const hspz_chunk &c = p->chunks[chunk];
    const uint64_t hits = (uint64_t)c.hit_end - c.hit_begin;
    if (cap < hits) return HSPZ_E_CAPACITY;
    if (hits && (!d_anchors || !d_flags)) return HSPZ_E_INVAL;
    SeqView r{p->index->d_ref, p->index->ref_len, p->index->d_ref_rev, p->index->has_n},
        q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    cudaError_t e = launch_expand_gate(p->d_P, p->d_lo, p->index->d_pos, c, p->index->shape.span, r, q, sa,
                                       d_anchors, d_flags, p->d_tiles, (cudaStream_t)stream);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_expand_gate");
}

int hspz_process_chunk(const hspz_plan *p, uint32_t chunk, const hspz_score_params *params, hspz_anchor *d_anchors,
                       uint8_t *d_flags, uint64_t cap_anchors, uint32_t *d_ids, hspz_segment_pair *d_records,
                       uint8_t *d_done, uint32_t *d_accepted, uint64_t cap_survivors, uint64_t *n_survivors,
                       uint64_t *n_accepted, float *gate_ms, void *stream) {
    if (!p || chunk >= p->chunks.size() || !n_survivors || !n_accepted) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    const hspz_chunk &c = p->chunks[chunk];
    const uint64_t hits = (uint64_t)c.hit_end - c.hit_begin;
    if (cap_anchors < hits) return HSPZ_E_CAPACITY;
    if (hits && (!d_anchors || !d_flags)) return HSPZ_E_INVAL;
    if (cap_survivors && (!d_ids || !d_records || !d_done || !d_accepted)) return HSPZ_E_INVAL;
    if (reinterpret_cast<uintptr_t>(d_records) & 15u) return HSPZ_E_INVAL;
    *n_survivors = *n_accepted = 0;
    if (gate_ms) *gate_ms = 0.f;
    if (!hits) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    const uint64_t words = compact_scratch_words(std::max(hits, cap_survivors)) + 8;
    uint32_t *scratch = nullptr;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    uint64_t totals[2] = {0, 0};
    SeqView r{p->index->d_ref, p->index->ref_len, p->index->d_ref_rev, p->index->has_n},
        q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    cudaError_t e = pool_alloc(&scratch, words * 4, st);
    // the two counts sit after the compaction scratch, 8-byte aligned
    uint64_t *tot = reinterpret_cast<uint64_t *>(scratch + ((words - 6) & ~1ull));
    if (e == cudaSuccess && gate_ms) {
        e = cudaEventCreate(&ev0);
        if (e == cudaSuccess) e = cudaEventCreate(&ev1);
        if (e == cudaSuccess) e = cudaEventRecord(ev0, st);
    }
    if (e == cudaSuccess)
        e = launch_expand_gate(p->d_P, p->d_lo, p->index->d_pos, c, p->index->shape.span, r, q, sa, d_anchors,
                               d_flags, p->d_tiles, st);
    if (e == cudaSuccess && gate_ms) e = cudaEventRecord(ev1, st);
    if (e == cudaSuccess) e = launch_compact(d_flags, hits, c.hit_begin, d_ids, cap_survivors, scratch, tot, st);
    if (e == cudaSuccess && cap_survivors) {
        e = launch_materialize(d_anchors, hits, c.hit_begin, d_ids, cap_survivors, r, q, sa, d_records, d_done, st,
                               tot);
        if (e == cudaSuccess)
            e = launch_compact(d_done, cap_survivors, 0, d_accepted, cap_survivors, scratch, tot + 1, st, tot);
    } else if (e == cudaSuccess) {
        e = cudaMemsetAsync(tot + 1, 0, 8, st);
    }
    if (e == cudaSuccess) e = read_back_launch(tot, 2, st);  // before the scratch holding them is freed
    cudaError_t ef = scratch ? pool_free(scratch, st) : cudaSuccess;
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = read_back_finish(totals, 2, st);
    if (e == cudaSuccess && gate_ms) e = cudaEventElapsedTime(gate_ms, ev0, ev1);
    if (ev0) cudaEventDestroy(ev0);
    if (ev1) cudaEventDestroy(ev1);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_process_chunk");
    *n_survivors = totals[0];
    if (totals[0] > cap_survivors) return HSPZ_E_CAPACITY;
    *n_accepted = totals[1];
    return HSPZ_OK;
}

int hspz_score_gate_plan(const hspz_index *ix, const hspz_plan *p, const hspz_anchor *d_anchors, uint64_t n,
                         const hspz_score_params *params, uint8_t *d_flags, void *stream) {
    if (!ix || !p || p->index != ix || (n && (!d_anchors || !d_flags))) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    SeqView r{ix->d_ref, ix->ref_len, ix->d_ref_rev, ix->has_n}, q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    cudaError_t e = launch_gate(d_anchors, nullptr, n, r, q, sa, d_flags, (cudaStream_t)stream);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_score_gate_plan");
}

// Packs the raw base codes of both sequences into one stream-ordered scratch
// buffer (forward copies, and the reversed copies when `reversed`) for the
// raw-sequence calls.  The copies are marked as holding N, so the kernels test
// every step for N instead of reading the N count back to the host.
static cudaError_t pack_raw_pair(const uint8_t *d_ref, uint64_t ref_len, const uint8_t *d_query, uint64_t query_len,
                                 bool reversed, cudaStream_t st, uint32_t **buf, SeqView *r, SeqView *q) {
    const uint64_t rw = packed_words(ref_len), qw = packed_words(query_len);
    cudaError_t e = pool_alloc(buf, (reversed ? 2 : 1) * (rw + qw) * 4, st);
    if (e != cudaSuccess) return e;
    uint32_t *p = *buf;
    *r = SeqView{p, ref_len, reversed ? p + rw + qw : nullptr, true};
    *q = SeqView{p + rw, query_len, reversed ? p + 2 * rw + qw : nullptr, true};
    e = launch_pack(d_ref, ref_len, 1, 0, const_cast<uint32_t *>(r->packed), rw, st);
    if (e == cudaSuccess) e = launch_pack(d_query, query_len, 0, 0, const_cast<uint32_t *>(q->packed), qw, st);
    if (e == cudaSuccess && reversed) e = launch_pack(d_ref, ref_len, 1, 1, const_cast<uint32_t *>(r->rev), rw, st);
    if (e == cudaSuccess && reversed) e = launch_pack(d_query, query_len, 0, 1, const_cast<uint32_t *>(q->rev), qw, st);
    return e;
}

int hspz_score_gate(const hspz_anchor *d_anchors, uint64_t n, const uint8_t *d_ref, uint64_t ref_len,
                    const uint8_t *d_query, uint64_t query_len, const hspz_score_params *params, uint8_t *d_flags,
                    void *stream) {
    if (n && (!d_anchors || !d_flags)) return HSPZ_E_INVAL;
    if ((ref_len && !d_ref) || (query_len && !d_query) || ref_len > kMaxSeqLen || query_len > kMaxSeqLen)
        return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    if (!n) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *buf = nullptr;
    SeqView r, q;
    cudaError_t e = pack_raw_pair(d_ref, ref_len, d_query, query_len, false, st, &buf, &r, &q);
    if (e == cudaSuccess) e = launch_gate(d_anchors, nullptr, n, r, q, sa, d_flags, st);
    cudaError_t ef = buf ? pool_free(buf, st) : cudaSuccess;
    if (e == cudaSuccess) e = ef;
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_score_gate");
}

int hspz_score_gate_bucketed(const hspz_index *ix, const hspz_plan *p, const hspz_anchor *d_anchors, uint64_t n,
                             const hspz_score_params *params, uint32_t n_buckets, uint8_t *d_flags, void *stream) {
    if (!ix || !p || p->index != ix || (n && (!d_anchors || !d_flags)) || n_buckets > 32 || n > (1ull << 32))
        return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    if (!sa.fast) {
        set_error("hspz_score_gate_bucketed: the matrix is not complement symmetric with int8 scores");
        return HSPZ_E_UNSUPPORTED;
    }
    if (!n) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (n_buckets == 0) {  // auto: windows of the packed reference (both directions) in 3/4 of the L2
        int dev = 0, l2 = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        const double window = 0.75 * (l2 > 0 ? l2 : (64 << 20));
        const double bytes = 2.0 * (double)ix->ref_words * 4.0;
        n_buckets = (uint32_t)std::min(32.0, std::max(1.0, std::ceil(bytes / window)));
    }
    const uint64_t Lr = std::max<uint64_t>(ix->ref_len, 1);
    const uint32_t span = (uint32_t)((Lr + n_buckets - 1) / n_buckets);
    hspz_anchor *sorted = nullptr;
    uint32_t *raw = nullptr, *scratch = nullptr;
    cudaError_t e = pool_alloc(&sorted, n * sizeof(hspz_anchor), st);
    if (e == cudaSuccess) e = pool_alloc(&raw, n * 4, st);
    if (e == cudaSuccess) e = pool_alloc(&scratch, bucket_scratch_words(n, n_buckets) * 4, st);
    if (e == cudaSuccess) e = launch_bucket_sort(d_anchors, n, span, n_buckets, sorted, raw, scratch, st);
    SeqView r{ix->d_ref, ix->ref_len, ix->d_ref_rev, ix->has_n}, q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    if (e == cudaSuccess) e = launch_gate(sorted, raw, n, r, q, sa, d_flags, st);
    for (void *ptr : {(void *)sorted, (void *)raw, (void *)scratch})
        if (ptr) pool_free(ptr, st);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_score_gate_bucketed");
}

int hspz_compact(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids, uint64_t cap,
                 uint64_t *n_out, void *stream) {
    if (!n_out || (n && !d_flags) || n > (1ull << 32) || (uint64_t)id_base + n > (1ull << 32)) return HSPZ_E_INVAL;
    if (cap && !d_ids) return HSPZ_E_INVAL;
    cudaStream_t st = (cudaStream_t)stream;
    *n_out = 0;
    if (!n) return HSPZ_OK;
    uint32_t *scratch = nullptr;
    const uint64_t words = compact_scratch_words(n) + 2;
    cudaError_t e = pool_alloc(&scratch, words * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_compact scratch");
    uint64_t *d_total = reinterpret_cast<uint64_t *>(scratch + ((words - 2) & ~1ull));
    uint64_t total = 0;
    e = launch_compact(d_flags, n, id_base, d_ids, cap, scratch, d_total, st);
    if (e == cudaSuccess) e = read_back_launch(d_total, 1, st);  // before the scratch holding it is freed
    cudaError_t ef = pool_free(scratch, st);
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = read_back_finish(&total, 1, st);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_compact");
    *n_out = total;
    return total > cap ? HSPZ_E_CAPACITY : HSPZ_OK;
}

int hspz_gather_records(const hspz_segment_pair *d_records, const uint32_t *d_idx, uint64_t n,
                        hspz_segment_pair *d_out, void *stream) {
    if (n && (!d_records || !d_idx || !d_out)) return HSPZ_E_INVAL;
    if ((reinterpret_cast<uintptr_t>(d_records) | reinterpret_cast<uintptr_t>(d_out)) & 15u) return HSPZ_E_INVAL;
    cudaError_t e = launch_gather_records(d_records, d_idx, n, d_out, (cudaStream_t)stream);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_gather_records");
}

int hspz_dedup(const hspz_segment_pair *d_records, uint64_t n, uint32_t *d_keep_ids, uint64_t cap, uint64_t *n_kept,
               void *stream) {
    if (!n_kept || (n && !d_records) || n > (1ull << 31)) return HSPZ_E_INVAL;
    if (reinterpret_cast<uintptr_t>(d_records) & 15u) return HSPZ_E_INVAL;
    if (cap && !d_keep_ids) return HSPZ_E_INVAL;
    *n_kept = 0;
    if (!n) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    // scratch: table | keep flags (n bytes, word-padded) | compaction scratch | total, error count
    // (the keep flags and the compaction scratch start on 16-byte boundaries)
    const uint64_t slots = dedup_table_slots(n), keep_words = (n + 15) / 16 * 4, cw = compact_scratch_words(n);
    const uint64_t words = slots + keep_words + cw + 6;
    uint32_t *scratch = nullptr;
    cudaError_t e = pool_alloc(&scratch, words * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_dedup scratch");
    uint32_t *d_tab = scratch;
    uint8_t *d_keep = reinterpret_cast<uint8_t *>(scratch + slots);
    uint32_t *d_cs = scratch + slots + keep_words;
    uint64_t *d_tail = reinterpret_cast<uint64_t *>(scratch + ((slots + keep_words + cw + 1) & ~1ull));
    uint64_t tail[2] = {0, 0};  // total kept, probe failures
    e = cudaMemsetAsync(d_tail, 0, 16, st);
    if (e == cudaSuccess)
        e = launch_dedup(d_records, n, d_tab, slots, d_keep, reinterpret_cast<unsigned long long *>(d_tail + 1), st);
    if (e == cudaSuccess) e = launch_compact(d_keep, n, 0, d_keep_ids, cap, d_cs, d_tail, st);
    if (e == cudaSuccess) e = read_back_launch(d_tail, 2, st);  // before the scratch holding them is freed
    cudaError_t ef = pool_free(scratch, st);
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = read_back_finish(tail, 2, st);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_dedup");
    if (tail[1]) {
        set_error("hspz_dedup: hash probe sequence exhausted");
        return HSPZ_E_UNSUPPORTED;
    }
    *n_kept = tail[0];
    return tail[0] > cap ? HSPZ_E_CAPACITY : HSPZ_OK;
}

int hspz_materialize_plan(const hspz_index *ix, const hspz_plan *p, const hspz_anchor *d_anchors, uint64_t n_anchors,
                          uint32_t id_base, const uint32_t *d_ids, uint64_t n_ids, const hspz_score_params *params,
                          hspz_segment_pair *d_out, uint8_t *d_done, void *stream) {
    if (!ix || !p || p->index != ix) return HSPZ_E_INVAL;
    if (n_ids && (!d_anchors || !d_ids || !d_out || !d_done)) return HSPZ_E_INVAL;
    if (reinterpret_cast<uintptr_t>(d_out) & 15u) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    SeqView r{ix->d_ref, ix->ref_len, ix->d_ref_rev, ix->has_n}, q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    cudaError_t e = launch_materialize(d_anchors, n_anchors, id_base, d_ids, n_ids, r, q, sa, d_out, d_done,
                                       (cudaStream_t)stream);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_materialize_plan");
}

int hspz_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                     uint64_t n_ids, const uint8_t *d_ref, uint64_t ref_len, const uint8_t *d_query,
                     uint64_t query_len, const hspz_score_params *params, hspz_segment_pair *d_out, uint8_t *d_done,
                     void *stream) {
    if (n_ids && (!d_anchors || !d_ids || !d_out || !d_done)) return HSPZ_E_INVAL;
    if ((ref_len && !d_ref) || (query_len && !d_query) || ref_len > kMaxSeqLen || query_len > kMaxSeqLen)
        return HSPZ_E_INVAL;
    if (reinterpret_cast<uintptr_t>(d_out) & 15u) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    if (!n_ids) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *buf = nullptr;
    SeqView r, q;
    cudaError_t e = pack_raw_pair(d_ref, ref_len, d_query, query_len, true, st, &buf, &r, &q);
    if (e == cudaSuccess)
        e = launch_materialize(d_anchors, n_anchors, id_base, d_ids, n_ids, r, q, sa, d_out, d_done, st);
    cudaError_t ef = buf ? pool_free(buf, st) : cudaSuccess;
    if (e == cudaSuccess) e = ef;
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_materialize");
}

int hspz_materialize_grouped(const hspz_index *ix, const hspz_plan *p, const hspz_anchor *d_anchors,
                             uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids, uint64_t n_ids,
                             const hspz_score_params *params, hspz_segment_pair *d_out, uint8_t *d_done,
                             void *stream) {
    if (!ix || !p || p->index != ix) return HSPZ_E_INVAL;
    if (n_ids && (!d_anchors || !d_ids || !d_out || !d_done)) return HSPZ_E_INVAL;
    if (reinterpret_cast<uintptr_t>(d_out) & 15u) return HSPZ_E_INVAL;
    ScoreArgs sa;
    if (make_score_args(params, &sa)) return HSPZ_E_INVAL;
    SeqView r{ix->d_ref, ix->ref_len, ix->d_ref_rev, ix->has_n}, q{p->d_qry, p->query_len, p->d_qry_rev, p->has_n};
    cudaError_t e = launch_materialize(d_anchors, n_anchors, id_base, d_ids, n_ids, r, q, sa, d_out, d_done,
                                       (cudaStream_t)stream, nullptr, true);
    return e == cudaSuccess ? HSPZ_OK : cuda_fail(e, "hspz_materialize_grouped");
}

int hspz_chunk_walk_host(const uint32_t *prefix, uint64_t n_seeds, uint64_t max_hits, int use_block_sums,
                         hspz_chunk *chunks, uint32_t cap, uint32_t *n_chunks) {
    if (!n_chunks || (n_seeds && !prefix)) return HSPZ_E_INVAL;
    const uint64_t total = n_seeds ? prefix[n_seeds - 1] : 0;
    const uint64_t nb = (n_seeds + kCountBlock - 1) / kCountBlock;
    std::vector<uint64_t> blk(nb);
    for (uint64_t b = 0; b < nb; b++) blk[b] = prefix[std::min<uint64_t>(n_seeds - 1, b * kCountBlock + kCountBlock - 1)];
    FetchBlock fetch = [&](uint64_t b, uint32_t *out, uint64_t *n) -> int {
        const uint64_t s0 = b * kCountBlock;
        *n = std::min<uint64_t>(kCountBlock, n_seeds - s0);
        memcpy(out, prefix + s0, *n * 4);
        return HSPZ_OK;
    };
    std::vector<hspz_chunk> out;
    int rc = chunk_walk(n_seeds, total, max_hits, use_block_sums ? blk.data() : nullptr, nb,
                        use_block_sums ? nullptr : prefix, fetch, out);
    if (rc) return rc;
    *n_chunks = (uint32_t)out.size();
    if (cap < out.size()) return HSPZ_E_CAPACITY;
    if (!out.empty()) memcpy(chunks, out.data(), out.size() * sizeof(hspz_chunk));
    return HSPZ_OK;
}

}  // extern "C"
