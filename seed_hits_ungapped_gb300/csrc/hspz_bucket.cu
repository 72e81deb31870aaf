// Reference-locality bucketing of the gate ("D. Score gate", D.5): a stable
// counting sort groups anchors into at most 32 reference-address buckets, so
// that the warps gating one bucket gather their reference windows from one
// range of the packed reference.  The gate then writes each flag at the
// anchor's raw id, so the flags (and every later output) equal the unbucketed
// gate's.
#include "hspz_internal.cuh"

namespace hspz {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 16;
constexpr int kTile = kThreads * kPerThread;
constexpr int kMaxBuckets = 32;

__device__ __forceinline__ uint32_t bucket_of(uint32_t ref_end, uint32_t span, uint32_t n_buckets) {
    const uint32_t b = ref_end / span;
    return b < n_buckets ? b : n_buckets - 1;
}

// Bucket counts of one tile, stored bucket-major: hist[b * n_tiles + tile].
__global__ void __launch_bounds__(kThreads) k_bucket_hist(const uint2 *__restrict__ a, uint64_t n, uint32_t span,
                                                          uint32_t n_buckets, uint32_t *__restrict__ hist,
                                                          uint64_t n_tiles) {
    __shared__ uint32_t h[kMaxBuckets];
    if (threadIdx.x < kMaxBuckets) h[threadIdx.x] = 0;
    __syncthreads();
    const uint64_t t0 = blockIdx.x * (uint64_t)kTile;
    for (int k = threadIdx.x; k < kTile; k += kThreads) {
        const uint64_t i = t0 + k;
        if (i < n) atomicAdd(&h[bucket_of(a[i].x, span, n_buckets)], 1u);
    }
    __syncthreads();
    if (threadIdx.x < n_buckets) hist[(uint64_t)threadIdx.x * n_tiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter: thread t owns tile items [16t, 16t+16) in order; an item's
// rank is its bucket's offset for the tile, plus the items of that bucket
// owned by earlier threads, plus the earlier items of the same thread.
__global__ void __launch_bounds__(kThreads) k_bucket_scatter(const uint2 *__restrict__ a, uint64_t n, uint32_t span,
                                                             uint32_t n_buckets, const uint32_t *__restrict__ off,
                                                             uint64_t n_tiles, uint2 *__restrict__ sorted,
                                                             uint32_t *__restrict__ raw) {
    __shared__ uint32_t cnt[kThreads][kMaxBuckets + 1];  // padded row: thread t, bucket b in bank (t + b) % 32
    uint32_t *row = cnt[threadIdx.x];
    for (int b = 0; b < kMaxBuckets; b++) row[b] = 0;
    const uint64_t i0 = blockIdx.x * (uint64_t)kTile + (uint64_t)threadIdx.x * kPerThread;
    uint2 v[kPerThread];
    uint8_t bk[kPerThread];
#pragma unroll
    for (int j = 0; j < kPerThread; j++) {
        const uint64_t i = i0 + j;
        v[j] = i < n ? a[i] : make_uint2(0, 0);
        bk[j] = (uint8_t)bucket_of(v[j].x, span, n_buckets);
        if (i < n) row[bk[j]]++;
    }
    __syncthreads();
    if (threadIdx.x < n_buckets) {  // thread b: exclusive scan of bucket b over the threads
        const int b = threadIdx.x;
        uint32_t run = 0;
        for (int t = 0; t < kThreads; t++) {
            const uint32_t c = cnt[t][b];
            cnt[t][b] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kPerThread; j++) {
        const uint64_t i = i0 + j;
        if (i < n) {
            const uint32_t b = bk[j];
            const uint64_t dst = (uint64_t)off[(uint64_t)b * n_tiles + blockIdx.x] + row[b];
            row[b]++;
            sorted[dst] = v[j];
            raw[dst] = (uint32_t)i;
        }
    }
}

}  // namespace

uint64_t bucket_scratch_words(uint64_t n, uint32_t n_buckets) {
    const uint64_t n_tiles = (n + kTile - 1) / kTile;
    return n_tiles * n_buckets + 1;
}

cudaError_t launch_bucket_sort(const hspz_anchor *d_anchors, uint64_t n, uint32_t span, uint32_t n_buckets,
                               hspz_anchor *d_sorted, uint32_t *d_raw, uint32_t *d_scratch, cudaStream_t st) {
    if (!n) return cudaSuccess;
    if (n_buckets < 1 || n_buckets > (uint32_t)kMaxBuckets || span < 1) return cudaErrorInvalidValue;
    const uint64_t n_tiles = (n + kTile - 1) / kTile;
    const uint2 *a = reinterpret_cast<const uint2 *>(d_anchors);
    k_bucket_hist<<<(unsigned)n_tiles, kThreads, 0, st>>>(a, n, span, n_buckets, d_scratch, n_tiles); count_launch();
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_scan_u32(d_scratch, n_tiles * n_buckets, d_scratch, st);
    if (e != cudaSuccess) return e;
    k_bucket_scatter<<<(unsigned)n_tiles, kThreads, 0, st>>>(a, n, span, n_buckets, d_scratch, n_tiles,
                                                             reinterpret_cast<uint2 *>(d_sorted), d_raw); count_launch();
    return cudaGetLastError();
}

}  // namespace hspz
