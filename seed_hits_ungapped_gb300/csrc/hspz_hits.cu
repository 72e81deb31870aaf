// Hit discovery kernels: sequence packing, reference index build, per-seed
// hit counting (find_num_hits), the 256-count block scan, and the two
// expansion mappings of "C. Hit discovery" (hspZ docs, C.1-C.5).
#include "hspz_internal.cuh"

namespace hspz {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t pack_nibble(uint32_t c, int parity) {
    if (c > 3) return kNibN;
    return c | (parity ? (((c ^ (c >> 1)) & 1u) << 2) : 0u);
}

// One thread per packed word: 8 bases, padded with N outside [0, len).  A
// word whose 8 bases lie inside the sequence at an 8-byte aligned place
// (forward: codes + 8w - padding; reversed: its mirror) takes them with one
// 8-byte load; the others (the ends, or unaligned codes) go byte by byte.
// N bases are counted per warp before one atomic add.
__global__ void k_pack(const uint8_t *__restrict__ codes, uint64_t len, int parity, int reverse,
                       uint32_t *__restrict__ out, uint64_t words, unsigned long long *__restrict__ n_count) {
    uint32_t ns = 0;
    const bool aligned = ((reinterpret_cast<uintptr_t>(reverse ? codes + len : codes)) & 7u) == 0;
    for (uint64_t w = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; w < words;
         w += (uint64_t)gridDim.x * blockDim.x) {
        const int64_t b0 = (int64_t)w * 8 - kPadBases;
        uint32_t v = 0;
        if (aligned && b0 >= 0 && (uint64_t)b0 + 8 <= len) {
            // reversed: bases b0 .. b0+7 are codes[len-1-b0] down to codes[len-8-b0]
            const uint2 raw = *reinterpret_cast<const uint2 *>(codes + (reverse ? len - 8 - (uint64_t)b0 : (uint64_t)b0));
            const uint32_t lo4 = reverse ? __byte_perm(raw.y, 0, 0x0123) : raw.x;
            const uint32_t hi4 = reverse ? __byte_perm(raw.x, 0, 0x0123) : raw.y;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t nib = pack_nibble(((i < 4 ? lo4 : hi4) >> (8 * (i & 3))) & 0xFFu, parity);
                ns += nib == kNibN;
                v |= nib << (4 * i);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int64_t b = b0 + i;
                uint32_t nib = kNibN;
                if (b >= 0 && (uint64_t)b < len) {
                    nib = pack_nibble(codes[reverse ? len - 1 - b : b], parity);
                    ns += nib == kNibN;
                }
                v |= nib << (4 * i);
            }
        }
        out[w] = v;
    }
    ns = __reduce_add_sync(kFull, ns);
    if (n_count && ns && (threadIdx.x & 31) == 0) atomicAdd(n_count, (unsigned long long)ns);
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        T y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// find_num_hits (C.1): one thread per seed; the block also emits its 64-bit
// count sum (C.2: 256 counts per block).
// Four 256-seed count blocks per CTA (C.1, and the per-block sums of C.2):
// thread t takes seeds t, t + 256, t + 512 and t + 768 of the CTA's span, so
// its four index lookups are in flight together, and each 256 seeds get their
// own sum in bsum.
constexpr int kCountPer = 4;

__global__ void __launch_bounds__(kCountBlock) k_count(const uint8_t *__restrict__ q, uint64_t n_seeds, SeedShape sh,
                                                       const uint32_t *__restrict__ idx, uint32_t *__restrict__ cnt,
                                                       uint32_t *__restrict__ lo, uint64_t *__restrict__ bsum) {
    __shared__ uint8_t tile[kCountPer * kCountBlock + kMaxSpan];
    __shared__ uint64_t wsum[kCountPer][kCountBlock / 32];
    const uint64_t s0 = blockIdx.x * (uint64_t)(kCountPer * kCountBlock);
    const uint64_t qlen = n_seeds + sh.span - 1;
    for (int i = threadIdx.x; i < kCountPer * kCountBlock + sh.span - 1; i += blockDim.x) {
        const uint64_t p = s0 + i;
        tile[i] = p < qlen ? q[p] : 4;
    }
    __syncthreads();
    uint32_t h[kCountPer];
    bool ok[kCountPer];
#pragma unroll
    for (int k = 0; k < kCountPer; k++) {
        const int t = threadIdx.x + k * kCountBlock;
        uint32_t v = 0;
        bool good = s0 + t < n_seeds;
#pragma unroll
        for (int i = 0; i < kMaxWeight; i++) {
            if (i < sh.weight) {
                const uint32_t b = tile[t + sh.care[i]];
                good &= (b <= 3);
                v = v * 4u + (b & 3u);
            }
        }
        h[k] = v;
        ok[k] = good;
    }
    uint32_t end[kCountPer], prev[kCountPer];
#pragma unroll
    for (int k = 0; k < kCountPer; k++) {
        end[k] = ok[k] ? __ldg(idx + h[k]) : 0u;
        prev[k] = (ok[k] && h[k]) ? __ldg(idx + h[k] - 1) : 0u;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < kCountPer; k++) {
        const uint64_t s = s0 + threadIdx.x + k * kCountBlock;
        const uint32_t c = end[k] - prev[k];  // 0 for a seed without a k-mer
        if (s < n_seeds) {
            cnt[s] = c;
            lo[s] = prev[k];
        }
        const uint64_t v = warp_sum<uint64_t>(c);
        if (lane == 0) wsum[k][warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < kCountPer) {
        const uint64_t b = blockIdx.x * (uint64_t)kCountPer + threadIdx.x;  // the 256-seed block
        if (b * kCountBlock < n_seeds) {
            uint64_t t = 0;
            for (int w = 0; w < kCountBlock / 32; w++) t += wsum[threadIdx.x][w];
            bsum[b] = t;
        }
    }
}

// Scan of n values in three launches (reduce, scan of the tile sums,
// downsweep), every access coalesced: a tile is 1024 values, read as 4 rows of
// 256 (thread t takes value 256k + t of row k).  `in` may be `excl` (scan in
// place): every value is read before it is written.
constexpr int kScanThreads = 256;
constexpr int kScanRows = 4;
constexpr int kScanTile = kScanThreads * kScanRows;

template <typename T>
__device__ __forceinline__ T block_excl_scan(T v, T *wtot, T *row_total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const T x = warp_incl_scan<T>(v, lane);
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    T pre = x - v, tot = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; w++) {
        pre += w < warp ? wtot[w] : (T)0;
        tot += wtot[w];
    }
    __syncthreads();
    *row_total = tot;
    return pre;
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kScanThreads) k_scan_reduce(const InT *in, uint64_t n, OutT *__restrict__ part) {
    __shared__ OutT wtot[kScanThreads / 32];
    const uint64_t base = blockIdx.x * (uint64_t)kScanTile + threadIdx.x;
    OutT v = 0;
#pragma unroll
    for (int k = 0; k < kScanRows; k++) {
        const uint64_t i = base + (uint64_t)k * kScanThreads;
        v += i < n ? (OutT)in[i] : (OutT)0;
    }
    OutT tot;
    block_excl_scan<OutT>(v, wtot, &tot);
    if (threadIdx.x == 0) part[blockIdx.x] = tot;
}

// Single-CTA scan of the tile sums (8 per thread per round), in place: the
// exclusive prefix of every tile, and the total.
template <typename OutT>
__global__ void __launch_bounds__(1024) k_scan_parts(OutT *part, uint64_t n, OutT *__restrict__ total) {
    constexpr int kItems = 8;
    __shared__ OutT wtot[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    OutT carry = 0;
    for (uint64_t base = 0; base < n; base += 1024ull * kItems) {
        OutT v[kItems];
        OutT run = 0;
        const uint64_t i0 = base + (uint64_t)threadIdx.x * kItems;
#pragma unroll
        for (int k = 0; k < kItems; k++) {
            v[k] = (i0 + k < n) ? part[i0 + k] : (OutT)0;
            run += v[k];
        }
        OutT x = warp_incl_scan<OutT>(run, lane);
        if (lane == 31) wtot[warp] = x;
        __syncthreads();
        if (warp == 0) wtot[lane] = warp_incl_scan<OutT>(wtot[lane], lane);
        __syncthreads();
        OutT pre = carry + (warp ? wtot[warp - 1] : (OutT)0) + (x - run);
#pragma unroll
        for (int k = 0; k < kItems; k++) {
            if (i0 + k < n) {
                part[i0 + k] = pre;
                pre += v[k];
            }
        }
        carry += wtot[31];
        __syncthreads();
    }
    if (threadIdx.x == 0 && total) *total = carry;
}

template <typename InT, typename OutT>
__global__ void __launch_bounds__(kScanThreads) k_scan_down(const InT *in, uint64_t n,
                                                            const OutT *__restrict__ part_excl, OutT *excl,
                                                            OutT *__restrict__ incl) {
    __shared__ OutT wtot[kScanThreads / 32];
    OutT off = part_excl[blockIdx.x];
    const uint64_t base = blockIdx.x * (uint64_t)kScanTile + threadIdx.x;
#pragma unroll
    for (int k = 0; k < kScanRows; k++) {
        const uint64_t i = base + (uint64_t)k * kScanThreads;
        const OutT v = i < n ? (OutT)in[i] : (OutT)0;
        OutT row;
        const OutT e = off + block_excl_scan<OutT>(v, wtot, &row);
        if (i < n) {
            if (excl) excl[i] = e;
            if (incl) incl[i] = e + v;
        }
        off += row;
    }
}

template <typename InT, typename OutT>
cudaError_t launch_scan(const InT *d_in, uint64_t n, OutT *d_excl, OutT *d_incl, OutT *d_total, cudaStream_t st) {
    if (!n) return d_total ? cudaMemsetAsync(d_total, 0, sizeof(OutT), st) : cudaSuccess;
    const uint64_t tiles = (n + kScanTile - 1) / kScanTile;
    OutT *part = nullptr;
    cudaError_t e = pool_alloc(&part, tiles * sizeof(OutT), st);
    if (e != cudaSuccess) return e;
    k_scan_reduce<InT, OutT><<<(unsigned)tiles, kScanThreads, 0, st>>>(d_in, n, part); count_launch();
    k_scan_parts<OutT><<<1, 1024, 0, st>>>(part, tiles, d_total); count_launch();
    k_scan_down<InT, OutT><<<(unsigned)tiles, kScanThreads, 0, st>>>(d_in, n, part, d_excl, d_incl); count_launch();
    e = cudaGetLastError();
    cudaError_t ef = pool_free(part, st);
    return e != cudaSuccess ? e : ef;
}

// Inclusive prefix (C.2): 1024 counts per CTA, 4 per thread, plus the
// exclusive offset of the CTA's first 256-count block.
constexpr int kPrefixPerThread = 4;
constexpr int kPrefixTile = kCountBlock * kPrefixPerThread;

__global__ void __launch_bounds__(kCountBlock) k_prefix(const uint32_t *__restrict__ cnt, uint64_t n,
                                                        const uint64_t *__restrict__ bexcl, uint32_t *__restrict__ P) {
    __shared__ uint64_t wtot[kCountBlock / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t s = blockIdx.x * (uint64_t)kPrefixTile + (uint64_t)threadIdx.x * kPrefixPerThread;
    uint32_t v[kPrefixPerThread];
    if (s + kPrefixPerThread <= n) {
        const uint4 q = *reinterpret_cast<const uint4 *>(cnt + s);
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    } else {
#pragma unroll
        for (int k = 0; k < kPrefixPerThread; k++) v[k] = s + k < n ? cnt[s + k] : 0u;
    }
    const uint64_t run = (uint64_t)v[0] + v[1] + v[2] + v[3];
    const uint64_t x = warp_incl_scan<uint64_t>(run, lane);
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    uint64_t pre = bexcl[(uint64_t)blockIdx.x * (kPrefixTile / kCountBlock)] + (x - run);
    for (int w = 0; w < warp; w++) pre += wtot[w];
    uint32_t o[kPrefixPerThread];
#pragma unroll
    for (int k = 0; k < kPrefixPerThread; k++) {
        pre += v[k];
        o[k] = (uint32_t)pre;
    }
    if (s + kPrefixPerThread <= n) {
        *reinterpret_cast<uint4 *>(P + s) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int k = 0; k < kPrefixPerThread; k++)
            if (s + k < n) P[s + k] = o[k];
    }
}

// C.5, thread-per-seed mapping: occurrence j goes to slot P[s] - 1 - hit_begin - j.
__global__ void k_expand_sparse(const uint32_t *__restrict__ P, const uint32_t *__restrict__ cnt,
                                const uint32_t *__restrict__ lo, const uint32_t *__restrict__ pos, uint32_t sb,
                                uint32_t se, uint32_t hb, uint32_t span, uint2 *__restrict__ out) {
    const uint64_t s = sb + blockIdx.x * (uint64_t)blockDim.x + threadIdx.x;
    if (s >= se) return;
    const uint32_t c = cnt[s];
    if (!c) return;
    const uint32_t end = P[s] - hb, l = lo[s], qe = (uint32_t)s + span - 1;
    for (uint32_t j = 0; j < c; j++) out[end - 1 - j] = make_uint2(__ldg(pos + l + j), qe);
}

// C.5, warp-per-seed mapping: the warp walks one bucket coalescently; same slots.
__global__ void k_expand_dense(const uint32_t *__restrict__ P, const uint32_t *__restrict__ cnt,
                               const uint32_t *__restrict__ lo, const uint32_t *__restrict__ pos, uint32_t sb,
                               uint32_t se, uint32_t hb, uint32_t span, uint2 *__restrict__ out) {
    const uint64_t s = sb + (blockIdx.x * (uint64_t)blockDim.x + threadIdx.x) / 32;
    const int lane = threadIdx.x & 31;
    if (s >= se) return;
    const uint32_t c = cnt[s];
    const uint32_t end = P[s] - hb, l = lo[s], qe = (uint32_t)s + span - 1;
    for (uint32_t j = lane; j < c; j += 32) out[end - 1 - j] = make_uint2(__ldg(pos + l + j), qe);
}

// ---------------------------------------------------------------- index build
// Valid-window flags, then (after a stable compaction of the window starts)
// the k-mer keys, a stable LSD radix sort on 3 x 8 key bits, and the bucket
// ends by binary search over the sorted keys.

__global__ void k_window_flags(const uint8_t *__restrict__ ref, uint64_t n_win, SeedShape sh,
                               uint8_t *__restrict__ flags) {
    for (uint64_t r = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; r < n_win;
         r += (uint64_t)gridDim.x * blockDim.x) {
        bool ok = true;
        for (int i = 0; i < sh.weight; i++) ok &= ref[r + sh.care[i]] <= 3;
        flags[r] = ok ? 1 : 0;
    }
}

__global__ void k_window_keys(const uint8_t *__restrict__ ref, const uint32_t *__restrict__ starts, uint64_t n,
                              SeedShape sh, uint32_t *__restrict__ keys, uint32_t *__restrict__ vals) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t r = starts[i];
        uint32_t h = 0;
        for (int k = 0; k < sh.weight; k++) h = h * 4u + (ref[(uint64_t)r + sh.care[k]] & 3u);
        keys[i] = h;
        vals[i] = r + (uint32_t)sh.span - 1;
    }
}

constexpr int kRadixThreads = 256;
constexpr int kRadixItems = 16;
constexpr int kRadixTile = kRadixThreads * kRadixItems;

// Digit histogram of one tile, stored digit-major: hist[d * n_tiles + tile].
__global__ void __launch_bounds__(kRadixThreads) k_radix_hist(const uint32_t *__restrict__ keys, uint64_t n, int shift,
                                                              uint32_t *__restrict__ hist, uint64_t n_tiles) {
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const uint64_t t0 = blockIdx.x * (uint64_t)kRadixTile;
    for (int k = threadIdx.x; k < kRadixTile; k += kRadixThreads) {
        uint64_t i = t0 + k;
        if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255u], 1u);
    }
    __syncthreads();
    hist[(uint64_t)threadIdx.x * n_tiles + blockIdx.x] = h[threadIdx.x];
}

// Stable scatter: thread t owns tile items [16t, 16t+16) in order, so the
// rank of an item is (items of its digit in earlier threads) + (earlier items
// of its digit in the same thread).
__global__ void __launch_bounds__(kRadixThreads) k_radix_scatter(const uint32_t *__restrict__ kin,
                                                                 const uint32_t *__restrict__ vin, uint64_t n,
                                                                 int shift, const uint32_t *__restrict__ off,
                                                                 uint64_t n_tiles, uint32_t *__restrict__ kout,
                                                                 uint32_t *__restrict__ vout) {
    extern __shared__ uint16_t sm[];  // [256 threads][256 digits]
    uint16_t *row = sm + threadIdx.x * 256;
    for (int d = 0; d < 256; d++) row[d] = 0;
    const uint64_t i0 = blockIdx.x * (uint64_t)kRadixTile + (uint64_t)threadIdx.x * kRadixItems;
    uint32_t k[kRadixItems], v[kRadixItems];
#pragma unroll
    for (int j = 0; j < kRadixItems; j++) {
        uint64_t i = i0 + j;
        k[j] = i < n ? kin[i] : 0u;
        v[j] = i < n ? vin[i] : 0u;
        if (i < n) row[(k[j] >> shift) & 255u]++;
    }
    __syncthreads();
    {  // thread d: exclusive scan of digit d over threads
        const int d = threadIdx.x;
        uint32_t run = 0;
        for (int t = 0; t < kRadixThreads; t++) {
            uint16_t c = sm[t * 256 + d];
            sm[t * 256 + d] = (uint16_t)run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRadixItems; j++) {
        uint64_t i = i0 + j;
        if (i < n) {
            uint32_t d = (k[j] >> shift) & 255u;
            uint64_t dst = (uint64_t)off[(uint64_t)d * n_tiles + blockIdx.x] + row[d];
            row[d]++;
            kout[dst] = k[j];
            vout[dst] = v[j];
        }
    }
}

// idx[h] = number of sorted keys <= h.
__global__ void k_bucket_ends(const uint32_t *__restrict__ keys, uint64_t n, uint64_t n_buckets,
                              uint32_t *__restrict__ idx) {
    for (uint64_t h = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; h < n_buckets;
         h += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t lo = 0, hi = n;
        while (lo < hi) {
            uint64_t mid = (lo + hi) >> 1;
            if (keys[mid] <= h) lo = mid + 1; else hi = mid;
        }
        idx[h] = (uint32_t)lo;
    }
}

unsigned grid_for(uint64_t n, int threads, unsigned cap = 152u * 32u) {
    uint64_t g = (n + threads - 1) / threads;
    if (g < 1) g = 1;
    return (unsigned)(g > cap ? cap : g);
}

}  // namespace

uint64_t packed_words(uint64_t len) {
    uint64_t w = (len + 2 * (uint64_t)kPadBases + 7) / 8;
    return (w + 3) & ~3ull;  // whole 16-byte vectors
}

cudaError_t launch_pack(const uint8_t *d_codes, uint64_t len, int with_parity, int reverse, uint32_t *d_packed,
                        uint64_t words, cudaStream_t st, unsigned long long *d_n_count) {
    k_pack<<<grid_for(words, 256), 256, 0, st>>>(d_codes, len, with_parity, reverse, d_packed, words, d_n_count); count_launch();
    return cudaGetLastError();
}

cudaError_t launch_count(const uint8_t *d_query, uint64_t n_seeds, const SeedShape &sh, const uint32_t *d_idx,
                         uint32_t *d_cnt, uint32_t *d_lo, uint64_t *d_block_sum, cudaStream_t st) {
    const uint64_t nb = (n_seeds + kCountBlock - 1) / kCountBlock;
    if (!nb) return cudaSuccess;
    k_count<<<(unsigned)((nb + kCountPer - 1) / kCountPer), kCountBlock, 0, st>>>(d_query, n_seeds, sh, d_idx, d_cnt,
                                                                                   d_lo, d_block_sum); count_launch();
    return cudaGetLastError();
}

cudaError_t launch_scan_u64(const uint64_t *d_in, uint64_t n, uint64_t *d_excl, uint64_t *d_incl, uint64_t *d_total,
                            cudaStream_t st) {
    return launch_scan<uint64_t, uint64_t>(d_in, n, d_excl, d_incl, d_total, st);
}

uint64_t radix_sort_scratch_words(uint64_t n) {
    const uint64_t n_tiles = (n + kRadixTile - 1) / kRadixTile;
    return 2 * n + n_tiles * 256;
}

cudaError_t launch_radix_sort_pairs(uint32_t *d_keys, uint32_t *d_vals, uint64_t n, int key_bits, uint32_t *d_scratch,
                                    cudaStream_t st) {
    if (!n) return cudaSuccess;
    const uint64_t n_tiles = (n + kRadixTile - 1) / kRadixTile;
    uint32_t *k0 = d_keys, *v0 = d_vals, *k1 = d_scratch, *v1 = d_scratch + n, *hist = d_scratch + 2 * n;
    const int smem = kRadixThreads * 256 * 2;
    cudaError_t e = cudaFuncSetAttribute(k_radix_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int passes = 0;
    for (int shift = 0; shift < key_bits && e == cudaSuccess; shift += 8, passes++) {
        k_radix_hist<<<(unsigned)n_tiles, kRadixThreads, 0, st>>>(k0, n, shift, hist, n_tiles); count_launch();
        e = cudaGetLastError();
        if (e == cudaSuccess) e = launch_scan_u32(hist, n_tiles * 256, hist, st);
        if (e != cudaSuccess) break;
        k_radix_scatter<<<(unsigned)n_tiles, kRadixThreads, smem, st>>>(k0, v0, n, shift, hist, n_tiles, k1, v1); count_launch();
        e = cudaGetLastError();
        uint32_t *t = k0; k0 = k1; k1 = t;
        t = v0; v0 = v1; v1 = t;
    }
    // an odd number of passes leaves the result in the scratch halves
    if (e == cudaSuccess && (passes & 1)) {
        e = cudaMemcpyAsync(d_keys, k0, n * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(d_vals, v0, n * 4, cudaMemcpyDeviceToDevice, st);
    }
    return e;
}

cudaError_t launch_scan_u32(const uint32_t *d_in, uint64_t n, uint32_t *d_excl, cudaStream_t st) {
    return launch_scan<uint32_t, uint32_t>(d_in, n, d_excl, (uint32_t *)nullptr, (uint32_t *)nullptr, st);
}

cudaError_t launch_prefix(const uint32_t *d_cnt, uint64_t n_seeds, const uint64_t *d_block_excl, uint32_t *d_P,
                          cudaStream_t st) {
    // cnt and P are 16-byte aligned (whole allocations); tiles of 1024 counts
    const uint64_t nt = (n_seeds + kPrefixTile - 1) / kPrefixTile;
    if (!nt) return cudaSuccess;
    k_prefix<<<(unsigned)nt, kCountBlock, 0, st>>>(d_cnt, n_seeds, d_block_excl, d_P); count_launch();
    return cudaGetLastError();
}

cudaError_t launch_expand(const uint32_t *d_P, const uint32_t *d_cnt, const uint32_t *d_lo, const uint32_t *d_pos,
                          const hspz_chunk &c, int span, int dense, hspz_anchor *d_out, cudaStream_t st) {
    uint64_t ns = (uint64_t)c.seed_end - c.seed_begin;
    if (!ns || c.hit_end == c.hit_begin) return cudaSuccess;
    uint2 *out = reinterpret_cast<uint2 *>(d_out);
    if (dense) {
        uint64_t threads = ns * 32;
        k_expand_dense<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(d_P, d_cnt, d_lo, d_pos, c.seed_begin,
                                                                          c.seed_end, c.hit_begin, span, out); count_launch();
    } else {
        k_expand_sparse<<<(unsigned)((ns + 255) / 256), 256, 0, st>>>(d_P, d_cnt, d_lo, d_pos, c.seed_begin,
                                                                      c.seed_end, c.hit_begin, span, out); count_launch();
    }
    return cudaGetLastError();
}

// Reference index on the device.  Temporary buffers come from the stream's
// memory pool and are released before return.
cudaError_t build_index_tables(const uint8_t *d_ref, uint64_t ref_len, const SeedShape &sh, uint32_t *d_idx,
                               uint32_t **d_pos_out, uint64_t *n_pos_out, cudaStream_t st) {
    cudaError_t e;
    const uint64_t n_buckets = 1ull << (2 * sh.weight);
    const uint64_t n_win = ref_len >= (uint64_t)sh.span ? ref_len - sh.span + 1 : 0;
    *d_pos_out = nullptr;
    *n_pos_out = 0;
    if (n_win == 0) {
        return cudaMemsetAsync(d_idx, 0, n_buckets * 4, st);
    }
    uint8_t *flags = nullptr;
    uint32_t *starts = nullptr, *scratch = nullptr, *k0 = nullptr, *v0 = nullptr, *k1 = nullptr, *v1 = nullptr,
             *hist = nullptr;
    uint64_t *d_n = nullptr;
    uint64_t n = 0;
    const uint64_t n_tiles_max = (n_win + kRadixTile - 1) / kRadixTile;
#define TRY(x)                        \
    do {                              \
        e = (x);                      \
        if (e != cudaSuccess) goto out; \
    } while (0)
    TRY(pool_alloc(&flags, n_win, st));
    TRY(pool_alloc(&starts, n_win * 4, st));
    TRY(pool_alloc(&scratch, compact_scratch_words(n_win) * 4, st));
    TRY(pool_alloc(&d_n, 8, st));
    k_window_flags<<<grid_for(n_win, 256), 256, 0, st>>>(d_ref, n_win, sh, flags); count_launch();
    TRY(cudaGetLastError());
    TRY(launch_compact(flags, n_win, 0, starts, n_win, scratch, d_n, st));
    TRY(cudaMemcpyAsync(&n, d_n, 8, cudaMemcpyDeviceToHost, st));
    TRY(cudaStreamSynchronize(st));
    if (n) {
        const uint64_t n_tiles = (n + kRadixTile - 1) / kRadixTile;
        (void)n_tiles_max;
        TRY(pool_alloc(&k0, n * 4, st));
        TRY(pool_alloc(&v0, n * 4, st));
        TRY(pool_alloc(&k1, n * 4, st));
        TRY(pool_alloc(&v1, n * 4, st));
        TRY(pool_alloc(&hist, n_tiles * 256 * 4, st));
        k_window_keys<<<grid_for(n, 256), 256, 0, st>>>(d_ref, starts, n, sh, k0, v0); count_launch();
        TRY(cudaGetLastError());
        const int smem = kRadixThreads * 256 * 2;
        TRY(cudaFuncSetAttribute(k_radix_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        for (int shift = 0; shift < 2 * sh.weight; shift += 8) {
            k_radix_hist<<<(unsigned)n_tiles, kRadixThreads, 0, st>>>(k0, n, shift, hist, n_tiles); count_launch();
            TRY(cudaGetLastError());
            TRY(launch_scan_u32(hist, n_tiles * 256, hist, st));
            k_radix_scatter<<<(unsigned)n_tiles, kRadixThreads, smem, st>>>(k0, v0, n, shift, hist, n_tiles, k1, v1); count_launch();
            TRY(cudaGetLastError());
            uint32_t *t = k0; k0 = k1; k1 = t;
            t = v0; v0 = v1; v1 = t;
        }
        k_bucket_ends<<<grid_for(n_buckets, 256), 256, 0, st>>>(k0, n, n_buckets, d_idx); count_launch();
        TRY(cudaGetLastError());
        TRY(cudaMalloc((void **)d_pos_out, n * 4));
        TRY(cudaMemcpyAsync(*d_pos_out, v0, n * 4, cudaMemcpyDeviceToDevice, st));
    } else {
        TRY(cudaMemsetAsync(d_idx, 0, n_buckets * 4, st));
    }
    *n_pos_out = n;
out:
#undef TRY
    for (void *p : {(void *)flags, (void *)starts, (void *)scratch, (void *)k0, (void *)v0, (void *)k1, (void *)v1,
                    (void *)hist, (void *)d_n})
        if (p) pool_free(p, st);
    cudaError_t e2 = cudaStreamSynchronize(st);
    return e != cudaSuccess ? e : e2;
}

}  // namespace hspz
