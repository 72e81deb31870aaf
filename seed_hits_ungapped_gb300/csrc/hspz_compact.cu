// Stable flag compaction ("D. Score gate", D.4): device blocks count their
// set flags, the block counts are scanned, and every block emits the original
// ids of its set flags at its exclusive offset in increasing order.
#include "hspz_internal.cuh"

namespace hspz {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 64;
constexpr int kTile = kThreads * kPerThread;  // 16384 flags per block
constexpr unsigned kFull = 0xFFFFFFFFu;

// The count of flags: n, or (when d_n is given) the count at d_n if it is at
// most n, else 0 (a count that overran its buffer yields nothing).
__device__ __forceinline__ uint64_t count_of(uint64_t n, const uint64_t *d_n) {
    if (!d_n) return n;
    const uint64_t v = *d_n;
    return v <= n ? v : 0;
}

// The 64 flags a thread owns, as a 64-bit mask (bit i = flag i != 0); with
// ALIGNED flags a full set comes in four 16-byte loads issued together.
template <bool ALIGNED>
__device__ __forceinline__ uint64_t load_mask(const uint8_t *__restrict__ f, uint64_t i0, uint64_t n) {
    uint64_t m = 0;
    if (ALIGNED && i0 + kPerThread <= n) {
        uint4 v[kPerThread / 16];
#pragma unroll
        for (int q = 0; q < kPerThread / 16; q++) v[q] = __ldg(reinterpret_cast<const uint4 *>(f + i0) + q);
#pragma unroll
        for (int q = 0; q < kPerThread / 16; q++) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const uint32_t nz = __vcmpne4(w[k], 0u);  // 0xFF per non-zero byte
#pragma unroll
                for (int b = 0; b < 4; b++) m |= (uint64_t)((nz >> (8 * b + 7)) & 1u) << (16 * q + 4 * k + b);
            }
        }
    } else {
#pragma unroll 16
        for (int k = 0; k < kPerThread; k++)
            if (i0 + k < n && f[i0 + k]) m |= 1ull << k;
    }
    return m;
}

template <bool ALIGNED>
__global__ void __launch_bounds__(kThreads) k_count_flags(const uint8_t *__restrict__ f, uint64_t n,
                                                          const uint64_t *__restrict__ d_n,
                                                          uint32_t *__restrict__ counts) {
    __shared__ uint32_t ws[kThreads / 32];
    n = count_of(n, d_n);
    const uint64_t i0 = blockIdx.x * (uint64_t)kTile + (uint64_t)threadIdx.x * kPerThread;
    uint32_t c = __popcll(load_mask<ALIGNED>(f, i0, n));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t t = 0;
        for (int w = 0; w < kThreads / 32; w++) t += ws[w];
        counts[blockIdx.x] = t;
    }
}

// Single-CTA exclusive scan of the block counts (64-bit offsets) and the total.
__global__ void __launch_bounds__(1024) k_scan_counts(const uint32_t *__restrict__ counts, uint64_t nb,
                                                      uint64_t *__restrict__ excl, uint64_t *__restrict__ total) {
    __shared__ uint64_t wt[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t carry = 0;
    for (uint64_t base = 0; base < nb; base += 1024) {
        const uint64_t i = base + threadIdx.x;
        const uint64_t v = i < nb ? counts[i] : 0;
        uint64_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wt[warp] = x;
        __syncthreads();
        if (warp == 0) {
            uint64_t t = wt[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint64_t y = __shfl_up_sync(kFull, t, o);
                if (lane >= o) t += y;
            }
            wt[lane] = t;
        }
        __syncthreads();
        const uint64_t pre = carry + (warp ? wt[warp - 1] : 0) + x - v;
        if (i < nb) excl[i] = pre;
        carry += wt[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) *total = carry;
}

template <bool ALIGNED>
__global__ void __launch_bounds__(kThreads) k_emit(const uint8_t *__restrict__ f, uint64_t n,
                                                   const uint64_t *__restrict__ d_n, uint32_t id_base,
                                                   const uint64_t *__restrict__ excl,
                                                   const uint64_t *__restrict__ total, uint64_t cap,
                                                   uint32_t *__restrict__ ids) {
    n = count_of(n, d_n);
    __shared__ uint32_t ws[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t i0 = blockIdx.x * (uint64_t)kTile + (uint64_t)threadIdx.x * kPerThread;
    // the flags, the block's offset and the total are independent loads: all in flight together
    uint64_t m = load_mask<ALIGNED>(f, i0, n);
    const uint64_t block_base = excl[blockIdx.x];
    if (*total > cap) return;  // nothing is written when the output does not fit (the same for every block)
    const uint32_t c = __popcll(m);
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    uint32_t pre = x - c;
    for (int w = 0; w < warp; w++) pre += ws[w];
    uint64_t dst = block_base + pre;
    while (m) {
        const int b = __ffsll((long long)m) - 1;
        m &= m - 1;
        ids[dst++] = id_base + (uint32_t)(i0 + b);
    }
}

}  // namespace

cudaError_t preload_compact_kernels() {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, k_count_flags<true>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, k_count_flags<false>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, k_scan_counts);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, k_emit<true>);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, k_emit<false>);
    return e;
}

uint64_t compact_scratch_words(uint64_t n) {
    const uint64_t nb = (n + kTile - 1) / kTile;
    return nb + 2 * nb + 2;  // counts (u32) + exclusive offsets (u64)
}

cudaError_t launch_compact(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids, uint64_t cap,
                           uint32_t *d_scratch, uint64_t *d_total, cudaStream_t st, const uint64_t *d_n) {
    if (!n) return cudaMemsetAsync(d_total, 0, 8, st);
    const uint64_t nb = (n + kTile - 1) / kTile;
    uint32_t *counts = d_scratch;
    // exclusive offsets start on an 8-byte boundary after the counts
    uint64_t *excl = reinterpret_cast<uint64_t *>(d_scratch + ((nb + 1) & ~1ull));
    const bool aligned = (reinterpret_cast<uintptr_t>(d_flags) & 15u) == 0;
    if (aligned) {
        k_count_flags<true><<<(unsigned)nb, kThreads, 0, st>>>(d_flags, n, d_n, counts); count_launch();
    } else {
        k_count_flags<false><<<(unsigned)nb, kThreads, 0, st>>>(d_flags, n, d_n, counts); count_launch();
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_scan_counts<<<1, 1024, 0, st>>>(counts, nb, excl, d_total); count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (aligned) {
        k_emit<true><<<(unsigned)nb, kThreads, 0, st>>>(d_flags, n, d_n, id_base, excl, d_total, cap, d_ids); count_launch();
    } else {
        k_emit<false><<<(unsigned)nb, kThreads, 0, st>>>(d_flags, n, d_n, id_base, excl, d_total, cap, d_ids); count_launch();
    }
    return cudaGetLastError();
}

}  // namespace hspz
