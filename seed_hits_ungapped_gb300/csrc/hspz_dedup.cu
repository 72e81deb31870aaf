// Duplicate removal over the accepted HSPs of one query batch (the dedup
// after materialization named in "D. Score gate": accepted raw HSPs become the
// final HSPs), and the record gather that collects a batch's accepted records
// chunk by chunk.
//
// The pages give only the funnel counts, not the criterion.  Reading taken: a
// record is dropped when an earlier record of the batch (raw order = index
// order of the input) has the same four fields.
//
// Method: one open-addressing table of record indices, twice the record count
// or more, rounded to a power of two.  Every record probes from the hash of
// its four fields; it claims the first empty slot, or meets the slot that
// already holds an equal record and lowers it to its own index (atomicMin).
// A key lands in exactly one slot: the slots before it on its probe sequence
// were full when the key was first inserted, and slots are never emptied.
// After the insert pass every slot holds the smallest index of its key, so a
// record is kept iff its slot holds its own index, whatever order the threads
// ran in.  The stable compaction then lists the kept indices in order.
#include "hspz_internal.cuh"

namespace hspz {
namespace {

constexpr uint32_t kEmpty = 0xFFFFFFFFu;
constexpr int kThreads = 256;

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
    // splitmix64 finalizer (Steele, Lea and Flood, "Fast splittable
    // pseudorandom number generators", 2014)
    x ^= x >> 30;
    x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27;
    x *= 0x94D049BB133111EBull;
    x ^= x >> 31;
    return x;
}

__device__ __forceinline__ uint32_t home_slot(uint4 r, uint32_t mask) {
    const uint64_t a = ((uint64_t)r.x << 32) | r.y, b = ((uint64_t)r.z << 32) | r.w;
    return (uint32_t)mix64(a ^ mix64(b)) & mask;
}

__device__ __forceinline__ bool same(uint4 a, uint4 b) {
    return ((a.x ^ b.x) | (a.y ^ b.y) | (a.z ^ b.z) | (a.w ^ b.w)) == 0;
}

// Insert pass.  A probe sequence longer than the table (impossible at load
// 1/2 or less) sets *err instead of looping.
__global__ void __launch_bounds__(kThreads) k_dedup_insert(const uint4 *__restrict__ rec, uint32_t n,
                                                           uint32_t *__restrict__ tab, uint32_t mask,
                                                           unsigned long long *__restrict__ err) {
    for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < n; i += gridDim.x * kThreads) {
        const uint4 r = rec[i];
        uint32_t s = home_slot(r, mask);
        bool placed = false;
        for (uint64_t probe = 0; probe <= (uint64_t)mask; probe++) {
            uint32_t cur = __ldcg(tab + s);
            if (cur == kEmpty) {
                cur = atomicCAS(tab + s, kEmpty, i);
                if (cur == kEmpty) {
                    placed = true;
                    break;
                }
            }
            // slots only go from empty to a key's index and then down to
            // smaller indices of the same key, so `cur` names the slot's key
            if (same(rec[cur], r)) {
                atomicMin(tab + s, i);
                placed = true;
                break;
            }
            s = (s + 1) & mask;
        }
        if (!placed) atomicAdd(err, 1ull);
    }
}

// Mark pass: keep[i] = 1 iff the slot of record i's key holds i.
__global__ void __launch_bounds__(kThreads) k_dedup_mark(const uint4 *__restrict__ rec, uint32_t n,
                                                         const uint32_t *__restrict__ tab, uint32_t mask,
                                                         uint8_t *__restrict__ keep,
                                                         unsigned long long *__restrict__ err) {
    for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < n; i += gridDim.x * kThreads) {
        const uint4 r = rec[i];
        uint32_t s = home_slot(r, mask);
        uint8_t k = 0;
        bool found = false;
        for (uint64_t probe = 0; probe <= (uint64_t)mask; probe++) {
            const uint32_t cur = tab[s];
            if (cur == kEmpty) break;
            if (same(rec[cur], r)) {
                k = cur == i ? 1 : 0;
                found = true;
                break;
            }
            s = (s + 1) & mask;
        }
        if (!found) atomicAdd(err, 1ull);
        keep[i] = k;
    }
}

__global__ void __launch_bounds__(kThreads) k_gather_records(const uint4 *__restrict__ rec,
                                                             const uint32_t *__restrict__ idx, uint64_t n,
                                                             uint4 *__restrict__ out) {
    for (uint64_t k = blockIdx.x * (uint64_t)kThreads + threadIdx.x; k < n; k += (uint64_t)gridDim.x * kThreads)
        out[k] = rec[idx[k]];
}

unsigned blocks_for(uint64_t n) {
    const uint64_t b = (n + kThreads - 1) / kThreads;
    return (unsigned)(b < 152ull * 32 ? b : 152ull * 32);
}

}  // namespace

uint64_t dedup_table_slots(uint64_t n) {
    uint64_t t = 1024;
    while (t < 2 * n) t <<= 1;
    return t;
}

cudaError_t launch_dedup(const hspz_segment_pair *d_records, uint64_t n, uint32_t *d_tab, uint64_t slots,
                         uint8_t *d_keep, unsigned long long *d_err, cudaStream_t st) {
    if (!n) return cudaSuccess;
    const uint4 *rec = reinterpret_cast<const uint4 *>(d_records);
    cudaError_t e = cudaMemsetAsync(d_tab, 0xFF, slots * sizeof(uint32_t), st);
    if (e != cudaSuccess) return e;
    const uint32_t mask = (uint32_t)(slots - 1);
    k_dedup_insert<<<blocks_for(n), kThreads, 0, st>>>(rec, (uint32_t)n, d_tab, mask, d_err); count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_dedup_mark<<<blocks_for(n), kThreads, 0, st>>>(rec, (uint32_t)n, d_tab, mask, d_keep, d_err); count_launch();
    return cudaGetLastError();
}

cudaError_t launch_gather_records(const hspz_segment_pair *d_records, const uint32_t *d_idx, uint64_t n,
                                  hspz_segment_pair *d_out, cudaStream_t st) {
    if (!n) return cudaSuccess;
    k_gather_records<<<blocks_for(n), kThreads, 0, st>>>(reinterpret_cast<const uint4 *>(d_records), d_idx, n,
                                                         reinterpret_cast<uint4 *>(d_out)); count_launch();
    return cudaGetLastError();
}

}  // namespace hspz
