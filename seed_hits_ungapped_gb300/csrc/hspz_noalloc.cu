// hspz_compact_noalloc: the stable flag compaction of hspz_compact with its
// scratch held in a fixed device array instead of memory allocated per call.
//
// Some callers cannot allocate device memory while they run: a host program
// whose device memory was handed in full to another allocator at start-up
// (so any cudaMalloc fails), or one that must not pay the implicit device
// synchronization that cudaMalloc/cudaFree can cause in a latency-bound loop.
// This entry point serves them: it calls no cudaMalloc, cudaFree or other
// allocating routine.  The scratch is a file-scope __device__ array.
//
// CUDA loads modules lazily by default, so the array (and the compaction
// kernels) would otherwise take their device memory at the first call that
// launches work, possibly after the caller has given all memory away.  Every
// call therefore first makes sure, for the current device, that the kernels
// are loaded and the array exists (the first call on a device loads them,
// even with n = 0), then looks up the array's device address.  The lookup is
// repeated on every call so the address always belongs to the device's
// current context (a cudaDeviceReset drops the old one).
#include "hspz_internal.cuh"

namespace hspz {
namespace {

// The scratch holds one 32-bit count and one 64-bit offset per compaction
// block plus the 64-bit total; sized here for blocks of 4096 flags, it has
// room to spare for the 16384-flag blocks of launch_compact.
constexpr uint64_t kNoAllocMaxFlags = 1ull << 28;
constexpr uint64_t kNoAllocWords = 3 * (kNoAllocMaxFlags / 4096) + 8;

static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocWords];

// Set-up on the current device: load the compaction kernels, then take the
// scratch array's device address (host code only ever sees a host-side
// stand-in for the symbol, never a device address).
int setup_scratch(uint32_t **out) {
    cudaError_t e = preload_compact_kernels();
    if (e != cudaSuccess) return cuda_fail(e, "hspz_compact_noalloc: loading the compaction kernels");
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_compact_noalloc: cudaGetSymbolAddress");
    *out = static_cast<uint32_t *>(p);
    return HSPZ_OK;
}

}  // namespace
}  // namespace hspz

using namespace hspz;

extern "C" uint64_t hspz_compact_noalloc_max_flags(void) { return kNoAllocMaxFlags; }

extern "C" int hspz_compact_noalloc(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids,
                                    uint64_t cap, uint64_t *n_out, void *stream) {
    if (!n_out || (n && !d_flags) || (uint64_t)id_base + n > (1ull << 32)) return HSPZ_E_INVAL;
    if (cap && !d_ids) return HSPZ_E_INVAL;
    if (n > kNoAllocMaxFlags) {
        set_error("hspz_compact_noalloc: n exceeds the fixed scratch limit of 2^28 flags");
        return HSPZ_E_INVAL;
    }
    *n_out = 0;
    uint32_t *scratch = nullptr;
    int rc = setup_scratch(&scratch);
    if (rc) return rc;
    if (!n) return HSPZ_OK;
    cudaStream_t st = (cudaStream_t)stream;
    // counts and offsets are rewritten in full by every call; the total sits
    // after the largest layout launch_compact can use
    uint64_t *d_total = reinterpret_cast<uint64_t *>(scratch + (kNoAllocWords - 4));
    uint64_t total = 0;
    cudaError_t e = launch_compact(d_flags, n, id_base, d_ids, cap, scratch, d_total, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&total, d_total, 8, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "hspz_compact_noalloc");
    *n_out = total;
    return total > cap ? HSPZ_E_CAPACITY : HSPZ_OK;
}
