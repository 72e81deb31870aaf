// Internal definitions shared by the CUDA translation units of libhspz.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "hspz.h"

namespace hspz {

// Packed sequences hold 8 bases per uint32 (one nibble each, base i of a word
// in bits 4i..4i+3) behind kPadBases bases of padding at both ends, so window
// loads around any in-range anchor stay inside the buffer: the widest read is
// a 256-base warp tile plus one word, starting inside the sequence.
//   reference nibble: bits 0-1 code, bit 2 = code0 ^ code1 (1 for C and G), bit 3 = N
//   query nibble:     bits 0-1 code, bit 2 = 0,                              bit 3 = N
// An N keeps code bits 0.  Padding nibbles are N.
constexpr int kPadBases = 512;
constexpr int kPadWords = kPadBases / 8;
constexpr uint32_t kNibN = 0x8u;
constexpr int kMaxSpan = 32;
constexpr int kMaxWeight = 12;
constexpr int kCountBlock = 256;  // seeds per count/scan block (C.2: 256 counts per block)

struct SeedShape {
    int span;
    int weight;
    int care[kMaxSpan];
};

struct ScoreArgs {
    int32_t m[25];
    int32_t xdrop;
    int32_t T;
    // complement-symmetric int8 table for the fast gate: entry (r ^ q) | parity(r) << 2
    uint32_t tab_lo, tab_hi;
    int fast;  // 1 when the fast table reproduces m exactly on A/C/G/T
    int exact; // 1 when fast and X >= 7 * max(0, largest entry of m): the gate's 8-base step needs no replay
};

struct SeqView {
    const uint32_t *packed;  // padded packed words
    uint64_t len;            // bases
    const uint32_t *rev;     // padded packed words of the reversed sequence (base i = base len-1-i)
    bool has_n;              // some base is N (not A/C/G/T)
};

int parse_pattern(const char *pat, SeedShape *sh);
int make_score_args(const hspz_score_params *p, ScoreArgs *out);
uint64_t packed_words(uint64_t len);

// stream-ordered allocation from the library's caching pool of the current device
cudaError_t pool_alloc(void **p, size_t bytes, cudaStream_t st);
template <typename T>
cudaError_t pool_alloc(T **p, size_t bytes, cudaStream_t st) {
    return pool_alloc(reinterpret_cast<void **>(p), bytes, st);
}
cudaError_t pool_free(void *p, cudaStream_t st);

// kernel launch accounting (every launch site calls count_launch(k) for k launches)
void count_launch(uint64_t k = 1);

// error plumbing
void set_error(const std::string &msg);
int cuda_fail(cudaError_t e, const char *what);
#define HSPZ_CUDA(call)                                          \
    do {                                                         \
        cudaError_t e_ = (call);                                 \
        if (e_ != cudaSuccess) return hspz::cuda_fail(e_, #call); \
    } while (0)

// launchers (each returns cudaError_t of the launch)
// d_n_count (nullable) is incremented by the number of N bases packed
cudaError_t launch_pack(const uint8_t *d_codes, uint64_t len, int with_parity, int reverse, uint32_t *d_packed,
                        uint64_t words, cudaStream_t st, unsigned long long *d_n_count = nullptr);
cudaError_t launch_count(const uint8_t *d_query, uint64_t n_seeds, const SeedShape &sh, const uint32_t *d_idx,
                         uint32_t *d_cnt, uint32_t *d_lo, uint64_t *d_block_sum, cudaStream_t st);
cudaError_t launch_scan_u64(const uint64_t *d_in, uint64_t n, uint64_t *d_excl, uint64_t *d_incl,
                            uint64_t *d_total, cudaStream_t st);
cudaError_t launch_prefix(const uint32_t *d_cnt, uint64_t n_seeds, const uint64_t *d_block_excl, uint32_t *d_P,
                          cudaStream_t st);
cudaError_t launch_expand(const uint32_t *d_P, const uint32_t *d_cnt, const uint32_t *d_lo, const uint32_t *d_pos,
                          const hspz_chunk &c, int span, int dense, hspz_anchor *d_out, cudaStream_t st);
// uint32 words of tile scratch the fused kernel needs for a chunk of max_chunk_hits anchors
uint64_t expand_gate_tile_words(uint64_t max_chunk_hits);
cudaError_t launch_expand_gate(const uint32_t *d_P, const uint32_t *d_lo, const uint32_t *d_pos,
                               const hspz_chunk &c, int span, SeqView ref, SeqView qry, const ScoreArgs &sa,
                               hspz_anchor *d_out, uint8_t *d_flags, uint32_t *d_tiles, cudaStream_t st);
// d_raw (nullable, fast matrices only): flag of anchor i goes to d_flags[d_raw[i]]
cudaError_t launch_gate(const hspz_anchor *d_anchors, const uint32_t *d_raw, uint64_t n, SeqView ref, SeqView qry,
                        const ScoreArgs &sa, uint8_t *d_flags, cudaStream_t st);
// reference-locality buckets (D.5): stable counting sort of n anchors by ref_end / span into n_buckets
// buckets; d_sorted/d_raw receive the anchors and their raw ids; d_scratch holds bucket_scratch_words(n)
uint64_t bucket_scratch_words(uint64_t n, uint32_t n_buckets);
cudaError_t launch_bucket_sort(const hspz_anchor *d_anchors, uint64_t n, uint32_t span, uint32_t n_buckets,
                               hspz_anchor *d_sorted, uint32_t *d_raw, uint32_t *d_scratch, cudaStream_t st);
cudaError_t launch_scan_u32(const uint32_t *d_in, uint64_t n, uint32_t *d_excl, cudaStream_t st);
// Stable LSD radix sort of n (key, value) pairs by the low key_bits bits of the
// key (8 bits per pass), in place; scratch of radix_sort_scratch_words(n) words.
uint64_t radix_sort_scratch_words(uint64_t n);
cudaError_t launch_radix_sort_pairs(uint32_t *d_keys, uint32_t *d_vals, uint64_t n, int key_bits, uint32_t *d_scratch,
                                    cudaStream_t st);
// With d_n, the survivor count is read on the device from *d_n (n_ids bounds it; a larger count means 0).
cudaError_t launch_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                               uint64_t n_ids, SeqView ref, SeqView qry, const ScoreArgs &sa,
                               hspz_segment_pair *d_out, uint8_t *d_done, cudaStream_t st,
                               const uint64_t *d_n = nullptr, bool grouped = false);
// stable compaction in three launches; d_scratch holds compact_scratch_words(n) uint32.
// With d_n, the flag count is read on the device from *d_n (n bounds it; a larger count means 0).
uint64_t compact_scratch_words(uint64_t n);
// Loads the compaction kernels onto the current device now (under lazy module
// loading a kernel is otherwise loaded, taking device memory, at its first launch).
cudaError_t preload_compact_kernels();
cudaError_t launch_compact(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids, uint64_t cap,
                           uint32_t *d_scratch, uint64_t *d_total, cudaStream_t st, const uint64_t *d_n = nullptr);

// duplicate removal (two passes over a table of dedup_table_slots(n) uint32, keep flags out)
uint64_t dedup_table_slots(uint64_t n);
cudaError_t launch_dedup(const hspz_segment_pair *d_records, uint64_t n, uint32_t *d_tab, uint64_t slots,
                         uint8_t *d_keep, unsigned long long *d_err, cudaStream_t st);
cudaError_t launch_gather_records(const hspz_segment_pair *d_records, const uint32_t *d_idx, uint64_t n,
                                  hspz_segment_pair *d_out, cudaStream_t st);

}  // namespace hspz

struct hspz_index {
    hspz::SeedShape shape;
    uint64_t ref_len;
    uint64_t n_pos;
    uint32_t *d_idx;  // 4^weight inclusive bucket ends
    uint32_t *d_pos;  // n_pos reference ends grouped by bucket
    uint32_t *d_ref;      // packed reference
    uint32_t *d_ref_rev;  // packed reversed reference (left walks run forward over it)
    uint64_t ref_words;
    int device;
    bool has_n;            // the reference holds N
};

struct hspz_plan {
    const hspz_index *index;
    uint64_t query_len;
    uint64_t n_seeds;
    uint64_t total;
    uint32_t *d_P;          // inclusive prefix, n_seeds
    uint32_t *d_lo;         // bucket start per seed
    uint32_t *d_cnt;        // hit count per seed
    uint64_t *d_blk;        // per 256-seed block: sums, exclusive and inclusive prefixes, total (3*nb + 1)
    uint64_t n_blocks;
    uint32_t *d_qry;        // packed query
    uint32_t *d_qry_rev;    // packed reversed query
    bool has_n;             // the query holds N
    uint64_t qry_words;
    std::vector<hspz_chunk> chunks;
    uint64_t max_chunk_hits;
    uint32_t *d_tiles;      // fused-kernel scratch: first/last seed of every tile of a chunk
    cudaStream_t stream;    // the stream the plan was made on; its buffers are freed in its order
};
