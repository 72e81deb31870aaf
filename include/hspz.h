/*
 * hspz.h -- C ABI of the GB300 (sm_103a) seed-hit -> ungapped X-drop HSP library.
 *
 * The library turns query spaced seeds into raw (reference-end, query-end)
 * anchors against a bucketed reference k-mer index, gates every anchor with an
 * exact score-only X-drop test, compacts the survivors stably and materializes
 * them into 16-byte SegmentPair records.  The operations follow the hspZ
 * v0.0.4 documentation:
 *   "C. Hit discovery"          C.1 count, C.2 prefix, C.3 MAX_HITS chunks,
 *                               C.4 sparse/dense choice, C.5 backward expansion
 *   "D. Score gate"             D.1 anchor feed, D.2 score-only X-drop + keep
 *                               threshold, D.3 byte flags, D.4 stable compaction
 *   "E. X-drop materialization" E.1 restore, E.2 right, E.3 left, E.4 closed
 *                               interval, E.5 store
 *
 * Conventions for every call
 *   - Base codes are uint8: A=0 C=1 G=2 T=3; any other value is N.
 *   - The substitution matrix is int32[25], row = reference base, column =
 *     query base, index 5*ref + query (row/column 4 = N).
 *   - Coordinates are 0-based.  An anchor holds the END of its seed window:
 *     reference end = window start + span - 1, query end = seed index + span - 1
 *     (seed s is the query window starting at position s; every query position
 *     is seeded).
 *   - Pointers named d_* are DEVICE pointers on the current CUDA device and
 *     stay owned by the caller.  Pointers without the prefix are host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are stream ordered; a call that returns counts to the
 *     host (hspz_build_index, hspz_find_hits, hspz_compact) synchronizes that
 *     stream before it returns.
 *   - Every call returns an hspz_status.  A non-zero status means no output
 *     of that call was written, except the *_needed / total counts documented
 *     below.  Arguments are checked before any launch; hspz_strerror() names
 *     the status, hspz_last_error() gives the last detailed message.
 *   - Every output slot a call owns is overwritten in full (the pages' "every
 *     active flag slot is overwritten before reuse", D.3, and "every active
 *     output slot is fully overwritten", E.5).
 *   - Limits: 1 <= K <= 2^30, 0 <= xdrop <= 2^30, |matrix entry| <= 2^16,
 *     sequences shorter than 2^32 - 2^10 bases.
 */
#ifndef HSPZ_H
#define HSPZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HSPZ_ABI_VERSION 1

typedef enum hspz_status {
    HSPZ_OK = 0,
    HSPZ_E_INVAL = 1,        /* bad argument (null pointer, bad pattern, limits)     */
    HSPZ_E_HIT_OVERFLOW = 2, /* total hits do not fit the 32-bit hit index (C.2)     */
    HSPZ_E_CAPACITY = 3,     /* output capacity too small; the needed size is given  */
    HSPZ_E_CUDA = 4,         /* a CUDA runtime call failed (see hspz_last_error)     */
    HSPZ_E_NOMEM = 5,        /* device or host allocation failed                      */
    HSPZ_E_UNSUPPORTED = 6   /* request outside what this build implements           */
} hspz_status;

/* Packed anchor, raw hit order (D.1 "packed (reference-end, query-end) anchors"). 8 bytes. */
typedef struct hspz_anchor {
    uint32_t ref_end;
    uint32_t query_end;
} hspz_anchor;

/* Materialized HSP (E.4/E.5): the closed interval ref_start..=ref_start+len on
 * the reference and query_start..=query_start+len on the query; score is the
 * substitution-score sum over that interval.  16 bytes, 16-byte aligned. */
typedef struct hspz_segment_pair {
    uint32_t ref_start;
    uint32_t query_start;
    uint32_t len;
    int32_t score;
} hspz_segment_pair;

/* One MAX_HITS chunk (C.3): seeds [seed_begin, seed_end) and global anchor
 * ids [hit_begin, hit_end).  A seed is never split across chunks. */
typedef struct hspz_chunk {
    uint32_t seed_begin;
    uint32_t seed_end;
    uint32_t hit_begin;
    uint32_t hit_end;
} hspz_chunk;

/* Scoring (D.2): substitution matrix, X-drop and hsp threshold K. */
typedef struct hspz_score_params {
    int32_t matrix[25];
    int32_t xdrop;
    int32_t K;
} hspz_score_params;

typedef struct hspz_index hspz_index; /* reference side: k-mer index + packed reference   */
typedef struct hspz_plan hspz_plan;   /* one query batch: seeds, prefix, chunks, packed query */

/* Expansion mappings (C.4). */
enum { HSPZ_EXPAND_AUTO = 0, HSPZ_EXPAND_SPARSE = 1, HSPZ_EXPAND_DENSE = 2 };
/* hspz_find_hits flags (C.3): locate chunk boundaries by copying the whole
 * prefix array instead of the block sums plus one 256-count block per cut. */
enum { HSPZ_WALK_FULL = 1 };

const char *hspz_strerror(int status);
const char *hspz_last_error(void);
int hspz_abi_version(void);
/* Number of CUDA kernels this library has launched in this process (all
 * devices, all threads); lets a caller count the launches of a region. */
uint64_t hspz_kernel_launches(void);
/* Device memory the library allocates per call (plans, scratch, index-build
 * temporaries) comes from one stream-ordered memory pool per device owned by
 * the library; memory freed back to it stays cached for the next call instead
 * of being returned to the driver.  This returns every pool's cached memory
 * that no allocation holds (cudaMemPoolTrimTo).  Memory still held by live
 * plans or by frees not yet reached on their streams stays in the pools.
 * Calls that hand a count back to the host (hspz_find_hits,
 * hspz_process_chunk, hspz_compact, hspz_dedup) read it through 64 bytes of
 * pinned, device-mapped host memory that each calling thread allocates on
 * its first such call and keeps for its lifetime (a one-thread kernel writes
 * it, so the read does not queue behind large copies on the copy engine). */
int hspz_release_cached_memory(void);

/* ------------------------------------------------------------------------ *
 * Keep threshold ("D. Score gate", D.2 invariant): the least integer total t
 * for which (float)t >= (float)K, i.e. the integer twin of KegAlign's f32 keep
 * comparison; computed once per engine on the host.  Returns HSPZ_E_INVAL for
 * K < 1 or K > 2^30.
 * ------------------------------------------------------------------------ */
int hspz_keep_threshold(int32_t K, int32_t *T_out);

/* ------------------------------------------------------------------------ *
 * Reference index ("C. Hit discovery", C.1 index table of cumulative bucket
 * ends; C.5 bucket start..end).  d_ref: ref_len base codes.  seed_pattern: a
 * string of '1' (care) and '0' (don't care), first and last '1', span <= 32,
 * weight <= 12 (default "1110100110010101111").  Every reference window
 * without N at a care offset is indexed by its packed k-mer (first care base
 * most significant); the index holds idx[4^weight] (inclusive bucket ends)
 * and pos[] (reference ends, ascending inside each bucket) plus a packed copy
 * of the reference for scoring.  The library owns the handle; free it with
 * hspz_index_free after every plan made from it.  Synchronizes `stream`.
 * ------------------------------------------------------------------------ */
int hspz_build_index(const uint8_t *d_ref, uint64_t ref_len, const char *seed_pattern,
                     hspz_index **index_out, void *stream);
void hspz_index_free(hspz_index *index);
/* Sizes and device views of the index tables (owned by the index). */
int hspz_index_info(const hspz_index *index, uint64_t *n_positions, uint32_t *span, uint32_t *weight);
int hspz_index_tables(const hspz_index *index, const uint32_t **d_idx, const uint32_t **d_pos);

/* ------------------------------------------------------------------------ *
 * Hit discovery for one query batch ("C. Hit discovery", C.1-C.3).
 * Seeds every query window (n_seeds = query_len - span + 1), counts each
 * seed's hits (find_num_hits: bucket end - previous bucket end; 0 for a seed
 * with N at a care offset), forms the global inclusive prefix and the total,
 * refuses a total above 2^32 - 1 with HSPZ_E_HIT_OVERFLOW (no plan is made;
 * *total_hits still reports the total), and cuts MAX_HITS chunks: one chunk if
 * total <= max_hits or max_hits == 0, else the lower-bound walk over the seed
 * prefixes that keeps the straddling seed whole.  flags: 0 or HSPZ_WALK_FULL.
 * The plan keeps pointers into `index`.  Its device buffers come from the
 * library's stream-ordered memory pool on `stream`, and hspz_plan_free returns
 * them in that stream's order, so free a plan only with its work queued on
 * that stream (or finished).  Synchronizes `stream`.
 * ------------------------------------------------------------------------ */
int hspz_find_hits(const hspz_index *index, const uint8_t *d_query, uint64_t query_len, uint64_t max_hits,
                   uint32_t flags, hspz_plan **plan_out, uint64_t *total_hits, void *stream);
void hspz_plan_free(hspz_plan *plan);
/* n_seeds, total hits, chunk count and the largest chunk's hit count. */
int hspz_plan_info(const hspz_plan *plan, uint64_t *n_seeds, uint64_t *total_hits, uint32_t *n_chunks,
                   uint64_t *max_chunk_hits);
/* Host copy of the chunk list; HSPZ_E_CAPACITY (with *n_chunks set) if cap is too small. */
int hspz_plan_chunks(const hspz_plan *plan, hspz_chunk *chunks, uint32_t cap, uint32_t *n_chunks);
/* Device view of the inclusive prefix P[n_seeds] (uint32, owned by the plan). */
int hspz_plan_prefix(const hspz_plan *plan, const uint32_t **d_prefix);

/* ------------------------------------------------------------------------ *
 * Backward expansion of one chunk ("C. Hit discovery", C.4-C.5): occurrence j
 * of seed s (j = 0 at the bucket start) goes to slot P[s] - 1 - hit_begin - j.
 * mode: HSPZ_EXPAND_AUTO picks the warp-per-seed mapping when the chunk holds
 * at least 16 hits per seed, else thread-per-seed; both write identical
 * anchors.  d_anchors needs cap >= chunk hits (else HSPZ_E_CAPACITY).
 * ------------------------------------------------------------------------ */
int hspz_expand(const hspz_plan *plan, uint32_t chunk, int mode, hspz_anchor *d_anchors, uint64_t cap,
                void *stream);

/* ------------------------------------------------------------------------ *
 * Fused expansion + score gate of one chunk (C.5 + D.1-D.3): writes the same
 * anchors as hspz_expand and, for each, the flag byte of hspz_score_gate_plan.
 * Uses a small tile table owned by the plan, so two hspz_expand_gate calls on
 * one plan must not run at the same time on the GPU.
 * ------------------------------------------------------------------------ */
int hspz_expand_gate(const hspz_plan *plan, uint32_t chunk, const hspz_score_params *params,
                     hspz_anchor *d_anchors, uint8_t *d_flags, uint64_t cap, void *stream);

/* ------------------------------------------------------------------------ *
 * One chunk through the rest of the path with a single host synchronization:
 * the fused expansion + gate (hspz_expand_gate), the stable compaction of the
 * flags into survivor ids (hspz_compact), their materialization
 * (hspz_materialize_plan) and the stable compaction of the done flags into
 * accepted indices (positions in the survivor list).  The survivor count
 * stays on the device between the steps.  d_anchors and d_flags need room
 * for the chunk's hits (cap_anchors); d_ids, d_records (16-byte aligned),
 * d_done and d_accepted for cap_survivors entries.  *n_survivors and
 * *n_accepted receive the counts.  If the survivors exceed cap_survivors,
 * HSPZ_E_CAPACITY is returned with *n_survivors set: the anchors and flags are
 * written, the survivor outputs are not; call again with more room.  gate_ms
 * (may be NULL) receives the fused kernel's own event-timed duration.  Uses
 * stream-ordered scratch; synchronizes `stream`.
 * ------------------------------------------------------------------------ */
int hspz_process_chunk(const hspz_plan *plan, uint32_t chunk, const hspz_score_params *params,
                       hspz_anchor *d_anchors, uint8_t *d_flags, uint64_t cap_anchors, uint32_t *d_ids,
                       hspz_segment_pair *d_records, uint8_t *d_done, uint32_t *d_accepted, uint64_t cap_survivors,
                       uint64_t *n_survivors, uint64_t *n_accepted, float *gate_ms, void *stream);

/* ------------------------------------------------------------------------ *
 * Score-only X-drop gate ("D. Score gate", D.1-D.3: anchors and the encoded
 * sequences in, one flag byte per anchor out) over n anchors of any origin.
 * d_anchors: n hspz_anchor (reference end, query end) in device memory;
 * d_ref / d_query: ref_len / query_len base codes (uint8, A0 C1 G2 T3, any
 * other value N) in device memory.  Per anchor (a_r, a_q): the right side
 * scores the anchor base and the bases after it, the left side the bases
 * before it; each side walks with S_0 = M_0 = 0, S_n = S_{n-1} +
 * m[ref][qry], stops before step n when M_{n-1} - S_n > xdrop or at a
 * sequence edge, and yields its maximum M.  d_flags[i] = 1 when M_left +
 * M_right >= T with T = hspz_keep_threshold(K), else 0; an anchor outside the
 * sequences gets 0.  The call packs both sequences into stream-ordered scratch
 * from the library's memory pool (about (ref_len + query_len) / 2 + 1 KiB
 * bytes, freed in stream order) and does not synchronize `stream`.
 * hspz_score_gate_plan gates against an index and a plan without packing.
 * ------------------------------------------------------------------------ */
int hspz_score_gate(const hspz_anchor *d_anchors, uint64_t n, const uint8_t *d_ref, uint64_t ref_len,
                    const uint8_t *d_query, uint64_t query_len, const hspz_score_params *params, uint8_t *d_flags,
                    void *stream);

/* The same gate against the packed reference of `index` and the packed query
 * of `plan` (made from that index); nothing is packed or allocated. */
int hspz_score_gate_plan(const hspz_index *index, const hspz_plan *plan, const hspz_anchor *d_anchors, uint64_t n,
                         const hspz_score_params *params, uint8_t *d_flags, void *stream);

/* ------------------------------------------------------------------------ *
 * Reference-bucketed score gate ("D. Score gate", D.5): the same flags as
 * hspz_score_gate_plan, computed after a stable counting sort of the anchors into
 * n_buckets reference-address windows (1..32; 0 = auto: enough windows that
 * one window of the packed reference, both directions, fits 3/4 of the L2).
 * The gate writes each flag at the anchor's raw position.  Needs a matrix the
 * fast gate takes (complement symmetric on A/C/G/T with int8 scores), else
 * HSPZ_E_UNSUPPORTED.  Uses stream-ordered scratch of 12 bytes per anchor.
 * ------------------------------------------------------------------------ */
int hspz_score_gate_bucketed(const hspz_index *index, const hspz_plan *plan, const hspz_anchor *d_anchors, uint64_t n,
                             const hspz_score_params *params, uint32_t n_buckets, uint8_t *d_flags, void *stream);

/* ------------------------------------------------------------------------ *
 * Stable compaction ("D. Score gate", D.4): d_ids receives id_base + i for
 * every i < n with d_flags[i] != 0, in increasing order; *n_out receives the
 * count.  If the count exceeds cap nothing is written and HSPZ_E_CAPACITY is
 * returned with *n_out set.  Uses stream-ordered scratch from the library's
 * memory pool.  Synchronizes `stream`.
 * ------------------------------------------------------------------------ */
int hspz_compact(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids, uint64_t cap,
                 uint64_t *n_out, void *stream);

/* ------------------------------------------------------------------------ *
 * hspz_compact without any device allocation.  The hspZ pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory while they run -- a program whose device memory was handed in full
 * to another allocator at start-up, so cudaMalloc would fail, or one that
 * must not take the implicit device synchronization cudaMalloc/cudaFree can
 * cause.  Same arguments, result and statuses as hspz_compact, for at most
 * hspz_compact_noalloc_max_flags() = 2^28 flags (larger n: HSPZ_E_INVAL with
 * a message in hspz_last_error).  Its scratch is one fixed device array of
 * about 768 KiB inside the library.  CUDA loads library code lazily, so that
 * array and the compaction kernels take their device memory on a device only
 * when this call first runs there (even with n = 0: that call loads them and
 * does nothing else); from then on they stay until the process exits.  Make
 * one call per device, n = 0 will do, before handing the device's memory to
 * another allocator, and before any stream capture.  Every call looks up the
 * array's device address for the current device, so a cudaDeviceReset does
 * not leave a stale address (the next call loads the code again).  All calls
 * share the one array, so calls that overlap on the GPU (different streams or
 * threads at the same time) race and must be serialized by the caller.
 * Synchronizes `stream` (except with n = 0).
 * ------------------------------------------------------------------------ */
int hspz_compact_noalloc(const uint8_t *d_flags, uint64_t n, uint32_t id_base, uint32_t *d_ids, uint64_t cap,
                         uint64_t *n_out, void *stream);
uint64_t hspz_compact_noalloc_max_flags(void);

/* ------------------------------------------------------------------------ *
 * Exact X-drop materialization ("E. X-drop materialization", E.1-E.5) against
 * raw device sequences (base codes as for hspz_score_gate).  For survivor k
 * with global id d_ids[k], the anchor d_anchors[d_ids[k] - id_base]
 * (n_anchors entries; an id outside [id_base, id_base + n_anchors), or an
 * anchor outside the sequences, yields a rejected slot) is walked right and
 * left as in hspz_score_gate, keeping on each side the EARLIEST step count n
 * attaining the maximum (0 for the empty prefix).  Then
 * ref_start = a_r - n_left, query_start = a_q - n_left,
 * len = n_left + n_right - 1 (closed interval start..=start+len) and
 * score = M_left + M_right (saturated at INT32_MAX).  done[k] = score >= T: an
 * accepted slot holds the record, a rejected slot is written as zeros with
 * done = 0.  d_out must be 16-byte aligned.  Any order of d_ids is allowed;
 * when the next entry is the next survivor on the same diagonal the two walks
 * share work (same records).  n_anchors is not in the pages' call: it bounds
 * the ids so that no id reads outside the caller's anchor array.  The call
 * packs both sequences forward and reversed into stream-ordered scratch
 * (about ref_len + query_len + 2 KiB bytes) and, when the 8-base stop test is
 * exact (xdrop >= 7 x the largest pair score), takes 48 bytes per id (at most
 * 2^25 ids at a time) more, all from the library's memory pool; it does not
 * synchronize `stream`.
 * ------------------------------------------------------------------------ */
int hspz_materialize(const hspz_anchor *d_anchors, uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids,
                     uint64_t n_ids, const uint8_t *d_ref, uint64_t ref_len, const uint8_t *d_query,
                     uint64_t query_len, const hspz_score_params *params, hspz_segment_pair *d_out, uint8_t *d_done,
                     void *stream);

/* The same materialization against the packed copies of `index` and `plan`
 * (made from that index); only the 48 bytes per id of the exact-test mode are
 * taken from the pool. */
int hspz_materialize_plan(const hspz_index *index, const hspz_plan *plan, const hspz_anchor *d_anchors,
                          uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids, uint64_t n_ids,
                          const hspz_score_params *params, hspz_segment_pair *d_out, uint8_t *d_done, void *stream);

/* ---------------------------------------------------------------------------
 * hspz_materialize_plan with the ids taken in diagonal order: the same records and
 * done flags, at the same places, for any id list.  Each slice of at most
 * 2^25 ids is sorted (stable radix sort) by the anchor's diagonal
 * (reference end - query end) first, so that survivors on one diagonal
 * become neighbours and share their walks (hspz_materialize_plan shares work only
 * between neighbouring entries of the list).  Worth it when many survivors
 * lie on the same diagonals but apart in the list, as in repeats: the ids of
 * one query position hit many reference positions, i.e. many diagonals.
 * Uses stream-ordered scratch of about 68 bytes per id (per slice) from the
 * library's memory pool; does not synchronize `stream`.
 * ------------------------------------------------------------------------ */
int hspz_materialize_grouped(const hspz_index *index, const hspz_plan *plan, const hspz_anchor *d_anchors,
                             uint64_t n_anchors, uint32_t id_base, const uint32_t *d_ids, uint64_t n_ids,
                             const hspz_score_params *params, hspz_segment_pair *d_out, uint8_t *d_done, void *stream);

/* ------------------------------------------------------------------------ *
 * Record gather: d_out[k] = d_records[d_idx[k]] for k < n (16-byte records;
 * both arrays 16-byte aligned; every d_idx[k] must index d_records).  Collects
 * a chunk's accepted records (d_idx = the accepted survivor indices written
 * by hspz_compact over the done flags) into a batch-wide array for
 * hspz_dedup, and the kept records after it.  Asynchronous on `stream`.
 * ------------------------------------------------------------------------ */
int hspz_gather_records(const hspz_segment_pair *d_records, const uint32_t *d_idx, uint64_t n,
                        hspz_segment_pair *d_out, void *stream);

/* ------------------------------------------------------------------------ *
 * Duplicate removal over the accepted HSPs of one query batch ("D. Score
 * gate": the accepted raw HSPs become the final HSPs after dedup; "C. Hit
 * discovery", C.5: the raw anchor order sets the dedup scope).  The pages do
 * not state the criterion.  Reading taken here: record i of d_records (the
 * batch's accepted records in raw order, n of them, 16-byte aligned) is
 * dropped when a record j < i has the same four fields.  d_keep_ids receives
 * the indices of the kept records in increasing order and *n_kept their
 * count; if the count exceeds cap nothing is written to d_keep_ids and
 * HSPZ_E_CAPACITY is returned with *n_kept set.  n <= 2^31 (else
 * HSPZ_E_INVAL).  Uses stream-ordered scratch of about 8n + n bytes from the
 * library's memory pool.  Synchronizes `stream`.
 * ------------------------------------------------------------------------ */
int hspz_dedup(const hspz_segment_pair *d_records, uint64_t n, uint32_t *d_keep_ids, uint64_t cap,
               uint64_t *n_kept, void *stream);

/* ------------------------------------------------------------------------ *
 * Host-only chunk walk over a host prefix array, exactly the walk
 * hspz_find_hits runs (use_block_sums != 0: lower bound located through the
 * 256-count block sums, then inside one block; 0: over the whole array).
 * For testing the host logic without a GPU.
 * ------------------------------------------------------------------------ */
int hspz_chunk_walk_host(const uint32_t *prefix, uint64_t n_seeds, uint64_t max_hits, int use_block_sums,
                         hspz_chunk *chunks, uint32_t cap, uint32_t *n_chunks);

#ifdef __cplusplus
}
#endif
#endif /* HSPZ_H */
