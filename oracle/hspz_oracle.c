/*
 * hspz_oracle.c -- plain, single-threaded CPU oracle for the hspZ seed-hit ->
 * ungapped X-drop HSP path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  It shares no
 * code, header, table or constant with the CUDA library: every step below is
 * written straight from the hspZ documentation pages, in their order, with no
 * blocking, fusion or reordering.
 *
 * Sources (hspZ v0.0.4 documentation):
 *   "C. Hit discovery"          hillerlab.github.io/hspZ/docs/algorithm/hit-discovery/
 *   "D. Score gate"             hillerlab.github.io/hspZ/docs/algorithm/score-gate/
 *   "E. X-drop materialization" hillerlab.github.io/hspZ/docs/algorithm/materialize/
 *
 * Base codes: A=0 C=1 G=2 T=3 N=4.  Substitution matrix: 5x5, row = reference
 * base, column = query base (m[5*r + q]).
 *
 * Parity pins (tests/test_oracle_pins.py): the worked prefix example of "C.
 * Hit discovery", brute-force seed matching, closed forms for all-match
 * segments, the maximum-prefix-sum brute force at infinite X-drop, hand cases
 * for the drop boundary and the earliest-maximum tie rule, an exhaustive f32
 * check of the keep threshold, and the exact 2^32 refusal edge.  The gate
 * flags are pinned by hand totals at exactly T and T - 1, by the best window
 * through each anchor at infinite X-drop (kept and rejected anchors), and by
 * a prefix-sum formulation of the X-drop stop at finite X; the rejected slot
 * of the materializer by a hand case below T.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_OK = 0, ORC_E_INVAL = 1, ORC_E_OVERFLOW = 2, ORC_E_CAPACITY = 3 };

#define ORC_MAX_SPAN 32
#define ORC_MAX_WEIGHT 12

/* ---------------------------------------------------------------------------
 * Spaced seed.  A pattern such as "1110100110010101111" lists care ('1') and
 * don't-care ('0') offsets of one window.  The packed k-mer of a window is the
 * base-4 number formed by its care bases, first care offset most significant
 * ("C.1 - packed k-mer per seed").  A window with N at a care offset has no
 * k-mer: it is never indexed and, as a query seed, it counts zero hits ("Empty
 * buckets contribute zero without changing seed order", C.1).
 * ------------------------------------------------------------------------- */
static int parse_pattern(const char *pat, int *care, int *weight, int *span)
{
    int n = 0, w = 0;
    if (!pat) return ORC_E_INVAL;
    for (; pat[n]; n++) {
        if (n >= ORC_MAX_SPAN) return ORC_E_INVAL;
        if (pat[n] == '1') care[w++] = n;
        else if (pat[n] != '0') return ORC_E_INVAL;
    }
    if (w < 1 || w > ORC_MAX_WEIGHT || pat[0] != '1' || pat[n - 1] != '1')
        return ORC_E_INVAL;
    *weight = w;
    *span = n;
    return ORC_OK;
}

int orc_pattern_info(const char *pat, int *weight, int *span)
{
    int care[ORC_MAX_SPAN];
    return parse_pattern(pat, care, weight, span);
}

/* k-mer of the window starting at p, or -1 if a care base is not A/C/G/T. */
static int64_t window_kmer(const uint8_t *seq, uint64_t p, const int *care, int w)
{
    int64_t h = 0;
    for (int i = 0; i < w; i++) {
        uint8_t b = seq[p + (uint64_t)care[i]];
        if (b > 3) return -1;
        h = h * 4 + b;
    }
    return h;
}

/* One entry per window start p = 0 .. len-span: its k-mer or -1. */
int orc_seed_buckets(const uint8_t *seq, uint64_t len, const char *pat, int64_t *out)
{
    int care[ORC_MAX_SPAN], w, span;
    if (parse_pattern(pat, care, &w, &span)) return ORC_E_INVAL;
    if (len < (uint64_t)span) return ORC_OK;
    for (uint64_t p = 0; p + (uint64_t)span <= len; p++) out[p] = window_kmer(seq, p, care, w);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Reference index ("C.1" and "C.5": index table of cumulative bucket ends,
 * bucket start..end of reference positions).  idx[h] = number of indexed
 * reference windows whose k-mer is <= h (inclusive cumulative bucket end).
 * pos[] lists, bucket by bucket, the reference END coordinate (window start +
 * span - 1) of every indexed window, ascending inside a bucket.
 * ------------------------------------------------------------------------- */
int orc_build_index(const uint8_t *ref, uint64_t len, const char *pat,
                    uint32_t *idx, uint32_t *pos, uint64_t pos_cap, uint64_t *n_pos)
{
    int care[ORC_MAX_SPAN], w, span;
    if (parse_pattern(pat, care, &w, &span)) return ORC_E_INVAL;
    uint64_t nb = 1ull << (2 * w);
    uint64_t *cnt = (uint64_t *)calloc(nb, sizeof(uint64_t));
    if (!cnt) return ORC_E_CAPACITY;
    uint64_t n = 0;
    if (len >= (uint64_t)span) {
        for (uint64_t p = 0; p + (uint64_t)span <= len; p++) {
            int64_t h = window_kmer(ref, p, care, w);
            if (h >= 0) { cnt[h]++; n++; }
        }
    }
    *n_pos = n;
    if (n > pos_cap || n > 0xFFFFFFFFull) { free(cnt); return ORC_E_CAPACITY; }
    /* inclusive cumulative bucket ends */
    uint64_t run = 0;
    for (uint64_t h = 0; h < nb; h++) { run += cnt[h]; idx[h] = (uint32_t)run; }
    /* fill each bucket from its start, scanning the reference left to right */
    for (uint64_t h = 0; h < nb; h++) cnt[h] = h ? idx[h - 1] : 0;
    if (len >= (uint64_t)span) {
        for (uint64_t p = 0; p + (uint64_t)span <= len; p++) {
            int64_t h = window_kmer(ref, p, care, w);
            if (h >= 0) pos[cnt[h]++] = (uint32_t)(p + (uint64_t)span - 1);
        }
    }
    free(cnt);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * find_num_hits ("C.1"): count = bucket end - previous bucket end, with the
 * previous end of bucket 0 taken as 0; a seed without a k-mer counts 0.
 * ------------------------------------------------------------------------- */
void orc_count_hits(const uint32_t *idx, const int64_t *buckets, uint64_t n_seeds, uint32_t *cnt)
{
    for (uint64_t s = 0; s < n_seeds; s++) {
        int64_t h = buckets[s];
        if (h < 0) { cnt[s] = 0; continue; }
        uint32_t end = idx[h];
        uint32_t prev = h ? idx[h - 1] : 0;
        cnt[s] = end - prev;
    }
}

/* ---------------------------------------------------------------------------
 * Global inclusive prefix ("C.2").  P[s] = sum of counts of seeds 0..s.  A
 * batch whose total does not fit the 32-bit hit index (total > 2^32 - 1) is
 * refused and P is left unspecified.
 * ------------------------------------------------------------------------- */
int orc_inclusive_prefix(const uint32_t *cnt, uint64_t n_seeds, uint32_t *P, uint64_t *total)
{
    uint64_t run = 0;
    for (uint64_t s = 0; s < n_seeds; s++) {
        run += cnt[s];
        if (run > 0xFFFFFFFFull) { *total = run; return ORC_E_OVERFLOW; }
        P[s] = (uint32_t)run;
    }
    *total = run;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * MAX_HITS chunk walk ("C.3").  max_hits == 0 means no cap.  Chunks cover the
 * seeds in order, each a non-empty seed range with its exact hit range.  If
 * the hits left from the current chunk start fit under the cap, one chunk
 * takes every remaining seed.  Otherwise the lower bound over the seed
 * prefixes finds the first seed e whose inclusive prefix reaches start + cap;
 * that seed is kept whole in the chunk, so a chunk may run past the cap by
 * less than one seed bucket.  chunks[] holds 4 words per chunk:
 * seed_begin, seed_end (exclusive), hit_begin, hit_end (exclusive).
 * ------------------------------------------------------------------------- */
int orc_chunk_walk(const uint32_t *P, uint64_t n_seeds, uint64_t max_hits,
                   uint32_t *chunks, uint64_t cap, uint64_t *n_chunks)
{
    uint64_t total = n_seeds ? P[n_seeds - 1] : 0;
    uint64_t sb = 0, hb = 0, n = 0;
    while (sb < n_seeds) {
        uint64_t se, he;
        if (max_hits == 0 || total - hb <= max_hits) {
            se = n_seeds;
            he = total;
        } else {
            uint64_t target = hb + max_hits;
            uint64_t lo = sb, hi = n_seeds; /* first s in [sb, n) with P[s] >= target */
            while (lo < hi) {
                uint64_t mid = lo + (hi - lo) / 2;
                if ((uint64_t)P[mid] < target) lo = mid + 1; else hi = mid;
            }
            se = lo + 1;
            he = P[lo];
        }
        if (n >= cap) { *n_chunks = n + 1; return ORC_E_CAPACITY; }
        chunks[4 * n + 0] = (uint32_t)sb;
        chunks[4 * n + 1] = (uint32_t)se;
        chunks[4 * n + 2] = (uint32_t)hb;
        chunks[4 * n + 3] = (uint32_t)he;
        n++;
        sb = se;
        hb = he;
    }
    *n_chunks = n;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Backward expansion ("C.5").  Occurrence j of seed s (j = 0 is the bucket
 * start) is written to slot P[s] - 1 - chunk_hit_begin - j.  The anchor is
 * (reference end, query end); a seed's query end is s + span - 1.
 * anchors[] holds 2 words per anchor.
 * ------------------------------------------------------------------------- */
void orc_expand(const uint32_t *idx, const uint32_t *pos, const int64_t *buckets,
                const uint32_t *P, const uint32_t *chunk, int span, uint32_t *anchors)
{
    uint32_t sb = chunk[0], se = chunk[1], hb = chunk[2];
    for (uint32_t s = sb; s < se; s++) {
        int64_t h = buckets[s];
        if (h < 0) continue;
        uint32_t start = h ? idx[h - 1] : 0;
        uint32_t count = idx[h] - start;
        for (uint32_t j = 0; j < count; j++) {
            uint64_t slot = (uint64_t)P[s] - 1 - hb - j;
            anchors[2 * slot + 0] = pos[start + j];
            anchors[2 * slot + 1] = s + (uint32_t)span - 1;
        }
    }
}

/* The anchor with global id g, found one by one (first seed whose inclusive
 * prefix exceeds g, then the backward slot rule solved for j). */
int orc_anchor_at(const uint32_t *idx, const uint32_t *pos, const int64_t *buckets,
                  const uint32_t *P, uint64_t n_seeds, int span, uint64_t g, uint32_t *out)
{
    uint64_t lo = 0, hi = n_seeds;
    while (lo < hi) {
        uint64_t mid = lo + (hi - lo) / 2;
        if ((uint64_t)P[mid] <= g) lo = mid + 1; else hi = mid;
    }
    if (lo >= n_seeds) return ORC_E_INVAL;
    int64_t h = buckets[lo];
    uint32_t start = h ? idx[h - 1] : 0;
    uint64_t j = (uint64_t)P[lo] - 1 - g;
    out[0] = pos[start + j];
    out[1] = (uint32_t)lo + (uint32_t)span - 1;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * One direction of the ungapped X-drop walk ("D.2", "E.2", "E.3").
 * The right side scores the anchor base and the bases after it; the left side
 * scores the bases before the anchor.  With S_0 = 0 and M_0 = 0, step n adds
 * the substitution score of the n-th base pair; the walk stops before step n
 * when M_{n-1} - S_n > X (a drop beyond X) or when a sequence edge is reached.
 * The side's result is the maximum M reached before the stop and the earliest
 * step count n at which it was first attained (0 when the maximum is the
 * empty prefix).
 * ------------------------------------------------------------------------- */
static void side_walk(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
                      uint64_t ar, uint64_t aq, int right, const int32_t *m, int64_t X,
                      int64_t *best, uint64_t *best_n)
{
    int64_t S = 0, M = 0;
    uint64_t nb = 0;
    for (uint64_t n = 1;; n++) {
        uint64_t rp, qp;
        if (right) {
            rp = ar + n - 1;
            qp = aq + n - 1;
            if (rp >= ref_len || qp >= qry_len) break;
        } else {
            if (n > ar || n > aq) break;
            rp = ar - n;
            qp = aq - n;
        }
        S += m[5 * ref[rp] + qry[qp]];
        if (M - S > X) break;
        if (S > M) { M = S; nb = n; }
    }
    *best = M;
    *best_n = nb;
}

/* Both sides of every anchor: out[4*i..] = M_left, n_left, M_right, n_right. */
void orc_side_scores(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
                     const uint32_t *anchors, uint64_t n, const int32_t *m, int32_t X, int64_t *out)
{
    for (uint64_t i = 0; i < n; i++) {
        int64_t ML, MR;
        uint64_t nL, nR;
        side_walk(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 0, m, X, &ML, &nL);
        side_walk(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 1, m, X, &MR, &nR);
        out[4 * i + 0] = ML;
        out[4 * i + 1] = (int64_t)nL;
        out[4 * i + 2] = MR;
        out[4 * i + 3] = (int64_t)nR;
    }
}

/* ---------------------------------------------------------------------------
 * Keep threshold ("D.2" invariant): the least integer t whose f32 rounding
 * compares >= the f32 rounding of K.  f32 rounding is monotone, so the set of
 * kept totals is upward closed; the search walks down from K.
 * ------------------------------------------------------------------------- */
int orc_keep_threshold(int32_t K, int32_t *T)
{
    if (K < 1) return ORC_E_INVAL;
    volatile float fk = (float)K;
    int64_t t = K;
    for (;;) {
        volatile float fprev = (float)(int32_t)(t - 1);
        if (t - 1 >= 0 && fprev >= fk) t--; else break;
    }
    *T = (int32_t)t;
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Score gate ("D.2", "D.3"): total = left maximum + right maximum; the flag
 * byte is 1 when total >= T, else 0.
 * ------------------------------------------------------------------------- */
void orc_gate(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
              const uint32_t *anchors, uint64_t n, const int32_t *m, int32_t X, int32_t T,
              uint8_t *flags)
{
    for (uint64_t i = 0; i < n; i++) {
        int64_t ML, MR;
        uint64_t nL, nR;
        side_walk(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 0, m, X, &ML, &nL);
        side_walk(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 1, m, X, &MR, &nR);
        flags[i] = (ML + MR >= (int64_t)T) ? 1 : 0;
    }
}

/* ---------------------------------------------------------------------------
 * Work of the gate decision, for measurement ("D.2", "D.3").  The flag is
 * known as soon as the running maxima reach T (total >= T is monotone in
 * either side's maximum), so the decision needs, per anchor: the left walk's
 * base pairs up to its stop, its edge, or the first pair at which its
 * maximum reaches T; then, unless that happened, the right walk's pairs up
 * to its stop, its edge, or the first pair at which the left maximum plus
 * its maximum reaches T.  Returns the sum of those pair counts over all
 * anchors.  The walk is the one side_walk takes, counted as it goes.
 * ------------------------------------------------------------------------- */
static uint64_t side_walk_pairs(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
                                uint64_t ar, uint64_t aq, int right, const int32_t *m, int64_t X,
                                int64_t need, int64_t *best)
{
    int64_t S = 0, M = 0;
    uint64_t scored = 0;
    for (uint64_t n = 1;; n++) {
        uint64_t rp, qp;
        if (right) {
            rp = ar + n - 1;
            qp = aq + n - 1;
            if (rp >= ref_len || qp >= qry_len) break;
        } else {
            if (n > ar || n > aq) break;
            rp = ar - n;
            qp = aq - n;
        }
        S += m[5 * ref[rp] + qry[qp]];
        scored = n;
        if (M - S > X) break;
        if (S > M) M = S;
        if (M >= need) break;
    }
    *best = M;
    return scored;
}

uint64_t orc_gate_pairs(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
                        const uint32_t *anchors, uint64_t n, const int32_t *m, int32_t X, int32_t T)
{
    uint64_t total = 0;
    for (uint64_t i = 0; i < n; i++) {
        int64_t ML, MR;
        total += side_walk_pairs(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 0, m, X,
                                 (int64_t)T, &ML);
        if (ML < (int64_t)T)
            total += side_walk_pairs(ref, ref_len, qry, qry_len, anchors[2 * i], anchors[2 * i + 1], 1, m, X,
                                     (int64_t)T - ML, &MR);
    }
    return total;
}

/* ---------------------------------------------------------------------------
 * Stable compaction ("D.4"): the ids (id_base + i) of every set flag, in
 * increasing order.
 * ------------------------------------------------------------------------- */
uint64_t orc_compact(const uint8_t *flags, uint64_t n, uint32_t id_base, uint32_t *ids)
{
    uint64_t k = 0;
    for (uint64_t i = 0; i < n; i++)
        if (flags[i]) ids[k++] = id_base + (uint32_t)i;
    return k;
}

/* ---------------------------------------------------------------------------
 * Materialization ("E.1" - "E.5").  For each survivor id, in order: restore
 * its anchor (anchors[] indexed by id - id_base), walk right and left keeping
 * the earliest maximum, then
 *   ref_start   = ref_end   - n_left
 *   query_start = query_end - n_left
 *   len         = n_left + n_right - 1   (closed interval start..=start+len)
 *   score       = M_left + M_right       (saturated at INT32_MAX)
 *   done        = score >= T
 * A rejected slot is written as all zeros with done = 0.
 * rec[] holds 4 words per record: ref_start, query_start, len, score.
 * ------------------------------------------------------------------------- */
void orc_materialize(const uint8_t *ref, uint64_t ref_len, const uint8_t *qry, uint64_t qry_len,
                     const uint32_t *anchors, uint32_t id_base, const uint32_t *ids, uint64_t n_ids,
                     const int32_t *m, int32_t X, int32_t T, int32_t *rec, uint8_t *done)
{
    for (uint64_t i = 0; i < n_ids; i++) {
        uint64_t a = (uint64_t)ids[i] - id_base;
        uint64_t ar = anchors[2 * a], aq = anchors[2 * a + 1];
        int64_t ML, MR;
        uint64_t nL, nR;
        side_walk(ref, ref_len, qry, qry_len, ar, aq, 0, m, X, &ML, &nL);
        side_walk(ref, ref_len, qry, qry_len, ar, aq, 1, m, X, &MR, &nR);
        int64_t score = ML + MR;
        if (score > 2147483647) score = 2147483647;
        if (score >= T) {
            rec[4 * i + 0] = (int32_t)(uint32_t)(ar - nL);
            rec[4 * i + 1] = (int32_t)(uint32_t)(aq - nL);
            rec[4 * i + 2] = (int32_t)(uint32_t)(nL + nR - 1);
            rec[4 * i + 3] = (int32_t)score;
            done[i] = 1;
        } else {
            rec[4 * i + 0] = rec[4 * i + 1] = rec[4 * i + 2] = rec[4 * i + 3] = 0;
            done[i] = 0;
        }
    }
}

/* ---------------------------------------------------------------------------
 * Duplicate removal over the accepted HSPs of one query batch ("D. Score
 * gate": the accepted raw HSPs become the final HSPs after dedup; "C. Hit
 * discovery" C.5: the raw anchor order fixes the dedup scope).  The pages do
 * not state the criterion; the reading taken here: a record is dropped when
 * an earlier record of the batch, in raw order, has the same four fields
 * (ref_start, query_start, len, score).  keep[i] = 1 for the first of every
 * group of equal records.  Method: sort the indices by (record, index) with
 * qsort; the first index of each run of equal records is the one kept.
 * PARITY OF THE CRITERION IS UNPINNED (the pages give only the funnel counts);
 * the function itself is pinned to that reading by brute force.
 * ------------------------------------------------------------------------- */
static const int32_t *dedup_rec;

static int dedup_cmp(const void *pa, const void *pb)
{
    uint64_t a = *(const uint64_t *)pa, b = *(const uint64_t *)pb;
    for (int f = 0; f < 4; f++) {
        int32_t x = dedup_rec[4 * a + f], y = dedup_rec[4 * b + f];
        if (x != y) return x < y ? -1 : 1;
    }
    return a < b ? -1 : (a > b ? 1 : 0);
}

int orc_dedup(const int32_t *rec, uint64_t n, uint8_t *keep)
{
    if (n == 0) return ORC_OK;
    uint64_t *order = (uint64_t *)malloc(n * sizeof(uint64_t));
    if (!order) return ORC_E_INVAL;
    for (uint64_t i = 0; i < n; i++) order[i] = i;
    dedup_rec = rec;
    qsort(order, n, sizeof(uint64_t), dedup_cmp);
    for (uint64_t k = 0; k < n; k++) {
        uint64_t i = order[k];
        int first = 1;
        if (k > 0) {
            uint64_t j = order[k - 1];
            first = memcmp(rec + 4 * i, rec + 4 * j, 4 * sizeof(int32_t)) != 0;
        }
        keep[i] = (uint8_t)first;
    }
    free(order);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * FNV-1a, 64-bit (Fowler, Noll and Vo): starting from h, for every byte b in
 * order, h = (h XOR b) * 1099511628211 mod 2^64.  The standard digest starts
 * from the offset basis 14695981039346656037.  Not part of the method: the
 * tests use it to compare the oracle's arrays with the CUDA path's arrays
 * at full size, segment by segment, without holding both in memory.
 * ------------------------------------------------------------------------- */
uint64_t orc_fnv1a64(uint64_t h, const uint8_t *p, uint64_t n)
{
    for (uint64_t i = 0; i < n; i++) {
        h ^= (uint64_t)p[i];
        h *= 1099511628211ull;
    }
    return h;
}
