/*
 * lookup_index.h -- a device-resident, incrementally updated n-gram index for
 * prompt-lookup drafting on GB300.
 *
 * Source: Strata engine article, gtnt.cn/news/124732, section 四 (the engine
 * keeps an n-gram -> position index of the prompt and of the confirmed output in
 * a fixed-size open-addressing hash table, a few tens of bytes per history token,
 * with O(1) appends, and drafts from the longest match it finds).  The result
 * returned here is not an approximation: lookup_index_draft returns exactly what
 * lookup_draft (include/lookup_draft.h; HyperQwen lookup-drafting article,
 * section "第1步") returns for the same histories -- the longest current suffix of
 * min_m..max_m tokens with an earlier occurrence, its most recent occurrence, and
 * the K tokens after it read from the self-extended history.
 *
 * What the index holds.  For every request r, every length n in [min_m, max_m]
 * and every history position q with n - 1 <= q <= L - 2 (every position but the
 * last), the n-gram ending at q is a key (r, n, t[q-n+1 .. q]).  Each key's slot
 * holds the largest such q.  The current suffix's own n-gram ends at L - 1, the
 * unindexed last position, so its slot gives the most recent earlier
 * occurrence: the longest n with a slot is the match length, q - n + 1 its
 * position.  Keys are 64-bit hashes of which a slot keeps a 32-bit fingerprint;
 * every candidate is checked against the history, and a request whose candidate
 * does not check out (two keys sharing a slot, or a table that overflowed) is
 * answered by a brute-force warp scan of its history, so the result is exact
 * whatever the hash does.
 *
 * Layout (device memory, caller-owned):
 *   tokens   int32 [N]: the slabs; request r's history is tokens[base[r] ..
 *            base[r] + len[r]) and may grow in place up to base[r] + cap[r].
 *            Positions are int32 indexes into tokens, so N < 2^31.
 *   base     int64 [B], len int32 [B], cap int32 [B] (len <= cap; slabs must not
 *            overlap)
 *   index    lookup_index_bytes(slots) bytes, 16-byte aligned (128-byte aligned
 *            for full speed): a 128-byte header then `slots` 8-byte slots
 *            (slots a power of two >= 16) in buckets of 4 slots, one 32-byte
 *            sector each; a key's bucket is read whole in one load round.
 *   The index remembers min_m, max_m, slots and hash_bits from the last build;
 *   a call with other values fails its requests (lookup_index_draft reports
 *   LOOKUP_DRAFT_LEN_FAILED, lookup_index_append status 2) instead of reading
 *   a table it did not build.
 *
 * Return codes are those of lookup_draft.h.  Every call enqueues its work on
 * `stream` and returns without synchronising; B == 0 enqueues nothing.
 */
#ifndef LOOKUP_INDEX_H
#define LOOKUP_INDEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

/* Slots for an index over `capacity_tokens` history tokens: the smallest power
 * of two >= 2 * (max_m - min_m + 1) * capacity_tokens (load factor <= 1/2).
 * Returns 0 for invalid arguments. */
int64_t lookup_index_slots_for(int64_t capacity_tokens, int32_t min_m, int32_t max_m);

/* Bytes of an index with `slots` slots: 128 + 8 * slots (0 if slots is not a
 * power of two >= 16). */
size_t lookup_index_bytes(int64_t slots);

/*
 * Build the index of the current histories: clears the table, then inserts every
 * n-gram (n in [min_m, max_m]) that ends before the last position of its
 * history.  The insertions run in parallel, in any order (a slot keeps the
 * largest position).
 * hash_bits in [1, 64] masks the 64-bit keys (64 in normal use; fewer bits make
 * keys share slots, which the exact fallback absorbs -- a test hook).
 * Scratch for the build comes from the library's stream-ordered pool.
 * 1 <= min_m <= max_m <= LOOKUP_DRAFT_MAX_M; returns LOOKUP_DRAFT_EINVAL otherwise.
 */
int lookup_index_build(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B,
                       int32_t min_m, int32_t max_m, void *index, int64_t slots, int32_t hash_bits,
                       struct CUstream_st *stream);

/*
 * Append request r's committed tokens commit[r][0 .. n) (n = ncommit[r] clamped
 * to [0, W]) at tokens[base[r] + len[r]], insert the n-grams that end at the old
 * last position and at every new position but the new last, and add n to
 * len[r].  out_status[r] (may be NULL): 0 = appended, 1 = the slab is full
 * (len + n > cap; nothing appended), 2 = the index was built with other
 * parameters (nothing appended).  O(n * (max_m - min_m + 1)) per request.
 */
int lookup_index_append(int32_t *tokens, const int64_t *base, int32_t *len, const int32_t *cap,
                        const int32_t *commit, const int32_t *ncommit, int32_t B, int32_t W,
                        int32_t min_m, int32_t max_m, void *index, int64_t slots, int32_t hash_bits,
                        int32_t *out_status, struct CUstream_st *stream);

/*
 * The draft step from the index: out_draft [B][K], out_len, out_pos, out_mlen
 * (may be NULL) exactly as lookup_draft_ex gives them for the histories
 * tokens[base[r] .. base[r] + len[r]).  out_fallback [B] (may be NULL): 1 where
 * the request was answered by the brute-force scan, else 0.  0 <= K <= 64.
 */
int lookup_index_draft(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B,
                       int32_t min_m, int32_t max_m, int32_t K, const void *index, int64_t slots,
                       int32_t hash_bits, int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                       int32_t *out_mlen, int32_t *out_fallback, struct CUstream_st *stream);

/*
 * lookup_index_draft followed by lookup_plan (include/lookup_loop.h), in one
 * launch: each request's warp answers the index query (K = H + T), keeps the
 * draft tokens in registers and applies the scheduling and fusion rules of
 * HyperQwen lookup-drafting article sections "第3步" and "第2步" to them.  The
 * draft itself is not written.
 *
 * tokens, base, len, B, min_m, max_m, index, slots, hash_bits   as for lookup_index_draft
 * model_draft, committed, H, T, replace_min, agree_min, agree_n, tail_min,
 * slack, enter_steps, sticky, state, out_long, out_block, out_len,
 * out_point_mass     as for lookup_plan; H + T <= LOOKUP_DRAFT_MAX_K
 * out_mlen, out_draft_len, out_fallback   int32 [B] or NULL: m, the length
 *                    lookup_index_draft would report, and its fallback flag
 * Every output equals lookup_index_draft (K = H + T) followed by lookup_plan.
 * Errors: those of the two calls.
 */
int lookup_index_draft_plan(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B,
                            int32_t min_m, int32_t max_m, const void *index, int64_t slots, int32_t hash_bits,
                            const int32_t *model_draft, const int32_t *committed, int32_t H, int32_t T,
                            int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                            int32_t slack, int32_t enter_steps, int32_t sticky, int32_t *state,
                            int32_t *out_long, int32_t *out_block, int32_t *out_len, int32_t *out_point_mass,
                            int32_t *out_mlen, int32_t *out_draft_len, int32_t *out_fallback,
                            struct CUstream_st *stream);

/*
 * lookup_verify (include/lookup_loop.h) followed by lookup_index_append with its
 * commit rows (W = P + 1): the verification of HyperQwen lookup-drafting article
 * section "第3步", then the in-place append of the committed tokens to the
 * histories and the index.  When every request gets a CTA in one wave (as for
 * lookup_index_append), one launch: each request's CTA verifies its block in one
 * warp and appends what it committed.  Otherwise the two calls, in order.
 *
 * block, block_len, target, probs, qprobs, point_mass, u, B, P, out_accepted,
 * out_commit, out_ncommit    as for lookup_verify (out_commit and out_ncommit
 *                            are written, then read by the append)
 * tokens, base, len, cap, min_m, max_m, index, slots, hash_bits, out_status
 *                            as for lookup_index_append
 * Every output equals lookup_verify followed by lookup_index_append(..., commit =
 * out_commit, ncommit = out_ncommit, W = P + 1, ...).
 * Errors: those of the two calls.
 */
int lookup_index_verify_append(const int32_t *block, const int32_t *block_len, const int32_t *target,
                               const float *probs, const float *qprobs, const int32_t *point_mass,
                               const float *u, int32_t B, int32_t P, int32_t *tokens, const int64_t *base,
                               int32_t *len, const int32_t *cap, int32_t min_m, int32_t max_m, void *index,
                               int64_t slots, int32_t hash_bits, int32_t *out_accepted, int32_t *out_commit,
                               int32_t *out_ncommit, int32_t *out_status, struct CUstream_st *stream);

/*
 * lookup_index_verify_append followed by lookup_index_draft (K tokens) on the
 * grown histories: the whole step after the target model in prompt-lookup
 * decoding without a draft model, where the next block is the lookup draft.
 * When every request gets a CTA in one wave, one launch: each request's CTA
 * verifies its block, appends what it committed, and drafts from its grown
 * history and the index.  The CTAs of other requests insert only their own
 * requests' keys, which never move or empty a slot, and an overflow anywhere
 * sends the query to the exact scan, so the draft is exact whatever the order.
 * Otherwise the two calls, in order.
 *
 * block ... out_status       as for lookup_index_verify_append
 * K, out_draft, out_draft_len, out_pos, out_mlen, out_fallback
 *                            as for lookup_index_draft (K, out_draft, out_len,
 *                            out_pos, out_mlen, out_fallback)
 * Every output equals lookup_index_verify_append followed by lookup_index_draft.
 * With K == P, out_draft may be the block array and out_draft_len the block
 * lengths (the next step's block, written in place): each request's block is
 * read before its draft is written.
 * Errors: those of the two calls.
 */
int lookup_index_verify_append_draft(const int32_t *block, const int32_t *block_len, const int32_t *target,
                                     const float *probs, const float *qprobs, const int32_t *point_mass,
                                     const float *u, int32_t B, int32_t P, int32_t *tokens, const int64_t *base,
                                     int32_t *len, const int32_t *cap, int32_t min_m, int32_t max_m, void *index,
                                     int64_t slots, int32_t hash_bits, int32_t K, int32_t *out_accepted,
                                     int32_t *out_commit, int32_t *out_ncommit, int32_t *out_status,
                                     int32_t *out_draft, int32_t *out_draft_len, int32_t *out_pos, int32_t *out_mlen,
                                     int32_t *out_fallback, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* LOOKUP_INDEX_H */
