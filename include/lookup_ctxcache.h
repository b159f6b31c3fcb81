/*
 * lookup_ctxcache.h -- context-cache drafting on GB300: the most frequent next
 * token of the longest recent n-gram, from device-resident n-gram statistics.
 *
 * Source: llama.cpp prompt-lookup article, ai-blog.deepmagic.app,
 * "從 165 微秒到 1.18 微秒", section "Prompt lookup decoding 到底是什麼": the
 * context cache tracks the n-grams of sizes 1 to 4 of the current token stream,
 * and a draft token is taken from an n-gram only when it passes fixed
 * thresholds (for the 4-gram: seen at least once, and its most frequent next
 * token following it at least half of the time).
 *
 * The result, per request, one draft token at a time:
 *   context = the history followed by the tokens drafted so far;
 *   for n = n_max down to n_min: g = the last n context tokens; over the
 *   occurrences of g in the history that have a next token, total = their
 *   number, c(x) = how many are followed by x, x* = the x with the largest c
 *   (equal counts: the smallest token id); g is accepted when
 *   total >= min_count[n-1] and c(x*) * share_den[n-1] >= share_num[n-1] * total;
 *   the first accepted n gives the next draft token x*; when none passes the
 *   draft ends.  Counts come from the history only.
 * out_len[r] is the number of tokens drafted (0..K); out_draft[r][len..K) = -1.
 *
 * Tokens compare as raw int32 values, as in lookup_draft.h: negative and
 * out-of-vocabulary values are counted and matched like any other.
 *
 * The cache holds, for every request r, n in [n_min, n_max] and history n-gram
 * g: the number of its occurrences with a next token, and the best (count, next
 * token) pair; and for every (g, next token) its count.  Keys are the exact
 * (r, n, g, x) packed into 128 bits -- no hashing of the identity, so no two
 * n-grams ever share counts.  A token enters a key as a 21-bit code: a value in
 * [0, 2^20) (the pages' Qwen vocabulary is 151,936) is its own code; any other
 * int32 value is given a code by a dictionary kept in the same table (2^20
 * codes; a value takes the first free code of a probe sequence of its own, so
 * up to about a million distinct such values per cache, its build and appends
 * together).  Limits: B <= 65,536, 1 <= n_min <= n_max <= 4.  A cache in which
 * some value found no code, or some key found no slot, fails every request of
 * its drafts (out_len LOOKUP_DRAFT_LEN_FAILED) instead of drafting from
 * incomplete counts.
 *
 * Layout (device memory, caller-owned): the slabs of include/lookup_index.h --
 * tokens int32 [N], base int64 [B], len int32 [B], cap int32 [B]; request r's
 * history is tokens[base[r] .. base[r] + len[r]) and grows in place.
 *   cache    lookup_ctx_bytes(slots) bytes, 16-byte aligned: a 128-byte header
 *            then `slots` 32-byte slots {key (16 bytes), two 64-bit values}.
 *   The cache remembers n_min, n_max and slots from its build; calls with other
 *   values fail their requests (out_len LOOKUP_DRAFT_LEN_FAILED, append
 *   status 2).  A table that overflowed is reported the same way.
 * Return codes are those of lookup_draft.h; every call is stream-ordered and
 * B == 0 enqueues nothing.
 */
#ifndef LOOKUP_CTXCACHE_H
#define LOOKUP_CTXCACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

/* Slots for `capacity_tokens` history tokens: the smallest power of two >=
 * 4 * (n_max - n_min + 1) * capacity_tokens (two keys per position and length,
 * load factor <= 1/2; dictionary keys, at most one per distinct token value
 * outside [0, 2^20), keep it <= 3/4).  0 for invalid arguments. */
int64_t lookup_ctx_slots_for(int64_t capacity_tokens, int32_t n_min, int32_t n_max);

/* 128 + 32 * slots (0 unless slots is a power of two >= 16). */
size_t lookup_ctx_bytes(int64_t slots);

/* Build the statistics of the current histories (clears the table first). */
int lookup_ctx_build(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t n_min,
                     int32_t n_max, void *cache, int64_t slots, struct CUstream_st *stream);

/* Append commit[r][0 .. n) (n = ncommit[r] clamped to [0, W]) in place, count
 * the new (n-gram, next token) pairs, add n to len[r].  out_status[r] (may be
 * NULL): 0 appended, 1 slab full (nothing appended), 2 cache built with other
 * parameters (nothing appended). */
int lookup_ctx_append(int32_t *tokens, const int64_t *base, int32_t *len, const int32_t *cap,
                      const int32_t *commit, const int32_t *ncommit, int32_t B, int32_t W, int32_t n_min,
                      int32_t n_max, void *cache, int64_t slots, int32_t *out_status, struct CUstream_st *stream);

/* Draft up to K (0..64) tokens per request.  min_count, share_num, share_den:
 * HOST arrays of 4 entries (index n - 1; share_num >= 0, share_den >= 1). */
int lookup_ctx_draft(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t n_min,
                     int32_t n_max, int32_t K, const int32_t *min_count, const int32_t *share_num,
                     const int32_t *share_den, const void *cache, int64_t slots, int32_t *out_draft,
                     int32_t *out_len, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* LOOKUP_CTXCACHE_H */
