/*
 * ctx_oracle.c -- plain CPU oracle of context-cache drafting.  TEST
 * INFRASTRUCTURE ONLY (see lookup_oracle.c for who may load it).
 *
 * Source: llama.cpp prompt-lookup article, ai-blog.deepmagic.app,
 * "從 165 微秒到 1.18 微秒", section "Prompt lookup decoding 到底是什麼": the
 * context cache keeps the statistics of the n-grams of sizes 1 to 4 of the
 * current token stream, and a draft token is taken from an n-gram only when it
 * passes fixed acceptance thresholds -- for the 4-gram, at least one earlier
 * occurrence, and the most frequent next token following it in at least half of
 * its occurrences.
 *
 * Written out per request, one draft token at a time:
 *   context = the history followed by the tokens drafted so far;
 *   for n = n_max down to n_min (longest first):
 *     g = the last n tokens of the context;
 *     the occurrences of g in the history that have a next token (start i with
 *       i + n <= L - 1), total = their number, and for each next token x its
 *       count c(x);
 *     x* = the x with the largest count (equal counts: the smallest token id);
 *     accepted when total >= min_count[n] and c(x*) * den[n] >= num[n] * total;
 *   the first accepted n gives the next draft token x*; when none does, the
 *   draft ends.  Statistics come from the history only: drafted tokens extend
 *   the context that is looked up, never the counts.
 * Everything is integer arithmetic; the share test is exact.
 */
#include <stdint.h>
#include <stdlib.h>

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* One request.  succ: scratch of L ints.  Returns the draft length. */
static int32_t ctx_draft_one(const int32_t *t, int64_t L, int32_t n_min, int32_t n_max, int32_t K,
                             const int32_t *min_count, const int32_t *num, const int32_t *den,
                             int32_t *draft, int32_t *succ)
{
    int32_t j = 0;
    while (j < K) {
        int accepted = 0;
        for (int32_t n = n_max; n >= n_min && !accepted; --n) {
            if (L + j < n)
                continue;                                    /* the context is shorter than n */
            int32_t g[4];
            for (int32_t k = 0; k < n; ++k) {                 /* the last n context tokens, oldest first */
                int64_t c = L + j - n + k;
                g[k] = c < L ? t[c] : draft[c - L];
            }
            int64_t total = 0;
            for (int64_t i = 0; i + n <= L - 1; ++i) {
                int same = 1;
                for (int32_t k = 0; k < n; ++k)
                    if (t[i + k] != g[k])
                        same = 0;
                if (same)
                    succ[total++] = t[i + n];
            }
            if (total == 0 || total < min_count[n - 1])
                continue;
            qsort(succ, (size_t)total, sizeof(int32_t), cmp_i32);
            int32_t best = succ[0];
            int64_t best_c = 0;
            for (int64_t a = 0; a < total;) {                /* runs of equal tokens, ascending */
                int64_t b = a;
                while (b < total && succ[b] == succ[a])
                    ++b;
                if (b - a > best_c) {                         /* strictly more: ties keep the smaller id */
                    best_c = b - a;
                    best = succ[a];
                }
                a = b;
            }
            if (best_c * (int64_t)den[n - 1] >= (int64_t)num[n - 1] * total) {
                draft[j] = best;
                accepted = 1;
            }
        }
        if (!accepted)
            break;
        ++j;
    }
    for (int32_t k = j; k < K; ++k)
        draft[k] = -1;
    return j;
}

/*
 * Requests [r_begin, r_end) of a CSR batch.  min_count, num, den: 4 entries each,
 * index n - 1.  Returns 0, or -1 for invalid arguments or no memory.
 */
int oracle_ctx_draft(const int32_t *tokens, const int64_t *offsets, int32_t r_begin, int32_t r_end,
                     int32_t n_min, int32_t n_max, int32_t K, const int32_t *min_count, const int32_t *num,
                     const int32_t *den, int32_t *out_draft, int32_t *out_len)
{
    if (n_min < 1 || n_min > n_max || n_max > 4 || K < 0)
        return -1;
    for (int32_t n = n_min; n <= n_max; ++n)
        if (num[n - 1] < 0 || den[n - 1] < 1)
            return -1;
    for (int32_t r = r_begin; r < r_end; ++r) {
        const int64_t L = offsets[r + 1] - offsets[r];
        int32_t *succ = (int32_t *)malloc(sizeof(int32_t) * (size_t)(L > 0 ? L : 1));
        if (!succ)
            return -1;
        out_len[r] = ctx_draft_one(tokens + offsets[r], L, n_min, n_max, K, min_count, num, den,
                                   out_draft + (int64_t)r * K, succ);
        free(succ);
    }
    return 0;
}
