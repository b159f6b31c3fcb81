/*
 * lookup_oracle.c -- plain CPU oracle for prompt-lookup (n-gram) drafting.
 *
 * TEST INFRASTRUCTURE ONLY. This file states, as directly as possible, what one
 * batched draft step computes, so that the CUDA library can be checked against
 * it element by element. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference legs load it; the library itself never does, and
 * nothing here is shared with the CUDA sources (no headers, helpers or tables).
 *
 * What is computed (HyperQwen lookup-drafting article, kwkr.cn/news/564408,
 * section "第1步"): before each decode step, every request scans its own token
 * history for the most recent earlier occurrence of its longest current suffix,
 * with suffix lengths from 4 to 12 tokens (here min_m..max_m), where the
 * occurrence is allowed to overlap the suffix; the tokens that follow that
 * occurrence are proposed as the draft.
 *
 * Readings taken where the page is silent (each one is listed in the design notes):
 *   - "longest first, then most recent": the search runs m = max_m .. min_m,
 *     and for each m the start p runs from the latest admissible one downwards;
 *   - "earlier occurrence": start p with p + m <= L - 1, i.e. the occurrence is
 *     not the suffix itself but may overlap it;
 *   - the draft is read from the history extended by its own draft,
 *     e[L + j] = e[p + m + j], so a match that runs into the suffix continues
 *     its own period; a matched request always gets exactly K draft tokens;
 *   - no match (or L <= min_m): length 0, position -1, every draft slot -1;
 *   - tokens are compared as raw int32 values; a match never leaves its request.
 *
 * Loop order is deliberately the plain one of the definition (length, then
 * position, then element by element) and has no blocking or early-out beyond it.
 */
#include <stdint.h>
#include <stddef.h>

/* 1 if t[a..a+n) equals t[b..b+n), element by element. */
static int same_tokens(const int32_t *t, int64_t a, int64_t b, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        if (t[a + i] != t[b + i])
            return 0;
    return 1;
}

/*
 * Longest-then-most-recent earlier occurrence of the current suffix of one
 * history t[0..L). Returns 1 and sets *m_out, *p_out when found, else 0.
 */
int oracle_find_match(const int32_t *t, int64_t L, int32_t min_m, int32_t max_m,
                      int32_t *m_out, int64_t *p_out)
{
    int64_t top = (int64_t)max_m;
    if (top > L - 1)
        top = L - 1;                       /* an earlier occurrence needs p >= 0 */
    for (int64_t m = top; m >= (int64_t)min_m; --m) {
        int64_t suffix_start = L - m;
        for (int64_t p = L - m - 1; p >= 0; --p) {   /* most recent first */
            if (same_tokens(t, p, suffix_start, m)) {
                *m_out = (int32_t)m;
                *p_out = p;
                return 1;
            }
        }
    }
    return 0;
}

/*
 * Draft of K tokens for a match (m, p) in t[0..L): draft[j] = e[L + j], where
 * e is t extended by the draft itself, e[L + j] = e[p + m + j].
 */
void oracle_fill_draft(const int32_t *t, int64_t L, int32_t m, int64_t p,
                       int32_t K, int32_t *draft)
{
    for (int32_t j = 0; j < K; ++j) {
        int64_t src = p + m + j;           /* index into e */
        draft[j] = (src < L) ? t[src] : draft[src - L];
    }
}

/*
 * Batched step over requests [r_begin, r_end) of a CSR batch:
 * request r's history is tokens[offsets[r] .. offsets[r+1]).
 * Outputs are indexed by the global request number r (out_draft row-major
 * [B][K]). out_m (may be NULL) receives the match length, 0 if none.
 * Returns 0, or -1 for arguments that do not describe a valid step.
 */
int oracle_lookup_draft(const int32_t *tokens, const int64_t *offsets,
                        int32_t r_begin, int32_t r_end,
                        int32_t min_m, int32_t max_m, int32_t K,
                        int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                        int32_t *out_m)
{
    if (min_m < 1 || max_m < min_m || K < 0 || r_begin < 0 || r_end < r_begin)
        return -1;
    for (int32_t r = r_begin; r < r_end; ++r) {
        const int32_t *t = tokens + offsets[r];
        int64_t L = offsets[r + 1] - offsets[r];
        int32_t *draft = out_draft + (int64_t)r * K;
        int32_t m = 0;
        int64_t p = -1;
        if (L < 0)
            return -1;
        if (oracle_find_match(t, L, min_m, max_m, &m, &p)) {
            oracle_fill_draft(t, L, m, p, K, draft);
            out_len[r] = K;
            out_pos[r] = (int32_t)p;
        } else {
            for (int32_t j = 0; j < K; ++j)
                draft[j] = -1;
            out_len[r] = 0;
            out_pos[r] = -1;
            m = 0;
        }
        if (out_m)
            out_m[r] = m;
    }
    return 0;
}
