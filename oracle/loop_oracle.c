/*
 * loop_oracle.c -- plain CPU oracle for the decode-loop steps around lookup
 * drafting.  TEST INFRASTRUCTURE ONLY (see lookup_oracle.c for who may load it).
 *
 * Source: HyperQwen lookup-drafting article, kwkr.cn/news/564408:
 *  - "第2步": in the head (positions the draft model proposed) a lookup match of
 *    >= replace_min tokens replaces the proposals; a match of >= agree_min is
 *    adopted only if the model's first agree_n tokens equal the lookup's; in the
 *    tail (positions nobody proposed) a match of >= tail_min fills them.
 *  - "第3步": the long block is entered when the match can fill the tail and the
 *    previous step's output was a nearly full block, on enter_steps consecutive
 *    steps, and is kept for `sticky` steps after that condition drops.  Greedy
 *    verification accepts the longest agreeing prefix; for sampled requests a
 *    lookup-filled position is a point mass on its token.
 * Each function is the rule written out for one request at a time, in the order
 * the article gives it.
 */
#include <stdint.h>
#include <stddef.h>

/* "第2步", one request.  Returns the number of proposals in the block. */
static int fuse_one(const int32_t *ld, int32_t m, const int32_t *md, int is_long, int32_t H, int32_t T,
                    int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                    int32_t *block, int32_t *pm)
{
    int agree = 1;
    for (int32_t i = 0; i < agree_n; ++i)
        if (ld[i] != md[i])
            agree = 0;
    int head_lookup = 0;
    if (m >= replace_min)
        head_lookup = 1;                         /* a long match replaces outright */
    else if (m >= agree_min && agree)
        head_lookup = 1;                         /* a shorter one needs the model to agree */
    for (int32_t i = 0; i < H; ++i) {
        block[i] = head_lookup ? ld[i] : md[i];
        pm[i] = head_lookup;
    }
    int tail = is_long && m >= tail_min;
    for (int32_t i = 0; i < T; ++i) {
        block[H + i] = tail ? ld[H + i] : -1;
        pm[H + i] = tail;
    }
    return tail ? H + T : H;
}

int oracle_fuse(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *long_block, int32_t B, int32_t K, int32_t H, int32_t T,
                int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                int32_t *out_block, int32_t *out_len, int32_t *out_pm)
{
    if (B < 0 || H < 1 || T < 0 || K < H + T || agree_n < 0 || agree_n > H)
        return -1;
    for (int32_t r = 0; r < B; ++r) {
        int is_long = long_block ? long_block[r] != 0 : 0;
        out_len[r] = fuse_one(lookup_draft + (int64_t)r * K, lookup_mlen[r], model_draft + (int64_t)r * H,
                              is_long, H, T, replace_min, agree_min, agree_n, tail_min,
                              out_block + (int64_t)r * (H + T), out_pm + (int64_t)r * (H + T));
    }
    return 0;
}

/* "第3步" scheduling, one request and one step.  st = {long, streak, hold}. */
static int schedule_one(int32_t m, int32_t committed, int32_t *st, int32_t H, int32_t T, int32_t tail_min,
                        int32_t slack, int32_t enter_steps, int32_t sticky)
{
    int32_t full = (st[0] ? H + T : H) + 1;      /* the block the previous step used */
    int cond = m >= tail_min && committed >= full - slack;
    st[1] = cond ? st[1] + 1 : 0;
    if (!st[0]) {
        if (st[1] >= enter_steps) {
            st[0] = 1;
            st[2] = sticky;
        }
    } else if (cond) {
        st[2] = sticky;
    } else if (st[2] > 0) {
        st[2] -= 1;                              /* sticky exit: keep the long block */
    } else {
        st[0] = 0;
    }
    return st[0];
}

int oracle_schedule(const int32_t *lookup_mlen, const int32_t *committed, int32_t B, int32_t H, int32_t T,
                    int32_t tail_min, int32_t slack, int32_t enter_steps, int32_t sticky,
                    int32_t *state, int32_t *out_long)
{
    if (B < 0 || H < 1 || T < 0 || enter_steps < 1 || sticky < 0 || slack < 0)
        return -1;
    for (int32_t r = 0; r < B; ++r)
        out_long[r] = schedule_one(lookup_mlen[r], committed[r], state + 3 * (int64_t)r, H, T, tail_min, slack,
                                   enter_steps, sticky);
    return 0;
}

/* Verification of one request's block; returns the accepted length. */
static int32_t verify_one(const int32_t *block, int32_t len, const int32_t *target, const float *p,
                          const float *q, const int32_t *pm, const float *u, int32_t P, int32_t *commit)
{
    int32_t a = 0;
    while (a < len) {
        int ok;
        if (!p) {
            ok = block[a] == target[a];          /* greedy: the target's own token */
        } else {
            float qa = q ? q[a] : 1.0f;
            if (pm && pm[a])
                qa = 1.0f;                       /* point mass on the lookup token */
            ok = u[a] * qa < p[a];               /* accept with probability min(1, p/q) */
        }
        if (!ok)
            break;
        ++a;
    }
    for (int32_t i = 0; i <= P; ++i)
        commit[i] = i < a ? block[i] : (i == a ? target[a] : -1);
    return a;
}

int oracle_verify(const int32_t *block, const int32_t *len, const int32_t *target, const float *probs,
                  const float *qprobs, const int32_t *point_mass, const float *u, int32_t B, int32_t P,
                  int32_t *out_accepted, int32_t *out_commit, int32_t *out_ncommit)
{
    if (B < 0 || P < 0 || (probs && !u))
        return -1;
    for (int32_t r = 0; r < B; ++r) {
        if (len[r] < 0 || len[r] > P)
            return -1;
        int64_t o = (int64_t)r * P;
        int32_t a = verify_one(block + o, len[r], target + (int64_t)r * (P + 1), probs ? probs + o : NULL,
                               qprobs ? qprobs + o : NULL, point_mass ? point_mass + o : NULL,
                               u ? u + o : NULL, P, out_commit + (int64_t)r * (P + 1));
        out_accepted[r] = a;
        out_ncommit[r] = a + 1;
    }
    return 0;
}

/* The next batch: each history followed by its committed tokens. */
int oracle_append(const int32_t *tokens, const int64_t *offsets, const int32_t *commit, const int32_t *ncommit,
                  int32_t B, int32_t W, int32_t *out_tokens, int64_t *out_offsets)
{
    if (B < 0 || W < 0)
        return -1;
    int64_t pos = 0;
    out_offsets[0] = 0;
    for (int32_t r = 0; r < B; ++r) {
        if (ncommit[r] < 0 || ncommit[r] > W)
            return -1;
        for (int64_t i = offsets[r]; i < offsets[r + 1]; ++i)
            out_tokens[pos++] = tokens[i];
        for (int32_t j = 0; j < ncommit[r]; ++j)
            out_tokens[pos++] = commit[(int64_t)r * W + j];
        out_offsets[r + 1] = pos;
    }
    return 0;
}
