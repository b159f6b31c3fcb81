/*
 * policy_oracle.c -- plain CPU oracle of the draft-source controller.  TEST
 * INFRASTRUCTURE ONLY (see lookup_oracle.c for who may load it).
 *
 * Source: Strata engine article, gtnt.cn/news/124732, section 五 ("在线成本-收益
 * 控制器"): every step the controller estimates, for the draft model's (MTP) draft
 * and for the prompt-lookup draft, the expected committed tokens divided by the
 * verify time; acceptance is estimated online with an EMA, per match-length
 * bucket (four buckets) for the lookup draft; the verify cost is the measured
 * round time; the lookup draft is used only when its expected benefit exceeds the
 * model's by more than a margin (5%), and when speculation does not pay at all the
 * controller falls back to plain decoding.
 *
 * Readings of what the section leaves open (each one a parameter or a plain
 * formula):
 *  - acceptance rate of a step = accepted / drafted tokens of the source that
 *    drafted it; EMA: acc = (1 - alpha) * acc + alpha * rate;
 *  - E[committed tokens] of n drafted tokens at per-token acceptance a is the
 *    accepted run plus the target's own token, 1 + a + a^2 + ... + a^n;
 *  - bucket of a match length m = the number of edges e[0] <= e[1] <= e[2] with
 *    m >= e[i] (0..3);
 *  - plain decoding commits one token per t_plain.
 * All arithmetic is float32, one operation at a time in the order written here
 * (the file is compiled as ISO C99, so nothing is contracted into a fused
 * multiply-add).
 *
 * Per request: acc[0..3] lookup acceptance per bucket, acc[4] the model's;
 * prev[0] last choice (0 plain, 1 model, 2 lookup), prev[1] its bucket, prev[2]
 * the tokens it drafted.  Returns the choice for this step.
 */
#include <stdint.h>

static int32_t bucket_of(int32_t m, const int32_t *edge)
{
    int32_t b = 0;
    for (int i = 0; i < 3; ++i)
        if (m >= edge[i])
            b += 1;
    return b;
}

/* 1 + a + a^2 + ... + a^n */
static float expected_committed(float a, int32_t n)
{
    float sum = 1.0f;
    float term = 1.0f;
    for (int32_t i = 1; i <= n; ++i) {
        term = term * a;
        sum = sum + term;
    }
    return sum;
}

static int32_t policy_one(int32_t m, int32_t accepted, int32_t n_lookup, int32_t n_model, float t_lookup,
                          float t_model, float t_plain, float alpha, float margin, const int32_t *edge,
                          float *acc, int32_t *prev)
{
    /* 1. the previous step's outcome updates the estimate of the source that drafted it */
    const int32_t last = prev[0], n = prev[2];
    if ((last == 1 || last == 2) && n > 0) {
        int32_t a = accepted;
        if (a < 0)
            a = 0;
        if (a > n)
            a = n;
        const float rate = (float)a / (float)n;
        const int32_t slot = last == 2 ? prev[1] : 4;
        const float kept = (1.0f - alpha) * acc[slot];
        const float added = alpha * rate;
        acc[slot] = kept + added;
    }
    /* 2. expected committed tokens per unit of verify time, per source */
    const float benefit_model = expected_committed(acc[4], n_model) / t_model;
    const int32_t b = bucket_of(m, edge);
    const int lookup_available = m > 0;
    const float benefit_lookup = lookup_available ? expected_committed(acc[b], n_lookup) / t_lookup : 0.0f;
    const float benefit_plain = 1.0f / t_plain;
    /* 3. lookup only when it beats the model by more than the margin */
    int32_t choice = 1;
    float best = benefit_model;
    if (lookup_available && benefit_lookup > (1.0f + margin) * benefit_model) {
        choice = 2;
        best = benefit_lookup;
    }
    /* 4. no speculation when it does not beat plain decoding */
    if (!(best > benefit_plain))
        choice = 0;
    prev[0] = choice;
    prev[1] = choice == 2 ? b : 0;
    prev[2] = choice == 2 ? n_lookup : (choice == 1 ? n_model : 0);
    return choice;
}

int oracle_policy(const int32_t *lookup_mlen, const int32_t *accepted, int32_t B, int32_t n_lookup,
                  int32_t n_model, float t_lookup, float t_model, float t_plain, float alpha, float margin,
                  int32_t edge1, int32_t edge2, int32_t edge3, float *acc, int32_t *prev, int32_t *out_choice)
{
    if (B < 0 || n_lookup < 0 || n_model < 0 || !(t_lookup > 0.0f) || !(t_model > 0.0f) || !(t_plain > 0.0f) ||
        !(alpha >= 0.0f && alpha <= 1.0f) || !(margin >= 0.0f) || edge1 > edge2 || edge2 > edge3)
        return -1;
    const int32_t edge[3] = {edge1, edge2, edge3};
    for (int32_t r = 0; r < B; ++r)
        out_choice[r] = policy_one(lookup_mlen[r], accepted[r], n_lookup, n_model, t_lookup, t_model, t_plain,
                                   alpha, margin, edge, acc + (int64_t)r * 5, prev + (int64_t)r * 3);
    return 0;
}
