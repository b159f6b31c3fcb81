/*
 * lookup_loop.h -- the decode-loop steps around prompt-lookup drafting, on GB300.
 *
 * Source: HyperQwen lookup-drafting article, kwkr.cn/news/564408.
 *  - "第2步" (fusion): the lookup draft is merged with the draft model's proposals,
 *    not written over them.  In the head (the positions the draft model proposes,
 *    7 in the article) a lookup match of >= 8 tokens replaces the proposals; a
 *    shorter match of >= 6 is adopted only when the draft model independently
 *    proposed the same first 2 tokens.  In the tail (8 further positions nobody
 *    proposed) a match of >= 4 tokens is enough.
 *  - "第3步" (scheduling): the long verify block (head + tail) is used only while
 *    the request is copying.  It is entered when the lookup match can fill the
 *    tail and the previous step's output was a nearly full block, on two
 *    consecutive steps; once entered it is kept for 3 more steps after the
 *    condition drops (sticky exit).
 *  - "第3步" (losslessness): greedy verification reads no proposal distribution;
 *    for sampled requests every lookup-filled position is rewritten as a point
 *    mass on the proposed token, a legal proposal for the rejection sampler.
 *
 * All arrays are device memory owned by the caller, row-major; every call
 * enqueues its work on `stream` and returns without synchronising.  Return
 * codes are those of lookup_draft.h (LOOKUP_DRAFT_OK, LOOKUP_DRAFT_EINVAL for
 * arguments that describe no valid call, LOOKUP_DRAFT_ECUDA for a failed
 * launch).  B == 0 enqueues nothing, except in lookup_append, which then
 * writes out_offsets[0] = 0.
 */
#ifndef LOOKUP_LOOP_H
#define LOOKUP_LOOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

/*
 * Fusion of the lookup draft with the draft model's proposals ("第2步").
 *
 * lookup_draft  int32 [B][K]: drafts from lookup_draft_ex (K >= H + T)
 * lookup_mlen   int32 [B]: their match lengths (0 = no match)
 * model_draft   int32 [B][H]: the draft model's proposals for the head
 * long_block    int32 [B]: nonzero = this step verifies head + tail; NULL = all 0
 * H, T          head and tail lengths (the article: 7 and 8); H >= 1, T >= 0,
 *               H + T <= 65536
 * replace_min   match length that replaces the head outright (8)
 * agree_min     shorter match length adopted when the model agrees (6)
 * agree_n       number of leading tokens that must agree (2), 0 <= agree_n <= H
 * tail_min      match length that fills the tail (4)
 * out_block     int32 [B][H + T]: the proposal block; unused tail slots -1
 * out_len       int32 [B]: proposals in the block, H or H + T
 * out_point_mass int32 [B][H + T]: 1 where the position holds a lookup token
 *               (its proposal distribution is a point mass), else 0
 *
 * Per request, with m = lookup_mlen[r], L = lookup_draft[r], M = model_draft[r]:
 *   head_lookup = m >= replace_min || (m >= agree_min && L[0..agree_n) == M[0..agree_n))
 *   block[i] = head_lookup ? L[i] : M[i] for i < H          (point mass = head_lookup)
 *   if long_block[r] and m >= tail_min: block[H + i] = L[H + i] for i < T, len = H + T
 *   else: block[H + i] = -1, len = H
 * The head and tail rules are applied independently, as the article states them.
 */
int lookup_fuse(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *long_block, int32_t B, int32_t K, int32_t H, int32_t T,
                int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                int32_t *out_block, int32_t *out_len, int32_t *out_point_mass,
                struct CUstream_st *stream);

/*
 * Long-block scheduling ("第3步"), one update per request and step.
 *
 * lookup_mlen   int32 [B]: this step's lookup match length
 * committed     int32 [B]: tokens the previous step committed (accepted + 1)
 * state         int32 [B][3] in/out: {long, streak, hold}; all zero initially
 * out_long      int32 [B]: 1 = verify the long block (head + tail) this step
 * H, T          head and tail lengths; a step's full block commits H + 1 tokens
 *               (short) or H + T + 1 (long)
 * tail_min      match length that can fill the tail (4)
 * slack         "nearly full": committed >= full - slack (1)
 * enter_steps   consecutive steps the condition must hold to enter (2)
 * sticky        steps the long block is kept after the condition drops (3)
 *
 * Per request: full = (long ? H + T : H) + 1 for the block the previous step used;
 *   cond = m >= tail_min && committed >= full - slack;
 *   streak = cond ? streak + 1 : 0;
 *   if !long: if streak >= enter_steps: long = 1, hold = sticky
 *   else if cond: hold = sticky
 *   else if hold > 0: hold -= 1            (kept: sticky exit)
 *   else: long = 0
 *   out_long = long
 */
int lookup_schedule(const int32_t *lookup_mlen, const int32_t *committed, int32_t B,
                    int32_t H, int32_t T, int32_t tail_min, int32_t slack, int32_t enter_steps,
                    int32_t sticky, int32_t *state, int32_t *out_long, struct CUstream_st *stream);

/*
 * lookup_schedule, then lookup_fuse with long_block = the new out_long, in one
 * launch (HyperQwen lookup-drafting article, sections "第3步" and "第2步"): the
 * per-request scheduling update and the block it selects, without a kernel
 * boundary between them.  Arguments, layouts and rules are those of the two
 * calls; tail_min serves both (the tail and the scheduling condition use the same
 * match length, m >= 4 in the article).  state is updated in place; out_long,
 * out_block, out_len and out_point_mass are exactly what lookup_schedule followed
 * by lookup_fuse write.  Errors: the union of the two calls' checks.
 */
int lookup_plan(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *committed, int32_t B, int32_t K, int32_t H, int32_t T,
                int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                int32_t slack, int32_t enter_steps, int32_t sticky, int32_t *state,
                int32_t *out_long, int32_t *out_block, int32_t *out_len, int32_t *out_point_mass,
                struct CUstream_st *stream);

/*
 * Draft-source controller (Strata engine article, gtnt.cn/news/124732, section
 * 五): per request and step, choose 2 = the lookup draft, 1 = the draft model's
 * draft, or 0 = plain decoding, by expected committed tokens per unit of verify
 * time.  This is the Strata engine's online cost-benefit rule.  A caller that
 * uses it with lookup_fuse passes lookup_mlen = 0 where the choice is not 2.
 *
 * lookup_mlen  int32 [B]: this step's lookup match length (0 = no match)
 * accepted     int32 [B]: tokens accepted at the previous step from the draft of
 *              the source chosen then (clamped to [0, the tokens it drafted])
 * acc          float [B][5] in/out: EMA acceptance rate of the lookup draft per
 *              match-length bucket (0..3), then of the model's draft; the caller
 *              sets the priors
 * prev         int32 [B][3] in/out: last choice, its bucket, tokens it drafted;
 *              all zero initially
 * out_choice   int32 [B]: 0, 1 or 2
 * n_lookup, n_model     tokens each source drafts per step (>= 0)
 * t_lookup, t_model     measured verify round time with each source's block (> 0)
 * t_plain               measured plain decoding step time (> 0)
 * alpha                 EMA weight of the newest rate, in [0, 1]
 * margin                lookup needs more than (1 + margin) x the model's benefit (0.05)
 * edge1 <= edge2 <= edge3   bucket of m = how many edges m reaches (6, 8, 12)
 *
 * Per request, in float32 with each operation rounded as written:
 *   if prev choice c is 1 or 2 and it drafted n > 0 tokens:
 *     rate = min(max(accepted, 0), n) / n;
 *     slot = c == 2 ? prev bucket : 4;  acc[slot] = (1 - alpha) * acc[slot] + alpha * rate
 *   E(a, n) = 1 + a + ... + a^n  (accepted run plus the target's own token)
 *   model  = E(acc[4], n_model) / t_model
 *   lookup = E(acc[bucket(m)], n_lookup) / t_lookup, only when m > 0
 *   choice = 2 if lookup > (1 + margin) * model, else 1;
 *            0 if the chosen source's value is not above 1 / t_plain
 *   prev = {choice, its bucket (lookup) or 0, the tokens it drafts}
 * Errors: LOOKUP_DRAFT_EINVAL for B < 0, negative n, non-positive times, alpha
 * outside [0, 1], a negative margin, decreasing edges, or a null pointer with B > 0.
 */
int lookup_policy(const int32_t *lookup_mlen, const int32_t *accepted, int32_t B, int32_t n_lookup,
                  int32_t n_model, float t_lookup, float t_model, float t_plain, float alpha, float margin,
                  int32_t edge1, int32_t edge2, int32_t edge3, float *acc, int32_t *prev, int32_t *out_choice,
                  struct CUstream_st *stream);

/*
 * A draft step followed by lookup_plan, in two launches instead of four
 * (HyperQwen lookup-drafting article, sections "第1步", "第3步", "第2步").  The
 * scan is lookup_draft's; the second kernel reduces each request's scan results
 * to its match (m, p), reads the draft tokens that lookup_draft_ex would write
 * with K = H + T, and applies lookup_plan's scheduling and fusion to them in the
 * same warp.  The draft itself is not written out.
 *
 * tokens, offsets, B, min_m, max_m   as for lookup_draft (device pointers)
 * model_draft, committed, H, T, replace_min, agree_min, agree_n, tail_min,
 * slack, enter_steps, sticky, state, out_long, out_block, out_len,
 * out_point_mass                     as for lookup_plan; H + T <= LOOKUP_DRAFT_MAX_K
 * out_mlen        int32 [B] or NULL: m, as lookup_draft_ex writes it
 * out_draft_len   int32 [B] or NULL: what lookup_draft's out_len would be (H + T,
 *                 0, or LOOKUP_DRAFT_LEN_FAILED); a failed request is planned as
 *                 one without a match
 * Scratch as for lookup_draft (the stream's buffer).  Errors: those of
 * lookup_draft and lookup_plan, and LOOKUP_DRAFT_EINVAL for a misaligned pointer.
 * Every output equals lookup_draft_ex (K = H + T) followed by lookup_plan.
 */
int lookup_draft_plan(const int32_t *tokens, const int64_t *offsets, int32_t B,
                      int32_t min_m, int32_t max_m,
                      const int32_t *model_draft, const int32_t *committed, int32_t H, int32_t T,
                      int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min,
                      int32_t slack, int32_t enter_steps, int32_t sticky, int32_t *state,
                      int32_t *out_long, int32_t *out_block, int32_t *out_len, int32_t *out_point_mass,
                      int32_t *out_mlen, int32_t *out_draft_len, struct CUstream_st *stream);

/*
 * Verification of a proposal block of width P (= H + T), greedy or sampled.
 *
 * block         int32 [B][P] (P <= 65536), len int32 [B] (proposals used,
 *               0 <= len <= P; a request with len outside that range gets the
 *               error row accepted = -1, ncommit = 0, commit all -1)
 * Greedy (probs == NULL): target int32 [B][P + 1] holds the target model's
 *   greedy token at each position given the block before it; accepted a is the
 *   largest a <= len with block[i] == target[i] for all i < a, and the step
 *   commits block[0..a) then target[a].
 * Sampled (probs != NULL): probs float [B][P] holds the target probability of
 *   each proposed token, qprobs float [B][P] the proposal probability of it (may
 *   be NULL = 1), point_mass int32 [B][P] (may be NULL) marks lookup positions,
 *   whose proposal probability is taken as exactly 1 (the point-mass rewrite),
 *   u float [B][P] uniform [0, 1) draws, and target int32 [B][P + 1] the tokens
 *   to commit at the first rejection (drawn by the caller from the residual
 *   distribution) or after a full acceptance (the bonus token).  Position i is
 *   accepted when u[i] * q[i] < p[i] (float32, as written); a is the first
 *   position not accepted (or len), and the step commits block[0..a) then
 *   target[a].
 * out_accepted  int32 [B]: a
 * out_commit    int32 [B][P + 1]: the committed tokens; slots past a + 1 are -1
 * out_ncommit   int32 [B]: a + 1
 */
int lookup_verify(const int32_t *block, const int32_t *len, const int32_t *target, const float *probs,
                  const float *qprobs, const int32_t *point_mass, const float *u, int32_t B, int32_t P,
                  int32_t *out_accepted, int32_t *out_commit, int32_t *out_ncommit,
                  struct CUstream_st *stream);

/*
 * The next step's histories: request r's history followed by its committed
 * tokens, as a new CSR batch.
 *
 * tokens, offsets  the current CSR batch (offsets[0] may be > 0)
 * commit           int32 [B][W], ncommit int32 [B] (0 <= ncommit <= W; a value
 *                  outside is clamped to that range)
 * out_offsets      int64 [B + 1]: new boundaries, out_offsets[0] = 0
 * out_tokens       int32 [offsets[B] - offsets[0] + sum(ncommit)]; a buffer of
 *                  offsets[B] - offsets[0] + B * W tokens always suffices, so
 *                  the caller need not read the counts back first
 * The new history of r is tokens[offsets[r] .. offsets[r+1]) then
 * commit[r][0 .. ncommit[r]).  Outputs must not overlap the inputs.
 */
int lookup_append(const int32_t *tokens, const int64_t *offsets, const int32_t *commit, const int32_t *ncommit,
                  int32_t B, int32_t W, int32_t *out_tokens, int64_t *out_offsets,
                  struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* LOOKUP_LOOP_H */
