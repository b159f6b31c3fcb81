/*
 * lookup_draft.h -- C ABI of the GB300 prompt-lookup (n-gram) drafting library.
 *
 * The operation (HyperQwen lookup-drafting article, kwkr.cn/news/564408, section
 * "第1步"): before a decode step, every request of a batch scans its own token
 * history for the most recent earlier occurrence of its longest current suffix,
 * trying suffix lengths from max_m down to min_m (the article uses 12 .. 4); the
 * occurrence may overlap the suffix, so periodic text (list items, indentation,
 * code fences) matches its own period.  The K tokens that follow the occurrence
 * are the draft.  The draft is read from the history extended by its own draft,
 * e[L + j] = e[p + m + j], so a match that runs into the suffix continues the
 * period.
 *
 * Precisely, for request r with history t[0..L):
 *   (m, p) = the largest m in [min_m, min(max_m, L-1)], then the largest p, such
 *            that p + m <= L - 1 and t[p .. p+m) == t[L-m .. L);
 *   found:    out_len[r] = K, out_pos[r] = p, out_mlen[r] = m,
 *             out_draft[r*K + j] = t[p + m + (j mod (L - p - m))] for j < K;
 *   none:     out_len[r] = 0, out_pos[r] = -1, out_mlen[r] = 0,
 *             out_draft[r*K + j] = -1.
 * Tokens compare as raw int32 values; a match never leaves its own request.
 *
 * Batch layout (CSR): request r's history is tokens[offsets[r] .. offsets[r+1]).
 * offsets has B+1 non-decreasing int64 entries, offsets[0] >= 0 (it need not be
 * 0), and every history is shorter than 2^31 tokens.  These preconditions are
 * not checked on the device pointers (the host never reads them); violating
 * them gives undefined results.  tokens needs only int32 alignment.
 *
 * Execution: every call enqueues its work on `stream` (NULL = the legacy
 * default stream) and returns without synchronising, except lookup_draft_host.
 * Device pointers must be valid on the current device.  The library keeps no
 * pointer to caller memory after a call returns.  Calls are thread-safe.  Calls
 * from several threads on one stream that use the stream's scratch (lookup_draft,
 * lookup_draft_ex, lookup_draft_plan, lookup_draft_host) hold the stream's lock
 * while they enqueue their kernels (lookup_draft_host: until it has synchronised),
 * so their kernels never interleave; they run in the order the threads take it.
 *
 * Return codes: LOOKUP_DRAFT_OK, or a negative LOOKUP_DRAFT_E* code.  A call that
 * returns an error may have enqueued nothing or part of its work; its outputs
 * are then unspecified.  Work that fails on the device after a successful return
 * is reported per request: out_len[r] = LOOKUP_DRAFT_LEN_FAILED.
 */
#ifndef LOOKUP_DRAFT_H
#define LOOKUP_DRAFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                     /* same type as cudaStream_t */

#define LOOKUP_DRAFT_MAX_M 32           /* largest accepted max_m */
#define LOOKUP_DRAFT_MAX_K 64           /* largest accepted K */

#define LOOKUP_DRAFT_OK 0
#define LOOKUP_DRAFT_EINVAL (-1)        /* arguments do not describe a valid step */
#define LOOKUP_DRAFT_ECUDA (-2)         /* a CUDA call failed; see lookup_draft_last_cuda_error */
#define LOOKUP_DRAFT_ERANGE (-3)        /* batch too large for lookup_draft_noalloc's fixed scratch */

#define LOOKUP_DRAFT_LEN_FAILED (-1)    /* out_len value: the scan for this request did not
                                           complete (a bounded wait on the device ran out) */

/*
 * One batched draft step (HyperQwen lookup-drafting article, section "第1步").
 *
 * tokens     device, int32 [offsets[B]]   concatenated histories (read only)
 * offsets    device, int64 [B + 1]        CSR boundaries (read only)
 * B          number of requests, >= 0; B == 0 enqueues nothing and returns OK
 * min_m      shortest suffix tried, 1 <= min_m <= max_m
 * max_m      longest suffix tried, max_m <= LOOKUP_DRAFT_MAX_M
 * K          draft tokens per request, 0 <= K <= LOOKUP_DRAFT_MAX_K
 * out_draft  device, int32 [B * K], row-major (may be NULL when K == 0)
 * out_len    device, int32 [B]: K on a match, 0 without, LOOKUP_DRAFT_LEN_FAILED
 * out_pos    device, int32 [B]: start p of the occurrence in the request, or -1
 * stream     CUDA stream all work is enqueued on
 *
 * Scratch: B + 16 * (number of scan CTAs, one per SM) 64-bit words, kept per
 * stream.  The first call on a stream, outside stream capture, allocates them
 * (cudaMalloc, rounded up to 64 KiB) and later calls on that stream reuse them,
 * so a run of calls has no allocation between its kernels.  A call with a larger
 * batch makes a buffer twice as large or more.  The library frees none of these
 * buffers before the process exits: a CUDA graph captured earlier may still use
 * an old one.  A call inside stream capture on a stream whose buffer is missing
 * or too small takes its scratch from a library-owned, stream-ordered memory
 * pool instead (memory nodes in the graph).
 * A graph captured from calls on a stream uses that stream's buffer, as it uses
 * its fixed output buffers: replays of it must not overlap in time with other
 * calls on that stream.  Buffers are keyed by the stream handle (the per-thread
 * default stream, cudaStreamPerThread, by the calling thread): synchronise a
 * stream before destroying it if calls on it may still run, since a stream
 * created later may receive the same handle, and with it the same buffer.
 * Set-up: the first call on a device sets up per-device state.  Make it outside
 * stream capture.  The first call on each stream (and one with a larger batch)
 * allocates: while another thread captures a stream in global capture mode, an
 * allocation may invalidate that capture, so make those calls first.
 * Errors: LOOKUP_DRAFT_EINVAL for null pointers (with B > 0), bad m range, K out of
 * range, or misaligned tokens/offsets; LOOKUP_DRAFT_ECUDA when an allocation or
 * launch fails.
 */
int lookup_draft(const int32_t *tokens, const int64_t *offsets, int32_t B,
                 int32_t min_m, int32_t max_m, int32_t K,
                 int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                 struct CUstream_st *stream);

/*
 * lookup_draft plus the match length: out_mlen (device, int32 [B], may be NULL)
 * receives m, or 0 when there is no match.  The article's fusion rules (section
 * "第2步") key on this length.
 */
int lookup_draft_ex(const int32_t *tokens, const int64_t *offsets, int32_t B,
                    int32_t min_m, int32_t max_m, int32_t K,
                    int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                    int32_t *out_mlen, struct CUstream_st *stream);

/*
 * Bytes of caller-provided scratch that lookup_draft_scan / lookup_draft_fill need
 * for a batch of B requests on the current device (a function of B and the
 * device's SM count).  Returns 0 when B < 0 or the device cannot be queried.
 */
size_t lookup_draft_workspace_bytes(int32_t B);

/*
 * The two stages of lookup_draft with caller-owned scratch, for callers that
 * manage their own memory or want to time the stages.  Run lookup_draft_scan,
 * then lookup_draft_fill with the same tokens, offsets, B, min_m and workspace,
 * on the same device and in stream order.
 *
 * lookup_draft_scan: the split-history scan.  Every history token is read once;
 *   each candidate end position tests the last suffix token first and extends
 *   survivors backwards; the best (m, p) per request and per scan warp range (16
 *   contiguous ranges per scan CTA) is left in
 *   `workspace` (device, >= lookup_draft_workspace_bytes(B) bytes, 8-byte aligned;
 *   needs no initialisation).
 * lookup_draft_fill: reduces those partial results and writes out_draft, out_len,
 *   out_pos and (if not NULL) out_mlen exactly as lookup_draft_ex does.
 * Errors as for lookup_draft, plus LOOKUP_DRAFT_EINVAL when the workspace is NULL,
 * misaligned or too small.
 */
int lookup_draft_scan(const int32_t *tokens, const int64_t *offsets, int32_t B,
                      int32_t min_m, int32_t max_m,
                      void *workspace, size_t workspace_bytes,
                      struct CUstream_st *stream);

int lookup_draft_fill(const int32_t *tokens, const int64_t *offsets, int32_t B,
                      int32_t min_m, int32_t max_m, int32_t K,
                      const void *workspace, size_t workspace_bytes,
                      int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                      int32_t *out_mlen, struct CUstream_st *stream);

/*
 * lookup_draft on HOST buffers: copies tokens[offsets[0] .. offsets[B]) and the
 * offsets to the current device, into the stream's scratch (the buffer
 * lookup_draft keeps per stream, grown to hold the copy, the outputs and the
 * scan's slots; the pool's stream-ordered memory inside stream capture, where
 * the final synchronisation fails), runs the step on `stream`, delivers the outputs into the host arrays and
 * synchronises the stream before returning.  Page-locked output arrays that the
 * device can address (cudaHostAlloc / cudaHostRegister memory) are written by
 * the draft-fill kernel directly; other host memory receives the outputs by
 * copies.  Page-locked input arrays that the device can address are read by the
 * device itself over the host link (a copy kernel, with the scan launched behind
 * it); other input memory goes through copy-engine transfers.  Pinned host
 * memory is fastest; pageable memory works.  The host offsets are checked
 * (non-decreasing, offsets[0] >= 0, every history < 2^31 tokens):
 * LOOKUP_DRAFT_EINVAL if not.
 */
int lookup_draft_host(const int32_t *h_tokens, const int64_t *h_offsets, int32_t B,
                      int32_t min_m, int32_t max_m, int32_t K,
                      int32_t *h_out_draft, int32_t *h_out_len, int32_t *h_out_pos,
                      struct CUstream_st *stream);

/*
 * lookup_draft without any allocation.  (The source article has no counterpart to
 * this entry point; it is a property of this library.)
 *
 * Some callers must not allocate device memory during a step: a serving loop whose
 * GPU memory is entirely handed out by another framework's allocator, a process
 * that runs under a fixed device-memory budget, or code that must not make the
 * driver calls an allocation implies while it is on a latency-critical path.  This
 * call computes exactly what lookup_draft computes, with the same arguments and
 * outputs, but it keeps the scan's scratch (one 64-bit slot per (request, warp
 * range) pair) in a fixed array of 65,536 slots (512 KiB) in device memory that is
 * part of the library: every GPU that loads the library holds that array until the
 * process exits.  It calls no cudaMalloc, cudaFree, memory-pool or other allocating
 * routine.
 *
 * Limit: B + 16 * (number of SMs) <= 65,536 (B <= 63,104 on a 152-SM GB300);
 * larger batches return LOOKUP_DRAFT_ERANGE and enqueue nothing.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address and sets kernel attributes; make that first call before
 * any stream capture on that device.
 * Sharing: every call on a device uses the same array and leaves its contents
 * behind.  Nothing in it needs clearing between calls (each scan writes every slot
 * it later reads), but calls whose GPU work overlaps in time race on the array and
 * give undefined results: issue them on one stream, or order them with events.
 * Errors as for lookup_draft, plus LOOKUP_DRAFT_ERANGE.
 */
int lookup_draft_noalloc(const int32_t *tokens, const int64_t *offsets, int32_t B,
                         int32_t min_m, int32_t max_m, int32_t K,
                         int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                         struct CUstream_st *stream);

/* Static description of a return code (never NULL). */
const char *lookup_draft_strerror(int code);

/* Message of the CUDA error behind the calling thread's last LOOKUP_DRAFT_ECUDA
 * ("" if none).  Valid until that thread's next call into the library. */
const char *lookup_draft_last_cuda_error(void);

/* Number of kernel launches this library has enqueued since it was loaded, on
 * every thread and stream (successful launches only; a failed call may have
 * enqueued some of its launches before the failure).  Inside a stream capture a
 * launch becomes a graph node and counts once, when it is captured: replays of
 * the graph are not counted.  The difference across a capture is the number of
 * kernels each replay runs.  Never fails; needs no GPU. */
uint64_t lookup_draft_launch_count(void);

/*
 * Diagnostics: the time limit, in nanoseconds, on the scan kernel's bounded waits
 * (default 1e9), counted from each scan CTA's start.  A CTA whose wait for the
 * TMA copy of the offsets runs out reads them from global memory instead (same
 * results).  A CTA whose wait for a history tile runs out lets its own copies
 * land (bounded again), marks its requests LOOKUP_DRAFT_LEN_FAILED and returns,
 * leaving the context usable.  Setting a tiny limit forces these paths, to test
 * them.  Process-wide; applies to launches made after the call.  0 restores the
 * default.
 */
void lookup_draft_set_wait_limit_ns(uint64_t ns);

/*
 * Measurement aid (the source article has no counterpart; it is part of this
 * library's measurement): one launch that streams `bytes` of device memory at
 * `data` and does nothing else with them.  The bytes are read once, with 16-byte
 * loads, each CTA a contiguous chunk, in a grid of ctas_per_sm CTAs per SM of
 * `threads` threads, launched like the draft step's kernels (programmatic
 * dependent launch).  Timed the way the scan is timed over the same bytes, it is
 * the floor that any kernel reading them once reaches in a launch here, so the
 * scan's time can be read against it as well as against the copy bandwidth.
 *
 * data         device, 16-byte aligned, `bytes` readable bytes (read only)
 * bytes        a multiple of 16; 0 enqueues nothing and returns OK
 * ctas_per_sm  1 .. 32;  threads: a multiple of 32 in 32 .. 1024
 * out_word     device, 4-byte aligned: receives a fold of the data only in the
 *              rare case that it equals a fixed pattern (so the loads cannot be
 *              optimised away); otherwise untouched
 * Errors: LOOKUP_DRAFT_EINVAL for a null or misaligned pointer, bytes not a
 * multiple of 16, or a launch shape out of range; LOOKUP_DRAFT_ECUDA when the
 * launch fails.
 */
int lookup_draft_read_floor(const void *data, size_t bytes, int32_t ctas_per_sm, int32_t threads,
                            uint32_t *out_word, struct CUstream_st *stream);

/*
 * The same measurement aid with 1-D bulk copies (TMA) into shared memory, the
 * way the scan reads its history: one CTA of 16 warps per SM, each warp
 * streaming a contiguous range of the buffer through a ring of three tiles of
 * up to 3 KB, each waited for on its mbarrier and folded from shared memory.
 * data/bytes/out_word as for lookup_draft_read_floor.  Its waits are bounded by
 * the limit lookup_draft_set_wait_limit_ns sets (1 s by default); a warp whose
 * wait runs out stores 0xFFFFFFFF in *out_word, waits (bounded again) for its
 * copies in flight and stops, leaving the context usable.
 */
int lookup_draft_read_floor_bulk(const void *data, size_t bytes, uint32_t *out_word, struct CUstream_st *stream);

/*
 * Checked build (a debugging aid; the source article has no counterpart).  The
 * drafting step's source also compiles with LOOKUP_DRAFT_CHECKED=1 into a second
 * library with the same entry points.  There, the scan and fill kernels check
 * the CSR offsets before they read any token through them, and check every
 * index they compute.  A failed check sets a bit in a per-device check word and
 * skips the access: no assert, no trap, no access out of bounds.  That covers
 * tile, suffix-table, token, scratch-slot, bulk-copy, offsets and output
 * indices.
 *
 * Invalid offsets: offsets[0] < 0, a decreasing pair, or a history of 2^31 tokens
 * or more.  Every CTA of the scan then returns before its first copy, and every
 * request of the call reports out_len = LOOKUP_DRAFT_LEN_FAILED, out_pos = -1,
 * out_draft = -1 (and out_mlen = 0).  An offsets[B] past the end of the tokens
 * buffer cannot be seen from the device and stays the caller's precondition.
 * In the regular build no check is compiled.
 *
 * The word is one per device, shared by all calls and streams, and it keeps
 * its bits until cleared.
 */
#define LOOKUP_DRAFT_CHECK_OFFSETS 0x01u  /* offsets are not a valid CSR (see above) */
#define LOOKUP_DRAFT_CHECK_TILE    0x02u  /* a read of a shared-memory tile outside the bytes copied into it */
#define LOOKUP_DRAFT_CHECK_SUFFIX  0x04u  /* a suffix-table index outside its rows or columns */
#define LOOKUP_DRAFT_CHECK_TOKENS  0x08u  /* a token read outside the batch or outside its request */
#define LOOKUP_DRAFT_CHECK_SLOTS   0x10u  /* a scratch-slot index outside the scratch */
#define LOOKUP_DRAFT_CHECK_COPY    0x20u  /* a bulk copy from outside the batch or into outside its ring buffer */
#define LOOKUP_DRAFT_CHECK_INDEX   0x40u  /* an offsets index outside [0, B] */
#define LOOKUP_DRAFT_CHECK_OUTPUT  0x80u  /* an output index outside the B x K outputs */

/* 1 in the checked build, 0 in the regular one. */
int lookup_draft_checked_build(void);

/*
 * Reads the check word of the current device into *out (device memory is
 * synchronised first: the word covers every call whose work has finished) and
 * clears it when `clear` is non-zero.  In the regular build *out = 0.
 * Errors: LOOKUP_DRAFT_EINVAL when out is NULL; LOOKUP_DRAFT_ECUDA when the copy
 * fails.
 */
int lookup_draft_check_word(uint32_t *out, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* LOOKUP_DRAFT_H */
