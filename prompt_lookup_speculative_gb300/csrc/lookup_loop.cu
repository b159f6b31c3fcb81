// lookup_loop.cu -- the decode-loop steps around prompt-lookup drafting, on GB300.
//
// Source: HyperQwen lookup-drafting article, kwkr.cn/news/564408, sections "第2步"
// (fusion of the lookup draft with the draft model's proposals) and "第3步"
// (long-block scheduling with sticky exit; lossless verification, where a
// lookup-filled position is a point mass on its token).  The exact contract of
// every entry point is in include/lookup_loop.h.
//
// fuse_kernel, schedule_kernel and verify_kernel are per-request integer work
// (a few hundred bytes per request), latency-bound.  The next step's histories
// are HBM-bound (4 bytes per history token read, 4 written): offsets_kernel
// turns the committed counts into the new CSR boundaries (one CTA, a block
// scan), then append_kernel copies each history and its committed tokens into
// the new batch, the output split into equal contiguous chunks per CTA.
//
// Every kernel is launched with programmatic dependent launch: it waits for the
// previous kernel on the stream before reading anything and lets the next one
// start its launch early.

#include "lookup_draft.h"
#include "lookup_loop.h"
#include "common.cuh"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

namespace {

using lkd::allow_dependent_launch;
using lkd::launch_pdl;
using lkd::wait_for_prerequisite_grid;

using lkd::kMaxBlock;                      // H + T (a verify block) at most
constexpr int kScanThreads = 1024;       // offsets_kernel
constexpr int kCopyThreads = 256;        // append_kernel
constexpr int kCopyCtasPerSm = 3;
constexpr int kCopyUnroll = 2;           // windows in flight per warp
constexpr int kSub = 4;                  // 128-token sub-windows per window (one int4 per lane each)
constexpr int kWin = 128 * kSub;         // tokens per window
constexpr int kCommitRegs = 1;           // committed tokens per lane held in registers
constexpr int kFusedLoads = 4;           // counts per thread in the fused append's prefix
constexpr int kFusedMaxB = kCopyThreads * kFusedLoads;   // batches up to this size: offsets inside append_kernel

// ------------------------------------------------------------------ fusion ----
struct FuseParams {
    const int32_t *lookup_draft;
    const int32_t *lookup_mlen;
    const int32_t *model_draft;
    const int32_t *long_block;
    int32_t *out_block;
    int32_t *out_len;
    int32_t *out_pm;
    int32_t B, K, H, T, replace_min, agree_min, agree_n, tail_min;
};

// The head rule of request r: its first H proposals come from the lookup draft
// (a long match, or a medium one whose first agree_n tokens the model agrees with).
__device__ inline bool head_from_lookup(const FuseParams &p, int r, int32_t m) {
    const int32_t *ld = p.lookup_draft + int64_t(r) * p.K;
    const int32_t *md = p.model_draft + int64_t(r) * p.H;
    bool agree = true;
    for (int j = 0; j < p.agree_n; ++j) agree = agree && ld[j] == md[j];
    return m >= p.replace_min || (m >= p.agree_min && agree);
}

// Block position i of request r: the proposal and its point-mass flag.
__device__ inline void fuse_position(const FuseParams &p, int r, int i, bool head_lookup, bool tail) {
    const int W = p.H + p.T;
    const int32_t *ld = p.lookup_draft + int64_t(r) * p.K;
    const int32_t *md = p.model_draft + int64_t(r) * p.H;
    int32_t v, pm;
    lkd::fuse_choice(i, p.H, head_lookup, tail, ld[i], i < p.H ? md[i] : -1, v, pm);
    p.out_block[int64_t(r) * W + i] = v;
    p.out_pm[int64_t(r) * W + i] = pm;
}

// One thread per (request, block position).
__global__ void fuse_kernel(FuseParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int W = p.H + p.T;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= int64_t(p.B) * W) return;
    const int r = int(idx / W), i = int(idx - int64_t(r) * W);
    const int32_t m = p.lookup_mlen[r];
    const bool head_lookup = head_from_lookup(p, r, m);
    const bool tail = p.long_block != nullptr && p.long_block[r] != 0 && m >= p.tail_min;
    fuse_position(p, r, i, head_lookup, tail);
    if (i == 0) p.out_len[r] = tail ? W : p.H;
}

// -------------------------------------------------------------- scheduling ----
struct ScheduleParams {
    const int32_t *lookup_mlen;
    const int32_t *committed;
    int32_t *state;
    int32_t *out_long;
    int32_t B, H, T, tail_min, slack, enter_steps, sticky;
};

// One scheduling update of a request's {long, streak, hold} from this step's
// match length m and the previous step's commit count.
__device__ inline void schedule_rule(const ScheduleParams &p, int32_t m, int32_t committed, int32_t &lng,
                                     int32_t &streak, int32_t &hold) {
    lkd::schedule_update(m, committed, p.H, p.T, p.tail_min, p.slack, p.enter_steps, p.sticky, lng, streak, hold);
}

// One thread per request: {long, streak, hold} updated in place.
__global__ void schedule_kernel(ScheduleParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= p.B) return;
    int32_t *st = p.state + 3 * int64_t(r);
    int32_t lng = st[0], streak = st[1], hold = st[2];
    schedule_rule(p, p.lookup_mlen[r], p.committed[r], lng, streak, hold);
    st[0] = lng;
    st[1] = streak;
    st[2] = hold;
    p.out_long[r] = lng;
}

// ---------------------------------------------------- schedule, then fuse ----
constexpr int kPlanWarps = 4;                   // requests per CTA

// One warp per request: every lane reads the old state and applies the
// scheduling rule (same values), the warp synchronises, lane 0 writes the new
// state and the long flag, and the lanes fuse the block's positions with that
// flag: lookup_schedule then lookup_fuse, in one launch.
__global__ void plan_kernel(ScheduleParams sp, FuseParams fp) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kPlanWarps + (threadIdx.x >> 5);
    if (r >= sp.B) return;                       // warp-uniform
    int32_t *st = sp.state + 3 * int64_t(r);
    int32_t lng = st[0], streak = st[1], hold = st[2];
    const int32_t m = sp.lookup_mlen[r];
    schedule_rule(sp, m, sp.committed[r], lng, streak, hold);
    __syncwarp();                                // every lane has read the old state
    if (lane == 0) {
        st[0] = lng;
        st[1] = streak;
        st[2] = hold;
        sp.out_long[r] = lng;
    }
    const bool head_lookup = head_from_lookup(fp, r, m);
    const bool tail = lng != 0 && m >= fp.tail_min;
    const int W = fp.H + fp.T;
    for (int i = lane; i < W; i += 32) fuse_position(fp, r, i, head_lookup, tail);
    if (lane == 0) fp.out_len[r] = tail ? W : fp.H;
}

// ---------------------------------------------------- draft-source controller ----
// Strata engine article, gtnt.cn/news/124732, section 五: per request and step,
// expected committed tokens per unit of verify time for the draft model's draft
// and for the lookup draft; acceptance estimated online by an EMA, per
// match-length bucket for the lookup draft; lookup only when it beats the model
// by more than the margin; plain decoding when neither beats one token per
// t_plain.  float32, each operation rounded as written (the intrinsics keep the
// compiler from fusing them), so every choice is reproducible bit for bit.
struct PolicyParams {
    const int32_t *lookup_mlen;
    const int32_t *accepted;
    float *acc;                  // [B][5]: lookup acceptance per bucket, then the model's
    int32_t *prev;               // [B][3]: last choice, its bucket, tokens it drafted
    int32_t *out_choice;
    int32_t B, n_lookup, n_model, edge1, edge2, edge3;
    float t_lookup, t_model, t_plain, alpha, margin;
};

// 1 + a + a^2 + ... + a^n
__device__ inline float expected_committed(float a, int32_t n) {
    float sum = 1.0f, term = 1.0f;
    for (int32_t i = 1; i <= n; ++i) {
        term = __fmul_rn(term, a);
        sum = __fadd_rn(sum, term);
    }
    return sum;
}

// One thread per request.  Its inputs, the five estimates included, are loaded in
// one round; the update and the choice work on registers (unrolled selects, no
// indexed local array), and the updated estimate is stored once.
__global__ void policy_kernel(PolicyParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= p.B) return;
    float *acc = p.acc + 5 * int64_t(r);
    int32_t *prev = p.prev + 3 * int64_t(r);
    float e[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) e[i] = acc[i];
    const int32_t last = prev[0], last_bucket = prev[1], n = prev[2];
    const int32_t m = p.lookup_mlen[r];
    int32_t a = p.accepted[r];
    // 1. the previous step's outcome updates the estimate of the source that drafted it
    if ((last == 1 || last == 2) && n > 0) {
        a = a < 0 ? 0 : (a > n ? n : a);
        const float rate = __fdiv_rn(__int2float_rn(a), __int2float_rn(n));
        const int32_t slot = last == 2 ? last_bucket : 4;
        float old = e[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (slot == i) old = e[i];
        const float kept = __fmul_rn(__fsub_rn(1.0f, p.alpha), old);
        const float added = __fmul_rn(p.alpha, rate);
        const float upd = __fadd_rn(kept, added);
#pragma unroll
        for (int i = 0; i < 5; ++i)
            if (slot == i) e[i] = upd;
        acc[slot] = upd;
    }
    // 2. expected committed tokens per unit of verify time, per source
    const int32_t b = int32_t(m >= p.edge1) + int32_t(m >= p.edge2) + int32_t(m >= p.edge3);
    float eb = e[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
        if (b == i) eb = e[i];
    const bool avail = m > 0;
    const float b_model = __fdiv_rn(expected_committed(e[4], p.n_model), p.t_model);
    const float b_lookup = avail ? __fdiv_rn(expected_committed(eb, p.n_lookup), p.t_lookup) : 0.0f;
    const float b_plain = __fdiv_rn(1.0f, p.t_plain);
    // 3. lookup only when it beats the model by more than the margin; 4. else plain
    int32_t choice = 1;
    float best = b_model;
    if (avail && b_lookup > __fmul_rn(__fadd_rn(1.0f, p.margin), b_model)) {
        choice = 2;
        best = b_lookup;
    }
    if (!(best > b_plain)) choice = 0;
    prev[0] = choice;
    prev[1] = choice == 2 ? b : 0;
    prev[2] = choice == 2 ? p.n_lookup : (choice == 1 ? p.n_model : 0);
    p.out_choice[r] = choice;
}

// ------------------------------------------------------------ verification ----
struct VerifyParams {
    lkd::VerifyIO io;
    int32_t B;
};

constexpr int kVerifyWarps = 4;

// One warp per request: lanes test positions, the first failure (a ballot)
// is the accepted length.
__global__ void verify_kernel(VerifyParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int r = blockIdx.x * kVerifyWarps + (threadIdx.x >> 5);
    if (r >= p.B) return;
    lkd::verify_warp(p.io, r, threadIdx.x & 31);
}

// ------------------------------------------------------------------ append ----
struct AppendParams {
    const int32_t *tokens;
    const int64_t *offsets;
    const int32_t *commit;
    const int32_t *ncommit;
    int32_t *out_tokens;
    int64_t *out_offsets;
    int32_t B, W;
};

__device__ inline int64_t clamped_count(const AppendParams &p, int64_t r) {
    return min(max(p.ncommit[r], 0), p.W);
}

// The new boundaries: out_offsets[r] = (offsets[r] - offsets[0]) + sum(ncommit[0..r)),
// one CTA: each thread sums a contiguous run of counts, a block-wide exclusive
// scan of the run sums, then each thread writes its run's boundaries.
__global__ void __launch_bounds__(kScanThreads) offsets_kernel(AppendParams p) {
    __shared__ int64_t warp_sums[kScanThreads / 32];
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t per = (int64_t(p.B) + kScanThreads - 1) / kScanThreads;
    const int64_t r0 = min(int64_t(tid) * per, int64_t(p.B)), r1 = min(r0 + per, int64_t(p.B));
    int64_t own = 0;
    for (int64_t r = r0; r < r1; ++r) own += clamped_count(p, r);
    int64_t incl = own;                                  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int64_t s = warp_sums[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        warp_sums[lane] = s;                             // inclusive over warps
    }
    __syncthreads();
    const int64_t base = p.offsets[0];
    int64_t before = (warp ? warp_sums[warp - 1] : 0) + incl - own;
    for (int64_t r = r0; r < r1; ++r) {
        p.out_offsets[r] = (p.offsets[r] - base) + before;
        before += clamped_count(p, r);
    }
    if (tid == kScanThreads - 1) p.out_offsets[p.B] = (p.offsets[p.B] - base) + warp_sums[kScanThreads / 32 - 1];
}

// The output quad at an aligned position: out[j] is run position 4l + 4 - a + j
// of the sub-window, i.e. cur[4 - a + j] for j < a, else nxt[j - a] (cur = this
// lane's input quad, nxt = the next one in the run).
__device__ inline int4 realign(int4 cur, int4 nxt, int a) {
    switch (a) {
    case 1: return make_int4(cur.w, nxt.x, nxt.y, nxt.z);
    case 2: return make_int4(cur.z, cur.w, nxt.x, nxt.y);
    default: return make_int4(cur.y, cur.z, cur.w, nxt.x);
    }
}

__device__ inline int comp(int4 q, int k) { return k == 0 ? q.x : k == 1 ? q.y : k == 2 ? q.z : q.w; }

__device__ inline int4 shfl_quad(int4 v, int src) {
    return make_int4(__shfl_sync(0xffffffffu, v.x, src), __shfl_sync(0xffffffffu, v.y, src),
                     __shfl_sync(0xffffffffu, v.z, src), __shfl_sync(0xffffffffu, v.w, src));
}

__device__ inline int4 shfl_quad_down(int4 v) {
    return make_int4(__shfl_down_sync(0xffffffffu, v.x, 1), __shfl_down_sync(0xffffffffu, v.y, 1),
                     __shfl_down_sync(0xffffffffu, v.z, 1), __shfl_down_sync(0xffffffffu, v.w, 1));
}

// The copy.  With FUSED (B <= kFusedMaxB = 1024 and sum(ncommit) < 2^31), every CTA
// first forms the exclusive prefix of the clamped counts in shared memory --
// what offsets_kernel computes -- and CTA 0 writes out_offsets from it; the
// shifts below then come from shared memory instead of a second kernel.
//
// The histories tokens[offsets[0] .. offsets[B]) are contiguous in
// the input, and each request's run moves as a block to out_offsets[r].  The
// input is cut into windows of kWin tokens aligned to 16 bytes; a window is
// kSub sub-windows of 128 tokens, one int4 per lane each, and each warp takes
// a contiguous range of windows, kCopyUnroll windows in flight.  A window inside
// one request and inside the batch is one contiguous output run: when the run
// is not 16-byte aligned, lanes pass their quads along the run (shuffles) and
// store aligned int4s, with the two partial quads at the run's ends stored
// token by token.  A window that holds a request boundary or an end of the
// batch is written token by token, one request at a time.
//
// Request boundaries come from a per-warp cache: lane i holds the end and the
// shift of request r_first + i, so walking to the next request is a shuffle
// (past 32 requests it falls back to loads).  Everything that reads only the
// inputs -- the window range, the first windows' loads, the request of the
// warp's first window (a 32-way search over offsets), the cache's ends and the
// warp's committed tokens -- is done before waiting for offsets_kernel (FUSED:
// after the previous kernel, since there is no offsets_kernel in between); after
// the wait, one load per lane completes the cache.  The committed tokens of
// request r are written by warp r (grid-stride).
template <bool FUSED>
__global__ void __launch_bounds__(kCopyThreads, kCopyCtasPerSm) append_kernel(AppendParams p) {
    extern __shared__ int32_t pre[];                     // FUSED: [B + 1] exclusive prefix of the counts
    __shared__ int32_t warp_tot[kCopyThreads / 32];
    const int tid = threadIdx.x;
    const int lane = threadIdx.x & 31;
    // FUSED: the previous kernel may still be writing any input (the verify step
    // lets its dependents launch before it writes the counts), so nothing is
    // read before it completes.  Unfused, the previous kernel is offsets_kernel,
    // which waited for the inputs' producer before letting this one launch.
    if (FUSED) wait_for_prerequisite_grid();
    const int64_t gwarp = (int64_t(blockIdx.x) * kCopyThreads + threadIdx.x) >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * (kCopyThreads / 32);
    const int B = p.B;
    const int64_t A0 = p.offsets[0], A1 = p.offsets[B];
    // e_base: the first window start, at or before A0, with tokens + e_base 16-byte aligned
    const int64_t mis_in = int64_t((reinterpret_cast<uintptr_t>(p.tokens) >> 2) & 3);
    const int64_t e_base = A0 - ((mis_in + A0) & 3);
    const int64_t nwin = A1 > A0 ? (A1 - e_base + kWin - 1) / kWin : 0;
    const int64_t per = nwin < (int64_t(1) << 32)      // windows per warp, rounded up
                            ? int64_t((uint32_t(nwin) + uint32_t(nwarps) - 1) / uint32_t(nwarps))
                            : (nwin + nwarps - 1) / nwarps;
    const int64_t k0 = min(gwarp * per, nwin), k1 = min(k0 + per, nwin);
    const int64_t mis_out = int64_t((reinterpret_cast<uintptr_t>(p.out_tokens) >> 2) & 3);

    int4 q[kCopyUnroll][kSub];
    auto load = [&](int64_t k, int u) {
#pragma unroll
        for (int s = 0; s < kSub; ++s) {
            const int64_t e = e_base + k * kWin + 128 * s + 4 * lane;   // this lane's quad
            if (e >= A0 && e + 4 <= A1) {
                q[u][s] = __ldg(reinterpret_cast<const int4 *>(p.tokens + e));
            } else {
                q[u][s] = make_int4(e >= A0 && e < A1 ? p.tokens[e] : 0,
                                    e + 1 >= A0 && e + 1 < A1 ? p.tokens[e + 1] : 0,
                                    e + 2 >= A0 && e + 2 < A1 ? p.tokens[e + 2] : 0,
                                    e + 3 >= A0 && e + 3 < A1 ? p.tokens[e + 3] : 0);
            }
        }
    };
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)                // first windows in flight before anything else
        if (k0 + u < k1) load(k0 + u, u);

    // this warp's committed tokens (request gwarp), into registers
    const int64_t rc0 = gwarp;
    int64_t nc0 = 0;
    int32_t cv[kCommitRegs];
    const int64_t rc0_end = (FUSED && rc0 < B) ? p.offsets[rc0 + 1] : 0;
    if (rc0 < B) {
        nc0 = clamped_count(p, rc0);
#pragma unroll
        for (int c = 0; c < kCommitRegs; ++c)
            cv[c] = lane + 32 * c < nc0 ? __ldg(p.commit + rc0 * p.W + lane + 32 * c) : 0;
    }

    // request holding the first valid token of window k0: largest r with offsets[r] <= e
    int r_first = 0;
    if (k0 < k1) {
        const int64_t e = max(e_base + k0 * kWin, A0);
        int lo = 0, hi = B;                              // offsets[lo] <= e < offsets[hi]
        while (hi - lo > 1) {
            const int step = (hi - lo + 31) / 32;
            const int idx = min(lo + lane * step, hi - 1);
            const unsigned le = __ballot_sync(0xffffffffu, p.offsets[idx] <= e);
            const int last = 31 - __clz(le);             // lane 0 always qualifies (idx = lo)
            const int nlo = min(lo + last * step, hi - 1);
            hi = min(nlo + step, hi);
            lo = nlo;
        }
        r_first = lo;
    }
    // the cache: lane i holds request r_first + i (its end, then its shift)
    const int rc = r_first + lane;
    const int64_t c_start = (k0 < k1 && rc < B) ? p.offsets[rc] : 0;
    const int64_t c_end = (k0 < k1 && rc < B) ? p.offsets[rc + 1] : 0;

    wait_for_prerequisite_grid();                        // FUSED: the counts; else: out_offsets
    allow_dependent_launch();

    // out_offsets[r] - offsets[r] (FUSED: from the shared prefix)
    auto shift_of = [&](int64_t r, int64_t off_r) -> int64_t {
        if (FUSED) return int64_t(pre[r]) - A0;
        return p.out_offsets[r] - off_r;
    };
    if (FUSED) {
        // counts into shared memory (coalesced), each thread's run summed, a block
        // scan of the run sums, then the runs rewritten as exclusive prefixes
        int32_t cnt_r[kFusedLoads];                      // independent loads, then the stores
#pragma unroll
        for (int u = 0; u < kFusedLoads; ++u) {
            const int i = tid + u * kCopyThreads;
            cnt_r[u] = i < B ? int32_t(clamped_count(p, i)) : 0;
        }
#pragma unroll
        for (int u = 0; u < kFusedLoads; ++u)
            if (tid + u * kCopyThreads < B) pre[tid + u * kCopyThreads] = cnt_r[u];
        __syncthreads();
        const int per = (B + kCopyThreads - 1) / kCopyThreads;
        const int i0 = min(tid * per, B), i1 = min(i0 + per, B);
        int own = 0;
        for (int i = i0; i < i1; ++i) own += pre[i];
        int incl = own;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == 31) warp_tot[tid >> 5] = incl;
        __syncthreads();
        int before = incl - own, total = 0;
#pragma unroll
        for (int w = 0; w < kCopyThreads / 32; ++w) {
            before += w < (tid >> 5) ? warp_tot[w] : 0;
            total += warp_tot[w];
        }
        for (int i = i0; i < i1; ++i) {
            const int cnt = pre[i];
            pre[i] = before;
            before += cnt;
        }
        if (tid == 0) pre[B] = total;
        __syncthreads();
        if (blockIdx.x == 0)
            for (int i = tid; i <= B; i += kCopyThreads) p.out_offsets[i] = (p.offsets[i] - A0) + pre[i];
    }

    int64_t c_shift = (k0 < k1 && rc < B) ? shift_of(rc, c_start) : 0;
    if (rc0 < B) {                                       // committed tokens after the history
        const int64_t dst = (FUSED ? (rc0_end - A0) + pre[rc0 + 1] : p.out_offsets[rc0 + 1]) - nc0;
#pragma unroll
        for (int c = 0; c < kCommitRegs; ++c)
            if (lane + 32 * c < nc0) p.out_tokens[dst + lane + 32 * c] = cv[c];
        for (int64_t j = lane + 32 * kCommitRegs; j < nc0; j += 32) p.out_tokens[dst + j] = __ldg(p.commit + rc0 * p.W + j);
    }
    for (int64_t rr = rc0 + nwarps; rr < B; rr += nwarps) {
        const int64_t n = clamped_count(p, rr);
        const int64_t dst = (FUSED ? (p.offsets[rr + 1] - A0) + pre[rr + 1] : p.out_offsets[rr + 1]) - n;
        for (int64_t j = lane; j < n; j += 32) p.out_tokens[dst + j] = __ldg(p.commit + rr * p.W + j);
    }
    if (k0 >= k1) return;

    // the current request r: tokens [.., r_end) move by shift (uniform across the warp)
    int r = r_first;
    int64_t r_end = __shfl_sync(0xffffffffu, c_end, 0);
    int64_t shift = __shfl_sync(0xffffffffu, c_shift, 0);
    auto next_request = [&]() {
        ++r;
        const int i = r - r_first;
        if (i < 32) {
            r_end = __shfl_sync(0xffffffffu, c_end, i);
            shift = __shfl_sync(0xffffffffu, c_shift, i);
        } else {
            r_end = p.offsets[r + 1];
            shift = shift_of(r, p.offsets[r]);
        }
    };

    for (int64_t kb = k0; kb < k1; kb += kCopyUnroll) {
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t k = kb + u;
            if (k >= k1) break;
            const int64_t w0 = e_base + k * kWin;
            const int64_t v0 = max(w0, A0), v1 = min(w0 + kWin, A1);
            while (r_end <= v0) next_request();          // the request of the window's first token
            if (w0 >= A0 && w0 + kWin <= A1 && r_end >= v1) {
                // one request, whole window: output run [w0 + shift, w0 + shift + kWin)
                int32_t *run = p.out_tokens + (w0 + shift);
                const int a = int((mis_out + w0 + shift) & 3);
                if (a == 0) {
#pragma unroll
                    for (int s = 0; s < kSub; ++s)
                        *reinterpret_cast<int4 *>(run + 128 * s + 4 * lane) = q[u][s];
                } else {
#pragma unroll
                    for (int s = 0; s < kSub; ++s) {
                        const int4 down = shfl_quad_down(q[u][s]);
                        const int4 wrap = shfl_quad(q[u][s + 1 < kSub ? s + 1 : s], 0);
                        const int4 nxt = lane < 31 ? down : wrap;
                        if (lane < 31 || s + 1 < kSub)
                            *reinterpret_cast<int4 *>(run - a + 128 * s + 4 * (lane + 1)) = realign(q[u][s], nxt, a);
                    }
                    if (lane == 0)
                        for (int j = 0; j < 4 - a; ++j) run[j] = comp(q[u][0], j);
                    if (lane == 31)
                        for (int j = 4 - a; j < 4; ++j) run[kWin - 4 + j] = comp(q[u][kSub - 1], j);
                }
            } else {
                // token by token, one request at a time: [seg0, seg1) moves by shift
                int64_t seg0 = v0;
                while (true) {
                    const int64_t seg1 = min(r_end, v1);
#pragma unroll
                    for (int s = 0; s < kSub; ++s) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int64_t e = w0 + 128 * s + 4 * lane + j;
                            if (e >= seg0 && e < seg1) p.out_tokens[e + shift] = comp(q[u][s], j);
                        }
                    }
                    if (r_end >= v1) break;
                    seg0 = r_end;
                    next_request();
                }
            }
            if (k + kCopyUnroll < k1) load(k + kCopyUnroll, u);   // the next pass's window
        }
    }
}

// ------------------------------------------------------------------- host ----
int cuda_fail(cudaError_t e, const char *what) { return lookup_record_cuda_error(e, what); }

unsigned blocks_for(int64_t n, int per) { return unsigned((n + per - 1) / per); }

}  // namespace

extern "C" {

int lookup_fuse(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *long_block, int32_t B, int32_t K, int32_t H, int32_t T, int32_t replace_min,
                int32_t agree_min, int32_t agree_n, int32_t tail_min, int32_t *out_block, int32_t *out_len,
                int32_t *out_point_mass, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_fuse");
    if (B < 0 || H < 1 || T < 0 || int64_t(H) + T > kMaxBlock || K < H + T || agree_n < 0 || agree_n > H)
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_draft || !lookup_mlen || !model_draft || !out_block || !out_len || !out_point_mass)
        return LOOKUP_DRAFT_EINVAL;
    FuseParams p{lookup_draft, lookup_mlen, model_draft, long_block, out_block, out_len, out_point_mass,
                 B, K, H, T, replace_min, agree_min, agree_n, tail_min};
    return launch_pdl(fuse_kernel, blocks_for(int64_t(B) * (H + T), 256), 256u, stream, p);
}

int lookup_schedule(const int32_t *lookup_mlen, const int32_t *committed, int32_t B, int32_t H, int32_t T,
                    int32_t tail_min, int32_t slack, int32_t enter_steps, int32_t sticky, int32_t *state,
                    int32_t *out_long, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_schedule");
    if (B < 0 || H < 1 || T < 0 || enter_steps < 1 || sticky < 0 || slack < 0) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_mlen || !committed || !state || !out_long) return LOOKUP_DRAFT_EINVAL;
    ScheduleParams p{lookup_mlen, committed, state, out_long, B, H, T, tail_min, slack, enter_steps, sticky};
    return launch_pdl(schedule_kernel, blocks_for(B, 256), 256u, stream, p);
}

int lookup_plan(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *committed, int32_t B, int32_t K, int32_t H, int32_t T, int32_t replace_min,
                int32_t agree_min, int32_t agree_n, int32_t tail_min, int32_t slack, int32_t enter_steps,
                int32_t sticky, int32_t *state, int32_t *out_long, int32_t *out_block, int32_t *out_len,
                int32_t *out_point_mass, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_plan");
    if (B < 0 || H < 1 || T < 0 || int64_t(H) + T > kMaxBlock || K < H + T || agree_n < 0 || agree_n > H ||
        enter_steps < 1 || sticky < 0 || slack < 0)
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_draft || !lookup_mlen || !model_draft || !committed || !state || !out_long || !out_block ||
        !out_len || !out_point_mass)
        return LOOKUP_DRAFT_EINVAL;
    ScheduleParams sp{lookup_mlen, committed, state, out_long, B, H, T, tail_min, slack, enter_steps, sticky};
    FuseParams fp{lookup_draft, lookup_mlen, model_draft, out_long, out_block, out_len, out_point_mass,
                  B, K, H, T, replace_min, agree_min, agree_n, tail_min};
    return lkd::launch_pdl2(plan_kernel, blocks_for(B, kPlanWarps), unsigned(kPlanWarps * 32), stream, sp, fp);
}

int lookup_policy(const int32_t *lookup_mlen, const int32_t *accepted, int32_t B, int32_t n_lookup, int32_t n_model,
                  float t_lookup, float t_model, float t_plain, float alpha, float margin, int32_t edge1,
                  int32_t edge2, int32_t edge3, float *acc, int32_t *prev, int32_t *out_choice,
                  struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_policy");
    if (B < 0 || n_lookup < 0 || n_model < 0 || !(t_lookup > 0.0f) || !(t_model > 0.0f) || !(t_plain > 0.0f) ||
        !(alpha >= 0.0f && alpha <= 1.0f) || !(margin >= 0.0f) || edge1 > edge2 || edge2 > edge3)
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_mlen || !accepted || !acc || !prev || !out_choice) return LOOKUP_DRAFT_EINVAL;
    PolicyParams p{lookup_mlen, accepted, acc, prev, out_choice, B, n_lookup, n_model, edge1, edge2, edge3,
                   t_lookup, t_model, t_plain, alpha, margin};
    return launch_pdl(policy_kernel, blocks_for(B, 256), 256u, stream, p);
}

int lookup_verify(const int32_t *block, const int32_t *len, const int32_t *target, const float *probs,
                  const float *qprobs, const int32_t *point_mass, const float *u, int32_t B, int32_t P,
                  int32_t *out_accepted, int32_t *out_commit, int32_t *out_ncommit, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_verify");
    if (B < 0 || P < 0 || P > kMaxBlock) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if ((P > 0 && !block) || !len || !target || (probs && !u) || !out_accepted || !out_commit || !out_ncommit)
        return LOOKUP_DRAFT_EINVAL;
    VerifyParams p{{block, len, target, probs, qprobs, point_mass, u, out_accepted, out_commit, out_ncommit, P}, B};
    return launch_pdl(verify_kernel, blocks_for(B, kVerifyWarps), unsigned(kVerifyWarps * 32), stream, p);
}

int lookup_append(const int32_t *tokens, const int64_t *offsets, const int32_t *commit, const int32_t *ncommit,
                  int32_t B, int32_t W, int32_t *out_tokens, int64_t *out_offsets, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_append");
    if (B < 0 || W < 0) return LOOKUP_DRAFT_EINVAL;
    if (!offsets || !out_offsets || (B > 0 && (!tokens || !ncommit || (W > 0 && !commit) || !out_tokens)))
        return LOOKUP_DRAFT_EINVAL;
    AppendParams p{tokens, offsets, commit, ncommit, out_tokens, out_offsets, B, W};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    if (B > 0 && ((reinterpret_cast<uintptr_t>(tokens) | reinterpret_cast<uintptr_t>(out_tokens)) & 3))
        return LOOKUP_DRAFT_EINVAL;
    const unsigned grid = unsigned(sms * kCopyCtasPerSm);
    if (B > 0 && B <= kFusedMaxB && int64_t(B) * W < (int64_t(1) << 31))
        return launch_pdl(append_kernel<true>, grid, unsigned(kCopyThreads), stream, p, size_t(B + 1) * sizeof(int32_t));
    int rc = launch_pdl(offsets_kernel, 1u, unsigned(kScanThreads), stream, p);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;      // B == 0: out_offsets = {0} only
    return launch_pdl(append_kernel<false>, grid, unsigned(kCopyThreads), stream, p);
}

}  // extern "C"
