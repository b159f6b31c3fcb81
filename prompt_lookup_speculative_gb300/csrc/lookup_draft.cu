// lookup_draft.cu -- prompt-lookup (n-gram) drafting on GB300 (sm_103a).
//
// What one call computes (HyperQwen lookup-drafting article, kwkr.cn/news/564408,
// section "第1步"): for every request of a CSR batch, the most recent earlier
// occurrence of the longest current suffix (max_m down to min_m tokens, overlap
// with the suffix allowed), and the K tokens that follow it, read from the history
// extended by its own draft (e[L+j] = e[p+m+j]).  The exact contract is in
// include/lookup_draft.h.
//
// A draft step is two kernels, both on the caller's stream:
//
//  scan_kernel -- the split-history scan, HBM bound (4 bytes per history token,
//    read once).  The whole batch is one array of 16-byte quads; the grid (one CTA
//    per SM, independent of the data so the host never reads the offsets) splits
//    it into equal contiguous chunks of at least 256 quads, and each CTA's chunk into 16 equal warp
//    ranges ("virtual chunks"), so long requests are shared by many warps and
//    short ones are packed into one.  The offsets arrive in shared memory with one
//    TMA bulk copy; from then on every warp works alone.  A warp first loads the
//    suffix tokens of the requests in its range (ahead of its bulk history reads,
//    so they are not queued behind them), then streams its range through a
//    private ring of shared-memory buffers filled by 1-D TMA bulk copies
//    (cp.async.bulk, mbarrier completion), each tile preceded by a halo of up to
//    31 tokens of backward context.  A tile is walked request by request; within
//    a request every lane takes 128-bit quads and runs the article's cheap
//    rejection test (section "第1步") branch-free: a token and the D - 1 tokens
//    before it against the last D suffix tokens, D = min(min_m, 4).  The rare
//    survivors are extended backwards, eight positions compared per round with
//    their shared-memory loads issued together.  A match of length k ending at
//    local position q gives the key (k << 32) | (q - k + 1): its maximum is the longest
//    match, then the most recent.  A warp keeps its current request and its
//    lanes' best keys across tiles and writes the warp's maximum into the
//    (request, virtual chunk) slot when it moves on.
//
//  fill_kernel -- one warp per request (fill_lanes_kernel: one request per lane,
//    for batches of 1,024 requests or more): max over the request's slots, then
//    the draft tokens t[p + m + (j mod d)], d = L - p - m, and the length/position.
//
// fill_plan_kernel is the fill's warp going on with the decode loop's next two
// steps, long-block scheduling and fusion (lookup_draft_plan).
//
// The kernels use programmatic dependent launch: each lets the next kernel on
// the stream start its prologue early and waits for its predecessor's results
// before reading them.  Compiled with LOOKUP_DRAFT_CHECKED=1, they also check
// every index they compute (the checked build, below).
//
// Partial-result slots.  Virtual chunk v owns slot (r + v) for every non-empty
// request r that has a token in its range.  Virtual chunks and requests are both
// ordered and disjoint, so the (v, r) pairs form a monotone staircase and r + v
// never repeats: every slot belongs to one warp, whose lanes fold their keys into
// it with atomicMax (no other warp contends on it), and it needs no clearing
// before a call (its warp zeroes it before use).
//
// No spin-wait is unbounded: every mbarrier wait gives up at a deadline.  A warp
// that gives up lets its own copies land (bounded), marks its requests as failed
// in their slots and stops, so the failure reaches the host as
// out_len = LOOKUP_DRAFT_LEN_FAILED instead of a hang.

#include "lookup_draft.h"
#include "lookup_loop.h"

#include "common.cuh"

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace {

using lkd::allow_dependent_launch;
using lkd::launch_pdl;
using lkd::TraceRange;
using lkd::wait_for_prerequisite_grid;

// ---------------------------------------------------------------- tuning ----
constexpr int kWarps = 16;             // scan warps per CTA; each owns a contiguous range
constexpr int kChunkMin = 256;         // quads per CTA chunk at least (small batches use fewer CTAs)
constexpr int kChunkSmall = 512;       // quads per CTA chunk below which it has 8 warp ranges
constexpr int kChunkMid = 2048;        // ... and below which 12 (else kWarps)
constexpr int kThreads = kWarps * 32;
constexpr int kBufs = 3;               // tiles in flight per warp
constexpr int kTileQuadsMax = 192;     // 3 KB of history per tile at most
constexpr int kTileQuadsMin = 32;
constexpr int kHaloQuads = 8;          // room for (LOOKUP_DRAFT_MAX_M - 1) tokens of context
constexpr int kSufRows = 8;            // requests per warp whose suffix is kept in smem
constexpr int kOffCap = 4097;          // offsets kept in smem when B + 1 <= kOffCap
constexpr int kFillWarps = 4;          // requests per fill CTA
constexpr int kFillUnroll = 4;         // slot loads in flight per fill lane
constexpr int kFillMinBlocks = 12;     // fill CTAs that fit beside a scan CTA on one SM
constexpr int kLaneFillThreads = 128;  // requests per CTA of the lane-per-request fill
constexpr int kLaneCover = 4;          // scan warps a lane folds by itself
constexpr int kLaneFillMinB = 1024;    // batches from this size use the lane-per-request fill

constexpr unsigned long long kKeyFailed = ~0ull;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

static_assert(4 * kHaloQuads >= LOOKUP_DRAFT_MAX_M - 1, "halo too small for LOOKUP_DRAFT_MAX_M");

// ---------------------------------------------------------- checked build ----
// Compiled with LOOKUP_DRAFT_CHECKED=1, every index the kernels compute is checked
// before use: a failed check sets its LOOKUP_DRAFT_CHECK_* bit in the device's
// check word and the access is skipped.  In the regular build LKD_OK(cond, bit)
// is the constant true and no check is compiled.
#ifndef LOOKUP_DRAFT_CHECKED
#define LOOKUP_DRAFT_CHECKED 0
#endif
#if LOOKUP_DRAFT_CHECKED
__device__ unsigned g_check_word;
__device__ __forceinline__ bool check_ok(bool ok, unsigned bit) {
    if (!ok) atomicOr(&g_check_word, bit);
    return ok;
}
#define LKD_OK(cond, bit) check_ok((cond), (bit))
#else
#define LKD_OK(cond, bit) true
#endif

constexpr size_t kBufBytes = size_t(kTileQuadsMax + kHaloQuads) * 16;

struct ScanParams {
    const int32_t *tokens;
    const int64_t *offsets;
    unsigned long long *slots;
    int32_t B;
    int32_t min_m;
    int32_t max_m;
    int32_t grid;
    uint32_t grid_magic;   // floor(n / grid) = umulhi(n, grid_magic) >> grid_shift for n < 2^31
    int32_t grid_shift;    // -1: grid == 1
    uint64_t wait_ns;
#if LOOKUP_DRAFT_CHECKED
    int64_t nslots;        // slots in the scratch
#endif
};

struct FillParams {
    const int32_t *tokens;
    const int64_t *offsets;
    const unsigned long long *slots;
    int32_t *out_draft;
    int32_t *out_len;
    int32_t *out_pos;
    int32_t *out_mlen;
    int32_t B;
    int32_t K;
    int32_t grid;
#if LOOKUP_DRAFT_CHECKED
    int64_t nslots;        // slots in the scratch
#endif
};

// ------------------------------------------------------ partition helpers ----
// The batch occupies aligned quads [q_lo, q_lo + nq) of the 16-byte-aligned view
// of `tokens`.  Chunk c (CTA c) is quads [c*S, (c+1)*S) of that range, clipped,
// with S = max(ceil(nq / G), kChunkMin): a small batch fills fewer CTAs, so its
// requests span fewer warp ranges (fewer slots for the fill to fold) and fewer
// warps repeat the per-warp prologue.  Warp w of chunk c takes quads [c*S + w*Sw, c*S + (w+1)*Sw)
// of it, clipped to the chunk, with Sw = warp_span32(S) (ceil(S / kWarps) unless
// the chunk is small).  Virtual chunk
// v = c*kWarps + w.  Empty chunks and empty warp ranges come last in their order.
// Quads per warp range for a CTA chunk of S quads.  Small chunks get fewer and
// longer ranges (8, or 12, of the kWarps; the other warps' ranges are empty), so
// a small batch starts fewer warps' request searches and suffix loads and leaves
// fewer slots to the fill.
__host__ __device__ __forceinline__ uint32_t warp_span32(uint32_t S) {
    if (S < uint32_t(kChunkSmall)) return (S + 7u) >> 3;
    if (S < uint32_t(kChunkMid)) return (S + 11u) / 12u;
    return (S + uint32_t(kWarps) - 1u) / uint32_t(kWarps);
}

struct Partition {
    int64_t q_lo;
    int64_t nq;
    int64_t S;          // quads per chunk
    int64_t Sw;         // quads per warp range
};

__host__ __device__ inline int tokens_shift(const int32_t *tokens) {
    return int((reinterpret_cast<uintptr_t>(tokens) & 15u) >> 2);
}

// x / y for y > 0, in 32-bit arithmetic whenever x allows it.
__device__ inline int64_t div_u(int64_t x, int64_t y) {
    if (((unsigned long long)x | (unsigned long long)y) < (1ull << 32)) return int64_t(uint32_t(x) / uint32_t(y));
    return int64_t((unsigned long long)x / (unsigned long long)y);
}

__device__ inline Partition make_partition(int64_t a_begin, int64_t a_end, int G) {
    Partition P;
    P.q_lo = a_begin >> 2;
    P.nq = ((a_end + 3) >> 2) - P.q_lo;
    P.S = div_u(P.nq + G - 1, G);
    P.S = P.S < kChunkMin ? kChunkMin : P.S;
    P.Sw = P.S < kChunkMid ? int64_t(warp_span32(uint32_t(P.S))) : div_u(P.S + kWarps - 1, kWarps);
    return P;
}

// Quads [lo, hi) of virtual chunk v, relative to q_lo (empty when lo >= hi).
__device__ inline void vchunk_range(const Partition &P, int64_t v, int64_t &lo, int64_t &hi) {
    const int64_t c = v / kWarps, w = v - c * kWarps;
    const int64_t c0 = c * P.S;
    const int64_t c1 = (c0 + P.S < P.nq) ? c0 + P.S : P.nq;
    lo = c0 + w * P.Sw;
    hi = (lo + P.Sw < c1) ? lo + P.Sw : c1;
}

// The virtual chunk holding quad x (relative to q_lo, 0 <= x < nq).
__device__ inline int64_t vchunk_of_quad(const Partition &P, int64_t x) {
    const int64_t c = div_u(x, P.S);
    return c * kWarps + div_u(x - c * P.S, P.Sw);
}

// ----------------------------------------------------------- PTX wrappers ----
// (common.cuh: shared memory addresses, mbarriers, 1-D bulk copies, the global timer)
using lkd::bulk_copy_g2s;
using lkd::bulk_copy_g2s_stream;
using lkd::fence_barrier_init;
using lkd::fence_proxy_async_smem;
using lkd::global_ns;
using lkd::mbar_expect_tx;
using lkd::mbar_init;
using lkd::mbar_try_wait;
using lkd::mbar_wait_until;
using lkd::prefetch_l2;
using lkd::smem_addr;

// ------------------------------------------------------------ scan kernel ----
// Dynamic shared memory: the warps' tile rings, their mbarriers (plus one for the
// offsets copy), the warps' suffix rows, and the offsets.  The rings alone exceed
// half of an SM's shared memory, so exactly one scan CTA runs per SM.
struct ScanSmemLayout {
    size_t bufs, bars, suf, offs, total;
};

__host__ __device__ inline ScanSmemLayout scan_smem_layout(int32_t B, int32_t max_m) {
    ScanSmemLayout L;
    L.bufs = 0;
    L.bars = L.bufs + size_t(kWarps) * kBufs * kBufBytes;
    L.suf = L.bars + (size_t(kWarps) * kBufs + 1) * sizeof(unsigned long long);
    L.offs = (L.suf + size_t(kWarps) * kSufRows * size_t(max_m) * 4 + 15) & ~size_t(15);
    // offsets copied as the 16-byte-aligned span covering them
    const size_t n_off = (int64_t(B) + 1 <= kOffCap) ? size_t(B) + 1 : 2;
    L.total = L.offs + ((n_off * 8 + 16 + 15) & ~size_t(15));
    return L;
}

// Rejection test on one quad: bit e is set when the token at element e of `cur`
// and the D - 1 tokens before it equal the last D suffix tokens s0, s1, ...  The
// tokens before cur.x are the last three of `prv`.
template <int D>
__device__ __forceinline__ unsigned quad_hits(const int4 &prv, const int4 &cur, int32_t s0, int32_t s1, int32_t s2,
                                              int32_t s3) {
    bool h0 = cur.x == s0, h1 = cur.y == s0, h2 = cur.z == s0, h3 = cur.w == s0;
    if (D >= 2) {
        h0 = h0 && prv.w == s1; h1 = h1 && cur.x == s1; h2 = h2 && cur.y == s1; h3 = h3 && cur.z == s1;
    }
    if (D >= 3) {
        h0 = h0 && prv.z == s2; h1 = h1 && prv.w == s2; h2 = h2 && cur.x == s2; h3 = h3 && cur.y == s2;
    }
    if (D >= 4) {
        h0 = h0 && prv.y == s3; h1 = h1 && prv.z == s3; h2 = h2 && prv.w == s3; h3 = h3 && cur.x == s3;
    }
    return unsigned(h0) | (unsigned(h1) << 1) | (unsigned(h2) << 2) | (unsigned(h3) << 3);
}

// Whether any element of the quad passes the D-token test (the common answer is
// no, so the per-element bits are only formed on the rare path).
template <int D>
__device__ __forceinline__ bool quad_any(const int4 &prv, const int4 &cur, int32_t s0, int32_t s1, int32_t s2,
                                         int32_t s3) {
    bool h0 = cur.x == s0, h1 = cur.y == s0, h2 = cur.z == s0, h3 = cur.w == s0;
    if (D >= 2) {
        h0 &= prv.w == s1; h1 &= cur.x == s1; h2 &= cur.y == s1; h3 &= cur.z == s1;
    }
    if (D >= 3) {
        h0 &= prv.z == s2; h1 &= prv.w == s2; h2 &= cur.x == s2; h3 &= cur.y == s2;
    }
    if (D >= 4) {
        h0 &= prv.y == s3; h1 &= prv.z == s3; h2 &= prv.w == s3; h3 &= cur.x == s3;
    }
    return (h0 | h1) | (h2 | h3);
}

// Length of the match ending at tile element e whose last k0 tokens already
// match: the largest k <= kmax with st[e - i] == suf[i] for every i < k.  Eight
// positions are compared per round, their loads issued together, so a full
// match of max_m = 12 costs one round of shared-memory latency instead of eight.
// st[e - k] stays inside the buffer (the halo holds 32 tokens and k < 32).
__device__ __forceinline__ int match_len(const int32_t *st, int e, const int32_t *suf, int k0, int kmax) {
    int kk = k0;
    while (kk < kmax) {
        unsigned ne = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = kk + i;
            if (k < kmax && st[e - k] != suf[k]) ne |= 1u << i;
        }
        const int left = kmax - kk;
        const unsigned stop = ne | (left < 8 ? (~0u << left) : 0u);
        if (stop) return kk + __ffs(int(stop)) - 1;
        kk += 8;
    }
    return kmax;
}

// Bit e set when element x4 + e lies in [lo, hi] (e = 0..3).
__device__ __forceinline__ unsigned range_mask(int x4, int lo, int hi) {
    const int a = lo - x4, b = hi - x4;
    if (b < 0 || a > 3) return 0u;
    const unsigned ma = a <= 0 ? 0xFu : (0xFu << a) & 0xFu;
    const unsigned mb = b >= 3 ? 0xFu : 0xFu >> (3 - b);
    return ma & mb;
}

// D = min(min_m, 4): how many suffix tokens the branch-free rejection test checks
// before a candidate is extended, eight positions per round.  OFFS_SMEM: B + 1 <= kOffCap,
// the offsets are copied into shared memory (otherwise read from global memory).
template <int D, bool OFFS_SMEM>
__global__ void __launch_bounds__(kThreads, 1) scan_kernel(ScanParams prm) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ unsigned long long sh_deadline;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int c = blockIdx.x;
    const int G = prm.grid;
    const int B = prm.B;
    const int min_m = prm.min_m;
    const int max_m = prm.max_m;

    const ScanSmemLayout lay = scan_smem_layout(B, max_m);
    unsigned long long *bars = reinterpret_cast<unsigned long long *>(smem + lay.bars);
    unsigned long long *offs_bar = bars + kWarps * kBufs;
    int32_t *suf_w = reinterpret_cast<int32_t *>(smem + lay.suf) + warp * kSufRows * max_m;

    const int shift = tokens_shift(prm.tokens);
    const int32_t *ta = reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(prm.tokens) & ~uintptr_t(15));
    constexpr bool offs_in_smem = OFFS_SMEM;
    const uintptr_t off_src = reinterpret_cast<uintptr_t>(prm.offsets) & ~uintptr_t(15);
    const int64_t *offs_s =
        reinterpret_cast<const int64_t *>(smem + lay.offs + (reinterpret_cast<uintptr_t>(prm.offsets) & 15u));

    // 0. Barriers (the offsets' by thread 0, each warp's ring by its lane 0), and
    //    the offsets warmed into L2 while the previous kernel on the stream
    //    finishes; then wait for it (it may have written the inputs).
    if (offs_in_smem && tid * 16 <= B) prefetch_l2(prm.offsets + tid * 16);
    unsigned long long *my_bars = bars + warp * kBufs;
    if (tid == 0) {
        sh_deadline = global_ns() + prm.wait_ns;         // every copy must land by then
        mbar_init(smem_addr(offs_bar), 1);
        fence_barrier_init();
    }
    if (lane == 0) {
        for (int i = 0; i < kBufs; ++i) mbar_init(smem_addr(&my_bars[i]), 1);
        fence_barrier_init();
    }
    wait_for_prerequisite_grid();
#if LOOKUP_DRAFT_CHECKED
    // The CSR offsets, before anything reads tokens through them: offsets[0] >= 0,
    // non-decreasing, every history shorter than 2^31 tokens.  Otherwise the CTA
    // returns before its first copy (the fill then fails every request).
    {
        bool bad = false;
        for (int i = tid; i <= B; i += kThreads) {
            const int64_t a = prm.offsets[i];
            bad |= i == 0 && a < 0;
            if (i < B) {
                const int64_t b = prm.offsets[i + 1];
                bad |= b < a || b - a >= (int64_t(1) << 31);
            }
        }
        if (__syncthreads_or(bad)) {
            if (tid == 0) atomicOr(&g_check_word, LOOKUP_DRAFT_CHECK_OFFSETS);
            return;
        }
    }
#endif

    // 1. Offsets -> shared memory: one bulk copy of the 16-byte span covering them,
    //    for the request searches.  Should the copy not land in time, the CTA reads
    //    the offsets from global memory instead (and lets the copy land before it
    //    exits).  The batch's two ends, all that the first copy of history needs,
    //    are read straight from memory meanwhile, through L1, which merges the
    //    CTA's 16 warps' requests for the same two lines.
    if (offs_in_smem && tid == 0) {
        const uintptr_t end = (reinterpret_cast<uintptr_t>(prm.offsets + B + 1) + 15) & ~uintptr_t(15);
        const uint32_t bytes = uint32_t(end - off_src);
        mbar_expect_tx(smem_addr(offs_bar), bytes);
        bulk_copy_g2s(smem_addr(smem + lay.offs), reinterpret_cast<const void *>(off_src), bytes,
                      smem_addr(offs_bar));
    }
    int64_t ends = 0;
    if (lane < 2) ends = __ldca(prm.offsets + (lane == 0 ? 0 : B));
    const int64_t a_begin = __shfl_sync(0xffffffffu, ends, 0) + shift;
    const int64_t a_end = __shfl_sync(0xffffffffu, ends, 1) + shift;
    allow_dependent_launch();
    bool failed = false;
    // 2. The warp's range, in 32-bit arithmetic whenever the batch allows it: this
    //    integer chain lies on the path to the warp's first copy.
    Partition P;
    int64_t wq0 = 0, wq1 = 0;
    P.q_lo = a_begin >> 2;
    P.nq = ((a_end + 3) >> 2) - P.q_lo;
    if (P.nq < (int64_t(1) << 31) - G) {
        const uint32_t nq = uint32_t(P.nq), n = nq + uint32_t(G - 1);
        uint32_t S = prm.grid_shift < 0 ? n : __umulhi(n, prm.grid_magic) >> prm.grid_shift;
        S = S < uint32_t(kChunkMin) ? uint32_t(kChunkMin) : S;
        const uint32_t Sw = warp_span32(S);
        P.S = S;
        P.Sw = Sw;
        const uint32_t c0 = uint32_t(c) * S;
        const uint32_t c1 = (c0 + S < nq) ? c0 + S : nq;
        const uint32_t lo = c0 + uint32_t(warp) * Sw;
        if (a_end > a_begin) {
            wq0 = lo;
            wq1 = (lo + Sw < c1) ? lo + Sw : c1;
        }
    } else {
        P = make_partition(a_begin, a_end, G);
        if (a_end > a_begin) vchunk_range(P, int64_t(c) * kWarps + warp, wq0, wq1);
    }

    // 3. Tiles: tile k is quads [k*tq, min((k+1)*tq, wn)) of the range (one tile
    //    when the range fits in one); the ring holds kBufs of them, tile k in buffer
    //    k % kBufs.  The first one is issued at once, the rest after the suffix
    //    loads below, so that only one tile per warp is queued ahead of those
    //    latency-critical loads.  Quads are counted from the range's first, and the
    //    halo reaches back at most `lead` quads (not before the batch).
    const int wn = wq0 < wq1 ? int(wq1 - wq0) : 0;
    const int halo = (max_m - 1 + 3) >> 2;
    int tq = wn <= kTileQuadsMax ? wn : (wn + 1) / 2;
    tq = tq < kTileQuadsMin ? kTileQuadsMin : (tq > kTileQuadsMax ? kTileQuadsMax : tq);
    // ceil(wn / tq): at most 2 unless tq is at its cap
    const int ntiles = tq == kTileQuadsMax ? (wn + kTileQuadsMax - 1) / kTileQuadsMax : (wn > tq ? 2 : 1);
    unsigned char *my_bufs = smem + lay.bufs + size_t(warp) * kBufs * kBufBytes;
    const int lead = wq0 < halo ? int(wq0) : halo;
    const int32_t *wsrc = ta + 4 * (P.q_lo + wq0);
    auto issue_tile = [&](int k, int slot) {             // lane 0 only
        const int t0 = k * tq;
        const int t1 = (t0 + tq < wn) ? t0 + tq : wn;
        const int ls = (t0 - halo > -lead) ? t0 - halo : -lead;
        const uint32_t bytes = uint32_t(t1 - ls) * 16u;
        unsigned char *buf = my_bufs + size_t(slot) * kBufBytes;
        const uint32_t bar = smem_addr(&my_bars[slot]);
        const int dq = kHaloQuads - (t0 - ls);           // first quad written in the buffer
        if (!LKD_OK(wq0 + ls >= 0 && wq0 + t1 <= P.nq && dq >= 0 && dq + (t1 - ls) <= kHaloQuads + kTileQuadsMax,
                    LOOKUP_DRAFT_CHECK_COPY)) {
            mbar_expect_tx(bar, 0u);                     // the phase completes with nothing copied
            return;
        }
        mbar_expect_tx(bar, bytes);
        bulk_copy_g2s_stream(smem_addr(buf + dq * 16), wsrc + ls * 4, bytes, bar);
    };
    if (wn > 0 && lane == 0) issue_tile(0, 0);

    __syncthreads();                                     // the offsets' barrier initialised before waiting
    const uint64_t deadline = sh_deadline;
    bool ok = true;
    if (offs_in_smem) ok = mbar_try_wait(smem_addr(offs_bar), 0) || mbar_wait_until(smem_addr(offs_bar), 0, deadline);
    const bool offs_smem = offs_in_smem && !__syncthreads_or(!ok);
    const bool offs_pending = offs_in_smem && !offs_smem;
    auto off_a = [&](int i) -> int64_t {
        if (!LKD_OK(i >= 0 && i <= B, LOOKUP_DRAFT_CHECK_INDEX)) i = 0;
        if (OFFS_SMEM && offs_smem) return offs_s[i] + shift;
        return __ldg(prm.offsets + i) + shift;
    };
    // Largest r in [lo, hi] with off_a(r) <= e, given off_a(lo) <= e: a 32-way
    // search, each lane testing one probe per round (warp-uniform result).
    auto owner = [&](int64_t e, int lo, int hi) -> int {
        while (hi > lo) {
            const int step = (hi - lo + 31) >> 5;
            const int probe = (lo + (lane + 1) * step < hi) ? lo + (lane + 1) * step : hi;
            const int cnt = __popc(__ballot_sync(0xffffffffu, off_a(probe) <= e));   // a prefix of lanes
            const int nlo = cnt == 0 ? lo : ((lo + cnt * step < hi) ? lo + cnt * step : hi);
            const int nhi = cnt == 32 ? hi : ((lo + (cnt + 1) * step < hi) ? lo + (cnt + 1) * step : hi) - 1;
            lo = nlo;
            hi = nhi;
        }
        return lo;
    };

    if (wn > 0) {                                        // warp-uniform: this warp has a range
        // The warp's range: elements [WA + wbeg, WA + wend) of the aligned view;
        // positions below are int32 relative to WA.
        const int64_t v = int64_t(c) * kWarps + warp;    // virtual chunk: slot column
        unsigned long long *slots = prm.slots + v;       // slot of request r: slots[r]
        const int64_t WA = 4 * (P.q_lo + wq0);
        const int wbeg = int(((WA > a_begin) ? WA : a_begin) - WA);
        const int wend = int(((4 * (P.q_lo + wq1) < a_end) ? 4 * (P.q_lo + wq1) : a_end) - WA);
        const int rw_lo = owner(WA + wbeg, 0, B - 1);

        // 4. Suffix tokens (row[j] = t[L-1-j], lane j) of requests rw_lo, rw_lo + 1, ...
        int64_t bound[kSufRows + 1];
#pragma unroll
        for (int row = 0; row <= kSufRows; ++row) bound[row] = off_a(rw_lo + row <= B ? rw_lo + row : B);
        int32_t sreg[kSufRows];
#pragma unroll
        for (int row = 0; row < kSufRows; ++row) {
            const int64_t src = bound[row + 1] - 1 - lane;
            const bool ld = rw_lo + row < B && lane < max_m && src >= bound[row] &&
                            LKD_OK(src >= a_begin && src < a_end, LOOKUP_DRAFT_CHECK_TOKENS);
            sreg[row] = ld ? __ldg(ta + src) : 0;
        }
        if (lane == 0) {
            const int first = ntiles < kBufs ? ntiles : kBufs;
            for (int k = 1; k < first; ++k) issue_tile(k, k);
        }
        const int rw_hi = owner(WA + wend - 1, rw_lo, B - 1);
        const int nrows = (rw_hi - rw_lo + 1 < kSufRows) ? rw_hi - rw_lo + 1 : kSufRows;
#pragma unroll
        for (int row = 0; row < kSufRows; ++row)
            if (row < nrows && lane < max_m) suf_w[row * max_m + lane] = sreg[row];
        // The slot of request r exists (checked build; the staircase keeps r + v below
        // B + the number of warp ranges).
        auto slot_ok = [&](int r) -> bool {
            return LKD_OK(r >= 0 && v + r < prm.nslots, LOOKUP_DRAFT_CHECK_SLOTS);
        };
        // this warp's slots: cleared before the warp writes its results into them
        for (int r = rw_lo + lane; r <= rw_hi; r += 32)
            if (off_a(r + 1) > off_a(r) && slot_ok(r)) slots[r] = 0ull;
        __syncwarp();

        // Suffix token j of request r (t[L-1-j]); 0 past the start of the history.
        auto suffix = [&](int r, int64_t o, int64_t n, int j) -> int32_t {
            const int row = r - rw_lo;
            if (!LKD_OK(row >= 0 && j >= 0 && j < max_m, LOOKUP_DRAFT_CHECK_SUFFIX)) return 0;
            if (row < kSufRows) return suf_w[row * max_m + j];
            return (n - 1 - j >= o && LKD_OK(n - 1 - j >= a_begin && n - 1 - j < a_end, LOOKUP_DRAFT_CHECK_TOKENS))
                       ? __ldg(ta + n - 1 - j)
                       : 0;
        };

        // 5. Stream the tiles.  The warp's current request (uniform across it) and
        //    each lane's best key for it carry over from tile to tile; the lanes'
        //    keys go into the request's slot when the warp moves on.
        int seg_r = rw_lo;                               // first request not yet finished
        int cur_r = -1;                                  // request of the cached state below
        int cur_o = 0, cur_nxt = 0;                      // its start and end, relative to WA
        int32_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
        unsigned long long best = 0ull;
        // A lane's best key goes into the request's slot with an atomic max (no
        // value returned, so nothing waits for it): the slot was zeroed above and
        // only this warp's lanes write it.
        auto flush = [&]() {
            if (best != 0ull && slot_ok(cur_r)) atomicMax(&slots[cur_r], best);
            best = 0ull;
        };
        auto set_request = [&](int r) {                  // warp-uniform, r in [rw_lo, rw_hi]
            if (r == cur_r) return;
            flush();
            cur_r = r;
            const int64_t o = off_a(r), n = off_a(r + 1);
            cur_o = int(o - WA);
            cur_nxt = int(n - WA);
            s0 = suffix(r, o, n, 0);
            if (D >= 2) s1 = suffix(r, o, n, 1);
            if (D >= 3) s2 = suffix(r, o, n, 2);
            if (D >= 4) s3 = suffix(r, o, n, 3);
        };
        set_request(rw_lo);
        int k = 0;
        for (; k < ntiles; ++k) {
            const int slot = k % kBufs;
            const uint32_t bar = smem_addr(&my_bars[slot]);
            const uint32_t parity = uint32_t(k / kBufs) & 1u;
            if (!mbar_try_wait(bar, parity) && !mbar_wait_until(bar, parity, deadline)) {
                failed = true;
                break;
            }
            const int t0 = k * tq;                       // tile's first quad, relative
            const int nq = (t0 + tq < wn) ? tq : wn - t0;
            const unsigned char *buf = my_bufs + size_t(slot) * kBufBytes + kHaloQuads * 16;
            const int4 *sq = reinterpret_cast<const int4 *>(buf);
            const int32_t *st = reinterpret_cast<const int32_t *>(buf);
            const int base = 4 * t0;                     // relative position of st[0]
            const int eb = base > wbeg ? base : wbeg;
            const int ee = (base + 4 * nq < wend) ? base + 4 * nq : wend;
#if LOOKUP_DRAFT_CHECKED
            const int qv = ((t0 - halo > -lead) ? t0 - halo : -lead) - t0;   // quads [qv, nq) were copied
#endif
            // Checked build: the tokens that the tests of candidate ends [lo, hi] depend
            // on (lo - D + 1 .. hi; the loops also load the rest of the quad before
            // lo's, whose masked values never count) lie in the tile's copied bytes;
            // a match ending at element e can be extended up to kmax tokens in them.
            auto tile_ok = [&](int lo, int hi) -> bool {
                return LKD_OK(((lo - (D - 1)) >> 2) >= qv && (hi >> 2) < nq, LOOKUP_DRAFT_CHECK_TILE);
            };
            auto elem_ok = [&](int e, int kmax) -> bool {
                return LKD_OK(kmax <= max_m, LOOKUP_DRAFT_CHECK_SUFFIX) &&
                       LKD_OK(e < 4 * nq && e - (kmax - 1) >= 4 * qv, LOOKUP_DRAFT_CHECK_TILE);
            };

            // Candidate ends [lo, hi] (tile elements, whole quads: lo and hi + 1 are
            // multiples of 4) of the current request: the D-token test on every quad.
            auto scan_range = [&](int lo, int hi) {
                const int qoff = base - cur_o;           // local position of st[0] in the request
                // Candidate end at tile element e whose last k0 tokens already
                // match: extend backwards, fold its key into `best`.
                auto extend = [&](int e, int k0) {
                    const int q = qoff + e;              // local end position in the request
                    const int kmax = max_m < q + 1 ? max_m : q + 1;
                    const int row = cur_r - rw_lo;
                    if (!elem_ok(e, kmax)) return;
                    int kk = k0;
                    if (row < kSufRows)
                        kk = match_len(st, e, suf_w + row * max_m, k0, kmax);
                    else
                        while (kk < kmax && st[e - kk] == suffix(cur_r, WA + cur_o, WA + cur_nxt, kk)) ++kk;
                    if (kk >= min_m) {
                        const unsigned long long key =
                            (static_cast<unsigned long long>(kk) << 32) | static_cast<uint32_t>(q - kk + 1);
                        best = key > best ? key : best;
                    }
                };
                auto extend_quad = [&](const int4 &p, const int4 &cq, int j) {   // rare path
                    unsigned h = quad_hits<D>(p, cq, s0, s1, s2, s3);
                    while (h) {
                        const int e = __ffs(h) - 1;
                        h &= h - 1;
                        extend(4 * j + e, D);
                    }
                };
                const int jq0 = (lo + 3) >> 2;           // first quad fully inside
                const int jq1 = ((hi + 1) >> 2) - 1;     // last quad fully inside
                if (jq0 <= jq1 && !tile_ok(4 * jq0, 4 * jq1 + 3)) return;
                // two quads per lane per iteration: independent loads and tests; the
                // previous quad (the halo when j == 0) supplies the tokens before each
                int j = jq0 + lane;
                for (; j + 32 <= jq1; j += 64) {
                    const int4 c0 = sq[j], c1 = sq[j + 32];
                    int4 p0 = make_int4(0, 0, 0, 0), p1 = make_int4(0, 0, 0, 0);
                    if (D >= 2) {
                        p0 = sq[j - 1];
                        p1 = sq[j + 31];
                    }
                    if (quad_any<D>(p0, c0, s0, s1, s2, s3) | quad_any<D>(p1, c1, s0, s1, s2, s3)) {
                        extend_quad(p0, c0, j);
                        extend_quad(p1, c1, j + 32);
                    }
                }
                if (j <= jq1) {
                    const int4 c0 = sq[j];
                    int4 p0 = make_int4(0, 0, 0, 0);
                    if (D >= 2) p0 = sq[j - 1];
                    if (quad_any<D>(p0, c0, s0, s1, s2, s3)) extend_quad(p0, c0, j);
                }
            };

            // Candidate ends [lo, hi] (tile elements) of the current request that cover
            // quads only in part (a tile shared by requests): one pass over every quad
            // the range touches, two per lane, the D-token test masked to the range.
            auto scan_partial = [&](int lo, int hi) {
                const int qoff = base - cur_o;           // local position of st[0] in the request
                const int row = cur_r - rw_lo;
                const int32_t *suf = row < kSufRows ? suf_w + row * max_m : nullptr;
                const int32_t *hist_last = ta + (WA + cur_nxt) - 1;
                auto extend = [&](int e) {               // the D tokens ending at e match
                    const int q = qoff + e;
                    const int kmax = max_m < q + 1 ? max_m : q + 1;
                    if (!elem_ok(e, kmax)) return;
                    int kk = D;
                    if (suf)
                        kk = match_len(st, e, suf, D, kmax);
                    else
                        while (kk < kmax &&
                               LKD_OK(cur_nxt - 1 - kk >= cur_o && WA + cur_nxt - 1 - kk < a_end,
                                      LOOKUP_DRAFT_CHECK_TOKENS) &&
                               st[e - kk] == __ldg(hist_last - kk))
                            ++kk;
                    if (kk >= min_m) {
                        const unsigned long long key =
                            (static_cast<unsigned long long>(kk) << 32) | static_cast<uint32_t>(q - kk + 1);
                        best = key > best ? key : best;
                    }
                };
                const int ja = lo >> 2, jb = hi >> 2;
                if (lo <= hi && !tile_ok(lo, hi)) return;
                const unsigned head = (0xFu << (lo & 3)) & 0xFu;   // elements >= lo in quad ja
                const unsigned tail = 0xFu >> (3 - (hi & 3));      // elements <= hi in quad jb
                for (int j = ja + lane; j <= jb; j += 64) {
                    const int j2 = j + 32;
                    const bool has2 = j2 <= jb;
                    const int jj2 = has2 ? j2 : jb;
                    const int4 c0 = sq[j], c1 = sq[jj2];
                    int4 p0 = make_int4(0, 0, 0, 0), p1 = make_int4(0, 0, 0, 0);
                    if (D >= 2) {
                        p0 = sq[j - 1];
                        p1 = sq[jj2 - 1];
                    }
                    const unsigned m0 = (j == ja ? head : 0xFu) & (j == jb ? tail : 0xFu);
                    const unsigned m1 = has2 ? (j2 == jb ? tail : 0xFu) : 0u;
                    unsigned h0 = quad_hits<D>(p0, c0, s0, s1, s2, s3) & m0;
                    unsigned h1 = quad_hits<D>(p1, c1, s0, s1, s2, s3) & m1;
                    while (h0) {
                        const int e = __ffs(h0) - 1;
                        h0 &= h0 - 1;
                        extend(4 * j + e);
                    }
                    while (h1) {
                        const int e = __ffs(h1) - 1;
                        h1 &= h1 - 1;
                        extend(4 * j2 + e);
                    }
                }
            };

            if (cur_r >= 0 && eb == base && ee == base + 4 * nq && cur_o + (min_m - 1) <= eb &&
                ee + 1 <= cur_nxt) {
                scan_range(0, 4 * nq - 1);               // the whole tile is candidates of cur_r
            } else {
                // Requests overlapping this tile, in order (uniform across the warp).
                while (seg_r < rw_hi && off_a(seg_r + 1) - WA <= eb) ++seg_r;
                // The common shared tile: request A = seg_r ends in it and B = seg_r + 1
                // reaches past its end.  With D >= 3, A's last candidate end and B's
                // first are more than 4 elements apart, so no quad holds candidates of
                // both: one pass over every quad of both ranges, each tested with its
                // own request's suffix.
                const int rA = seg_r, rB = seg_r + 1;
                const int oA = int(off_a(rA) - WA), nA = int(off_a(rA + 1) - WA);
                const int nB = rB <= rw_hi ? int(off_a(rB + 1) - WA) : nA;
                if (D >= 3 && rB <= rw_hi && nA < ee && nB >= ee && nB > nA) {
                    flush();                             // the keys pending for cur_r
                    const int oB = nA;
                    const int loA = ((oA + (min_m - 1) > eb) ? oA + (min_m - 1) : eb) - base;
                    const int hiA = ((nA - 2 < ee - 1) ? nA - 2 : ee - 1) - base;
                    const int loB = ((oB + (min_m - 1) > eb) ? oB + (min_m - 1) : eb) - base;
                    const int hiB = ((nB - 2 < ee - 1) ? nB - 2 : ee - 1) - base;
                    const int32_t a0 = suffix(rA, WA + oA, WA + nA, 0), a1 = suffix(rA, WA + oA, WA + nA, 1),
                                  a2 = suffix(rA, WA + oA, WA + nA, 2);
                    const int32_t a3 = D >= 4 ? suffix(rA, WA + oA, WA + nA, 3) : 0;
                    const int32_t b0 = suffix(rB, WA + oB, WA + nB, 0), b1 = suffix(rB, WA + oB, WA + nB, 1),
                                  b2 = suffix(rB, WA + oB, WA + nB, 2);
                    const int32_t b3 = D >= 4 ? suffix(rB, WA + oB, WA + nB, 3) : 0;
                    // candidate end at tile element e of A or B whose last D tokens match
                    unsigned long long bestA = 0ull, bestB = 0ull;
                    auto extend2 = [&](int e, bool inB) {
                        const int r = inB ? rB : rA;
                        const int q = base + e - (inB ? oB : oA);      // local end position
                        const int kmax = max_m < q + 1 ? max_m : q + 1;
                        const int64_t o_abs = WA + (inB ? oB : oA), n_abs = WA + (inB ? nB : nA);
                        if (!elem_ok(e, kmax)) return;
                        int kk = D;
                        if (r - rw_lo < kSufRows)
                            kk = match_len(st, e, suf_w + (r - rw_lo) * max_m, D, kmax);
                        else
                            while (kk < kmax && st[e - kk] == suffix(r, o_abs, n_abs, kk)) ++kk;
                        if (kk >= min_m) {
                            const unsigned long long key =
                                (static_cast<unsigned long long>(kk) << 32) | static_cast<uint32_t>(q - kk + 1);
                            if (inB) bestB = key > bestB ? key : bestB;
                            else bestA = key > bestA ? key : bestA;
                        }
                    };
                    // every quad the two ranges touch, once: a quad holds candidate ends of
                    // A or of B, never of both (D >= 3 leaves 3 elements between A's last
                    // and B's first), so it is tested with that request's suffix and its
                    // rare hits are masked to that request's range
                    const bool hasA = loA <= hiA, hasB = loB <= hiB;
                    const int jlo = (hasA ? loA : loB) >> 2, jhi = (hasB ? hiB : hiA) >> 2;
                    const bool pass_ok = (!hasA && !hasB) || tile_ok(hasA ? loA : loB, hasB ? hiB : hiA);
                    // a quad is B's when it reaches B's first candidate (the gap before it
                    // is at least 3 elements), else A's; the range masks apply on the rare
                    // path only, so a gap or edge quad costs nothing extra
                    auto test2 = [&](int j, const int4 &p, const int4 &c) {
                        const bool inB = hasB && 4 * j + 3 >= loB;
                        unsigned h = quad_hits<D>(p, c, inB ? b0 : a0, inB ? b1 : a1, inB ? b2 : a2, inB ? b3 : a3) &
                                     range_mask(4 * j, inB ? loB : loA, inB ? hiB : hiA);
                        if (!inB && !hasA) h = 0u;
                        while (h) {
                            const int e = __ffs(h) - 1;
                            h &= h - 1;
                            extend2(4 * j + e, inB);
                        }
                    };
                    for (int j = jlo + lane; pass_ok && j <= jhi; j += 64) {
                        const int j2 = j + 32;
                        const bool has2 = j2 <= jhi;
                        const int jj2 = has2 ? j2 : j;
                        const int4 c0 = sq[j], c1 = sq[jj2], p0 = sq[j - 1], p1 = sq[jj2 - 1];
                        const bool b0q = hasB && 4 * j + 3 >= loB, b1q = hasB && 4 * j2 + 3 >= loB;
                        const bool any0 =
                            quad_any<D>(p0, c0, b0q ? b0 : a0, b0q ? b1 : a1, b0q ? b2 : a2, b0q ? b3 : a3);
                        const bool any1 =   // the test runs either way: no branch on has2
                            quad_any<D>(p1, c1, b1q ? b0 : a0, b1q ? b1 : a1, b1q ? b2 : a2, b1q ? b3 : a3) & has2;
                        if (any0 | any1) {
                            if (any0) test2(j, p0, c0);
                            if (any1) test2(j2, p1, c1);
                        }
                    }
                    // A ends here; B continues into the next tile with its keys pending
                    if (bestA != 0ull && slot_ok(rA)) atomicMax(&slots[rA], bestA);
                    cur_r = rB;
                    cur_o = oB;
                    cur_nxt = nB;
                    s0 = b0;
                    s1 = b1;
                    s2 = b2;
                    s3 = b3;
                    best = bestB;
                } else for (int r = seg_r; r <= rw_hi; ++r) {
                    const int o_r = int(off_a(r) - WA);
                    if (o_r >= ee) break;
                    const int nxt = int(off_a(r + 1) - WA);
                    const int lo = (o_r + (min_m - 1) > eb) ? o_r + (min_m - 1) : eb;   // candidate end range
                    const int hi = (nxt - 2 < ee - 1) ? nxt - 2 : ee - 1;               // within this tile
                    if (lo > hi) continue;
                    set_request(r);
                    scan_partial(lo - base, hi - base);
                }
            }
            // Refill this buffer with the warp's tile k + kBufs.
            __syncwarp();
            if (lane == 0 && k + kBufs < ntiles) {
                fence_proxy_async_smem();
                issue_tile(k + kBufs, slot);
            }
        }
        if (!failed) {
            flush();                                     // the last request's result
        } else {
            // 6. A wait ran out: let this warp's copies land (bounded), then mark
            //    its requests as failed.  Copies k .. min(k + kBufs, ntiles) - 1 may
            //    still be in flight.
            if (lane == 0) {
                const uint64_t drain_deadline = global_ns() + kDefaultWaitNs;
                const int stop = (k + kBufs < ntiles) ? k + kBufs : ntiles;
                for (int kk = k; kk < stop; ++kk)
                    (void)mbar_wait_until(smem_addr(&my_bars[kk % kBufs]), uint32_t(kk / kBufs) & 1u,
                                          drain_deadline);
            }
            __syncwarp();
            for (int r = rw_lo + lane; r <= rw_hi; r += 32)
                if (off_a(r + 1) > off_a(r) && slot_ok(r)) slots[r] = kKeyFailed;
        }
    }
    if (offs_pending && tid == 0) (void)mbar_wait_until(smem_addr(offs_bar), 0, global_ns() + kDefaultWaitNs);
}

// ------------------------------------------------------------ fill kernel ----
// The outputs of request r (history start o0, length L) from its reduced key.  A
// key that does not describe an admissible match (1 <= m, p + m <= L - 1) can only
// come from a failed scan; it is reported as such and never dereferenced.  Draft
// token j is t[p + m + (j mod d)], d = L - p - m >= 1: the history extended by
// its own draft.  Lanes first, first + step, ... of the row are written here.
__device__ inline void write_draft(const FillParams &prm, int r, int64_t o0, int64_t L, unsigned long long key,
                                   int first, int step, bool head) {
    if (!LKD_OK(r >= 0 && r < prm.B, LOOKUP_DRAFT_CHECK_OUTPUT)) return;
    const int64_t km = int64_t(key >> 32), kp = int64_t(uint32_t(key));
    const bool failed = key != 0ull && (key == kKeyFailed || km < 1 || kp + km > L - 1);
    const bool found = key != 0ull && !failed;
    const int32_t m = found ? int32_t(km) : 0;
    const int64_t p = found ? kp : -1;
    const int d = found ? int(L - p - m) : 1;            // L < 2^31
    const int K = prm.K;
    int32_t *row = prm.out_draft + int64_t(r) * K;
    const int32_t *src = prm.tokens + o0 + p + m;
    for (int j = first; j < K; j += step)
        row[j] = found && LKD_OK(p + m + (j < d ? j : j % d) < L, LOOKUP_DRAFT_CHECK_TOKENS)
                     ? __ldg(src + (j < d ? j : j % d))
                     : -1;
    if (head) {
        prm.out_len[r] = found ? K : (failed ? LOOKUP_DRAFT_LEN_FAILED : 0);
        prm.out_pos[r] = int32_t(p);
        if (prm.out_mlen) prm.out_mlen[r] = m;
    }
}

#if LOOKUP_DRAFT_CHECKED
// Checked build: whether the offsets are not a valid CSR (offsets[0] < 0, a
// decreasing pair, a history of 2^31 tokens or more).  Every thread of the CTA
// takes part; the answer is the CTA's.
__device__ bool offsets_invalid(const int64_t *offsets, int B) {
    bool bad = false;
    for (int i = threadIdx.x; i <= B; i += blockDim.x) {
        const int64_t a = offsets[i];
        bad |= i == 0 && a < 0;
        if (i < B) {
            const int64_t b = offsets[i + 1];
            bad |= b < a || b - a >= (int64_t(1) << 31);
        }
    }
    bad = __syncthreads_or(bad) != 0;
    if (bad && threadIdx.x == 0) atomicOr(&g_check_word, LOOKUP_DRAFT_CHECK_OFFSETS);
    return bad;
}

#endif

// One warp per request, for small batches: the request's slots lie in the scan
// warps v0 .. v1 holding its first and last quads, and the lanes load them in
// parallel.  The reduced key (in every lane) goes to tail(r, lane, o0, L, key),
// which writes the request's outputs; invalid offsets (checked build) arrive as a
// failed key.
template <class Tail>
__device__ __forceinline__ void fold_request(const FillParams &prm, Tail &&tail) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kFillWarps + (threadIdx.x >> 5);
#if LOOKUP_DRAFT_CHECKED
    const bool csr_bad = offsets_invalid(prm.offsets, prm.B);
#else
    constexpr bool csr_bad = false;
#endif
    // Inputs the scan does not write: read them before waiting for it.
    int64_t o0 = 0, o1 = 0, first = 0, end = 0;
    if (r < prm.B && !csr_bad) {
        o0 = __ldg(prm.offsets + r);
        o1 = __ldg(prm.offsets + r + 1);
        first = __ldg(prm.offsets);
        end = __ldg(prm.offsets + prm.B);
    }
    const int shift = tokens_shift(prm.tokens);
    const int64_t L = o1 - o0;
    // The request's slots are those of warps v0 .. v1, the ones holding its first
    // and last quads (empty warp ranges own none).  All of that follows from the
    // offsets, so it is worked out before the wait, with which of the first round's
    // loads to make.
    Partition P{};
    int64_t v0 = 0, v1 = -1;
    if (r < prm.B && L > 0) {
        P = make_partition(first + shift, end + shift, prm.grid);
        v0 = vchunk_of_quad(P, ((o0 + shift) >> 2) - P.q_lo);
        v1 = vchunk_of_quad(P, ((o1 - 1 + shift) >> 2) - P.q_lo);
    }
    bool take[kFillUnroll];
#pragma unroll
    for (int u = 0; u < kFillUnroll; ++u) {
        const int64_t v = v0 + lane + u * 32;
        int64_t lo = 0, hi = 0;
        if (v <= v1) vchunk_range(P, v, lo, hi);
        take[u] = v <= v1 && lo < hi && LKD_OK(int64_t(r) + v < prm.nslots, LOOKUP_DRAFT_CHECK_SLOTS);
    }
    allow_dependent_launch();
    wait_for_prerequisite_grid();
    if (r >= prm.B) return;
#if LOOKUP_DRAFT_CHECKED
    if (csr_bad) {
        tail(r, lane, int64_t(0), int64_t(0), kKeyFailed);
        return;
    }
#endif

    unsigned long long key = 0ull;
    if (L > 0) {
        // Lane i folds the slots of warps v0 + i, v0 + i + 32, ...: kFillUnroll
        // independent loads at a time.
        unsigned long long x[kFillUnroll];
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) x[u] = take[u] ? prm.slots[int64_t(r) + v0 + lane + u * 32] : 0ull;
#pragma unroll
        for (int u = 0; u < kFillUnroll; ++u) key = x[u] > key ? x[u] : key;
        for (int64_t vb = v0 + lane + kFillUnroll * 32; vb <= v1; vb += kFillUnroll * 32) {   // long requests
#pragma unroll
            for (int u = 0; u < kFillUnroll; ++u) {
                const int64_t v = vb + u * 32;
                int64_t lo, hi;
                vchunk_range(P, v, lo, hi);
                x[u] = (v <= v1 && lo < hi && LKD_OK(int64_t(r) + v < prm.nslots, LOOKUP_DRAFT_CHECK_SLOTS))
                           ? prm.slots[int64_t(r) + v]
                           : 0ull;
            }
#pragma unroll
            for (int u = 0; u < kFillUnroll; ++u) key = x[u] > key ? x[u] : key;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xffffffffu, key, o);
            key = x > key ? x : key;
        }
    }
    tail(r, lane, o0, L, key);
}

__global__ void __launch_bounds__(kFillWarps * 32, kFillMinBlocks) fill_kernel(FillParams prm) {
    fold_request(prm, [&](int r, int lane, int64_t o0, int64_t L, unsigned long long key) {
        write_draft(prm, r, o0, L, key, lane, 32, lane == 0);
    });
}

// ------------------------------------------------- draft, then schedule and fuse ----
// The decode loop's next two steps on the fill's result, in the fill's warp:
// long-block scheduling and fusion with the draft model's head (HyperQwen
// lookup-drafting article, sections "第3步" and "第2步"), the rules lookup_plan
// applies, on the draft lookup_draft_ex would write (K = H + T <= 64).
struct PlanArgs {
    lkd::PlanIO io;
    int32_t *out_mlen;            // may be null
    int32_t *out_draft_len;       // may be null
};

__global__ void __launch_bounds__(kFillWarps * 32, kFillMinBlocks) fill_plan_kernel(FillParams prm, PlanArgs pa) {
    // The rules' own inputs (the model's proposals, the commit count, the state)
    // are not written by the scan, this kernel's only predecessor in the call, and
    // everything before the scan had completed when it let this kernel launch: read
    // them now, before the wait inside fold_request.
    const int rq = blockIdx.x * kFillWarps + (threadIdx.x >> 5);
    lkd::PlanIn in{};
    if (rq < prm.B) in = lkd::plan_load(pa.io, rq, threadIdx.x & 31);
    fold_request(prm, [&](int r, int lane, int64_t o0, int64_t L, unsigned long long key) {
        const int64_t km = int64_t(key >> 32), kp = int64_t(uint32_t(key));
        const bool failed = key != 0ull && (key == kKeyFailed || km < 1 || kp + km > L - 1);
        const bool found = key != 0ull && !failed;
        const int32_t m = found ? int32_t(km) : 0;
        const int64_t p = found ? kp : 0;
        const int d = found ? int(L - p - m) : 1;
        const int W = pa.io.H + pa.io.T;
        // Draft tokens lane and lane + 32 (-1 without a match), as write_draft forms them.
        const int32_t *src = prm.tokens + o0 + p + m;
        const int j1 = lane + 32;
        const int32_t tok0 = (found && lane < W && LKD_OK(p + m + (lane < d ? lane : lane % d) < L,
                                                          LOOKUP_DRAFT_CHECK_TOKENS))
                                 ? __ldg(src + (lane < d ? lane : lane % d))
                                 : -1;
        const int32_t tok1 = (found && j1 < W && LKD_OK(p + m + (j1 < d ? j1 : j1 % d) < L, LOOKUP_DRAFT_CHECK_TOKENS))
                                 ? __ldg(src + (j1 < d ? j1 : j1 % d))
                                 : -1;
        lkd::plan_apply(pa.io, r, lane, m, tok0, tok1, in);
        if (lane == 0) {
            if (pa.out_mlen) pa.out_mlen[r] = m;
            if (pa.out_draft_len) pa.out_draft_len[r] = found ? W : (failed ? LOOKUP_DRAFT_LEN_FAILED : 0);
        }
    });
}

// One request per lane, for large batches: there most requests' slots lie in one
// or two scan warps, and a warp per request would spend its issue slots on idle
// lanes.  A lane folds up to kLaneCover slots itself; the few requests whose
// slots span more scan warps are folded by the whole warp, one at a time.
__global__ void __launch_bounds__(kLaneFillThreads) fill_lanes_kernel(FillParams prm) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kLaneFillThreads + threadIdx.x;
#if LOOKUP_DRAFT_CHECKED
    const bool csr_bad = offsets_invalid(prm.offsets, prm.B);
#else
    constexpr bool csr_bad = false;
#endif
    const bool live = r < prm.B;
    int64_t o0 = 0, o1 = 0;
    if (live && !csr_bad) {
        o0 = __ldg(prm.offsets + r);
        o1 = __ldg(prm.offsets + r + 1);
    }
    const int64_t first = __ldg(prm.offsets);
    const int64_t end = __ldg(prm.offsets + prm.B);
    const int shift = tokens_shift(prm.tokens);
    const int64_t L = o1 - o0;
    // The request's scan warps and which of them own a slot follow from the
    // offsets alone: worked out before the wait.
    const Partition P = make_partition(first + shift, end + shift, prm.grid);
    int64_t v0 = 0, v1 = -1;                             // no slots: empty request or no request
    if (L > 0 && !csr_bad) {
        v0 = vchunk_of_quad(P, ((o0 + shift) >> 2) - P.q_lo);
        v1 = vchunk_of_quad(P, ((o1 - 1 + shift) >> 2) - P.q_lo);
    }
    const bool own = v1 - v0 < kLaneCover;
    bool take[kLaneCover];
#pragma unroll
    for (int u = 0; u < kLaneCover; ++u) {
        const int64_t v = v0 + u;
        int64_t lo = 0, hi = 0;
        if (own && v <= v1) vchunk_range(P, v, lo, hi);
        take[u] = own && v <= v1 && lo < hi && LKD_OK(int64_t(r) + v < prm.nslots, LOOKUP_DRAFT_CHECK_SLOTS);
    }
    allow_dependent_launch();
    wait_for_prerequisite_grid();
#if LOOKUP_DRAFT_CHECKED
    if (csr_bad) {
        if (live) write_draft(prm, r, 0, 0, kKeyFailed, 0, 1, true);   // every output marked failed
        return;
    }
#endif
    if (__all_sync(0xffffffffu, !live)) return;          // warp-uniform

    unsigned long long key = 0ull;
    if (own) {
        unsigned long long x[kLaneCover];
#pragma unroll
        for (int u = 0; u < kLaneCover; ++u) x[u] = take[u] ? prm.slots[int64_t(r) + v0 + u] : 0ull;
#pragma unroll
        for (int u = 0; u < kLaneCover; ++u) key = x[u] > key ? x[u] : key;
    }
    for (unsigned wide = __ballot_sync(0xffffffffu, !own); wide != 0u; wide &= wide - 1) {
        const int src = __ffs(int(wide)) - 1;
        const int64_t a = __shfl_sync(0xffffffffu, v0, src);
        const int64_t b = __shfl_sync(0xffffffffu, v1, src);
        const int rs = __shfl_sync(0xffffffffu, r, src);
        unsigned long long kw = 0ull;
        for (int64_t v = a + lane; v <= b; v += 32) {
            int64_t lo, hi;
            vchunk_range(P, v, lo, hi);
            const unsigned long long x =
                (lo < hi && LKD_OK(int64_t(rs) + v < prm.nslots, LOOKUP_DRAFT_CHECK_SLOTS)) ? prm.slots[int64_t(rs) + v]
                                                                                           : 0ull;
            kw = x > kw ? x : kw;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long x = __shfl_xor_sync(0xffffffffu, kw, o);
            kw = x > kw ? x : kw;
        }
        if (lane == src) key = kw;
    }
    if (live) write_draft(prm, r, o0, L, key, 0, 1, true);
}

// ------------------------------------------------------ host-input copy ----
// lookup_draft_host with page-locked inputs: the device reads the batch straight
// from host memory over the host link, with 16-byte loads, kCopyUnroll of them in
// flight per thread, and writes the device copies the scan reads.  A kernel starts
// sooner than a copy-engine transfer, and the scan behind it is launched while it
// runs (programmatic dependent launch) and only waits for its results.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopyCtasPerSm = 2;      // fit beside a scan CTA (its registers leave room for two)

struct CopyParams {
    const int4 *src;                   // host memory the device can address, 16-byte units
    int4 *dst;                         // device
    int64_t n16;
    const int64_t *src_off;            // host offsets (B + 1 of them), device-addressable
    int64_t *dst_off;
    int32_t n_off;
};

__global__ void __launch_bounds__(kCopyThreads) host_copy_kernel(CopyParams prm) {
    allow_dependent_launch();
    wait_for_prerequisite_grid();      // the destination is stream-ordered scratch
    const int64_t stride = int64_t(gridDim.x) * kCopyThreads;
    const int64_t t = int64_t(blockIdx.x) * kCopyThreads + threadIdx.x;
    for (int64_t i = t; i < prm.n_off; i += stride) prm.dst_off[i] = prm.src_off[i];
    int64_t i = t;
    for (; i + (kCopyUnroll - 1) * stride < prm.n16; i += kCopyUnroll * stride) {
        int4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) v[u] = prm.src[i + u * stride];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) prm.dst[i + u * stride] = v[u];
    }
    for (; i < prm.n16; i += stride) prm.dst[i] = prm.src[i];
}

// ------------------------------------------------------------- host side ----
}  // namespace

#include <unordered_map>                       // per-stream scratch (host code only)

namespace {

thread_local char g_cuda_msg[256] = "";

int cuda_fail(cudaError_t e, const char *what) {
    std::snprintf(g_cuda_msg, sizeof g_cuda_msg, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
    return LOOKUP_DRAFT_ECUDA;
}

#define LD_CUDA(call)                                  \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

// The device address of page-locked host memory the device can address, else
// nullptr (pageable or unknown memory).
const void *mapped_host_const(const void *p) {
    if (!p) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();                              // clear the error state of the query
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

int32_t *mapped_host(int32_t *p) { return static_cast<int32_t *>(const_cast<void *>(mapped_host_const(p))); }

// Every scan instantiation may use the shared memory of the largest batch the
// offsets copy serves and the largest max_m (more than the 48 KB default).
int scan_attributes() {
    const int smem_max = int(scan_smem_layout(kOffCap - 1, LOOKUP_DRAFT_MAX_M).total);
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<3, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<3, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    LD_CUDA(cudaFuncSetAttribute(scan_kernel<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max));
    return LOOKUP_DRAFT_OK;
}

struct DeviceState {
    std::atomic<bool> ready{false};     // set (release) once the fields below are final
    int sms = 0;
    cudaMemPool_t pool = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device set-up, once: SM count, shared-memory opt-in, scratch pool.  After
// it, a call only reads the ready flag; the lock is taken for the set-up alone.
int device_state(DeviceState **out) {
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
    DeviceState &st = g_dev[dev];
    if (st.ready.load(std::memory_order_acquire)) {
        *out = &st;
        return LOOKUP_DRAFT_OK;
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
        int sms = 0;
        LD_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        const int rc_attr = scan_attributes();
        if (rc_attr != LOOKUP_DRAFT_OK) return rc_attr;
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        LD_CUDA(cudaMemPoolCreate(&pool, &props));
        uint64_t keep = ~0ull;                         // keep freed scratch for reuse
        LD_CUDA(cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep));
        st.sms = sms;
        st.pool = pool;
        st.ready.store(true, std::memory_order_release);
    }
    *out = &st;
    return LOOKUP_DRAFT_OK;
}

// One scan CTA per SM (its shared-memory rings admit no second one).
int grid_for(const DeviceState &st) { return st.sms; }

// Division of n < 2^31 by the grid size G >= 2 as a multiply-high and a shift:
// magic = ceil(2^k / G) with k = 31 + ceil(log2 G), so that magic < 2^32 and
// n * magic / 2^k = n / G + n * err / (G * 2^k), err < G, stays below the next
// integer whenever n * G <= 2^k (the method of division by invariant integers).
void grid_divider(int G, uint32_t &magic, int32_t &shift) {
    if (G <= 1) {
        magic = 0;
        shift = -1;
        return;
    }
    int l = 0;
    while ((int64_t(1) << l) < G) ++l;
    const int k = 31 + l;
    magic = uint32_t(((uint64_t(1) << k) + uint64_t(G) - 1) / uint64_t(G));
    shift = k - 32;
}

// One 64-bit slot per (request, virtual chunk) pair on the staircase: at most
// B + (number of virtual chunks) of them.
size_t workspace_bytes_for(int32_t B, int grid) {
    return (size_t(B) + size_t(grid) * kWarps) * sizeof(unsigned long long);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_common(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                 int32_t K) {
    if (B < 0 || min_m < 1 || max_m < min_m || max_m > LOOKUP_DRAFT_MAX_M || K < 0 || K > LOOKUP_DRAFT_MAX_K)
        return LOOKUP_DRAFT_EINVAL;
    if (B > 0 && (!tokens || !offsets || !aligned(tokens, 4) || !aligned(offsets, 8))) return LOOKUP_DRAFT_EINVAL;
    if (B > INT32_MAX - 65536) return LOOKUP_DRAFT_EINVAL;
    return LOOKUP_DRAFT_OK;
}

int check_outputs(int32_t B, int32_t K, const int32_t *out_draft, const int32_t *out_len, const int32_t *out_pos,
                  const int32_t *out_mlen) {
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!out_len || !out_pos || (K > 0 && !out_draft)) return LOOKUP_DRAFT_EINVAL;
    if (!aligned(out_len, 4) || !aligned(out_pos, 4) || (out_draft && !aligned(out_draft, 4)) ||
        (out_mlen && !aligned(out_mlen, 4)))
        return LOOKUP_DRAFT_EINVAL;
    return LOOKUP_DRAFT_OK;
}

int launch_scan(const DeviceState &st, const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m,
                int32_t max_m, unsigned long long *slots, cudaStream_t stream) {
    ScanParams prm;
    prm.tokens = tokens;
    prm.offsets = offsets;
    prm.slots = slots;
    prm.B = B;
    prm.min_m = min_m;
    prm.max_m = max_m;
    prm.grid = grid_for(st);
    grid_divider(prm.grid, prm.grid_magic, prm.grid_shift);
    prm.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
#if LOOKUP_DRAFT_CHECKED
    prm.nslots = int64_t(B) + int64_t(prm.grid) * kWarps;
#endif
    const ScanSmemLayout lay = scan_smem_layout(B, max_m);
    const bool offs_smem = int64_t(B) + 1 <= kOffCap;
    void (*kernel)(ScanParams) = nullptr;
    switch ((min_m < 4 ? min_m : 4) * 2 + (offs_smem ? 1 : 0)) {
    case 2: kernel = scan_kernel<1, false>; break;
    case 3: kernel = scan_kernel<1, true>; break;
    case 4: kernel = scan_kernel<2, false>; break;
    case 5: kernel = scan_kernel<2, true>; break;
    case 6: kernel = scan_kernel<3, false>; break;
    case 7: kernel = scan_kernel<3, true>; break;
    case 8: kernel = scan_kernel<4, false>; break;
    default: kernel = scan_kernel<4, true>; break;
    }
    return launch_pdl(kernel, unsigned(prm.grid), unsigned(kThreads), stream, prm, lay.total);
}

int launch_fill(const DeviceState &st, const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t K,
                const unsigned long long *slots, int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                int32_t *out_mlen, cudaStream_t stream) {
    FillParams prm;
    prm.tokens = tokens;
    prm.offsets = offsets;
    prm.slots = slots;
    prm.out_draft = out_draft;
    prm.out_len = out_len;
    prm.out_pos = out_pos;
    prm.out_mlen = out_mlen;
    prm.B = B;
    prm.K = K;
    prm.grid = grid_for(st);
#if LOOKUP_DRAFT_CHECKED
    prm.nslots = int64_t(B) + int64_t(prm.grid) * kWarps;
#endif
    if (B >= kLaneFillMinB)
        return launch_pdl(fill_lanes_kernel, unsigned((int64_t(B) + kLaneFillThreads - 1) / kLaneFillThreads),
                          unsigned(kLaneFillThreads), stream, prm);
    return launch_pdl(fill_kernel, unsigned((int64_t(B) + kFillWarps - 1) / kFillWarps), unsigned(kFillWarps * 32),
                      stream, prm);
}

int launch_host_copy(const DeviceState &st, const CopyParams &cp, cudaStream_t stream) {
    const int64_t want = (cp.n16 + kCopyThreads - 1) / kCopyThreads;
    const int64_t cap = int64_t(st.sms) * kCopyCtasPerSm;
    return launch_pdl(host_copy_kernel, unsigned(want < 1 ? 1 : (want < cap ? want : cap)), unsigned(kCopyThreads),
                      stream, cp);
}

// Scratch kept per stream.  A call takes the result slots from its stream's
// buffer, so consecutive calls in a CUDA graph have no memory nodes between them
// and the next call's scan launches early behind the previous fill (a pool
// allocation and free per call, captured as memory nodes, cost ~0.4 us per step).
// Buffers are keyed by the stream handle and made outside stream capture only (a
// hit makes no CUDA call at all, so it is safe inside a capture; a miss asks
// cudaStreamIsCapturing, which capture allows).  They grow geometrically and are
// never freed before exit: a captured graph may still refer to a buffer that a
// larger batch later replaced.
// Calls on one stream are ordered, so they never overlap on its buffer.
struct StreamScratch {
    unsigned long long *slots = nullptr;
    size_t bytes = 0;
    // Held by a call while it enqueues the kernels that use the buffer (the host
    // entry point: until its stream synchronisation), so that calls from several
    // threads on one stream never interleave their kernels on it.  One per stream
    // key, kept across growth; never freed.
    std::mutex *mu = nullptr;
};
std::mutex g_scratch_mu;
std::unordered_map<uintptr_t, StreamScratch> g_scratch[kMaxDevices];

// The calling thread's last stream and its buffer: a repeat call on that stream
// takes no lock.  A buffer is never freed, so this copy stays valid even after
// another thread has given the stream a larger one (calls on one stream are
// ordered whichever buffer each uses).
struct LastScratch {
    int dev = -1;
    uintptr_t stream = 0;
    StreamScratch sc;
};
thread_local LastScratch t_last;

// The scratch of `stream` on device `dev`, holding at least `need` bytes, and the
// stream's lock (*mu) to hold while enqueuing work on it; nullptr for both (no
// error) when it has none and cannot make one now: the stream is capturing.
int stream_scratch(int dev, cudaStream_t stream, size_t need, unsigned long long **out, std::mutex **mu) {
    // cudaStreamPerThread is one handle for a different stream in every thread:
    // keyed by the calling thread instead (an address of its own, never a handle).
    const uintptr_t key = stream == cudaStreamPerThread ? reinterpret_cast<uintptr_t>(&t_last) | 1u
                                                        : reinterpret_cast<uintptr_t>(stream);
    if (t_last.dev == dev && t_last.stream == key && t_last.sc.bytes >= need) {
        *out = t_last.sc.slots;
        *mu = t_last.sc.mu;
        return LOOKUP_DRAFT_OK;
    }
    *out = nullptr;
    *mu = nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    StreamScratch &sc = g_scratch[dev][key];
    if (sc.bytes >= need) {
        *out = sc.slots;
        *mu = sc.mu;
        t_last.dev = dev;
        t_last.stream = key;
        t_last.sc = sc;
        return LOOKUP_DRAFT_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    LD_CUDA(cudaStreamIsCapturing(stream, &cs));
    if (cs != cudaStreamCaptureStatusNone) return LOOKUP_DRAFT_OK;
    size_t bytes = sc.bytes * 2 > need ? sc.bytes * 2 : need;
    bytes = (bytes + 65535) & ~size_t(65535);
    if (!sc.mu) sc.mu = new std::mutex;
    void *p = nullptr;
    LD_CUDA(cudaMalloc(&p, bytes));                     // valid on every stream at once
    sc.slots = static_cast<unsigned long long *>(p);    // the old buffer, if any, stays allocated
    sc.bytes = bytes;
    *out = sc.slots;
    *mu = sc.mu;
    t_last.dev = dev;
    t_last.stream = key;
    t_last.sc = sc;
    return LOOKUP_DRAFT_OK;
}

int run_step(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m, int32_t K,
             int32_t *out_draft, int32_t *out_len, int32_t *out_pos, int32_t *out_mlen, cudaStream_t stream) {
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    const size_t need = workspace_bytes_for(B, grid_for(*st));
    unsigned long long *slots = nullptr;
    std::mutex *mu = nullptr;
    rc = stream_scratch(dev, stream, need, &slots, &mu);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    if (slots) {
        std::lock_guard<std::mutex> hold(*mu);
        rc = launch_scan(*st, tokens, offsets, B, min_m, max_m, slots, stream);
        if (rc == LOOKUP_DRAFT_OK)
            rc = launch_fill(*st, tokens, offsets, B, K, slots, out_draft, out_len, out_pos, out_mlen, stream);
        return rc;
    }
    // No stream scratch (a capture on a stream without one): stream-ordered scratch
    // from the library pool for this call.
    void *ws = nullptr;
    LD_CUDA(cudaMallocFromPoolAsync(&ws, need, st->pool, stream));
    slots = static_cast<unsigned long long *>(ws);
    rc = launch_scan(*st, tokens, offsets, B, min_m, max_m, slots, stream);
    if (rc == LOOKUP_DRAFT_OK)
        rc = launch_fill(*st, tokens, offsets, B, K, slots, out_draft, out_len, out_pos, out_mlen, stream);
    cudaError_t fe = cudaFreeAsync(ws, stream);
    if (rc == LOOKUP_DRAFT_OK && fe != cudaSuccess) return cuda_fail(fe, "cudaFreeAsync");
    return rc;
}

// The scan, then the fill with scheduling and fusion, on the stream's scratch (the
// pool's when a capture finds none), as run_step does.
int run_plan(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
             const PlanArgs &pa, cudaStream_t stream) {
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    const size_t need = workspace_bytes_for(B, grid_for(*st));
    unsigned long long *slots = nullptr;
    std::mutex *mu = nullptr;
    rc = stream_scratch(dev, stream, need, &slots, &mu);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    std::unique_lock<std::mutex> hold;
    if (mu) hold = std::unique_lock<std::mutex>(*mu);
    void *ws = nullptr;
    if (!slots) {
        LD_CUDA(cudaMallocFromPoolAsync(&ws, need, st->pool, stream));
        slots = static_cast<unsigned long long *>(ws);
    }
    FillParams fp{};
    fp.tokens = tokens;
    fp.offsets = offsets;
    fp.slots = slots;
    fp.B = B;
    fp.K = pa.io.H + pa.io.T;
    fp.grid = grid_for(*st);
#if LOOKUP_DRAFT_CHECKED
    fp.nslots = int64_t(B) + int64_t(fp.grid) * kWarps;
#endif
    rc = launch_scan(*st, tokens, offsets, B, min_m, max_m, slots, stream);
    if (rc == LOOKUP_DRAFT_OK)
        rc = lkd::launch_pdl2(fill_plan_kernel, unsigned((int64_t(B) + kFillWarps - 1) / kFillWarps),
                              unsigned(kFillWarps * 32), stream, fp, pa);
    if (ws) {
        cudaError_t fe = cudaFreeAsync(ws, stream);
        if (rc == LOOKUP_DRAFT_OK && fe != cudaSuccess) return cuda_fail(fe, "cudaFreeAsync");
    }
    return rc;
}

// ------------------------------------------------- no-allocation entry point ----
// lookup_draft_noalloc keeps the scan's result slots in one fixed array in device
// memory instead of taking them from a pool, so a call makes no allocation at
// all.  The host needs the array's device address, which it takes once per device
// (with that device current) from cudaGetSymbolAddress; the array's name in host
// code is only a host-side stand-in and must never be handed to a kernel.
constexpr size_t kStaticSlots = size_t(1) << 16;   // 64-bit slots: 512 KiB per device

struct StaticState {
    std::atomic<bool> ready{false};                     // set (release) once the fields below are final
    int sms = 0;
    unsigned long long *slots = nullptr;                // device address of the array
};
StaticState g_static[kMaxDevices];
std::mutex g_static_mu;

}  // namespace

// The error record shared with the loop-step entry points of lookup_loop.cu
// (same library; not exported from it).
__attribute__((visibility("hidden"))) int lookup_record_cuda_error(cudaError_t e, const char *what) {
    return cuda_fail(e, what);
}

// Kernel launches the library has enqueued, process-wide (lookup_draft_launch_count).
static std::atomic<uint64_t> g_launches{0};

__attribute__((visibility("hidden"))) void lookup_note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

__attribute__((visibility("hidden"))) uint64_t lookup_wait_limit_ns() {
    return g_wait_ns.load(std::memory_order_relaxed);
}

// Fixed scratch of lookup_draft_noalloc (file scope; every GPU that loads the
// library holds it until the process exits).
static __device__ __align__(256) unsigned long long g_static_slots[kStaticSlots];

namespace {

// Per-device set-up of lookup_draft_noalloc, once: SM count, the scan kernels'
// shared-memory opt-in, and the device address of g_static_slots.  No allocation.
// After it, a call only reads the ready flag; the lock is taken for the set-up alone.
int static_state(StaticState **out) {
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
    StaticState &st = g_static[dev];
    if (st.ready.load(std::memory_order_acquire)) {
        *out = &st;
        return LOOKUP_DRAFT_OK;
    }
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!st.ready.load(std::memory_order_relaxed)) {
        int sms = 0;
        LD_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        const int rc_attr = scan_attributes();
        if (rc_attr != LOOKUP_DRAFT_OK) return rc_attr;
        void *ptr = nullptr;
        LD_CUDA(cudaGetSymbolAddress(&ptr, g_static_slots));
        st.sms = sms;
        st.slots = static_cast<unsigned long long *>(ptr);
        st.ready.store(true, std::memory_order_release);
    }
    *out = &st;
    return LOOKUP_DRAFT_OK;
}

}  // namespace

// ------------------------------------------------------------------ C ABI ----
extern "C" {

int lookup_draft_ex(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                    int32_t K, int32_t *out_draft, int32_t *out_len, int32_t *out_pos, int32_t *out_mlen,
                    struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_ex");
    g_cuda_msg[0] = '\0';
    int rc = check_common(tokens, offsets, B, min_m, max_m, K);
    if (rc == LOOKUP_DRAFT_OK) rc = check_outputs(B, K, out_draft, out_len, out_pos, out_mlen);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    return run_step(tokens, offsets, B, min_m, max_m, K, out_draft, out_len, out_pos, out_mlen, stream);
}

int lookup_draft(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m, int32_t K,
                 int32_t *out_draft, int32_t *out_len, int32_t *out_pos, struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft");
    return lookup_draft_ex(tokens, offsets, B, min_m, max_m, K, out_draft, out_len, out_pos, nullptr, stream);
}

size_t lookup_draft_workspace_bytes(int32_t B) {
    g_cuda_msg[0] = '\0';
    if (B < 0) return 0;
    DeviceState *st = nullptr;
    if (device_state(&st) != LOOKUP_DRAFT_OK) return 0;
    return workspace_bytes_for(B, grid_for(*st));
}

int lookup_draft_scan(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                      void *workspace, size_t workspace_bytes, struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_scan");
    g_cuda_msg[0] = '\0';
    int rc = check_common(tokens, offsets, B, min_m, max_m, 0);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    if (!workspace || !aligned(workspace, 8)) return LOOKUP_DRAFT_EINVAL;
    DeviceState *st = nullptr;
    rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    if (workspace_bytes < workspace_bytes_for(B, grid_for(*st))) return LOOKUP_DRAFT_EINVAL;
    return launch_scan(*st, tokens, offsets, B, min_m, max_m, static_cast<unsigned long long *>(workspace), stream);
}

int lookup_draft_fill(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                      int32_t K, const void *workspace, size_t workspace_bytes, int32_t *out_draft, int32_t *out_len,
                      int32_t *out_pos, int32_t *out_mlen, struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_fill");
    g_cuda_msg[0] = '\0';
    int rc = check_common(tokens, offsets, B, min_m, max_m, K);
    if (rc == LOOKUP_DRAFT_OK) rc = check_outputs(B, K, out_draft, out_len, out_pos, out_mlen);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    if (!workspace || !aligned(workspace, 8)) return LOOKUP_DRAFT_EINVAL;
    DeviceState *st = nullptr;
    rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    if (workspace_bytes < workspace_bytes_for(B, grid_for(*st))) return LOOKUP_DRAFT_EINVAL;
    return launch_fill(*st, tokens, offsets, B, K, static_cast<const unsigned long long *>(workspace), out_draft,
                       out_len, out_pos, out_mlen, stream);
}

int lookup_draft_host(const int32_t *h_tokens, const int64_t *h_offsets, int32_t B, int32_t min_m, int32_t max_m,
                      int32_t K, int32_t *h_out_draft, int32_t *h_out_len, int32_t *h_out_pos,
                      struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_host");
    g_cuda_msg[0] = '\0';
    int rc = check_common(h_tokens, h_offsets, B, min_m, max_m, K);
    if (rc == LOOKUP_DRAFT_OK) rc = check_outputs(B, K, h_out_draft, h_out_len, h_out_pos, nullptr);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    if (h_offsets[0] < 0) return LOOKUP_DRAFT_EINVAL;
    for (int32_t r = 0; r < B; ++r) {
        const int64_t L = h_offsets[r + 1] - h_offsets[r];
        if (L < 0 || L >= (int64_t(1) << 31)) return LOOKUP_DRAFT_EINVAL;
    }
    DeviceState *st = nullptr;
    rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;

    const int64_t first = h_offsets[0];
    const size_t n_tok = size_t(h_offsets[B] - first);
    // Page-locked inputs the device can address are read by host_copy_kernel: the
    // whole 16-byte units of their device-side address range (never past the
    // pages that hold the tokens), so the device copy keeps the tokens' 16-byte
    // phase.  Other host memory goes through copy-engine transfers.
    const void *m_tok = n_tok ? mapped_host_const(h_tokens + first) : nullptr;
    const void *m_off = mapped_host_const(h_offsets);
    const bool kernel_copy = m_off && (n_tok == 0 || m_tok);
    const uintptr_t src_t = kernel_copy && n_tok ? reinterpret_cast<uintptr_t>(m_tok) : 0;
    const uintptr_t src_lo = src_t & ~uintptr_t(15);
    const uintptr_t src_hi = (src_t + n_tok * 4 + 15) & ~uintptr_t(15);
    const size_t phase = size_t(src_t - src_lo);
    const size_t tok_bytes = kernel_copy ? size_t(src_hi - src_lo) : ((n_tok * 4 + 15) & ~size_t(15));
    const size_t off_bytes = (size_t(B) + 1) * 8;
    const size_t out_words = size_t(B) * size_t(K) + 2 * size_t(B);
    const size_t ws_bytes = workspace_bytes_for(B, grid_for(*st));
    const size_t total = tok_bytes + ((off_bytes + 15) & ~size_t(15)) + ((out_words * 4 + 15) & ~size_t(15)) + ws_bytes;
    // The stream's scratch holds the staging buffer: calls on one stream are
    // ordered and this one synchronises before it returns, so the buffer is idle
    // between calls.  Without one (a capturing stream, where the synchronisation
    // below fails anyway) the buffer comes from the pool for this call.
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    unsigned long long *staging = nullptr;
    std::mutex *mu = nullptr;
    rc = stream_scratch(dev, stream, total, &staging, &mu);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    std::unique_lock<std::mutex> hold;                  // until the synchronisation below
    if (mu) hold = std::unique_lock<std::mutex>(*mu);
    void *buf = staging;
    if (!buf) LD_CUDA(cudaMallocFromPoolAsync(&buf, total, st->pool, stream));
    unsigned char *base = static_cast<unsigned char *>(buf);
    int32_t *d_tok = reinterpret_cast<int32_t *>(base + phase);
    int64_t *d_off = reinterpret_cast<int64_t *>(base + tok_bytes);
    int32_t *d_out = reinterpret_cast<int32_t *>(base + tok_bytes + ((off_bytes + 15) & ~size_t(15)));
    auto *d_ws = reinterpret_cast<unsigned long long *>(reinterpret_cast<unsigned char *>(d_out) +
                                                        ((out_words * 4 + 15) & ~size_t(15)));
    int32_t *d_draft = d_out;
    int32_t *d_len = d_out + size_t(B) * size_t(K);
    int32_t *d_pos = d_len + B;
    // Page-locked, device-mapped output buffers are written by the fill kernel
    // directly (no copies back); any other host memory gets them by copies.
    int32_t *m_draft = mapped_host(h_out_draft), *m_len = mapped_host(h_out_len), *m_pos = mapped_host(h_out_pos);
    const bool direct = m_len && m_pos && (K == 0 || m_draft);
    if (direct) {
        d_draft = K > 0 ? m_draft : d_draft;
        d_len = m_len;
        d_pos = m_pos;
    }
    // The device copy holds tokens[first .. end); index it with the caller's offsets
    // through a base pointer moved back by `first` elements (never dereferenced there).
    const int32_t *d_tok_base =
        reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(d_tok) - uintptr_t(first) * 4u);

    cudaError_t e = cudaSuccess;
    if (kernel_copy) {
        CopyParams cp;
        cp.src = reinterpret_cast<const int4 *>(src_lo);
        cp.dst = reinterpret_cast<int4 *>(base);
        cp.n16 = int64_t(tok_bytes / 16);
        cp.src_off = static_cast<const int64_t *>(m_off);
        cp.dst_off = d_off;
        cp.n_off = B + 1;
        rc = launch_host_copy(*st, cp, stream);
    } else {
        if (n_tok) e = cudaMemcpyAsync(d_tok, h_tokens + first, n_tok * 4, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync(d_off, h_offsets, off_bytes, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync (host to device)");
    }
    if (rc == LOOKUP_DRAFT_OK) {
        rc = launch_scan(*st, d_tok_base, d_off, B, min_m, max_m, d_ws, stream);
        if (rc == LOOKUP_DRAFT_OK)
            rc = launch_fill(*st, d_tok_base, d_off, B, K, d_ws, d_draft, d_len, d_pos, nullptr, stream);
    }
    if (rc == LOOKUP_DRAFT_OK && !direct && K > 0)
        e = cudaMemcpyAsync(h_out_draft, d_draft, size_t(B) * size_t(K) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && !direct && e == cudaSuccess)
        e = cudaMemcpyAsync(h_out_len, d_len, size_t(B) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && !direct && e == cudaSuccess)
        e = cudaMemcpyAsync(h_out_pos, d_pos, size_t(B) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync (device to host)");
    cudaError_t fe = staging ? cudaSuccess : cudaFreeAsync(buf, stream);
    cudaError_t se = cudaStreamSynchronize(stream);
    if (rc == LOOKUP_DRAFT_OK && fe != cudaSuccess) rc = cuda_fail(fe, "cudaFreeAsync");
    if (rc == LOOKUP_DRAFT_OK && se != cudaSuccess) rc = cuda_fail(se, "cudaStreamSynchronize");
    return rc;
}

int lookup_draft_noalloc(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                         int32_t K, int32_t *out_draft, int32_t *out_len, int32_t *out_pos,
                         struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_noalloc");
    g_cuda_msg[0] = '\0';
    int rc = check_common(tokens, offsets, B, min_m, max_m, K);
    if (rc == LOOKUP_DRAFT_OK) rc = check_outputs(B, K, out_draft, out_len, out_pos, nullptr);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    StaticState *st = nullptr;
    rc = static_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    DeviceState ds;                                     // SM count only: no pool is made or used
    ds.sms = st->sms;
    if (size_t(B) + size_t(grid_for(ds)) * kWarps > kStaticSlots) return LOOKUP_DRAFT_ERANGE;
    rc = launch_scan(ds, tokens, offsets, B, min_m, max_m, st->slots, stream);
    if (rc == LOOKUP_DRAFT_OK)
        rc = launch_fill(ds, tokens, offsets, B, K, st->slots, out_draft, out_len, out_pos, nullptr, stream);
    return rc;
}

const char *lookup_draft_strerror(int code) {
    switch (code) {
    case LOOKUP_DRAFT_OK: return "ok";
    case LOOKUP_DRAFT_EINVAL: return "invalid argument";
    case LOOKUP_DRAFT_ECUDA: return "CUDA error";
    case LOOKUP_DRAFT_ERANGE: return "batch too large for the fixed scratch of lookup_draft_noalloc";
    default: return "unknown lookup_draft status";
    }
}

const char *lookup_draft_last_cuda_error(void) { return g_cuda_msg; }

uint64_t lookup_draft_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void lookup_draft_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

int lookup_draft_plan(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                      const int32_t *model_draft, const int32_t *committed, int32_t H, int32_t T,
                      int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min, int32_t slack,
                      int32_t enter_steps, int32_t sticky, int32_t *state, int32_t *out_long, int32_t *out_block,
                      int32_t *out_len, int32_t *out_point_mass, int32_t *out_mlen, int32_t *out_draft_len,
                      struct CUstream_st *stream) {
    TraceRange trace_("lookup_draft_plan");
    g_cuda_msg[0] = '\0';
    if (H < 1 || T < 0 || int64_t(H) + T > LOOKUP_DRAFT_MAX_K || agree_n < 0 || agree_n > H || enter_steps < 1 ||
        sticky < 0 || slack < 0)
        return LOOKUP_DRAFT_EINVAL;
    int rc = check_common(tokens, offsets, B, min_m, max_m, H + T);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    if (!model_draft || !committed || !state || !out_long || !out_block || !out_len || !out_point_mass)
        return LOOKUP_DRAFT_EINVAL;
    const int32_t *ptrs[] = {model_draft, committed, state, out_long, out_block, out_len, out_point_mass, out_mlen,
                             out_draft_len};
    for (const int32_t *q : ptrs)
        if (q && !aligned(q, 4)) return LOOKUP_DRAFT_EINVAL;
    PlanArgs pa{{model_draft, committed, state, out_long, out_block, out_len, out_point_mass, H, T, replace_min,
                 agree_min, agree_n, tail_min, slack, enter_steps, sticky},
                out_mlen, out_draft_len};
    return run_plan(tokens, offsets, B, min_m, max_m, pa, stream);
}

int lookup_draft_checked_build(void) { return LOOKUP_DRAFT_CHECKED ? 1 : 0; }

int lookup_draft_check_word(uint32_t *out, int32_t clear) {
    g_cuda_msg[0] = '\0';
    if (!out) return LOOKUP_DRAFT_EINVAL;
#if LOOKUP_DRAFT_CHECKED
    LD_CUDA(cudaDeviceSynchronize());
    unsigned w = 0;
    LD_CUDA(cudaMemcpyFromSymbol(&w, g_check_word, sizeof w));
    if (clear) {
        const unsigned zero = 0;
        LD_CUDA(cudaMemcpyToSymbol(g_check_word, &zero, sizeof zero));
    }
    *out = w;
#else
    (void)clear;
    *out = 0;
#endif
    return LOOKUP_DRAFT_OK;
}

}  // extern "C"
