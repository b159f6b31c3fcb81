// lookup_draft.cu -- prompt-lookup (n-gram) drafting on GB300 (sm_103a).
//
// What one call computes (HyperQwen lookup-drafting article, kwkr.cn/news/564408,
// section "第1步"): for every request of a CSR batch, the most recent earlier
// occurrence of the longest current suffix (max_m down to min_m tokens, overlap
// with the suffix allowed), and the K tokens that follow it, read from the history
// extended by its own draft (e[L+j] = e[p+m+j]).  The exact contract is in
// include/lookup_draft.h.
//
// Two kernels, both on the caller's stream:
//
//  scan_kernel -- the split-history scan, HBM bound (4 bytes per history token,
//    read once).  The whole batch is one array of 16-byte quads; the grid (a fixed
//    number of CTAs per SM, independent of the data so the host never reads the
//    offsets) splits it into equal contiguous chunks, so long requests are shared
//    by many CTAs and short ones are packed into one.  Each CTA streams its chunk
//    through shared memory in tiles moved by 1-D TMA bulk copies (cp.async.bulk,
//    mbarrier completion, a ring of stages), each tile preceded by a halo of up to
//    31 tokens of backward context.  A thread reads one quad (128-bit) at a time
//    and compares its tokens with the last suffix token of their request; the rare
//    survivors are extended backwards against the suffix kept in shared memory
//    (the article's cheap rejection test, section "第1步").  A match of length k
//    ending at local position q gives the key (k << 32) | (q - k + 1): its maximum
//    is the longest match, then the most recent.  Each thread keeps its best key
//    for its current request and folds it into a per-(request, CTA) slot with one
//    red.max when it moves on.
//
//  fill_kernel -- one warp per request: max over the request's slots, then the
//    draft tokens t[p + m + (j mod d)], d = L - p - m, and the length/position.
//    Launched with programmatic dependent launch so its launch and its reads of
//    the offsets overlap the scan's tail.
//
// Partial-result slots.  CTA c owns slot (r + c) for every request r that has a
// token in its chunk.  Chunks and requests are both ordered and disjoint, so the
// (c, r) pairs form a monotone staircase and r + c never repeats: no slot is shared
// and none needs clearing before a call (each CTA zeroes its own before use).
//
// No spin-wait is unbounded: every mbarrier wait gives up after a time limit, and
// a CTA that gives up waits (bounded) for its own copies, marks its requests as
// failed in their slots and exits, so the failure reaches the host as
// out_len = LOOKUP_DRAFT_LEN_FAILED instead of a hang.

#include "lookup_draft.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace {

// ---------------------------------------------------------------- tuning ----
constexpr int kThreads = 256;          // scan CTA size
constexpr int kTileQuads = 1024;       // 16 KB of history per tile
constexpr int kHaloQuads = 8;          // room for (LOOKUP_DRAFT_MAX_M - 1) tokens of context
constexpr int kStages = 4;             // tiles in flight per CTA
constexpr int kSufCap = 64;            // requests per CTA whose suffix is kept in smem
constexpr int kOffCap = 4097;          // offsets kept in smem when B + 1 <= kOffCap
constexpr int kCtasPerSm = 2;
constexpr int kFillWarps = 4;          // requests per fill CTA

constexpr unsigned long long kKeyFailed = ~0ull;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

static_assert(4 * kHaloQuads >= LOOKUP_DRAFT_MAX_M - 1, "halo too small for LOOKUP_DRAFT_MAX_M");

constexpr size_t kStageBytes = size_t(kTileQuads + kHaloQuads) * 16;

struct ScanParams {
    const int32_t *tokens;
    const int64_t *offsets;
    unsigned long long *slots;
    int32_t B;
    int32_t min_m;
    int32_t max_m;
    int32_t grid;
    uint64_t wait_ns;
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
};

// ------------------------------------------------------ partition helpers ----
// The batch occupies aligned quads [q_lo, q_lo + nq) of the 16-byte-aligned view
// of `tokens`; chunk c is quads [q_lo + c*nq/G, q_lo + (c+1)*nq/G).
struct Partition {
    int64_t a_begin;    // first history token, index in the aligned view
    int64_t a_end;      // one past the last
    int64_t q_lo;
    int64_t nq;
};

__host__ __device__ inline int tokens_shift(const int32_t *tokens) {
    return int((reinterpret_cast<uintptr_t>(tokens) & 15u) >> 2);
}

__device__ inline Partition make_partition(int64_t a_begin, int64_t a_end) {
    Partition P;
    P.a_begin = a_begin;
    P.a_end = a_end;
    P.q_lo = a_begin >> 2;
    P.nq = ((a_end + 3) >> 2) - P.q_lo;
    return P;
}

__device__ inline int64_t chunk_start(const Partition &P, int64_t c, int G) {
    return P.q_lo + int64_t((unsigned long long)c * (unsigned long long)P.nq / (unsigned long long)G);
}

// The chunk holding aligned quad x: the largest c with chunk_start(c) <= x.
__device__ inline int64_t chunk_of_quad(const Partition &P, int64_t x, int G) {
    unsigned long long rel = (unsigned long long)(x - P.q_lo);
    return int64_t(((rel + 1) * (unsigned long long)G - 1) / (unsigned long long)P.nq);
}

// ----------------------------------------------------------- PTX wrappers ----
__device__ inline uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ inline void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ inline void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ inline void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ inline bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ inline uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` to complete; false if `limit_ns` ran out first.
__device__ inline bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

__device__ inline void red_max_u64(unsigned long long *p, unsigned long long v) {
    atomicMax(p, v);   // result unused: compiles to a fire-and-forget reduction
}

__device__ inline void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ inline void wait_for_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ scan kernel ----
struct ScanSmemLayout {
    size_t stages, bars, suf, offs, total;
};

__host__ __device__ inline ScanSmemLayout scan_smem_layout(int32_t B, int32_t max_m) {
    ScanSmemLayout L;
    L.stages = 0;
    L.bars = L.stages + kStages * kStageBytes;
    L.suf = L.bars + kStages * sizeof(unsigned long long);
    L.offs = L.suf + ((size_t(kSufCap) * size_t(max_m) * 4 + 15) & ~size_t(15));
    size_t n_off = (int64_t(B) + 1 <= kOffCap) ? size_t(B) + 1 : 2;
    L.total = L.offs + n_off * 8;
    return L;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) scan_kernel(ScanParams prm) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int c = blockIdx.x;
    const int G = prm.grid;
    const int B = prm.B;
    const int min_m = prm.min_m;
    const int max_m = prm.max_m;

    const ScanSmemLayout lay = scan_smem_layout(B, max_m);
    unsigned long long *bars = reinterpret_cast<unsigned long long *>(smem + lay.bars);
    int32_t *suf_s = reinterpret_cast<int32_t *>(smem + lay.suf);
    int64_t *offs_s = reinterpret_cast<int64_t *>(smem + lay.offs);

    const int shift = tokens_shift(prm.tokens);
    const int32_t *ta = reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(prm.tokens) & ~uintptr_t(15));
    const bool offs_in_smem = int64_t(B) + 1 <= kOffCap;

    // 1. Offsets (shifted into the aligned view) -> shared memory, one burst.
    if (offs_in_smem) {
        for (int i = tid; i <= B; i += kThreads) offs_s[i] = __ldg(prm.offsets + i) + shift;
    } else if (tid < 2) {
        offs_s[tid] = __ldg(prm.offsets + (tid == 0 ? 0 : B)) + shift;
    }
    __syncthreads();

    auto off_a = [&](int i) -> int64_t {
        return offs_in_smem ? offs_s[i] : __ldg(prm.offsets + i) + shift;
    };

    const int64_t a_begin = offs_s[0];
    const int64_t a_end = offs_in_smem ? offs_s[B] : offs_s[1];
    if (a_end <= a_begin) return;                       // no history tokens at all
    const Partition P = make_partition(a_begin, a_end);
    const int64_t qa = chunk_start(P, c, G);
    const int64_t qb = chunk_start(P, c + 1, G);
    if (qa >= qb) return;                               // empty chunk: owns no slot

    // 2. Tile plan and the first copies (one elected thread).
    const int halo = (max_m - 1 + 3) >> 2;
    const int ntiles = int((qb - qa + kTileQuads - 1) / kTileQuads);
    auto issue_tile = [&](int i) {
        const int s = i % kStages;
        const int64_t t0 = qa + int64_t(i) * kTileQuads;
        const int64_t t1 = (t0 + kTileQuads < qb) ? t0 + kTileQuads : qb;
        const int64_t ls = (t0 - halo > P.q_lo) ? t0 - halo : P.q_lo;
        const uint32_t bytes = uint32_t(t1 - ls) * 16u;
        unsigned char *stage = smem + lay.stages + size_t(s) * kStageBytes;
        const uint32_t dst = smem_addr(stage + size_t(kHaloQuads - (t0 - ls)) * 16);
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_expect_tx(bar, bytes);
        bulk_copy_g2s(dst, ta + ls * 4, bytes, bar);
    };
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        fence_barrier_init();
        const int first = ntiles < kStages ? ntiles : kStages;
        for (int i = 0; i < first; ++i) issue_tile(i);
    }
    allow_dependent_launch();

    // 3. Requests with a token in this chunk: [r_lo, r_hi].
    const int64_t e_first = (4 * qa > a_begin) ? 4 * qa : a_begin;
    const int64_t e_last = ((4 * qb < a_end) ? 4 * qb : a_end) - 1;
    auto owner = [&](int64_t a) -> int {                // largest r with off_a(r) <= a
        int lo = 0, hi = B;                             // off_a(0) <= a < off_a(B)
        while (hi - lo > 1) {
            const int mid = lo + ((hi - lo) >> 1);
            if (off_a(mid) <= a) lo = mid; else hi = mid;
        }
        return lo;
    };
    const int r_lo = owner(e_first);
    const int r_hi = owner(e_last);

    // 4. Suffix rows (row[j] = t[L-1-j]) of the first kSufCap requests, and this
    //    CTA's slots cleared.
    {
        const int nrows = (r_hi - r_lo + 1 < kSufCap) ? r_hi - r_lo + 1 : kSufCap;
        for (int idx = tid; idx < nrows * max_m; idx += kThreads) {
            const int row = idx / max_m, j = idx - row * max_m;
            const int r = r_lo + row;
            const int64_t src = off_a(r + 1) - 1 - j;
            suf_s[idx] = (src >= off_a(r)) ? ta[src] : 0;
        }
        for (int r = r_lo + tid; r <= r_hi; r += kThreads) prm.slots[int64_t(r) + c] = 0ull;
    }
    __syncthreads();

    auto suffix = [&](int r, int64_t nxt, int j) -> int32_t {
        const int row = r - r_lo;
        return row < kSufCap ? suf_s[row * max_m + j] : ta[nxt - 1 - j];
    };

    // Per-thread position in the batch: current request and its candidate range.
    int r = r_lo;
    int64_t nxt = off_a(r + 1);
    int64_t lo = off_a(r) + (min_m - 1);    // first candidate end position
    int64_t hi = nxt - 2;                    // last candidate end position (p + m <= L - 1)
    int32_t last = suffix(r, nxt, 0);
    int best_r = -1;
    unsigned long long best_key = 0ull;

    auto flush = [&]() {
        if (best_key) red_max_u64(prm.slots + (int64_t(best_r) + c), best_key);
    };
    // Candidate end at aligned index a (its token equals `last`): extend backwards.
    auto extend = [&](const int32_t *st, int64_t st_base, int64_t a) {
        const int64_t q = a - off_a(r);                 // local end position
        const int kmax = (int64_t(max_m) < q + 1) ? max_m : int(q + 1);
        int k = 1;
        while (k < kmax && st[a - k - st_base] == suffix(r, nxt, k)) ++k;
        if (k >= min_m) {
            const unsigned long long key =
                (static_cast<unsigned long long>(k) << 32) | static_cast<uint32_t>(q - k + 1);
            if (r != best_r) {
                flush();
                best_r = r;
                best_key = key;
            } else if (key > best_key) {
                best_key = key;
            }
        }
    };
    auto advance_to = [&](int64_t a) {                 // make r the request holding a
        if (a < nxt) return;
        do {
            ++r;
            nxt = off_a(r + 1);
        } while (a >= nxt);
        lo = off_a(r) + (min_m - 1);
        hi = nxt - 2;
        last = suffix(r, nxt, 0);
    };

    // 5. Stream the tiles.
    bool failed = false;
    int i = 0;
    for (; i < ntiles; ++i) {
        const int s = i % kStages;
        const uint32_t parity = uint32_t(i / kStages) & 1u;
        const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), parity, prm.wait_ns);
        const int64_t t0 = qa + int64_t(i) * kTileQuads;
        const int nq = int(((t0 + kTileQuads < qb) ? t0 + kTileQuads : qb) - t0);
        if (ok) {
            const unsigned char *stage = smem + lay.stages + size_t(s) * kStageBytes + kHaloQuads * 16;
            const int4 *sq = reinterpret_cast<const int4 *>(stage);
            const int32_t *st = reinterpret_cast<const int32_t *>(stage);
            const int64_t st_base = 4 * t0;              // aligned index of st[0]
            for (int j = tid; j < nq; j += kThreads) {
                const int64_t a0 = st_base + 4 * int64_t(j);
                const int4 v = sq[j];
                if (a0 >= lo && a0 + 3 <= hi) {          // the whole quad is candidates of r
                    if ((v.x == last) | (v.y == last) | (v.z == last) | (v.w == last)) {
                        if (v.x == last) extend(st, st_base, a0);
                        if (v.y == last) extend(st, st_base, a0 + 1);
                        if (v.z == last) extend(st, st_base, a0 + 2);
                        if (v.w == last) extend(st, st_base, a0 + 3);
                    }
                } else {
                    const int32_t vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int64_t a = a0 + e;
                        if (a < a_begin) continue;
                        if (a >= a_end) break;
                        advance_to(a);
                        if (a >= lo && a <= hi && vals[e] == last) extend(st, st_base, a);
                    }
                }
            }
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        if (tid == 0 && i + kStages < ntiles) {
            fence_proxy_async_smem();
            issue_tile(i + kStages);
        }
    }

    if (!failed) {
        flush();
        return;
    }
    // 6. A wait ran out: let this CTA's copies land (bounded), then mark every
    //    request it owns as failed.  The stage of tile i is still outstanding, and
    //    so are tiles i+1 .. min(i + kStages, ntiles) - 1.
    if (tid == 0) {
        const int stop = (i + kStages < ntiles) ? i + kStages : ntiles;
        for (int k = i; k < stop; ++k)
            (void)mbar_wait_bounded(smem_addr(&bars[k % kStages]), uint32_t(k / kStages) & 1u,
                                    kDefaultWaitNs);
    }
    __syncthreads();
    for (int rr = r_lo + tid; rr <= r_hi; rr += kThreads) red_max_u64(prm.slots + (int64_t(rr) + c), kKeyFailed);
}

// ------------------------------------------------------------ fill kernel ----
__global__ void __launch_bounds__(kFillWarps * 32) fill_kernel(FillParams prm) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kFillWarps + (threadIdx.x >> 5);
    if (r >= prm.B) {
        wait_for_prerequisite_grid();
        return;
    }
    // Inputs the scan does not write: read them before waiting for it.
    const int64_t o0 = __ldg(prm.offsets + r);
    const int64_t o1 = __ldg(prm.offsets + r + 1);
    const int64_t first = __ldg(prm.offsets);
    const int64_t end = __ldg(prm.offsets + prm.B);
    const int shift = tokens_shift(prm.tokens);
    const int64_t L = o1 - o0;
    wait_for_prerequisite_grid();

    unsigned long long key = 0ull;
    if (L > 0) {
        const Partition P = make_partition(first + shift, end + shift);
        const int64_t c0 = chunk_of_quad(P, (o0 + shift) >> 2, prm.grid);
        const int64_t c1 = chunk_of_quad(P, (o1 - 1 + shift) >> 2, prm.grid);
        for (int64_t cc = c0 + lane; cc <= c1; cc += 32) {
            // With fewer quads than CTAs some chunks are empty; their CTAs own no slot.
            if (chunk_start(P, cc, prm.grid) == chunk_start(P, cc + 1, prm.grid)) continue;
            const unsigned long long v = prm.slots[int64_t(r) + cc];
            key = v > key ? v : key;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long v = __shfl_xor_sync(0xffffffffu, key, o);
            key = v > key ? v : key;
        }
    }
    // A key that does not describe an admissible match (1 <= m, p + m <= L - 1) can
    // only come from a failed scan; it is reported as such and never dereferenced.
    const int64_t km = int64_t(key >> 32), kp = int64_t(uint32_t(key));
    const bool failed = key != 0ull && (key == kKeyFailed || km < 1 || kp + km > L - 1);
    const bool found = key != 0ull && !failed;
    const int32_t m = found ? int32_t(km) : 0;
    const int64_t p = found ? kp : -1;
    const int64_t d = found ? L - p - m : 1;
    const int K = prm.K;
    int32_t *row = prm.out_draft + int64_t(r) * K;
    for (int j = lane; j < K; j += 32) row[j] = found ? __ldg(prm.tokens + o0 + p + m + (j % d)) : -1;
    if (lane == 0) {
        prm.out_len[r] = found ? K : (failed ? LOOKUP_DRAFT_LEN_FAILED : 0);
        prm.out_pos[r] = int32_t(p);
        if (prm.out_mlen) prm.out_mlen[r] = m;
    }
}

// ------------------------------------------------------------- host side ----
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

struct DeviceState {
    bool ready = false;
    int sms = 0;
    cudaMemPool_t pool = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device set-up, once: SM count, shared-memory opt-in, scratch pool.
int device_state(DeviceState **out) {
    int dev = 0;
    LD_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device index");
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        int sms = 0;
        LD_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        const ScanSmemLayout worst = scan_smem_layout(kOffCap - 1, LOOKUP_DRAFT_MAX_M);
        LD_CUDA(cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(worst.total)));
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
        st.ready = true;
    }
    *out = &st;
    return LOOKUP_DRAFT_OK;
}

int grid_for(const DeviceState &st) { return st.sms * kCtasPerSm; }

size_t workspace_bytes_for(int32_t B, int grid) { return (size_t(B) + size_t(grid)) * sizeof(unsigned long long); }

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
    prm.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    const ScanSmemLayout lay = scan_smem_layout(B, max_m);
    scan_kernel<<<prm.grid, kThreads, lay.total, stream>>>(prm);
    LD_CUDA(cudaGetLastError());
    return LOOKUP_DRAFT_OK;
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
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(unsigned((int64_t(B) + kFillWarps - 1) / kFillWarps));
    cfg.blockDim = dim3(kFillWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    LD_CUDA(cudaLaunchKernelEx(&cfg, fill_kernel, prm));
    return LOOKUP_DRAFT_OK;
}

int run_step(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m, int32_t K,
             int32_t *out_draft, int32_t *out_len, int32_t *out_pos, int32_t *out_mlen, cudaStream_t stream) {
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    void *ws = nullptr;
    LD_CUDA(cudaMallocFromPoolAsync(&ws, workspace_bytes_for(B, grid_for(*st)), st->pool, stream));
    auto *slots = static_cast<unsigned long long *>(ws);
    rc = launch_scan(*st, tokens, offsets, B, min_m, max_m, slots, stream);
    if (rc == LOOKUP_DRAFT_OK)
        rc = launch_fill(*st, tokens, offsets, B, K, slots, out_draft, out_len, out_pos, out_mlen, stream);
    cudaError_t fe = cudaFreeAsync(ws, stream);
    if (rc == LOOKUP_DRAFT_OK && fe != cudaSuccess) return cuda_fail(fe, "cudaFreeAsync");
    return rc;
}

}  // namespace

// ------------------------------------------------------------------ C ABI ----
extern "C" {

int lookup_draft_ex(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m,
                    int32_t K, int32_t *out_draft, int32_t *out_len, int32_t *out_pos, int32_t *out_mlen,
                    struct CUstream_st *stream) {
    g_cuda_msg[0] = '\0';
    int rc = check_common(tokens, offsets, B, min_m, max_m, K);
    if (rc == LOOKUP_DRAFT_OK) rc = check_outputs(B, K, out_draft, out_len, out_pos, out_mlen);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;
    return run_step(tokens, offsets, B, min_m, max_m, K, out_draft, out_len, out_pos, out_mlen, stream);
}

int lookup_draft(const int32_t *tokens, const int64_t *offsets, int32_t B, int32_t min_m, int32_t max_m, int32_t K,
                 int32_t *out_draft, int32_t *out_len, int32_t *out_pos, struct CUstream_st *stream) {
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
    const size_t tok_bytes = (n_tok * 4 + 15) & ~size_t(15);
    const size_t off_bytes = (size_t(B) + 1) * 8;
    const size_t out_words = size_t(B) * size_t(K) + 2 * size_t(B);
    const size_t ws_bytes = workspace_bytes_for(B, grid_for(*st));
    const size_t total = tok_bytes + ((off_bytes + 15) & ~size_t(15)) + ((out_words * 4 + 15) & ~size_t(15)) + ws_bytes;
    void *buf = nullptr;
    LD_CUDA(cudaMallocFromPoolAsync(&buf, total, st->pool, stream));
    unsigned char *base = static_cast<unsigned char *>(buf);
    int32_t *d_tok = reinterpret_cast<int32_t *>(base);
    int64_t *d_off = reinterpret_cast<int64_t *>(base + tok_bytes);
    int32_t *d_out = reinterpret_cast<int32_t *>(base + tok_bytes + ((off_bytes + 15) & ~size_t(15)));
    auto *d_ws = reinterpret_cast<unsigned long long *>(reinterpret_cast<unsigned char *>(d_out) +
                                                        ((out_words * 4 + 15) & ~size_t(15)));
    int32_t *d_draft = d_out;
    int32_t *d_len = d_out + size_t(B) * size_t(K);
    int32_t *d_pos = d_len + B;
    // The device copy holds tokens[first .. end); index it with the caller's offsets
    // through a base pointer moved back by `first` elements (never dereferenced there).
    const int32_t *d_tok_base =
        reinterpret_cast<const int32_t *>(reinterpret_cast<uintptr_t>(d_tok) - uintptr_t(first) * 4u);

    cudaError_t e = cudaSuccess;
    if (n_tok) e = cudaMemcpyAsync(d_tok, h_tokens + first, n_tok * 4, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_off, h_offsets, off_bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) {
        rc = launch_scan(*st, d_tok_base, d_off, B, min_m, max_m, d_ws, stream);
        if (rc == LOOKUP_DRAFT_OK)
            rc = launch_fill(*st, d_tok_base, d_off, B, K, d_ws, d_draft, d_len, d_pos, nullptr, stream);
    } else {
        rc = cuda_fail(e, "cudaMemcpyAsync (host to device)");
    }
    if (rc == LOOKUP_DRAFT_OK && K > 0)
        e = cudaMemcpyAsync(h_out_draft, d_draft, size_t(B) * size_t(K) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && e == cudaSuccess)
        e = cudaMemcpyAsync(h_out_len, d_len, size_t(B) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && e == cudaSuccess)
        e = cudaMemcpyAsync(h_out_pos, d_pos, size_t(B) * 4, cudaMemcpyDeviceToHost, stream);
    if (rc == LOOKUP_DRAFT_OK && e != cudaSuccess) rc = cuda_fail(e, "cudaMemcpyAsync (device to host)");
    cudaError_t fe = cudaFreeAsync(buf, stream);
    cudaError_t se = cudaStreamSynchronize(stream);
    if (rc == LOOKUP_DRAFT_OK && fe != cudaSuccess) rc = cuda_fail(fe, "cudaFreeAsync");
    if (rc == LOOKUP_DRAFT_OK && se != cudaSuccess) rc = cuda_fail(se, "cudaStreamSynchronize");
    return rc;
}

const char *lookup_draft_strerror(int code) {
    switch (code) {
    case LOOKUP_DRAFT_OK: return "ok";
    case LOOKUP_DRAFT_EINVAL: return "invalid argument";
    case LOOKUP_DRAFT_ECUDA: return "CUDA error";
    default: return "unknown lookup_draft status";
    }
}

const char *lookup_draft_last_cuda_error(void) { return g_cuda_msg; }

void lookup_draft_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : kDefaultWaitNs); }

}  // extern "C"
