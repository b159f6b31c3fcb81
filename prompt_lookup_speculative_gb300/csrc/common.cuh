// common.cuh -- device and host helpers shared by the library's kernels (private).
#pragma once

#include "lookup_draft.h"

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

// Records a CUDA failure for lookup_draft_last_cuda_error (lookup_draft.cu);
// returns LOOKUP_DRAFT_ECUDA.
int lookup_record_cuda_error(cudaError_t e, const char *what);
// Counts one enqueued kernel launch (lookup_draft_launch_count, lookup_draft.cu).
void lookup_note_launch();
// The limit on a kernel's bounded waits, in ns (lookup_draft_set_wait_limit_ns).
uint64_t lookup_wait_limit_ns();

namespace lkd {

// Programmatic dependent launch: wait for the previous kernel on the stream
// (its writes visible), and let the next one start launching.
__device__ inline void wait_for_prerequisite_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ inline void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Long-block scheduling (HyperQwen lookup-drafting article, section "第3步"): one
// update of a request's {long, streak, hold} from this step's match length m and
// the previous step's commit count.  full = the tokens a fully accepted block of
// the previous step commits; the condition is a usable match and a nearly full
// commit; `enter_steps` consecutive steps enter the long block, and it is kept for
// `sticky` steps after the condition first fails.
__device__ inline void schedule_update(int32_t m, int32_t committed, int32_t H, int32_t T, int32_t tail_min,
                                       int32_t slack, int32_t enter_steps, int32_t sticky, int32_t &lng,
                                       int32_t &streak, int32_t &hold) {
    const int32_t full = (lng ? H + T : H) + 1;
    const bool cond = m >= tail_min && committed >= full - slack;
    streak = cond ? streak + 1 : 0;
    if (!lng) {
        if (streak >= enter_steps) {
            lng = 1;
            hold = sticky;
        }
    } else if (cond) {
        hold = sticky;
    } else if (hold > 0) {
        --hold;                                          // sticky exit: the long block is kept
    } else {
        lng = 0;
    }
}

// Fusion ("第2步"), block position i: the head (i < H) takes the lookup token when
// the head rule holds, else the model's; the tail takes the lookup token when the
// tail rule holds, else -1.  A lookup token is a point mass.
__device__ inline void fuse_choice(int32_t i, int32_t H, bool head_lookup, bool tail, int32_t lookup_tok,
                                   int32_t model_tok, int32_t &v, int32_t &pm) {
    if (i < H) {
        v = head_lookup ? lookup_tok : model_tok;
        pm = head_lookup;
    } else {
        v = tail ? lookup_tok : -1;
        pm = tail;
    }
}

// The decode loop's scheduling and fusion for one request, in the warp that holds
// its lookup draft: lanes hold draft tokens j = lane and lane + 32 (-1 without a
// match), m is the match length (0 without one), W = H + T <= 64.  Every lane
// reads the old state and applies the rule, the warp synchronises, lane 0 writes
// the new state, the long flag and the block length, and the lanes write the
// block's positions: lookup_schedule then lookup_fuse, for that request.
struct PlanIO {
    const int32_t *model_draft;   // [B][H]
    const int32_t *committed;     // [B]
    int32_t *state;               // [B][3] in/out
    int32_t *out_long;
    int32_t *out_block;           // [B][H + T]
    int32_t *out_len;
    int32_t *out_pm;              // [B][H + T]
    int32_t H, T, replace_min, agree_min, agree_n, tail_min, slack, enter_steps, sticky;
};

// A request's inputs to the rules, read by each lane: the model's proposals j =
// lane and lane + 32, the commit count and the old state.
struct PlanIn {
    int32_t md0, md1, committed, lng, streak, hold;
};

__device__ inline PlanIn plan_load(const PlanIO &pa, int r, int lane) {
    const int32_t *md = pa.model_draft + int64_t(r) * pa.H;
    const int32_t *st = pa.state + 3 * int64_t(r);
    const int j1 = lane + 32;
    return PlanIn{lane < pa.H ? md[lane] : -1, j1 < pa.H ? md[j1] : -1, pa.committed[r], st[0], st[1], st[2]};
}

__device__ inline void plan_apply(const PlanIO &pa, int r, int lane, int32_t m, int32_t tok0, int32_t tok1,
                                  const PlanIn &in) {
    const int W = pa.H + pa.T;
    const int j1 = lane + 32;
    // head rule: the model agrees with the draft's first agree_n tokens
    const bool ne = (lane < pa.agree_n && tok0 != in.md0) || (j1 < pa.agree_n && tok1 != in.md1);
    const bool agree = __all_sync(0xffffffffu, !ne);
    const bool head = m >= pa.replace_min || (m >= pa.agree_min && agree);
    // scheduling: every lane holds the old state, then lane 0 writes the new one
    int32_t *st = pa.state + 3 * int64_t(r);
    int32_t lng = in.lng, streak = in.streak, hold = in.hold;
    schedule_update(m, in.committed, pa.H, pa.T, pa.tail_min, pa.slack, pa.enter_steps, pa.sticky, lng, streak,
                    hold);
    __syncwarp();
    const bool tail = lng != 0 && m >= pa.tail_min;
    if (lane == 0) {
        st[0] = lng;
        st[1] = streak;
        st[2] = hold;
        pa.out_long[r] = lng;
        pa.out_len[r] = tail ? W : pa.H;
    }
    // fusion of the block's positions
    int32_t v, pm;
    if (lane < W) {
        fuse_choice(lane, pa.H, head, tail, tok0, in.md0, v, pm);
        pa.out_block[int64_t(r) * W + lane] = v;
        pa.out_pm[int64_t(r) * W + lane] = pm;
    }
    if (j1 < W) {
        fuse_choice(j1, pa.H, head, tail, tok1, in.md1, v, pm);
        pa.out_block[int64_t(r) * W + j1] = v;
        pa.out_pm[int64_t(r) * W + j1] = pm;
    }
}

__device__ inline void plan_warp(const PlanIO &pa, int r, int lane, int32_t m, int32_t tok0, int32_t tok1) {
    plan_apply(pa, r, lane, m, tok0, tok1, plan_load(pa, r, lane));
}

// Verification of request r's proposal block by one warp (HyperQwen lookup-drafting
// article, "第3步"): the accepted length a is the first position that fails, greedy
// (the target's token differs) or sampled (u * q >= p in float32, q = 1 at a
// point mass); the commit row holds the accepted tokens, then the target's token
// at a, then -1.  A block length outside [0, P] gives an error row (accepted -1,
// no committed token).  Blocks are [B, P], the target rows [B, P + 1].
constexpr int kMaxBlock = 1 << 16;        // positions of a verify block (H + T) at most

struct VerifyIO {
    const int32_t *block, *len, *target;
    const float *probs, *qprobs;
    const int32_t *point_mass;
    const float *u;
    int32_t *out_accepted, *out_commit, *out_ncommit;
    int32_t P;
};

__device__ inline void verify_warp(const VerifyIO &v, int r, int lane) {
    const int64_t o = int64_t(r) * v.P;
    const int32_t len = v.len[r];
    int32_t *commit = v.out_commit + int64_t(r) * (v.P + 1);
    if (len < 0 || len > v.P) {                          // no valid block: an error row
        for (int i = lane; i <= v.P; i += 32) commit[i] = -1;
        if (lane == 0) {
            v.out_accepted[r] = -1;
            v.out_ncommit[r] = 0;
        }
        return;
    }
    int32_t a = len;
    for (int base = 0; base < len; base += 32) {
        const int i = base + lane;
        bool ok = true;
        if (i < len) {
            if (v.probs == nullptr) {
                ok = v.block[o + i] == v.target[int64_t(r) * (v.P + 1) + i];
            } else {
                float q = v.qprobs ? v.qprobs[o + i] : 1.0f;
                if (v.point_mass && v.point_mass[o + i]) q = 1.0f;   // the point-mass rewrite
                ok = __fmul_rn(v.u[o + i], q) < v.probs[o + i];
            }
        }
        const unsigned bad = __ballot_sync(0xffffffffu, !ok);
        if (bad) {
            a = base + __ffs(bad) - 1;
            break;
        }
    }
    for (int i = lane; i <= v.P; i += 32)
        commit[i] = i < a ? v.block[o + i] : (i == a ? v.target[int64_t(r) * (v.P + 1) + a] : -1);
    if (lane == 0) {
        v.out_accepted[r] = a;
        v.out_ncommit[r] = a + 1;
    }
}

// Shared memory addresses, mbarriers, 1-D bulk copies (TMA) and the global timer.
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

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.  Both
// addresses and the size are multiples of 16 bytes.
__device__ inline void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// The same copy with an L2 evict-first policy, for history tiles: each is read
// once, so the lines that are used again across launches (the kernels' code, the
// slots, the offsets) are the ones kept in L2.
__device__ inline void bulk_copy_g2s_stream(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ inline void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
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

// Wait for phase `parity` of `bar` to complete; false once the global timer has
// passed `deadline_ns` (checked before every try, so a past deadline fails at once).
__device__ inline bool mbar_wait_until(uint32_t bar, uint32_t parity, uint64_t deadline_ns) {
    for (;;) {
        if (global_ns() > deadline_ns) return false;
        if (mbar_try_wait(bar, parity)) return true;
    }
}

// splitmix64's output mix (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014).
__device__ inline uint64_t mix64(uint64_t x) {
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    x ^= x >> 31;
    return x;
}

// 128-bit compare-and-swap at a 16-byte aligned global address (atom.cas.b128,
// sm_90 and later); returns the previous 128 bits.
__device__ inline void cas128(void *addr, uint64_t cmp_lo, uint64_t cmp_hi, uint64_t new_lo, uint64_t new_hi,
                              uint64_t &old_lo, uint64_t &old_hi) {
    asm volatile(
        "{\n\t.reg .b128 d, c, v;\n\t"
        "mov.b128 c, {%2, %3};\n\t"
        "mov.b128 v, {%4, %5};\n\t"
        "atom.global.cas.b128 d, [%6], c, v;\n\t"
        "mov.b128 {%0, %1}, d;\n\t}"
        : "=l"(old_lo), "=l"(old_hi)
        : "l"(cmp_lo), "l"(cmp_hi), "l"(new_lo), "l"(new_hi), "l"(addr)
        : "memory");
}

// Host: launch with programmatic stream serialization allowed (and `smem` bytes
// of dynamic shared memory).
template <typename Params>
inline int launch_pdl(void (*kernel)(Params), unsigned grid, unsigned block, cudaStream_t stream, const Params &prm,
                      size_t smem = 0) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
    if (e != cudaSuccess) return lookup_record_cuda_error(e, "kernel launch");
    lookup_note_launch();
    return LOOKUP_DRAFT_OK;
}

// The same for a kernel of two parameter structs.
template <typename P1, typename P2>
inline int launch_pdl2(void (*kernel)(P1, P2), unsigned grid, unsigned block, cudaStream_t stream, const P1 &a,
                       const P2 &b) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, b);
    if (e != cudaSuccess) return lookup_record_cuda_error(e, "kernel launch");
    lookup_note_launch();
    return LOOKUP_DRAFT_OK;
}

inline int sm_count(int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    return e == cudaSuccess ? LOOKUP_DRAFT_OK : lookup_record_cuda_error(e, "device query");
}

inline bool pow2_at_least(int64_t x, int64_t lo) { return x >= lo && (x & (x - 1)) == 0; }

inline unsigned capped_grid(int64_t want, int64_t cap) {
    if (want < 1) want = 1;
    return unsigned(want < cap ? want : cap);
}

// An NVTX range over one library call: a span per call in a timeline tool,
// nearly free when no tool is attached (header-only NVTX).
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

}  // namespace lkd
