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

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

// Records a CUDA failure for lookup_draft_last_cuda_error (lookup_draft.cu);
// returns LOOKUP_DRAFT_ECUDA.
int lookup_record_cuda_error(cudaError_t e, const char *what);

namespace {

constexpr int kMaxBlock = 1 << 16;        // H + T (a verify block) at most
constexpr int kScanThreads = 1024;       // offsets_kernel
constexpr int kCopyThreads = 512;        // append_kernel
constexpr int kCopyCtasPerSm = 4;
constexpr int kCopyUnroll = 2;

__device__ inline void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ inline void wait_for_prerequisite_grid() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

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

// One thread per (request, block position).
__global__ void fuse_kernel(FuseParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int W = p.H + p.T;
    const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= int64_t(p.B) * W) return;
    const int r = int(idx / W), i = int(idx - int64_t(r) * W);
    const int32_t *ld = p.lookup_draft + int64_t(r) * p.K;
    const int32_t *md = p.model_draft + int64_t(r) * p.H;
    const int32_t m = p.lookup_mlen[r];
    bool agree = true;
    for (int j = 0; j < p.agree_n; ++j) agree = agree && ld[j] == md[j];
    const bool head_lookup = m >= p.replace_min || (m >= p.agree_min && agree);
    const bool tail = p.long_block != nullptr && p.long_block[r] != 0 && m >= p.tail_min;
    int32_t v, pm;
    if (i < p.H) {
        v = head_lookup ? ld[i] : md[i];
        pm = head_lookup;
    } else {
        v = tail ? ld[i] : -1;
        pm = tail;
    }
    p.out_block[idx] = v;
    p.out_pm[idx] = pm;
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

// One thread per request: {long, streak, hold} updated in place.
__global__ void schedule_kernel(ScheduleParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= p.B) return;
    int32_t *st = p.state + 3 * int64_t(r);
    int32_t lng = st[0], streak = st[1], hold = st[2];
    const int32_t full = (lng ? p.H + p.T : p.H) + 1;
    const bool cond = p.lookup_mlen[r] >= p.tail_min && p.committed[r] >= full - p.slack;
    streak = cond ? streak + 1 : 0;
    if (!lng) {
        if (streak >= p.enter_steps) {
            lng = 1;
            hold = p.sticky;
        }
    } else if (cond) {
        hold = p.sticky;
    } else if (hold > 0) {
        --hold;                                          // sticky exit: the long block is kept
    } else {
        lng = 0;
    }
    st[0] = lng;
    st[1] = streak;
    st[2] = hold;
    p.out_long[r] = lng;
}

// ------------------------------------------------------------ verification ----
struct VerifyParams {
    const int32_t *block;
    const int32_t *len;
    const int32_t *target;
    const float *probs;
    const float *qprobs;
    const int32_t *point_mass;
    const float *u;
    int32_t *out_accepted;
    int32_t *out_commit;
    int32_t *out_ncommit;
    int32_t B, P;
};

constexpr int kVerifyWarps = 4;

// One warp per request: lanes test positions, the first failure (a ballot)
// is the accepted length.
__global__ void verify_kernel(VerifyParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kVerifyWarps + (threadIdx.x >> 5);
    if (r >= p.B) return;
    const int64_t o = int64_t(r) * p.P;
    const int32_t len = p.len[r];
    int32_t *commit = p.out_commit + int64_t(r) * (p.P + 1);
    if (len < 0 || len > p.P) {                          // no valid block: an error row
        for (int i = lane; i <= p.P; i += 32) commit[i] = -1;
        if (lane == 0) {
            p.out_accepted[r] = -1;
            p.out_ncommit[r] = 0;
        }
        return;
    }
    int32_t a = len;
    for (int base = 0; base < len; base += 32) {
        const int i = base + lane;
        bool ok = true;
        if (i < len) {
            if (p.probs == nullptr) {
                ok = p.block[o + i] == p.target[int64_t(r) * (p.P + 1) + i];
            } else {
                float q = p.qprobs ? p.qprobs[o + i] : 1.0f;
                if (p.point_mass && p.point_mass[o + i]) q = 1.0f;   // the point-mass rewrite
                ok = __fmul_rn(p.u[o + i], q) < p.probs[o + i];
            }
        }
        const unsigned bad = __ballot_sync(0xffffffffu, !ok);
        if (bad) {
            a = base + __ffs(bad) - 1;
            break;
        }
    }
    for (int i = lane; i <= p.P; i += 32)
        commit[i] = i < a ? p.block[o + i] : (i == a ? p.target[int64_t(r) * (p.P + 1) + a] : -1);
    if (lane == 0) {
        p.out_accepted[r] = a;
        p.out_ncommit[r] = a + 1;
    }
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

// The new boundaries: out_offsets[r] = (offsets[r] - offsets[0]) + sum(ncommit[0..r)),
// one CTA scanning the counts in blocks of kScanThreads.
__global__ void __launch_bounds__(kScanThreads) offsets_kernel(AppendParams p) {
    __shared__ int64_t warp_sums[kScanThreads / 32];
    __shared__ int64_t carry_s;
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t base = p.offsets[0];
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int64_t r0 = 0; r0 < p.B; r0 += kScanThreads) {
        const int64_t r = r0 + tid;
        int64_t x = r < p.B ? int64_t(min(max(p.ncommit[r], 0), p.W)) : 0;   // clamped to [0, W]
        int64_t incl = x;                                // inclusive scan within the warp
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
            warp_sums[lane] = s;                         // inclusive over warps
        }
        __syncthreads();
        const int64_t carry = carry_s;
        const int64_t before = carry + (warp ? warp_sums[warp - 1] : 0) + incl - x;   // exclusive
        if (r < p.B) p.out_offsets[r] = (p.offsets[r] - base) + before;
        __syncthreads();
        if (tid == kScanThreads - 1) carry_s = carry + warp_sums[kScanThreads / 32 - 1];
        __syncthreads();
    }
    if (tid == 0) p.out_offsets[p.B] = (p.offsets[p.B] - base) + carry_s;
}

// Copy: CTA c writes the output quads [c*Sq, (c+1)*Sq) (4 tokens each).  Thread
// t takes quads t, t + kCopyThreads, ... of its CTA's range, kCopyUnroll of them
// per pass, so a warp reads and writes 512 contiguous bytes per quad step; the
// request of each token comes from a monotone walk over the new boundaries.
// Sources are read token by token (a history's shift into the new batch is the
// running sum of earlier commits, so it has no fixed alignment); with kVec the
// quad is written with one 16-byte store (out_tokens 16-byte aligned).
template <bool kVec>
__global__ void __launch_bounds__(kCopyThreads, kCopyCtasPerSm) append_kernel(AppendParams p) {
    wait_for_prerequisite_grid();                        // out_offsets are ready
    allow_dependent_launch();
    const int64_t total = p.out_offsets[p.B];
    const int64_t nquad = (total + 3) >> 2;
    const int64_t Sq = (nquad + gridDim.x - 1) / gridDim.x;
    const int64_t x0 = int64_t(blockIdx.x) * Sq * 4;
    const int64_t x1 = (x0 + Sq * 4 < total) ? x0 + Sq * 4 : total;
    if (x0 >= x1) return;
    // the request holding x0: the largest r with out_offsets[r] <= x0
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
        const int mid = lo + ((hi - lo) >> 1);
        if (p.out_offsets[mid] <= x0) lo = mid; else hi = mid;
    }
    int r = lo;
    int64_t nstart = p.out_offsets[r], nend = p.out_offsets[r + 1];
    int64_t hist = p.offsets[r + 1] - p.offsets[r];
    const int32_t *src = p.tokens + p.offsets[r];
    const int32_t *crow = p.commit + int64_t(r) * p.W;
    for (int64_t xb = x0 + 4 * threadIdx.x; xb < x1; xb += int64_t(4) * kCopyThreads * kCopyUnroll) {
        int32_t v[kCopyUnroll][4];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t x = xb + int64_t(4) * kCopyThreads * u + k;
                v[u][k] = 0;
                if (x < x1) {
                    while (x >= nend) {                  // into the next request
                        ++r;
                        nstart = nend;
                        nend = p.out_offsets[r + 1];
                        hist = p.offsets[r + 1] - p.offsets[r];
                        src = p.tokens + p.offsets[r];
                        crow = p.commit + int64_t(r) * p.W;
                    }
                    const int64_t i = x - nstart;        // position in the new history
                    v[u][k] = i < hist ? __ldg(src + i) : __ldg(crow + (i - hist));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t x = xb + int64_t(4) * kCopyThreads * u;
            if (kVec && x + 4 <= x1) {
                *reinterpret_cast<int4 *>(p.out_tokens + x) = make_int4(v[u][0], v[u][1], v[u][2], v[u][3]);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (x + k < x1) p.out_tokens[x + k] = v[u][k];
            }
        }
    }
}

// ------------------------------------------------------------------- host ----
int cuda_fail(cudaError_t e, const char *what) { return lookup_record_cuda_error(e, what); }

template <typename Params>
int launch_pdl(void (*kernel)(Params), dim3 grid, dim3 block, cudaStream_t stream, const Params &prm) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
    return e == cudaSuccess ? LOOKUP_DRAFT_OK : cuda_fail(e, "kernel launch");
}

unsigned blocks_for(int64_t n, int per) { return unsigned((n + per - 1) / per); }

}  // namespace

extern "C" {

int lookup_fuse(const int32_t *lookup_draft, const int32_t *lookup_mlen, const int32_t *model_draft,
                const int32_t *long_block, int32_t B, int32_t K, int32_t H, int32_t T, int32_t replace_min,
                int32_t agree_min, int32_t agree_n, int32_t tail_min, int32_t *out_block, int32_t *out_len,
                int32_t *out_point_mass, struct CUstream_st *stream) {
    if (B < 0 || H < 1 || T < 0 || int64_t(H) + T > kMaxBlock || K < H + T || agree_n < 0 || agree_n > H)
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_draft || !lookup_mlen || !model_draft || !out_block || !out_len || !out_point_mass)
        return LOOKUP_DRAFT_EINVAL;
    FuseParams p{lookup_draft, lookup_mlen, model_draft, long_block, out_block, out_len, out_point_mass,
                 B, K, H, T, replace_min, agree_min, agree_n, tail_min};
    return launch_pdl(fuse_kernel, dim3(blocks_for(int64_t(B) * (H + T), 256)), dim3(256), stream, p);
}

int lookup_schedule(const int32_t *lookup_mlen, const int32_t *committed, int32_t B, int32_t H, int32_t T,
                    int32_t tail_min, int32_t slack, int32_t enter_steps, int32_t sticky, int32_t *state,
                    int32_t *out_long, struct CUstream_st *stream) {
    if (B < 0 || H < 1 || T < 0 || enter_steps < 1 || sticky < 0 || slack < 0) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!lookup_mlen || !committed || !state || !out_long) return LOOKUP_DRAFT_EINVAL;
    ScheduleParams p{lookup_mlen, committed, state, out_long, B, H, T, tail_min, slack, enter_steps, sticky};
    return launch_pdl(schedule_kernel, dim3(blocks_for(B, 256)), dim3(256), stream, p);
}

int lookup_verify(const int32_t *block, const int32_t *len, const int32_t *target, const float *probs,
                  const float *qprobs, const int32_t *point_mass, const float *u, int32_t B, int32_t P,
                  int32_t *out_accepted, int32_t *out_commit, int32_t *out_ncommit, struct CUstream_st *stream) {
    if (B < 0 || P < 0 || P > kMaxBlock) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if ((P > 0 && !block) || !len || !target || (probs && !u) || !out_accepted || !out_commit || !out_ncommit)
        return LOOKUP_DRAFT_EINVAL;
    VerifyParams p{block, len, target, probs, qprobs, point_mass, u, out_accepted, out_commit, out_ncommit, B, P};
    return launch_pdl(verify_kernel, dim3(blocks_for(B, kVerifyWarps)), dim3(kVerifyWarps * 32), stream, p);
}

int lookup_append(const int32_t *tokens, const int64_t *offsets, const int32_t *commit, const int32_t *ncommit,
                  int32_t B, int32_t W, int32_t *out_tokens, int64_t *out_offsets, struct CUstream_st *stream) {
    if (B < 0 || W < 0) return LOOKUP_DRAFT_EINVAL;
    if (!offsets || !out_offsets || (B > 0 && (!tokens || !ncommit || (W > 0 && !commit) || !out_tokens)))
        return LOOKUP_DRAFT_EINVAL;
    AppendParams p{tokens, offsets, commit, ncommit, out_tokens, out_offsets, B, W};
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    int rc = launch_pdl(offsets_kernel, dim3(1), dim3(kScanThreads), stream, p);
    if (rc != LOOKUP_DRAFT_OK || B == 0) return rc;      // B == 0: out_offsets = {0} only
    const bool vec = (reinterpret_cast<uintptr_t>(out_tokens) & 15) == 0;
    return launch_pdl(vec ? append_kernel<true> : append_kernel<false>, dim3(unsigned(sms * kCopyCtasPerSm)),
                      dim3(kCopyThreads), stream, p);
}

}  // extern "C"
