// read_floor.cu -- a measurement aid: the time to stream a buffer from device
// memory with nothing else done, launched the way the draft step's kernels are
// (programmatic dependent launch).  Timed the same way as the scan over the same
// bytes, it gives the floor a single launch of any kernel that reads them once
// can reach here, against which the scan's fraction of the copy bandwidth is
// read.  The contract is in include/lookup_draft.h.

#include "lookup_draft.h"

#include "common.cuh"

namespace {

using lkd::allow_dependent_launch;
using lkd::launch_pdl;
using lkd::sm_count;
using lkd::wait_for_prerequisite_grid;

constexpr int kUnroll = 4;                       // 16-byte loads in flight per thread
constexpr uint32_t kNeverWritten = 0x5eed1e55u;  // the result is stored only if it equals this

// A 16-byte read-only load with an L2 evict-first policy, the policy the scan's
// history copies use.
__device__ __forceinline__ int4 load_stream(const int4 *p, uint64_t policy) {
    int4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.s32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

struct FloorParams {
    const int4 *p;
    int64_t n16;
    uint32_t *out;
};

// Contiguous chunk per CTA, kUnroll independent 16-byte loads per thread per
// iteration (L2 evict-first, as the scan's copies), all folded by XOR.  The fold
// is stored only when it equals a fixed pattern, so the loads cannot be dropped
// and almost no launch writes anything.
__global__ void read_floor_kernel(FloorParams prm) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int4 *__restrict__ p = prm.p;
    const int64_t n16 = prm.n16;
    const int64_t per = (n16 + gridDim.x - 1) / gridDim.x;
    const int64_t b = int64_t(blockIdx.x) * per;
    const int64_t e = b + per < n16 ? b + per : n16;
    const int64_t step = blockDim.x;
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    uint32_t acc = 0;
    int64_t i = b + threadIdx.x;
    for (; i + (kUnroll - 1) * step < e; i += kUnroll * step) {
        int4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = load_stream(p + i + u * step, policy);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc ^= uint32_t(v[u].x ^ v[u].y ^ v[u].z ^ v[u].w);
    }
    for (; i < e; i += step) {
        const int4 v = load_stream(p + i, policy);
        acc ^= uint32_t(v.x ^ v.y ^ v.z ^ v.w);
    }
    acc = __reduce_xor_sync(0xffffffffu, acc);
    if (acc == kNeverWritten && (threadIdx.x & 31) == 0) *prm.out = acc;
}

}  // namespace

extern "C" int lookup_draft_read_floor(const void *data, size_t bytes, int32_t ctas_per_sm, int32_t threads,
                                       uint32_t *out_word, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_draft_read_floor");
    if (!out_word || (reinterpret_cast<uintptr_t>(out_word) & 3u) != 0 || (bytes > 0 && !data) ||
        (reinterpret_cast<uintptr_t>(data) & 15u) != 0 || (bytes & 15u) != 0 || ctas_per_sm < 1 ||
        ctas_per_sm > 32 || threads < 32 || threads > 1024 || (threads & 31) != 0)
        return LOOKUP_DRAFT_EINVAL;
    if (bytes == 0) return LOOKUP_DRAFT_OK;
    int sms = 0;
    const int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    FloorParams prm;
    prm.p = static_cast<const int4 *>(data);
    prm.n16 = int64_t(bytes / 16);
    prm.out = out_word;
    return launch_pdl(read_floor_kernel, unsigned(sms * ctas_per_sm), unsigned(threads), stream, prm);
}
