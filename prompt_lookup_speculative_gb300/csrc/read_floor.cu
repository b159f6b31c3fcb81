// read_floor.cu -- a measurement aid: the time to stream a buffer from device
// memory with nothing else done, launched the way the draft step's kernels are
// (programmatic dependent launch).  Timed the same way as the scan over the same
// bytes, it gives the floor a single launch of any kernel that reads them once
// can reach here, against which the scan's fraction of the copy bandwidth is
// read.  The contract is in include/lookup_draft.h.

#include "lookup_draft.h"

#include "common.cuh"

#include <atomic>

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

// The same read with 1-D bulk copies (TMA) into shared memory, the way the scan
// reads its history: one CTA per SM (its rings pin one), each warp a contiguous
// range of the buffer streamed through a ring of kBulkBufs tiles of up to
// kBulkTileQuads quads, each waited for on its mbarrier and folded from shared
// memory.  Every wait is bounded by wait_ns from the CTA's start; a warp whose
// wait runs out stores kBulkTimedOut, waits for its copies in flight (bounded by
// kBulkDrainNs, never by the caller's limit: the CTA must not end while a copy
// still writes its shared memory) and stops.
constexpr int kBulkWarps = 16, kBulkBufs = 3, kBulkTileQuads = 192;
constexpr int kBulkTileBytes = kBulkTileQuads * 16;
constexpr size_t kBulkSmem = size_t(kBulkWarps) * kBulkBufs * (kBulkTileBytes + 8);
constexpr uint32_t kBulkTimedOut = 0xffffffffu;
constexpr uint64_t kBulkDrainNs = 1000000000ull;

struct BulkParams {
    const int4 *p;
    int64_t n16;
    uint32_t *out;
    uint64_t wait_ns;
};

__global__ void __launch_bounds__(kBulkWarps * 32) read_floor_bulk_kernel(BulkParams prm) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char *buf = smem + size_t(warp) * kBulkBufs * kBulkTileBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + size_t(kBulkWarps) * kBulkBufs * kBulkTileBytes) +
                     warp * kBulkBufs;
    const uint64_t deadline = lkd::global_ns() + prm.wait_ns;
    if (lane == 0) {
        for (int k = 0; k < kBulkBufs; ++k) lkd::mbar_init(lkd::smem_addr(&bars[k]), 1);
        lkd::fence_barrier_init();
    }
    __syncwarp();
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int64_t n16 = prm.n16;
    const int64_t nw = int64_t(gridDim.x) * kBulkWarps, v = int64_t(blockIdx.x) * kBulkWarps + warp;
    const int64_t per = (n16 + nw - 1) / nw;
    const int64_t lo = v * per < n16 ? v * per : n16;
    const int64_t hi = lo + per < n16 ? lo + per : n16;
    const int64_t ntile = (hi - lo + kBulkTileQuads - 1) / kBulkTileQuads;
    auto issue = [&](int64_t k) {                      // lane 0: tile k of the warp's range into buffer k mod kBulkBufs
        const int64_t q0 = lo + k * kBulkTileQuads;
        const int64_t nq = hi - q0 < kBulkTileQuads ? hi - q0 : kBulkTileQuads;
        const uint32_t bar = lkd::smem_addr(&bars[k % kBulkBufs]);
        lkd::mbar_expect_tx(bar, uint32_t(nq * 16));
        lkd::bulk_copy_g2s_stream(lkd::smem_addr(buf + (k % kBulkBufs) * kBulkTileBytes), prm.p + q0,
                                  uint32_t(nq * 16), bar);
    };
    if (lane == 0)
        for (int64_t k = 0; k < ntile && k < kBulkBufs; ++k) issue(k);
    uint32_t acc = 0;
    int64_t k = 0;
    bool ok = true;
    for (; k < ntile; ++k) {
        const uint32_t bar = lkd::smem_addr(&bars[k % kBulkBufs]), parity = uint32_t(k / kBulkBufs) & 1u;
        // the deadline is checked before every try (mbarrier.try_wait itself may
        // suspend until the copy lands), so a limit that has passed always fails
        if (!lkd::mbar_wait_until(bar, parity, deadline)) {
            ok = false;
            break;
        }
        const int64_t q0 = lo + k * kBulkTileQuads;
        const int nq = int(hi - q0 < kBulkTileQuads ? hi - q0 : kBulkTileQuads);
        const int4 *t = reinterpret_cast<const int4 *>(buf + (k % kBulkBufs) * kBulkTileBytes);
        for (int i = lane; i < nq; i += 32) {
            const int4 x = t[i];
            acc ^= uint32_t(x.x ^ x.y ^ x.z ^ x.w);
        }
        __syncwarp();                                   // every lane has read the buffer
        if (lane == 0 && k + kBulkBufs < ntile) {
            lkd::fence_proxy_async_smem();              // its next copy comes after those reads
            issue(k + kBulkBufs);
        }
    }
    if (!ok) {                                          // the copies issued from tile k on are still in flight
        if (lane == 0) *prm.out = kBulkTimedOut;
        const uint64_t drain = lkd::global_ns() + kBulkDrainNs;
        for (int64_t j = k; j < ntile && j < k + kBulkBufs; ++j)
            (void)lkd::mbar_wait_until(lkd::smem_addr(&bars[j % kBulkBufs]), uint32_t(j / kBulkBufs) & 1u, drain);
        return;
    }
    acc = __reduce_xor_sync(0xffffffffu, acc);
    if (acc == kNeverWritten && lane == 0) *prm.out = acc;
}

}  // namespace

extern "C" int lookup_draft_read_floor_bulk(const void *data, size_t bytes, uint32_t *out_word,
                                            struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_draft_read_floor_bulk");
    if (!out_word || (reinterpret_cast<uintptr_t>(out_word) & 3u) != 0 || (bytes > 0 && !data) ||
        (reinterpret_cast<uintptr_t>(data) & 15u) != 0 || (bytes & 15u) != 0)
        return LOOKUP_DRAFT_EINVAL;
    if (bytes == 0) return LOOKUP_DRAFT_OK;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    // the shared-memory opt-in is a per-device attribute: set once on each device
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> attr_set[kMaxDevices];
    int dev = 0;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess) return lookup_record_cuda_error(ge, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return lookup_record_cuda_error(cudaErrorInvalidDevice, "device index");
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            cudaFuncSetAttribute(read_floor_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kBulkSmem));
        if (e != cudaSuccess) return lookup_record_cuda_error(e, "cudaFuncSetAttribute");
        attr_set[dev].store(true, std::memory_order_release);
    }
    BulkParams prm;
    prm.p = static_cast<const int4 *>(data);
    prm.n16 = int64_t(bytes / 16);
    prm.out = out_word;
    prm.wait_ns = lookup_wait_limit_ns();
    return launch_pdl(read_floor_bulk_kernel, unsigned(sms), unsigned(kBulkWarps * 32), stream, prm, kBulkSmem);
}

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
