// lookup_ctxcache.cu -- context-cache drafting (the most frequent next token of
// the longest recent n-gram) from device-resident n-gram statistics.
//
// Source: llama.cpp prompt-lookup article, ai-blog.deepmagic.app, "從 165 微秒到
// 1.18 微秒", section "Prompt lookup decoding 到底是什麼".  The contract is in
// include/lookup_ctxcache.h.
//
// Table: a 128-byte header, then 32-byte slots {key (two 64-bit words), v0, v1}
// in buckets of 2.  A key is the exact (r, n, g, x) packed into 128 bits, so two
// n-grams never share a slot; only the bucket is hashed.  Tokens enter keys as
// 21-bit codes: a token in [0, 2^20) is its own code, and any other int32 value
// gets a code in [2^20, 2^21) from a dictionary kept in the same table, so the
// statistics are exact on every int32 value.  Three kinds of key:
//   COUNT (r, n, g, x): v0 = how many occurrences of g are followed by x;
//   CTX   (r, n, g):    v0 = occurrences of g that have a next token,
//                       v1 = max over x of (count(g, x) << 32 | order(x)),
//                       order(x) = 2^32 - 1 - (x + 2^31) as unsigned, so the
//                       maximum is the smallest signed token with the count;
//   CODE  (c):          v0 = 2^32 | the token value that owns dictionary code c.
// Counting an occurrence of g followed by x is an atomicAdd on COUNT (giving the
// new count c), an atomicAdd on CTX.v0 and an atomicMax of (c << 32 | order(x))
// on CTX.v1.  Counts only grow, so v1 ends as (the largest count, the smallest
// token with that count) in any order of updates: the build counts every
// position of every history in parallel.  A slot is claimed with one 128-bit CAS
// of its key.  A value outside [0, 2^20) owns the first code of its probe
// sequence (a hash of the value, then the following codes) that was free when it
// asked or already is its own; a code is taken with one CAS of its CODE slot's
// value, so racing claimants of one value agree and no code is wasted.  The draft is one
// warp per request, one token per round: lane l reads the CTX slot of the
// context's last (n_max - l) tokens, the longest length that passes the
// thresholds gives the token, and the context window (four tokens and their
// codes, one per lane) shifts by a shuffle.

#include "lookup_ctxcache.h"

#include "common.cuh"

namespace {

using lkd::allow_dependent_launch;
using lkd::cas128;
using lkd::launch_pdl;
using lkd::mix64;
using lkd::sm_count;
using lkd::wait_for_prerequisite_grid;

constexpr uint32_t kMagic = 0x4c4b4358u;        // "LKCX"
constexpr int kBucket = 2;                      // slots per bucket: one 64-byte pair of sectors
constexpr int kMaxProbe = 2048;                 // buckets probed before the overflow flag
constexpr int kCodeBits = 21;                   // token code width in a key
constexpr int32_t kDirect = 1 << 20;            // tokens in [0, kDirect) are their own code
constexpr uint32_t kMaxCodes = 1u << 20;        // dictionary codes: kDirect + [0, kMaxCodes)
constexpr int kCodeProbe = 4096;                // codes tried per value before the overflow flag
constexpr int kThreads = 256;
constexpr int kDraftThreads = 128;              // 4 warps per CTA, one request each
constexpr int kScanThreads = 1024;
constexpr int kMaxN = 4;

struct __align__(16) Header {
    uint32_t magic;
    int32_t n_min, n_max, pad0;
    int64_t slots;
    uint32_t overflow;                          // a key found no slot, or a value found no code
    uint32_t pad[25];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

struct __align__(32) Slot {
    unsigned long long lo, hi, v0, v1;
};
static_assert(sizeof(Slot) == 32, "slot is 32 bytes");

enum Kind { kCount = 0, kCtx = 1 };

// g: the codes of the n tokens, oldest first (unused entries 0); x: a code.  Bits:
// lo = g0 | g1 << 21 | g2 << 42 | kind << 63, hi = g3 | x << 21 | n << 42 | r << 45.
// n >= 1 keeps every such key non-zero and apart from the dictionary's CODE keys (n = 0).
__device__ inline void make_key(int r, int n, const int32_t (&g)[kMaxN], int kind, int32_t x, uint64_t &lo,
                                uint64_t &hi) {
    lo = uint64_t(uint32_t(g[0])) | (uint64_t(uint32_t(g[1])) << kCodeBits) |
         (uint64_t(uint32_t(g[2])) << (2 * kCodeBits)) | (uint64_t(kind) << 63);
    hi = uint64_t(uint32_t(g[3])) | (uint64_t(uint32_t(x)) << kCodeBits) | (uint64_t(n) << (2 * kCodeBits)) |
         (uint64_t(uint32_t(r)) << (2 * kCodeBits + 3));
}

// The key of dictionary code c (bit 61 of hi; n = 0), and the mark of its owner v.
__device__ inline void code_key(uint32_t c, uint64_t &lo, uint64_t &hi) {
    lo = c;
    hi = 1ull << 61;
}
__device__ inline unsigned long long owner_mark(int32_t v) { return (1ull << 32) | uint32_t(v); }
__device__ inline uint32_t first_code(int32_t v) { return uint32_t(mix64(uint32_t(v))) & (kMaxCodes - 1u); }

// Order of a token among equal counts: larger for smaller signed values.
__device__ inline uint64_t tie_order(int32_t x) { return 0xffffffffull - uint64_t(uint32_t(x) ^ 0x80000000u); }
__device__ inline int32_t from_tie_order(uint64_t low) { return int32_t(uint32_t(0xffffffffull - low) ^ 0x80000000u); }

__device__ inline int64_t bucket_of(uint64_t lo, uint64_t hi, int64_t bmask) {
    return int64_t(mix64(lo ^ mix64(hi)) & uint64_t(bmask));
}

__device__ inline bool header_ok(const Header *hd, int n_min, int n_max, int64_t slots) {
    return hd->magic == kMagic && hd->n_min == n_min && hd->n_max == n_max && hd->slots == slots;
}

// The slot of key (lo, hi), claimed if absent; nullptr (and the overflow flag)
// when no slot was found.  Slots never empty again and every claim scans in the
// same order, so an empty slot means the key is not stored further on.
__device__ inline Slot *claim(Slot *tab, int64_t bmask, uint64_t lo, uint64_t hi, Header *hd) {
    int64_t b = bucket_of(lo, hi, bmask);
    for (int probe = 0; probe < kMaxProbe; ++probe) {
        Slot *sb = tab + b * kBucket;
        int4 k[kBucket];
#pragma unroll
        for (int s = 0; s < kBucket; ++s) k[s] = __ldcg(reinterpret_cast<const int4 *>(sb + s));
#pragma unroll
        for (int s = 0; s < kBucket; ++s) {
            uint64_t klo = uint64_t(uint32_t(k[s].x)) | (uint64_t(uint32_t(k[s].y)) << 32);
            uint64_t khi = uint64_t(uint32_t(k[s].z)) | (uint64_t(uint32_t(k[s].w)) << 32);
            if (klo == 0ull && khi == 0ull) cas128(sb + s, 0ull, 0ull, lo, hi, klo, khi);
            if ((klo == 0ull && khi == 0ull) || (klo == lo && khi == hi)) return sb + s;
        }
        b = (b + 1) & bmask;
    }
    atomicOr(&hd->overflow, 1u);
    return nullptr;
}

// Values of key (lo, hi): false when absent.
__device__ inline bool find(const Slot *tab, int64_t bmask, uint64_t lo, uint64_t hi, unsigned long long &v0,
                            unsigned long long &v1) {
    int64_t b = bucket_of(lo, hi, bmask);
    for (int probe = 0; probe < kMaxProbe; ++probe) {
        const int4 *sb = reinterpret_cast<const int4 *>(tab + b * kBucket);
        int4 w[2 * kBucket];
#pragma unroll
        for (int s = 0; s < 2 * kBucket; ++s) w[s] = __ldcg(sb + s);
#pragma unroll
        for (int s = 0; s < kBucket; ++s) {
            const uint64_t klo = uint64_t(uint32_t(w[2 * s].x)) | (uint64_t(uint32_t(w[2 * s].y)) << 32);
            const uint64_t khi = uint64_t(uint32_t(w[2 * s].z)) | (uint64_t(uint32_t(w[2 * s].w)) << 32);
            if (klo == lo && khi == hi) {
                v0 = uint64_t(uint32_t(w[2 * s + 1].x)) | (uint64_t(uint32_t(w[2 * s + 1].y)) << 32);
                v1 = uint64_t(uint32_t(w[2 * s + 1].z)) | (uint64_t(uint32_t(w[2 * s + 1].w)) << 32);
                return true;
            }
            if (klo == 0ull && khi == 0ull) return false;
        }
        b = (b + 1) & bmask;
    }
    return false;
}

// The code of token v if it has one (read only); -1 when v owns no code, so no
// counted n-gram holds it.  A free code met before v's means v never asked for
// one: codes are never released, so v would have taken it.
__device__ inline int32_t encode_find(const Slot *tab, int64_t bmask, int32_t v) {
    if (v >= 0 && v < kDirect) return v;
    const unsigned long long mark = owner_mark(v);
    uint32_t c = first_code(v);
    for (int probe = 0; probe < kCodeProbe; ++probe) {
        uint64_t lo, hi;
        code_key(c, lo, hi);
        unsigned long long owner = 0ull, unused = 0ull;
        if (!find(tab, bmask, lo, hi, owner, unused) || owner == 0ull) return -1;
        if (owner == mark) return kDirect + int32_t(c);
        c = (c + 1u) & (kMaxCodes - 1u);
    }
    return -1;
}

// The code of token v, taking a dictionary code when v is outside [0, kDirect);
// -1 (with the overflow flag) when the table ran out of slots or no code of v's
// probe sequence could be had.
__device__ inline int32_t encode_claim(Slot *tab, int64_t bmask, Header *hd, int32_t v) {
    if (v >= 0 && v < kDirect) return v;
    const unsigned long long mark = owner_mark(v);
    uint32_t c = first_code(v);
    for (int probe = 0; probe < kCodeProbe; ++probe) {
        uint64_t lo, hi;
        code_key(c, lo, hi);
        Slot *sl = claim(tab, bmask, lo, hi, hd);
        if (!sl) return -1;
        unsigned long long owner = __ldcg(&sl->v0);
        if (owner == 0ull) {
            owner = atomicCAS(&sl->v0, 0ull, mark);
            if (owner == 0ull) owner = mark;                 // taken now
        }
        if (owner == mark) return kDirect + int32_t(c);
        c = (c + 1u) & (kMaxCodes - 1u);
    }
    atomicOr(&hd->overflow, 1u);
    return -1;
}

// One occurrence of g (codes, length n) followed by the token x (code cx).
__device__ inline void count_pair(Slot *tab, int64_t bmask, Header *hd, int r, int n, const int32_t (&g)[kMaxN],
                                  int32_t x, int32_t cx) {
    uint64_t lo, hi;
    make_key(r, n, g, kCount, cx, lo, hi);
    Slot *c_slot = claim(tab, bmask, lo, hi, hd);
    make_key(r, n, g, kCtx, 0, lo, hi);
    Slot *g_slot = claim(tab, bmask, lo, hi, hd);
    if (!c_slot || !g_slot) return;
    const unsigned long long c = atomicAdd(&c_slot->v0, 1ull) + 1ull;
    atomicAdd(&g_slot->v0, 1ull);
    atomicMax(&g_slot->v1, (c << 32) | tie_order(x));
}

// ------------------------------------------------------------------ build ----
struct BuildParams {
    const int32_t *tokens;
    const int64_t *base;
    const int32_t *len;
    int64_t *pref;                                       // [B + 1] scratch: prefix of len
    Slot *tab;
    Header *hd;
    int64_t slots;
    int32_t B, n_min, n_max;
};

__global__ void clear_kernel(BuildParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < p.slots; i += stride) {
        Slot s;
        s.lo = s.hi = s.v0 = s.v1 = 0ull;
        p.tab[i] = s;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        Header h;
        memset(&h, 0, sizeof h);
        h.magic = kMagic;
        h.n_min = p.n_min;
        h.n_max = p.n_max;
        h.slots = p.slots;
        *p.hd = h;
    }
}

// pref[r] = sum of len[0..r) (negative lengths count as 0), one CTA.
__global__ void __launch_bounds__(kScanThreads) prefix_kernel(BuildParams p) {
    __shared__ int64_t warp_sums[kScanThreads / 32];
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t per = (int64_t(p.B) + kScanThreads - 1) / kScanThreads;
    const int64_t r0 = min(int64_t(tid) * per, int64_t(p.B)), r1 = min(r0 + per, int64_t(p.B));
    int64_t own = 0;
    for (int64_t r = r0; r < r1; ++r) own += max(p.len[r], 0);
    int64_t incl = own;
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
        warp_sums[lane] = s;
    }
    __syncthreads();
    int64_t before = (warp ? warp_sums[warp - 1] : 0) + incl - own;
    for (int64_t r = r0; r < r1; ++r) {
        p.pref[r] = before;
        before += max(p.len[r], 0);
    }
    if (tid == kScanThreads - 1) p.pref[p.B] = warp_sums[kScanThreads / 32 - 1];
}

// Every position i >= 1 of every history (its token follows the n-grams that
// end at i - 1), flattened; warp w takes a contiguous range of the virtual
// positions and each lane walks its request forward.
__global__ void __launch_bounds__(kThreads) build_kernel(BuildParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * (kThreads / 32);
    const int64_t total = p.pref[p.B];
    const int64_t per = ((total + nwarps - 1) / nwarps + 31) & ~int64_t(31);
    const int64_t v0 = min(gwarp * per, total), v1 = min(v0 + per, total);
    if (v0 >= v1) return;
    int lo = 0, hi = p.B;                                // pref[lo] <= v0 < pref[hi]
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = min(lo + lane * step, hi - 1);
        const unsigned le = __ballot_sync(0xffffffffu, p.pref[idx] <= v0);
        const int last = 31 - __clz(le);
        const int nlo = min(lo + last * step, hi - 1);
        hi = min(nlo + step, hi);
        lo = nlo;
    }
    int r = lo;
    int64_t r_end = p.pref[r + 1], r_start = p.pref[r], base = p.base[r];
    const int64_t bmask = p.slots / kBucket - 1;
    for (int64_t v = v0 + lane; v < v1; v += 32) {
        while (r_end <= v) {
            ++r;
            r_start = r_end;
            r_end = p.pref[r + 1];
            base = p.base[r];
        }
        const int i = int(v - r_start);
        if (i < 1) continue;
        const int32_t *t = p.tokens + base;
        const int32_t x = t[i];
        const int span = i < p.n_max ? i : p.n_max;      // tokens before x that an n-gram uses
        int32_t w[kMaxN];                                // w[k] = t[i - 1 - k]
#pragma unroll
        for (int k = 0; k < kMaxN; ++k) w[k] = k < span ? t[i - 1 - k] : 0;
        const int32_t cx = encode_claim(p.tab, bmask, p.hd, x);
        if (cx < 0) continue;                            // out of room: flagged, every draft fails
        int32_t cw[kMaxN];                               // their codes
#pragma unroll
        for (int k = 0; k < kMaxN; ++k) cw[k] = k < span ? encode_claim(p.tab, bmask, p.hd, w[k]) : 0;
        for (int n = p.n_min; n <= span; ++n) {
            int32_t g[kMaxN] = {0, 0, 0, 0};
            bool ok = true;
#pragma unroll
            for (int k = 0; k < kMaxN; ++k)
                if (k < n) {
                    g[k] = cw[n - 1 - k];                // oldest first
                    ok = ok && g[k] >= 0;
                }
            if (ok) count_pair(p.tab, bmask, p.hd, r, n, g, x, cx);
        }
    }
}

// ----------------------------------------------------------------- append ----
struct AppendParams {
    int32_t *tokens;
    const int64_t *base;
    int32_t *len;
    const int32_t *cap;
    const int32_t *commit;
    const int32_t *ncommit;
    Slot *tab;
    Header *hd;
    int32_t *status;
    int64_t slots;
    int32_t B, W, n_min, n_max;
};

__device__ inline int append_status(const AppendParams &p, bool ok, int r, int &L, int &n, int64_t &base) {
    L = p.len[r];
    n = min(max(p.ncommit[r], 0), p.W);
    base = p.base[r];
    return !ok ? 2 : (int64_t(L) + n > int64_t(p.cap[r]) ? 1 : 0);
}

// One thread per (request, new position, length): write the token (once) and
// count the pair (the n tokens before it, it).  The tokens come from the old
// history or straight from `commit`, so nothing waits for a write.
__global__ void __launch_bounds__(kThreads) ctx_append_kernel(AppendParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.n_min, p.n_max, p.slots);
    const int64_t bmask = p.slots / kBucket - 1;
    const int nl = p.n_max - p.n_min + 1;
    const int64_t per_r = int64_t(p.W) * nl;
    const int64_t total = int64_t(p.B) * per_r;
    for (int64_t task = int64_t(blockIdx.x) * kThreads + threadIdx.x; task < total;
         task += int64_t(gridDim.x) * kThreads) {
        const int r = int(task / per_r);
        const int rest = int(task - int64_t(r) * per_r);
        const int j = rest / nl, n = p.n_min + rest % nl;
        int L, cnt;
        int64_t base;
        if (append_status(p, ok, r, L, cnt, base) != 0 || j >= cnt) continue;
        const int32_t *crow = p.commit + int64_t(r) * p.W;
        const int32_t x = crow[j];
        if (n == p.n_min) p.tokens[base + L + j] = x;      // one writer per new token
        const int i = L + j;                                 // x's position
        if (i < n) continue;
        const int32_t cx = encode_claim(p.tab, bmask, p.hd, x);
        if (cx < 0) continue;                                // out of room: flagged
        int32_t g[kMaxN] = {0, 0, 0, 0};
        bool okg = true;
#pragma unroll
        for (int k = 0; k < kMaxN; ++k)
            if (k < n) {
                const int src = i - n + k;
                g[k] = encode_claim(p.tab, bmask, p.hd, src >= L ? crow[src - L] : p.tokens[base + src]);
                okg = okg && g[k] >= 0;
            }
        if (okg) count_pair(p.tab, bmask, p.hd, r, n, g, x, cx);
    }
}

// Batches that fit in one wave: one CTA per request at a time (grid-stride over
// requests) takes that request's tasks as above; every thread reads the old
// length first, and after a barrier one thread writes the new length and the
// status, so the append is one launch.  (Larger batches use the kernel above and
// then the length pass below.)
__global__ void __launch_bounds__(kThreads) ctx_append_request_kernel(AppendParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.n_min, p.n_max, p.slots);
    const int64_t bmask = p.slots / kBucket - 1;
    const int nl = p.n_max - p.n_min + 1;
    const int64_t per_r = int64_t(p.W) * nl;
    for (int r = blockIdx.x; r < p.B; r += gridDim.x) {
        int L, cnt;
        int64_t base;
        const int st = append_status(p, ok, r, L, cnt, base);
        const int32_t *crow = p.commit + int64_t(r) * p.W;
        for (int64_t t = threadIdx.x; st == 0 && t < per_r; t += blockDim.x) {
            const int j = int(t / nl), n = p.n_min + int(t % nl);
            if (j >= cnt) break;                                 // tasks are ordered by j
            const int32_t x = crow[j];
            if (n == p.n_min) p.tokens[base + L + j] = x;      // one writer per new token
            const int i = L + j;                                 // x's position
            if (i < n) continue;
            const int32_t cx = encode_claim(p.tab, bmask, p.hd, x);
            if (cx < 0) continue;                                // out of room: flagged
            int32_t g[kMaxN] = {0, 0, 0, 0};
            bool okg = true;
#pragma unroll
            for (int k = 0; k < kMaxN; ++k)
                if (k < n) {
                    const int src = i - n + k;
                    g[k] = encode_claim(p.tab, bmask, p.hd, src >= L ? crow[src - L] : p.tokens[base + src]);
                    okg = okg && g[k] >= 0;
                }
            if (okg) count_pair(p.tab, bmask, p.hd, r, n, g, x, cx);
        }
        __syncthreads();                                     // every reader of len[r] is done
        if (threadIdx.x == 0) {
            if (st == 0) p.len[r] = L + cnt;
            if (p.status) p.status[r] = st;
        }
    }
}

__global__ void __launch_bounds__(kThreads) append_len_kernel(AppendParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.n_min, p.n_max, p.slots);
    for (int r = blockIdx.x * kThreads + threadIdx.x; r < p.B; r += gridDim.x * kThreads) {
        int L, n;
        int64_t base;
        const int st = append_status(p, ok, r, L, n, base);
        if (st == 0) p.len[r] = L + n;
        if (p.status) p.status[r] = st;
    }
}

// ------------------------------------------------------------------ draft ----
struct DraftParams {
    const int32_t *tokens;
    const int64_t *base;
    const int32_t *len;
    const Slot *tab;
    const Header *hd;
    int32_t *out_draft;
    int32_t *out_len;
    int64_t slots;
    int32_t B, n_min, n_max, K;
    int32_t min_count[kMaxN], num[kMaxN], den[kMaxN];
};

__global__ void __launch_bounds__(kDraftThreads) ctx_draft_kernel(DraftParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kDraftThreads / 32);
    const bool ok = header_ok(p.hd, p.n_min, p.n_max, p.slots) && p.hd->overflow == 0u;
    const int64_t bmask = p.slots / kBucket - 1;
    const int nl = p.n_max - p.n_min + 1;
    for (int r = (blockIdx.x * kDraftThreads + threadIdx.x) >> 5; r < p.B; r += nwarps) {
        const int L = max(p.len[r], 0);
        const int32_t *t = p.tokens + p.base[r];
        int32_t *row = p.out_draft + int64_t(r) * p.K;
        // the context window: lane k < 4 holds the code of the k-th token from the
        // end (-1: a value that no counted n-gram holds)
        int32_t c = -1;
        if (ok && lane < kMaxN && lane < L) c = encode_find(p.tab, bmask, t[L - 1 - lane]);
        int j = 0;
        while (ok && j < p.K) {
            const int n = p.n_max - lane;                // lane 0: the longest length
            int32_t g[kMaxN] = {0, 0, 0, 0};
            bool okg = lane < nl && L + j >= n;
#pragma unroll
            for (int k = 0; k < kMaxN; ++k) {
                const int src = min(max(n - 1 - k, 0), kMaxN - 1);   // oldest first: distance n-1-k from the end
                const int32_t v = __shfl_sync(0xffffffffu, c, src);
                if (k < n) {
                    g[k] = v;
                    okg = okg && v >= 0;
                }
            }
            bool pass = false;
            unsigned long long best = 0ull;
            if (okg) {
                uint64_t lo, hi;
                make_key(r, n, g, kCtx, 0, lo, hi);
                unsigned long long total = 0ull;
                if (find(p.tab, bmask, lo, hi, total, best) && total > 0ull) {
                    const unsigned long long cbest = best >> 32;
                    pass = total >= (unsigned long long)max(p.min_count[n - 1], 0) &&
                           cbest * (unsigned long long)p.den[n - 1] >= (unsigned long long)p.num[n - 1] * total;
                }
            }
            const unsigned ballot = __ballot_sync(0xffffffffu, pass);
            if (!ballot) break;
            const int src = __ffs(ballot) - 1;           // the longest passing length
            const unsigned long long b = __shfl_sync(0xffffffffu, best, src);
            const int32_t x = from_tie_order(b & 0xffffffffull);
            if (lane == 0) row[j] = x;
            const int32_t up = __shfl_up_sync(0xffffffffu, c, 1);
            c = lane == 0 ? encode_find(p.tab, bmask, x) : up;   // x was counted, so it has a code
            ++j;
        }
        for (int k = j + lane; k < p.K; k += 32) row[k] = -1;
        if (lane == 0) p.out_len[r] = ok ? j : LOOKUP_DRAFT_LEN_FAILED;
    }
}

bool params_ok(int32_t n_min, int32_t n_max, int64_t slots) {
    return n_min >= 1 && n_min <= n_max && n_max <= kMaxN && lkd::pow2_at_least(slots, 16);
}

bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; }

}  // namespace

extern "C" {

int64_t lookup_ctx_slots_for(int64_t capacity_tokens, int32_t n_min, int32_t n_max) {
    if (capacity_tokens < 0 || n_min < 1 || n_min > n_max || n_max > kMaxN) return 0;
    const int64_t want = 4 * int64_t(n_max - n_min + 1) * capacity_tokens;
    int64_t s = 16;
    while (s < want) {
        if (s > (int64_t(1) << 40)) return 0;
        s <<= 1;
    }
    return s;
}

size_t lookup_ctx_bytes(int64_t slots) {
    if (!lkd::pow2_at_least(slots, 16) || slots > (int64_t(1) << 40)) return 0;
    return sizeof(Header) + sizeof(Slot) * size_t(slots);
}

int lookup_ctx_build(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t n_min,
                     int32_t n_max, void *cache, int64_t slots, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_ctx_build");
    if (B < 0 || B > 65536 || !params_ok(n_min, n_max, slots) || !cache || !aligned16(cache))
        return LOOKUP_DRAFT_EINVAL;
    if (B > 0 && (!tokens || !base || !len)) return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    BuildParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.hd = static_cast<Header *>(cache);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(cache) + sizeof(Header));
    p.slots = slots;
    p.B = B;
    p.n_min = n_min;
    p.n_max = n_max;
    void *pref = nullptr;
    if (B > 0) {                                         // scratch first: the kernels then follow one another
        const cudaError_t e = cudaMallocAsync(&pref, sizeof(int64_t) * (size_t(B) + 1), stream);
        if (e != cudaSuccess) return lookup_record_cuda_error(e, "build scratch");
    }
    p.pref = static_cast<int64_t *>(pref);
    rc = launch_pdl(clear_kernel, unsigned(sms * 8), 256u, stream, p);
    if (B == 0) return rc;
    if (rc == LOOKUP_DRAFT_OK) rc = launch_pdl(prefix_kernel, 1u, unsigned(kScanThreads), stream, p);
    if (rc == LOOKUP_DRAFT_OK) rc = launch_pdl(build_kernel, unsigned(sms * 8), unsigned(kThreads), stream, p);
    const cudaError_t e = cudaFreeAsync(pref, stream);
    if (rc == LOOKUP_DRAFT_OK && e != cudaSuccess) rc = lookup_record_cuda_error(e, "build scratch");
    return rc;
}

int lookup_ctx_append(int32_t *tokens, const int64_t *base, int32_t *len, const int32_t *cap, const int32_t *commit,
                      const int32_t *ncommit, int32_t B, int32_t W, int32_t n_min, int32_t n_max, void *cache,
                      int64_t slots, int32_t *out_status, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_ctx_append");
    if (B < 0 || B > 65536 || W < 0 || !params_ok(n_min, n_max, slots)) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!tokens || !base || !len || !cap || !ncommit || (W > 0 && !commit) || !cache || !aligned16(cache))
        return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    AppendParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.cap = cap;
    p.commit = commit;
    p.ncommit = ncommit;
    p.hd = static_cast<Header *>(cache);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(cache) + sizeof(Header));
    p.status = out_status;
    p.slots = slots;
    p.B = B;
    p.W = W;
    p.n_min = n_min;
    p.n_max = n_max;
    // a CTA per request (sized to its tasks) when the batch fits in one wave of
    // them: one launch; else dense tasks, then the lengths
    const int64_t per_r = int64_t(W) * (n_max - n_min + 1);
    const int64_t block = per_r < 32 ? 32 : (per_r >= kThreads ? kThreads : (per_r + 31) / 32 * 32);
    const int64_t wave = int64_t(sms) * (2048 / block < 32 ? 2048 / block : 32);   // resident CTAs
    if (B <= wave) return launch_pdl(ctx_append_request_kernel, unsigned(B), unsigned(block), stream, p);
    const int64_t tasks = int64_t(B) * per_r;
    rc = launch_pdl(ctx_append_kernel, lkd::capped_grid((tasks + kThreads - 1) / kThreads, int64_t(sms) * 8),
                    unsigned(kThreads), stream, p);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    return launch_pdl(append_len_kernel, lkd::capped_grid((int64_t(B) + kThreads - 1) / kThreads, int64_t(sms) * 4),
                      unsigned(kThreads), stream, p);
}

int lookup_ctx_draft(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t n_min,
                     int32_t n_max, int32_t K, const int32_t *min_count, const int32_t *share_num,
                     const int32_t *share_den, const void *cache, int64_t slots, int32_t *out_draft,
                     int32_t *out_len, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_ctx_draft");
    if (B < 0 || B > 65536 || K < 0 || K > LOOKUP_DRAFT_MAX_K || !params_ok(n_min, n_max, slots))
        return LOOKUP_DRAFT_EINVAL;
    if (!min_count || !share_num || !share_den) return LOOKUP_DRAFT_EINVAL;
    for (int n = n_min; n <= n_max; ++n)
        if (share_num[n - 1] < 0 || share_den[n - 1] < 1) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!tokens || !base || !len || !cache || !aligned16(cache) || (K > 0 && !out_draft) || !out_len)
        return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    DraftParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.hd = static_cast<const Header *>(cache);
    p.tab = reinterpret_cast<const Slot *>(static_cast<const char *>(cache) + sizeof(Header));
    p.out_draft = out_draft;
    p.out_len = out_len;
    p.slots = slots;
    p.B = B;
    p.n_min = n_min;
    p.n_max = n_max;
    p.K = K;
    for (int k = 0; k < kMaxN; ++k) {
        p.min_count[k] = min_count[k];
        p.num[k] = share_num[k];
        p.den[k] = share_den[k];
    }
    const int64_t warps_per_cta = kDraftThreads / 32;
    return launch_pdl(ctx_draft_kernel, lkd::capped_grid((int64_t(B) + warps_per_cta - 1) / warps_per_cta,
                                                         int64_t(sms) * 16),
                      unsigned(kDraftThreads), stream, p);
}

}  // extern "C"
