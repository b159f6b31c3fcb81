// lookup_index.cu -- device-resident n-gram index for exact prompt-lookup drafting.
//
// Source: Strata engine article, gtnt.cn/news/124732, section 四 (an n-gram ->
// position index of the prompt and confirmed output, open addressing, O(1)
// appends); the result is the exact draft of HyperQwen lookup-drafting article,
// section "第1步".  The contract is in include/lookup_index.h.
//
// Table: a 128-byte header, then `slots` 8-byte slots in buckets of 4 (one
// 32-byte sector: one DRAM access per probe).  The key of the n-gram ending at q
// in request r is a 64-bit hash of (r, n, t[q], t[q-1], ..., t[q-n+1]); its home
// bucket comes from the key's low bits, and its slot holds the key's high half
// as a fingerprint (low bit set, so a used slot is never 0) above the largest
// end position inserted under it.  Only positions before each request's last
// are indexed, so that largest position is the most recent EARLIER occurrence
// the query asks for.  An insertion claims an empty slot with a 64-bit CAS, and
// a slot holding its fingerprint takes the position with one 64-bit atomicMax
// (equal high halves: the maximum keeps the larger position), in any order.
//
// Query (one warp per request): lane j probes the key of the suffix's n-gram
// for n = min_m + j and gets the latest earlier end of that n-gram, if any; the
// longest n with a position is the match, checked against the history.  Keys
// that share a fingerprint and a probe sequence merge their positions, so a
// candidate that does not check out (or a table that overflowed) sends the
// request to a warp brute-force scan instead: the result never depends on the
// hash.
//
// Decode loop: the append writes the committed tokens in place and inserts
// their n-grams, one CTA per request when the batch fits one wave of them.  The
// same kernel can first verify the request's block (lookup_index_verify_append)
// and, after the new length is written, draft its next block from the grown
// history (lookup_index_verify_append_draft); the query is the one device
// function the draft kernels use, so every fused form returns what the separate
// calls would.

#include "lookup_index.h"
#include "lookup_loop.h"

#include "common.cuh"

namespace {

using lkd::allow_dependent_launch;
using lkd::launch_pdl;
using lkd::mix64;
using lkd::sm_count;
using lkd::wait_for_prerequisite_grid;

constexpr uint32_t kMagic = 0x4c4b4959u;        // "LKIY": 8-byte slots
constexpr int kBucket = 4;                      // slots per bucket: one 32-byte sector
constexpr int kMaxProbe = 2048;                 // buckets probed before the overflow flag
constexpr int kBuildThreads = 256;
constexpr int kWarpThreads = 128;               // draft kernel: 4 warps per CTA
constexpr int kAppendThreads = 256;             // append kernels
constexpr int kScanThreads = 1024;

struct __align__(16) Header {
    uint32_t magic;
    int32_t min_m, max_m, hash_bits;
    int64_t slots;
    uint32_t overflow;                          // set when an insertion found no slot
    uint32_t pad[25];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes: the slots start on a 128-byte line");

using Slot = unsigned long long;                // fingerprint << 32 | latest end position; 0 = empty

__device__ inline uint64_t seed_of(int r) { return mix64(uint64_t(uint32_t(r)) * 0x9e3779b97f4a7c15ull + 0x632be59bd9b4e019ull); }
__device__ inline uint64_t step_hash(uint64_t h, int32_t tok) { return mix64(h ^ uint64_t(uint32_t(tok))); }
__device__ inline unsigned long long key_of(uint64_t h, int n, int hash_bits) {
    uint64_t k = mix64(h ^ (uint64_t(n) << 40));
    if (hash_bits < 64) k &= (uint64_t(1) << hash_bits) - 1;
    return k;
}
__device__ inline uint32_t fingerprint(unsigned long long key) { return uint32_t(key >> 32) | 1u; }

__device__ inline bool header_ok(const Header *hd, int min_m, int max_m, int hash_bits, int64_t slots) {
    return hd->magic == kMagic && hd->min_m == min_m && hd->max_m == max_m && hd->hash_bits == hash_bits &&
           hd->slots == slots;
}

// Buckets: a key's home is bucket (key & bmask), kBucket consecutive slots in
// one 32-byte sector, read whole in one round of loads; a full bucket moves on
// to the next.  Every insertion scans in that same order and slots never empty again,
// so an empty slot seen during a scan means the key is not stored further on.
__device__ inline void read_bucket(const Slot *tab, int64_t b, Slot (&v)[kBucket]) {
    const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(tab + b * kBucket);
    const ulonglong2 a = __ldcg(p), c = __ldcg(p + 1);
    v[0] = a.x;
    v[1] = a.y;
    v[2] = c.x;
    v[3] = c.y;
}

// Insert end position q under key; false (and the overflow flag) if no slot was
// found.  Any order of insertions leaves each slot at its largest position.
__device__ inline bool insert(Slot *tab, int64_t bmask, unsigned long long key, int q, Header *hd) {
    const unsigned long long fp = (unsigned long long)fingerprint(key) << 32;
    const unsigned long long word = fp | uint32_t(q);
    int64_t b = int64_t(key & uint64_t(bmask));
    for (int probe = 0; probe < kMaxProbe; ++probe) {
        Slot v[kBucket];
        read_bucket(tab, b, v);
#pragma unroll
        for (int s = 0; s < kBucket; ++s) {
            Slot *sl = tab + b * kBucket + s;
            unsigned long long k = v[s];
            if (k == 0ull) {
                k = atomicCAS(sl, 0ull, word);
                if (k == 0ull) return true;              // claimed with q
            }
            if ((k & 0xffffffff00000000ull) == fp) {
                if (uint32_t(k) < uint32_t(q)) atomicMax(sl, word);
                return true;
            }
        }
        b = (b + 1) & bmask;
    }
    atomicOr(&hd->overflow, 1u);
    return false;
}

// The latest end position stored under key; false when an empty slot or the
// probe limit is reached first.
__device__ inline bool find(const Slot *tab, int64_t bmask, unsigned long long key, int &pos) {
    const unsigned long long fp = (unsigned long long)fingerprint(key) << 32;
    int64_t b = int64_t(key & uint64_t(bmask));
    for (int probe = 0; probe < kMaxProbe; ++probe) {
        Slot v[kBucket];
        read_bucket(tab, b, v);
#pragma unroll
        for (int s = 0; s < kBucket; ++s) {
            if ((v[s] & 0xffffffff00000000ull) == fp) {
                pos = int(uint32_t(v[s]));
                return true;
            }
            if (v[s] == 0ull) return false;
        }
        b = (b + 1) & bmask;
    }
    return false;
}

// Insert the n-grams (n in [min_m, max_m]) that end at position q = base + i.
// The tokens are loaded first, all at once (the hash chain would otherwise wait
// for each load in turn).
__device__ inline void insert_position(const int32_t *tokens, int64_t base, int i, int r, int min_m, int max_m,
                                       int hash_bits, Slot *tab, int64_t mask, Header *hd) {
    const int64_t q = base + i;
    const int top = min(max_m, i + 1);
    int32_t v[LOOKUP_DRAFT_MAX_M];
#pragma unroll
    for (int k = 0; k < LOOKUP_DRAFT_MAX_M; ++k) v[k] = k < top ? tokens[q - k] : 0;
    uint64_t h = seed_of(r);
#pragma unroll
    for (int k = 0; k < LOOKUP_DRAFT_MAX_M; ++k) {
        if (k < top) {
            h = step_hash(h, v[k]);
            if (k + 1 >= min_m) insert(tab, mask, key_of(h, k + 1, hash_bits), int(q), hd);
        }
    }
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
    int32_t B, min_m, max_m, hash_bits;
};

__global__ void clear_kernel(BuildParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < p.slots; i += stride) p.tab[i] = 0ull;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        Header h;
        memset(&h, 0, sizeof h);
        h.magic = kMagic;
        h.min_m = p.min_m;
        h.max_m = p.max_m;
        h.hash_bits = p.hash_bits;
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

// Every history position but each request's last, flattened: warp w takes a
// contiguous range of the virtual positions [0, pref[B]); each lane walks its
// request forward.
__global__ void __launch_bounds__(kBuildThreads) build_kernel(BuildParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = (int64_t(blockIdx.x) * kBuildThreads + threadIdx.x) >> 5;
    const int64_t nwarps = int64_t(gridDim.x) * (kBuildThreads / 32);
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
    const int64_t mask = (p.slots / kBucket) - 1;       // bucket mask
    for (int64_t v = v0 + lane; v < v1; v += 32) {
        while (r_end <= v) {
            ++r;
            r_start = r_end;
            r_end = p.pref[r + 1];
            base = p.base[r];
        }
        if (v + 1 == r_end) continue;                    // the last position: not indexed
        insert_position(p.tokens, base, int(v - r_start), r, p.min_m, p.max_m, p.hash_bits, p.tab, mask, p.hd);
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
    int32_t B, W, min_m, max_m, hash_bits;
};

__device__ inline int append_status(const AppendParams &p, bool ok, int r, int &L, int &n, int64_t &base) {
    L = p.len[r];
    n = min(max(p.ncommit[r], 0), p.W);
    base = p.base[r];
    return !ok ? 2 : (int64_t(L) + n > int64_t(p.cap[r]) ? 1 : 0);
}

// Large batches (more requests than one wave of per-request CTAs): the writes
// and insertions with one thread per (request, new token, length) task,
// grid-stride over B * W * (max_m - min_m + 1) tasks, then the lengths in a
// second kernel.  The tokens that
// end at a new position come from the old history or straight from `commit`,
// so no insertion waits for a write.  len is only read here.
template <int kMaxLen>
__global__ void __launch_bounds__(kAppendThreads) index_append_dense_kernel(AppendParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.min_m, p.max_m, p.hash_bits, p.slots);
    const int64_t mask = (p.slots / kBucket) - 1;       // bucket mask
    const int nl = p.max_m - p.min_m + 1;
    const int64_t per_r = int64_t(p.W) * nl;
    const int64_t total = int64_t(p.B) * per_r;
    for (int64_t task = int64_t(blockIdx.x) * kAppendThreads + threadIdx.x; task < total;
         task += int64_t(gridDim.x) * kAppendThreads) {
        const int r = int(task / per_r);
        const int rest = int(task - int64_t(r) * per_r);
        const int j = rest / nl, len_n = p.min_m + rest % nl;   // new token j, length len_n
        int L, n;
        int64_t base;
        if (append_status(p, ok, r, L, n, base) != 0 || j >= n) continue;
        const int32_t *crow = p.commit + int64_t(r) * p.W;
        if (len_n == p.min_m) p.tokens[base + L + j] = crow[j];  // one writer per new token
        const int i = L - 1 + j;                             // the n-gram's end: one before the new token
        if (i + 1 < len_n) continue;                         // no n-gram of that length ends here
        // the len_n tokens ending at i, from the old history or from commit, loaded at once
        int32_t v[kMaxLen];
#pragma unroll
        for (int k = 0; k < kMaxLen; ++k) {
            const int src = i - k;
            v[k] = k >= len_n ? 0 : (src >= L ? crow[src - L] : p.tokens[base + src]);
        }
        uint64_t h = seed_of(r);
#pragma unroll
        for (int k = 0; k < kMaxLen; ++k)
            if (k < len_n) h = step_hash(h, v[k]);
        insert(p.tab, mask, key_of(h, len_n, p.hash_bits), int(base + i), p.hd);
    }
}

// Then the lengths and the status, one thread per request (after every reader
// of len in the kernel above).
__global__ void __launch_bounds__(kAppendThreads) append_len_kernel(AppendParams p) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.min_m, p.max_m, p.hash_bits, p.slots);
    for (int r = blockIdx.x * kAppendThreads + threadIdx.x; r < p.B; r += gridDim.x * kAppendThreads) {
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
    int32_t *out_pos;
    int32_t *out_mlen;
    int32_t *out_fallback;
    int64_t slots;
    int32_t B, min_m, max_m, K, hash_bits;
};

// The exact answer by brute force: candidate ends q = L-2, L-3, ... in batches of
// 32 (one per lane), each extended backwards up to max_m tokens; the largest key
// (m << 32 | p) wins, and a batch holding a max_m match ends the search.
__device__ unsigned long long brute_force(const int32_t *t, int L, int tok, int min_m, int max_m, int lane) {
    unsigned long long best = 0ull;
    for (int qe = L - 2; qe >= min_m - 1; qe -= 32) {
        const int q = qe - lane;
        int k = 0;
        bool alive = q >= min_m - 1;
        for (int i = 0; i < max_m; ++i) {
            const int s = __shfl_sync(0xffffffffu, tok, i);    // suffix token i (from the end)
            alive = alive && q - i >= 0 && t[q - i] == s;
            k += alive;
        }
        unsigned long long key = 0ull;
        if (k >= min_m) key = (uint64_t(uint32_t(k)) << 32) | uint32_t(q - k + 1);
#pragma unroll
        for (int d = 16; d; d >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, d);
            key = o > key ? o : key;
        }
        best = key > best ? key : best;
        if (int(best >> 32) == max_m) break;
    }
    return best;
}

// One request's index query in the calling warp (all 32 lanes): the longest
// suffix n-gram with a stored earlier end, checked against the history, else
// the brute-force scan; the draft row, length, position, m and fallback flag,
// or with PLAN the decode loop's scheduling and fusion on the draft tokens.
template <bool PLAN>
__device__ __forceinline__ void index_draft_request(const DraftParams &p, const lkd::PlanIO &pio, int r, int lane,
                                                    bool hd_ok, bool overflow, int64_t mask, int nl) {
    const int L = max(p.len[r], 0);
    const int64_t base = p.base[r];
    const int32_t *t = p.tokens + base;
    // suffix token i (counted from the end) in lane i
    const int tok = (lane < p.max_m && lane < L) ? t[L - 1 - lane] : 0;
    int32_t *row = PLAN ? nullptr : p.out_draft + int64_t(r) * p.K;
    unsigned long long best = 0ull;
    bool fallback = overflow, drafted = false;
    int32_t tok0 = -1, tok1 = -1;                    // PLAN: draft tokens lane and lane + 32
    if (hd_ok && !overflow && L >= p.min_m + 1) {
        // keys: lane j hashes the n-gram of length n = min_m + j
        const int n = p.min_m + lane;
        unsigned long long key = 0ull;
        uint64_t h = seed_of(r);
        const int top = min(p.max_m, L);
        for (int k = 0; k < top; ++k) {
            h = step_hash(h, __shfl_sync(0xffffffffu, tok, k));
            if (k + 1 == n) key = key_of(h, n, p.hash_bits);
        }
        // 0 none, 1 candidate, 2 inconsistent (a position outside the request:
        // the slot is shared with another key)
        int state = 0, cand = -1;
        if (lane < nl && n <= L - 1) {
            int pos = -1;
            if (find(p.tab, mask, key, pos)) {
                const int64_t c = int64_t(pos) - base;       // relative end position
                if (c < n - 1 || c > L - 2) state = 2;
                else { state = 1; cand = int(c); }
            }
        }
        const unsigned cmask = __ballot_sync(0xffffffffu, state == 1);
        const unsigned incons = __ballot_sync(0xffffffffu, state == 2);
        const int jbest = cmask ? 31 - __clz(cmask) : -1;
        // a longer length whose slot is inconsistent may hide the true match
        const unsigned above = jbest >= 0 ? (jbest < 31 ? ~((2u << jbest) - 1) : 0u) : 0xffffffffu;
        if (incons & above) {
            fallback = true;
        } else if (jbest >= 0) {
            // check the candidate and gather its draft in the same round of loads
            const int m = p.min_m + jbest;
            const int c = __shfl_sync(0xffffffffu, cand, jbest);
            const int d = L - 1 - c;                         // L - pos - m
            const bool bad = lane < m && t[c - lane] != tok;
            const int32_t d0 = lane < p.K ? t[c + 1 + lane % d] : 0;
            const int32_t d1 = lane + 32 < p.K ? t[c + 1 + (lane + 32) % d] : 0;
            if (__ballot_sync(0xffffffffu, bad)) {
                fallback = true;                             // the slot was shared with another key
            } else {
                best = (uint64_t(uint32_t(m)) << 32) | uint32_t(c - m + 1);
                if (PLAN) {
                    tok0 = lane < p.K ? d0 : -1;
                    tok1 = lane + 32 < p.K ? d1 : -1;
                } else {
                    if (lane < p.K) row[lane] = d0;
                    if (lane + 32 < p.K) row[lane + 32] = d1;
                }
                drafted = true;
            }
        }
    }
    if (fallback && hd_ok) best = brute_force(t, L, tok, p.min_m, p.max_m, lane);
    const int m = int(best >> 32);
    const int pos = int(uint32_t(best));
    const bool found = hd_ok && m > 0;
    if (!drafted) {                                         // the draft from the self-extended history
        const int d = L - pos - m;
        if (PLAN) {
            tok0 = (found && lane < p.K) ? t[pos + m + (lane % d)] : -1;
            tok1 = (found && lane + 32 < p.K) ? t[pos + m + ((lane + 32) % d)] : -1;
        } else {
            for (int j = lane; j < p.K; j += 32) row[j] = found ? t[pos + m + (j % d)] : -1;
        }
    }
    if (PLAN) lkd::plan_warp(pio, r, lane, found ? m : 0, tok0, tok1);
    if (lane == 0) {
        // PLAN: out_len (the draft length) is optional and no position is written
        if (!PLAN || p.out_len) p.out_len[r] = !hd_ok ? LOOKUP_DRAFT_LEN_FAILED : (found ? p.K : 0);
        if (!PLAN) p.out_pos[r] = found ? pos : -1;
        if (p.out_mlen) p.out_mlen[r] = found ? m : 0;
        if (p.out_fallback) p.out_fallback[r] = fallback ? 1 : 0;
    }
}

// PLAN: the draft tokens stay in the warp's registers and the decode loop's
// scheduling and fusion follow (lkd::plan_warp); out_len then receives the length
// lookup_index_draft would report, and no draft row is written.
template <bool PLAN>
__global__ void __launch_bounds__(kWarpThreads) index_draft_kernel(DraftParams p, lkd::PlanIO pio) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * (kWarpThreads / 32);
    const bool hd_ok = header_ok(p.hd, p.min_m, p.max_m, p.hash_bits, p.slots);
    const bool overflow = hd_ok && p.hd->overflow != 0u;
    const int64_t mask = (p.slots / kBucket) - 1;       // bucket mask
    const int nl = p.max_m - p.min_m + 1;
    for (int r = (blockIdx.x * kWarpThreads + threadIdx.x) >> 5; r < p.B; r += nwarps)
        index_draft_request<PLAN>(p, pio, r, lane, hd_ok, overflow, mask, nl);
}

// ------------------------------------------------------- append, per request ----
struct AppendExtra {
    lkd::VerifyIO v;                                     // VERIFY
    DraftParams d;                                       // DRAFT
};

// Batches that fit in one wave: one CTA per request at a time (grid-stride over
// requests), the CTA's threads take the request's (new token j, length) tasks:
// write token j at position L + j and insert the n-gram that ends one position
// earlier, at L - 1 + j (the old last position first; the new last position is
// indexed by the next append).  The tokens of an n-gram come from the old
// history or straight from `commit`, so no insertion waits for a write.  Every
// thread reads the request's old length first; after a barrier (no thread reads
// it any more) one thread writes the new length and the status, so the append
// is one launch.  VERIFY: warp 0 first verifies the request's block into x.v's
// outputs (lookup_verify's rule, for that request), which p.commit and p.ncommit
// point at; after a barrier the CTA appends what it committed.  DRAFT: after the
// new length is written, warp 0 drafts the request from the grown history and
// the index (lookup_index_draft's answer, into x.d's outputs).
template <int kMaxLen, bool VERIFY, bool DRAFT>
__global__ void __launch_bounds__(kAppendThreads) index_append_request_kernel(AppendParams p, AppendExtra x) {
    wait_for_prerequisite_grid();
    allow_dependent_launch();
    const bool ok = header_ok(p.hd, p.min_m, p.max_m, p.hash_bits, p.slots);
    const int64_t mask = (p.slots / kBucket) - 1;       // bucket mask
    const int nl = p.max_m - p.min_m + 1;
    const int64_t per_r = int64_t(p.W) * nl;
    for (int r = blockIdx.x; r < p.B; r += gridDim.x) {
        if (VERIFY) {
            if (threadIdx.x < 32) lkd::verify_warp(x.v, r, threadIdx.x);
            __syncthreads();                                 // the commit row and count are written
        }
        int L, n;
        int64_t base;
        const int st = append_status(p, ok, r, L, n, base);
        const int32_t *crow = p.commit + int64_t(r) * p.W;
        for (int64_t t = threadIdx.x; st == 0 && t < per_r; t += blockDim.x) {
            const int j = int(t / nl), len_n = p.min_m + int(t % nl);   // new token j, length len_n
            if (j >= n) break;                                   // tasks are ordered by j
            if (len_n == p.min_m) p.tokens[base + L + j] = crow[j];  // one writer per new token
            const int i = L - 1 + j;                             // the n-gram's end: one before the new token
            if (i + 1 < len_n) continue;                         // no n-gram of that length ends here
            // the len_n tokens ending at i, from the old history or from commit, loaded at once
            int32_t v[kMaxLen];
#pragma unroll
            for (int k = 0; k < kMaxLen; ++k) {
                const int src = i - k;
                v[k] = k >= len_n ? 0 : (src >= L ? crow[src - L] : p.tokens[base + src]);
            }
            uint64_t h = seed_of(r);
#pragma unroll
            for (int k = 0; k < kMaxLen; ++k)
                if (k < len_n) h = step_hash(h, v[k]);
            insert(p.tab, mask, key_of(h, len_n, p.hash_bits), int(base + i), p.hd);
        }
        __syncthreads();                                     // every reader of len[r] is done
        if (threadIdx.x == 0) {
            if (st == 0) p.len[r] = L + n;
            if (p.status) p.status[r] = st;
        }
        if (DRAFT) {
            // The new tokens, the request's insertions and its length are written;
            // the table is read through L2, where the insertions' atomics land.
            // Other CTAs insert only other requests' keys, which never move or
            // empty a slot, and an overflow anywhere sends the query to the exact
            // scan.
            __syncthreads();
            if (threadIdx.x < 32) {
                const bool overflow = ok && __ldcg(&p.hd->overflow) != 0u;
                index_draft_request<false>(x.d, lkd::PlanIO{}, r, threadIdx.x, ok, overflow, mask, nl);
            }
            __syncthreads();                                 // before the next request reuses the CTA
        }
    }
}



// ------------------------------------------------------------------- host ----
bool pow2(int64_t x) { return x >= 16 && (x & (x - 1)) == 0; }

bool params_ok(int32_t min_m, int32_t max_m, int32_t hash_bits, int64_t slots) {
    return min_m >= 1 && min_m <= max_m && max_m <= LOOKUP_DRAFT_MAX_M && hash_bits >= 1 && hash_bits <= 64 &&
           pow2(slots);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

unsigned warp_grid(int B, int sms) {
    const int64_t need = (int64_t(B) + kWarpThreads / 32 - 1) / (kWarpThreads / 32);
    return unsigned(need < int64_t(sms) * 16 ? need : int64_t(sms) * 16);
}

}  // namespace

extern "C" {

int64_t lookup_index_slots_for(int64_t capacity_tokens, int32_t min_m, int32_t max_m) {
    if (capacity_tokens < 0 || min_m < 1 || min_m > max_m || max_m > LOOKUP_DRAFT_MAX_M) return 0;
    const int64_t want = 2 * int64_t(max_m - min_m + 1) * capacity_tokens;
    int64_t s = 16;
    while (s < want) {
        if (s > (int64_t(1) << 40)) return 0;
        s <<= 1;
    }
    return s;
}

size_t lookup_index_bytes(int64_t slots) {
    if (!pow2(slots) || slots > (int64_t(1) << 40)) return 0;
    return sizeof(Header) + sizeof(Slot) * size_t(slots);
}

int lookup_index_build(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t min_m,
                       int32_t max_m, void *index, int64_t slots, int32_t hash_bits, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_build");
    if (B < 0 || !params_ok(min_m, max_m, hash_bits, slots) || !index || !aligned16(index)) return LOOKUP_DRAFT_EINVAL;
    if (B > 0 && (!tokens || !base || !len)) return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    cudaStream_t st = stream;
    BuildParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.hd = static_cast<Header *>(index);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(index) + sizeof(Header));
    p.slots = slots;
    p.B = B;
    p.min_m = min_m;
    p.max_m = max_m;
    p.hash_bits = hash_bits;
    void *pref = nullptr;
    if (B > 0) {                                         // scratch first: the kernels then follow one another
        const cudaError_t e = cudaMallocAsync(&pref, sizeof(int64_t) * (size_t(B) + 1), st);
        if (e != cudaSuccess) return lookup_record_cuda_error(e, "build scratch");
    }
    p.pref = static_cast<int64_t *>(pref);
    rc = launch_pdl(clear_kernel, unsigned(sms * 8), 256u, st, p);
    if (B == 0) return rc;
    if (rc == LOOKUP_DRAFT_OK) rc = launch_pdl(prefix_kernel, 1u, unsigned(kScanThreads), st, p);
    if (rc == LOOKUP_DRAFT_OK) rc = launch_pdl(build_kernel, unsigned(sms * 8), unsigned(kBuildThreads), st, p);
    const cudaError_t e = cudaFreeAsync(pref, st);
    if (rc == LOOKUP_DRAFT_OK && e != cudaSuccess) rc = lookup_record_cuda_error(e, "build scratch");
    return rc;
}

// A CTA per request, sized to its tasks (a warp at least, kAppendThreads at most),
// when every request gets one in a single wave: the append is one launch.  Larger
// batches spread the tasks densely over the threads and set the lengths in a
// second launch (one CTA per request would take several waves).
bool one_wave_append(int32_t B, int32_t W, int32_t min_m, int32_t max_m, int sms, unsigned &block) {
    const int64_t per_r = int64_t(W) * (max_m - min_m + 1);
    const int64_t b = per_r < 32 ? 32 : (per_r >= kAppendThreads ? kAppendThreads : (per_r + 31) / 32 * 32);
    const int64_t wave = int64_t(sms) * (2048 / b < 32 ? 2048 / b : 32);   // resident CTAs
    block = unsigned(b);
    return B <= wave;
}

int lookup_index_append(int32_t *tokens, const int64_t *base, int32_t *len, const int32_t *cap, const int32_t *commit,
                        const int32_t *ncommit, int32_t B, int32_t W, int32_t min_m, int32_t max_m, void *index,
                        int64_t slots, int32_t hash_bits, int32_t *out_status, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_append");
    if (B < 0 || W < 0 || !params_ok(min_m, max_m, hash_bits, slots)) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!tokens || !base || !len || !cap || !ncommit || (W > 0 && !commit) || !index || !aligned16(index))
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
    p.hd = static_cast<Header *>(index);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(index) + sizeof(Header));
    p.status = out_status;
    p.slots = slots;
    p.B = B;
    p.W = W;
    p.min_m = min_m;
    p.max_m = max_m;
    p.hash_bits = hash_bits;
    unsigned block = 0;
    // the token window in registers: 16 entries when max_m allows, else 32
    if (one_wave_append(B, W, min_m, max_m, sms, block))
        return lkd::launch_pdl2(max_m <= 16 ? index_append_request_kernel<16, false, false>
                                            : index_append_request_kernel<LOOKUP_DRAFT_MAX_M, false, false>,
                                unsigned(B), block, stream, p, AppendExtra{});
    const int64_t per_r = int64_t(W) * (max_m - min_m + 1);
    const int64_t tasks = int64_t(B) * per_r;
    const int64_t want = (tasks + kAppendThreads - 1) / kAppendThreads;
    const unsigned grid = unsigned(want < int64_t(sms) * 8 ? (want > 0 ? want : 1) : int64_t(sms) * 8);
    rc = launch_pdl(max_m <= 16 ? index_append_dense_kernel<16> : index_append_dense_kernel<LOOKUP_DRAFT_MAX_M>, grid,
                    unsigned(kAppendThreads), stream, p);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    const unsigned grid2 = unsigned((int64_t(B) + kAppendThreads - 1) / kAppendThreads);
    return launch_pdl(append_len_kernel, grid2 < unsigned(sms * 4) ? grid2 : unsigned(sms * 4), unsigned(kAppendThreads),
                      stream, p);
}

int lookup_index_verify_append(const int32_t *block, const int32_t *block_len, const int32_t *target,
                               const float *probs, const float *qprobs, const int32_t *point_mass, const float *u,
                               int32_t B, int32_t P, int32_t *tokens, const int64_t *base, int32_t *len,
                               const int32_t *cap, int32_t min_m, int32_t max_m, void *index, int64_t slots,
                               int32_t hash_bits, int32_t *out_accepted, int32_t *out_commit, int32_t *out_ncommit,
                               int32_t *out_status, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_verify_append");
    if (B < 0 || P < 0 || P > lkd::kMaxBlock || !params_ok(min_m, max_m, hash_bits, slots)) return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if ((P > 0 && !block) || !block_len || !target || (probs && !u) || !out_accepted || !out_commit || !out_ncommit)
        return LOOKUP_DRAFT_EINVAL;
    if (!tokens || !base || !len || !cap || !index || !aligned16(index)) return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    const int32_t W = P + 1;
    unsigned threads = 0;
    if (!one_wave_append(B, W, min_m, max_m, sms, threads)) {
        // several waves: the two steps as two calls (the dense append reads every
        // request's commit row, so all of them are verified first)
        rc = lookup_verify(block, block_len, target, probs, qprobs, point_mass, u, B, P, out_accepted, out_commit,
                           out_ncommit, stream);
        if (rc != LOOKUP_DRAFT_OK) return rc;
        return lookup_index_append(tokens, base, len, cap, out_commit, out_ncommit, B, W, min_m, max_m, index, slots,
                                   hash_bits, out_status, stream);
    }
    AppendParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.cap = cap;
    p.commit = out_commit;
    p.ncommit = out_ncommit;
    p.hd = static_cast<Header *>(index);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(index) + sizeof(Header));
    p.status = out_status;
    p.slots = slots;
    p.B = B;
    p.W = W;
    p.min_m = min_m;
    p.max_m = max_m;
    p.hash_bits = hash_bits;
    AppendExtra x{};
    x.v = lkd::VerifyIO{block, block_len, target, probs, qprobs, point_mass, u, out_accepted, out_commit,
                        out_ncommit, P};
    return lkd::launch_pdl2(max_m <= 16 ? index_append_request_kernel<16, true, false>
                                        : index_append_request_kernel<LOOKUP_DRAFT_MAX_M, true, false>,
                            unsigned(B), threads, stream, p, x);
}

int lookup_index_verify_append_draft(const int32_t *block, const int32_t *block_len, const int32_t *target,
                                     const float *probs, const float *qprobs, const int32_t *point_mass,
                                     const float *u, int32_t B, int32_t P, int32_t *tokens, const int64_t *base,
                                     int32_t *len, const int32_t *cap, int32_t min_m, int32_t max_m, void *index,
                                     int64_t slots, int32_t hash_bits, int32_t K, int32_t *out_accepted,
                                     int32_t *out_commit, int32_t *out_ncommit, int32_t *out_status,
                                     int32_t *out_draft, int32_t *out_draft_len, int32_t *out_pos, int32_t *out_mlen,
                                     int32_t *out_fallback, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_verify_append_draft");
    if (B < 0 || P < 0 || P > lkd::kMaxBlock || K < 0 || K > LOOKUP_DRAFT_MAX_K ||
        !params_ok(min_m, max_m, hash_bits, slots))
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if ((P > 0 && !block) || !block_len || !target || (probs && !u) || !out_accepted || !out_commit || !out_ncommit)
        return LOOKUP_DRAFT_EINVAL;
    if (!tokens || !base || !len || !cap || !index || !aligned16(index) || (K > 0 && !out_draft) ||
        !out_draft_len || !out_pos)
        return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    const int32_t W = P + 1;
    unsigned threads = 0;
    if (!one_wave_append(B, W, min_m, max_m, sms, threads)) {
        // several waves: verification and the append, then the draft, as calls
        rc = lookup_index_verify_append(block, block_len, target, probs, qprobs, point_mass, u, B, P, tokens, base,
                                        len, cap, min_m, max_m, index, slots, hash_bits, out_accepted, out_commit,
                                        out_ncommit, out_status, stream);
        if (rc != LOOKUP_DRAFT_OK) return rc;
        return lookup_index_draft(tokens, base, len, B, min_m, max_m, K, index, slots, hash_bits, out_draft,
                                  out_draft_len, out_pos, out_mlen, out_fallback, stream);
    }
    AppendParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.cap = cap;
    p.commit = out_commit;
    p.ncommit = out_ncommit;
    p.hd = static_cast<Header *>(index);
    p.tab = reinterpret_cast<Slot *>(static_cast<char *>(index) + sizeof(Header));
    p.status = out_status;
    p.slots = slots;
    p.B = B;
    p.W = W;
    p.min_m = min_m;
    p.max_m = max_m;
    p.hash_bits = hash_bits;
    AppendExtra x{};
    x.v = lkd::VerifyIO{block, block_len, target, probs, qprobs, point_mass, u, out_accepted, out_commit,
                        out_ncommit, P};
    x.d.tokens = tokens;
    x.d.base = base;
    x.d.len = len;
    x.d.hd = p.hd;
    x.d.tab = p.tab;
    x.d.out_draft = out_draft;
    x.d.out_len = out_draft_len;
    x.d.out_pos = out_pos;
    x.d.out_mlen = out_mlen;
    x.d.out_fallback = out_fallback;
    x.d.slots = slots;
    x.d.B = B;
    x.d.min_m = min_m;
    x.d.max_m = max_m;
    x.d.K = K;
    x.d.hash_bits = hash_bits;
    return lkd::launch_pdl2(max_m <= 16 ? index_append_request_kernel<16, true, true>
                                        : index_append_request_kernel<LOOKUP_DRAFT_MAX_M, true, true>,
                            unsigned(B), threads, stream, p, x);
}

int lookup_index_draft(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t min_m,
                       int32_t max_m, int32_t K, const void *index, int64_t slots, int32_t hash_bits,
                       int32_t *out_draft, int32_t *out_len, int32_t *out_pos, int32_t *out_mlen,
                       int32_t *out_fallback, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_draft");
    if (B < 0 || K < 0 || K > LOOKUP_DRAFT_MAX_K || !params_ok(min_m, max_m, hash_bits, slots))
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!tokens || !base || !len || !index || !aligned16(index) || (K > 0 && !out_draft) || !out_len || !out_pos)
        return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    DraftParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.hd = static_cast<const Header *>(index);
    p.tab = reinterpret_cast<const Slot *>(static_cast<const char *>(index) + sizeof(Header));
    p.out_draft = out_draft;
    p.out_len = out_len;
    p.out_pos = out_pos;
    p.out_mlen = out_mlen;
    p.out_fallback = out_fallback;
    p.slots = slots;
    p.B = B;
    p.min_m = min_m;
    p.max_m = max_m;
    p.K = K;
    p.hash_bits = hash_bits;
    return lkd::launch_pdl2(index_draft_kernel<false>, warp_grid(B, sms), unsigned(kWarpThreads), stream, p,
                            lkd::PlanIO{});
}

int lookup_index_draft_plan(const int32_t *tokens, const int64_t *base, const int32_t *len, int32_t B, int32_t min_m,
                            int32_t max_m, const void *index, int64_t slots, int32_t hash_bits,
                            const int32_t *model_draft, const int32_t *committed, int32_t H, int32_t T,
                            int32_t replace_min, int32_t agree_min, int32_t agree_n, int32_t tail_min, int32_t slack,
                            int32_t enter_steps, int32_t sticky, int32_t *state, int32_t *out_long,
                            int32_t *out_block, int32_t *out_len, int32_t *out_point_mass, int32_t *out_mlen,
                            int32_t *out_draft_len, int32_t *out_fallback, struct CUstream_st *stream) {
    lkd::TraceRange trace_("lookup_index_draft_plan");
    if (B < 0 || !params_ok(min_m, max_m, hash_bits, slots) || H < 1 || T < 0 ||
        int64_t(H) + T > LOOKUP_DRAFT_MAX_K || agree_n < 0 || agree_n > H || enter_steps < 1 || sticky < 0 ||
        slack < 0)
        return LOOKUP_DRAFT_EINVAL;
    if (B == 0) return LOOKUP_DRAFT_OK;
    if (!tokens || !base || !len || !index || !aligned16(index) || !model_draft || !committed || !state ||
        !out_long || !out_block || !out_len || !out_point_mass)
        return LOOKUP_DRAFT_EINVAL;
    int sms = 0;
    int rc = sm_count(&sms);
    if (rc != LOOKUP_DRAFT_OK) return rc;
    DraftParams p{};
    p.tokens = tokens;
    p.base = base;
    p.len = len;
    p.hd = static_cast<const Header *>(index);
    p.tab = reinterpret_cast<const Slot *>(static_cast<const char *>(index) + sizeof(Header));
    p.out_draft = nullptr;                               // the draft stays in registers
    p.out_len = out_draft_len;
    p.out_pos = nullptr;
    p.out_mlen = out_mlen;
    p.out_fallback = out_fallback;
    p.slots = slots;
    p.B = B;
    p.min_m = min_m;
    p.max_m = max_m;
    p.K = H + T;
    p.hash_bits = hash_bits;
    const lkd::PlanIO pio{model_draft, committed, state, out_long, out_block, out_len, out_point_mass, H, T,
                          replace_min, agree_min, agree_n, tail_min, slack, enter_steps, sticky};
    return lkd::launch_pdl2(index_draft_kernel<true>, warp_grid(B, sms), unsigned(kWarpThreads), stream, p, pio);
}

}  // extern "C"
