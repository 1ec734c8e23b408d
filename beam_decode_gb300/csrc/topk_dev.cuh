// Device building blocks of the item-constrained top-K, shared by the batch
// path (k_topk.cu) and the allocation-free entry point (k_noalloc.cu), so that
// both compute the same keys and the same selection from one copy of the code.
//
// The ranking comes from the output logits (zhiding.cn recsys-examples
// article, section "语义ID：解决稀疏性与长尾问题"); the top-K is item-constrained
// and the beam width dynamic (section "语义ID生成式推荐专用推理框架").
//
// Keys.  key(b, c) = S_b + (x_bc - LSE_b) in float32, each operation rounded
// once, stored as an order-preserving uint32 (larger key -> larger integer;
// -0.0 counts as +0.0); 0 marks "not a candidate".  The flat index of a
// candidate is f = b*C + c.  The order is key descending, then f ascending,
// so every selection is unique.
//
// Two stages.
//   stage 1 (per beam, inside the log-softmax kernel): when W < C a beam can
//     contribute at most W candidates, so each row keeps only its own top W
//     keys (rank counted against the row's other keys, same order) and
//     clears the rest.  The global top W is unchanged: every key above a
//     selected key in its own row is selected too.
//   stage 2 (cross-beam merge, one cluster of 8 CTAs per request, or of 4 when
//     the requests' clusters of 8 would not fit the GPU at once):
//     each CTA takes a contiguous flat range of the request's keys into shared
//     memory.  The threshold -- the W-th largest key -- is found by
//     range-adaptive bucketing: kNB equal-width buckets over [a0, largest
//     key], where a0 is the smallest key, or, when the request has at least W
//     rows, the smallest of the rows' largest keys if that is higher (those W
//     maxima lie at or above it, so the W-th largest key does too); each warp
//     counts its keys into its own histogram, and after a cluster barrier
//     every CTA sums the CTAs' histograms through distributed shared memory
//     and finds the same bucket holding the W-th key.  While that bucket
//     holds more than kThrCap keys (and more than one key value) it is
//     bucketed again (levels of kNBBits bits cover 32).  Keys above the
//     bucket are taken; the bucket's keys are collected and its top kk (key
//     desc, flat asc) taken too; each taken entry's output position is its
//     rank among them.  A bucket of more than kThrCap equal keys takes its
//     first kk in flat order instead.  Every exchange goes through the
//     cluster's shared memory: the merge needs no global scratch.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <float.h>
#include <math_constants.h>
#include <stdint.h>

#include "grbeam_internal.h"

namespace grb {
namespace topk {

namespace cg = cooperative_groups;

__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unorder_key(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// (m, s) pair: running maximum and sum of exp(x - m)
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 > m) {
        s = s * exp2f((m - m2) * CUDART_L2E_F) + s2;
        m = m2;
    } else if (m2 > -CUDART_INF_F) {
        s = s + s2 * exp2f((m2 - m) * CUDART_L2E_F);
    }
}

constexpr int kLsThreads = 256;  // threads of a log-softmax CTA

// Natural-log log-sum-exp of one logit row of V floats (16-byte aligned), split over the
// kLogitCluster CTAs of a cluster: each CTA reduces its part of the row with 16-byte loads
// into a running (max, sum), the cluster combines the partials through distributed
// shared memory in a fixed order, and every CTA returns the same value.
__device__ __forceinline__ float cluster_row_lse(const float* __restrict__ x, int V, cg::cluster_group& cluster,
                                                 int part, float* red_m, float* red_s, float* part_ms) {
    const int n4 = V >> 2;
    const int b0 = (int)((int64_t)n4 * part / kLogitCluster);
    const int b1 = (int)((int64_t)n4 * (part + 1) / kLogitCluster);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    // Each term is exp2((x - m) * log2 e): the difference first, so that a value equal or close
    // to the running max m gives an exact small argument whatever its magnitude (a product
    // m * log2 e rounded on its own is off by ~1e22 at |m| ~ 1e30).  m starts at the most
    // negative finite value, so that -inf logits add exactly 0 and a row of -inf has
    // log-sum-exp -inf.
    float m = -FLT_MAX, s = 0.f;
    int i = b0 + threadIdx.x;
    // 4 independent 16-byte loads in flight per thread
    for (; i + 3 * kLsThreads < b1; i += 4 * kLsThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(x4 + i + u * kLsThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float cm = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
            if (cm > m) { s *= exp2f((m - cm) * CUDART_L2E_F); m = cm; }
            s += exp2f((v[u].x - m) * CUDART_L2E_F) + exp2f((v[u].y - m) * CUDART_L2E_F) +
                 exp2f((v[u].z - m) * CUDART_L2E_F) + exp2f((v[u].w - m) * CUDART_L2E_F);
        }
    }
    for (; i < b1; i += kLsThreads) {
        float4 v = __ldcs(x4 + i);
        float cm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (cm > m) { s *= exp2f((m - cm) * CUDART_L2E_F); m = cm; }
        s += exp2f((v.x - m) * CUDART_L2E_F) + exp2f((v.y - m) * CUDART_L2E_F) +
             exp2f((v.z - m) * CUDART_L2E_F) + exp2f((v.w - m) * CUDART_L2E_F);
    }
    if (part == kLogitCluster - 1) {  // ragged tail of a row whose length is not a multiple of 4
        for (int j = (n4 << 2) + threadIdx.x; j < V; j += kLsThreads) lse_merge(m, s, x[j], 1.f);
    }
    // warp, then block
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        lse_merge(m, s, m2, s2);
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { red_m[w] = m; red_s[w] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = red_m[0], ss = red_s[0];
        for (int k = 1; k < kLsThreads / 32; ++k) lse_merge(mm, ss, red_m[k], red_s[k]);
        part_ms[0] = mm;
        part_ms[1] = ss;
    }
    cluster.sync();
    // every CTA combines the partials in the same order
    float mm = -CUDART_INF_F, ss = 0.f;
    for (int k = 0; k < kLogitCluster; ++k) {
        const float* pk = cluster.map_shared_rank(part_ms, k);
        lse_merge(mm, ss, pk[0], pk[1]);
    }
    cluster.sync();  // keep every CTA's shared memory alive until all have read it
    return mm + logf(ss);
}

// The ordered key of one (beam, code) candidate, or 0 when it is not one.  *nan is set when
// a valid candidate's key is NaN (it is then not a candidate either).
__device__ __forceinline__ uint32_t candidate_key(float S, float x, float lse, bool valid, bool* nan) {
    float key = __fadd_rn(S, __fsub_rn(x, lse));
    if (!valid) return 0u;
    if (key != key) {
        *nan = true;
        return 0u;
    }
    if (key == 0.f) key = 0.f;  // -0.0 -> +0.0
    return order_key(key);
}

// Stage 1 for one row whose C keys sit in shared memory (row_keys, every CTA of the row's
// cluster holding all of them): the key of code c survives when fewer than `keep` keys of
// the row come before it in the order (key desc, code asc).  Returns the key to store for
// code c (0 when it does not survive).
__device__ __forceinline__ uint32_t row_keep(const uint32_t* row_keys, int C, int c, int keep) {
    const uint32_t u = row_keys[c];
    if (u == 0u || keep >= C) return u;
    int before = 0;
    for (int j = 0; j < C; ++j) {
        const uint32_t v = row_keys[j];
        before += (v > u) || (v == u && j < c);
    }
    return before < keep ? u : 0u;
}

// The level gather of one live row for one CTA of its kLogitCluster cluster (`part`): the
// candidate keys of the C codes (xc = the row's logits of the level's codes, mk = the row's
// mask of valid codes, S = the beam's score, lse = the row's log-sum-exp), stage 1 when
// keep < C, and this CTA's part of the row written to out[0..C).  on_code(c, valid, lp)
// is called for the CTA's codes (lp = x - LSE).  The request's bound of candidate keys,
// range[0..1] = (~lower, upper), is raised to cover them (fire-and-forget atomics, one pair
// per warp of the row's first CTA), and range[2] to ~(this row's largest key): over the
// request's rows it holds ~(the smallest row maximum).  Returns whether a valid key was NaN.  Every thread of the CTA
// calls it; row_keys is kMaxCodes uint32 of shared memory.
template <typename OnCode>
__device__ __forceinline__ bool gather_row(const float* __restrict__ xc, const uint32_t* __restrict__ mk, float S,
                                           float lse, int C, int keep, int part, uint32_t* row_keys,
                                           uint32_t* __restrict__ out, uint32_t* range, OnCode&& on_code) {
    const int c0 = (int)((int64_t)C * part / kLogitCluster);
    const int c1 = (int)((int64_t)C * (part + 1) / kLogitCluster);
    const bool prune = keep < C;
    // Every CTA forms all C keys of the row: stage 1 ranks each against the whole row, and the
    // row's largest key feeds the bound below.  Only this CTA's part is written.
    bool nan = false;
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int c = (int)threadIdx.x; c < C; c += kLsThreads) {
        const bool valid = (mk[c >> 5] >> (c & 31)) & 1u;
        const float x = xc[c];
        const uint32_t u = candidate_key(S, x, lse, valid, &nan);
        if (u != 0u) {
            lo = min(lo, u);
            hi = max(hi, u);
        }
        row_keys[c] = u;
        if (!prune && c >= c0 && c < c1) {
            out[c] = u;
            on_code(c, valid, __fsub_rn(x, lse));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
    }
    __shared__ uint32_t warp_hi[kLsThreads / 32];
    if ((threadIdx.x & 31) == 0) {
        warp_hi[threadIdx.x >> 5] = hi;
        if (hi != 0u && part == 0) {
            atomicMax(range, ~lo);
            atomicMax(range + 1, hi);
        }
    }
    __syncthreads();
    if (part == 0 && threadIdx.x == 0) {
        // range[2] = ~(the smallest of the rows' largest keys); a row without a candidate
        // counts as 0, which turns the bound off
        uint32_t m = 0u;
#pragma unroll
        for (int k = 0; k < kLsThreads / 32; ++k) m = max(m, warp_hi[k]);
        atomicMax(range + 2, ~m);
    }
    if (prune) {
        for (int c = c0 + (int)threadIdx.x; c < c1; c += kLsThreads) {
            out[c] = row_keep(row_keys, C, c, keep);  // the beam's own top `keep`
            on_code(c, (mk[c >> 5] >> (c & 31)) & 1u, __fsub_rn(xc[c], lse));
        }
    }
    return nan;
}

// ---------------------------------------------------------------------------
// stage 2: cross-beam merge
// ---------------------------------------------------------------------------
constexpr int kMergeCTAs = 8;         // the largest cluster of a request (portable)
constexpr int kNBBits = 8;
constexpr int kNB = 1 << kNBBits;     // buckets per level (one per thread)
constexpr int kMergeThreads = kNB;
constexpr int kMergeStage = 16384;    // keys of a CTA's range kept in shared memory (else re-read)
// levels of kNBBits bits cover the 32-bit key: the last level's buckets are single values
constexpr int kLevels = (32 + kNBBits - 1) / kNBBits;
constexpr int kThrCap = 1024;         // threshold-bucket keys ranked directly

// Shared memory of a merge CTA (dynamic, followed by kMergeStage staged keys).  The fields
// other CTAs of the cluster read are marked "published".
struct MergeSmem {
    int hist[2][kNB];                   // published: this CTA's bucket counts, by level parity
    int hsub[kMergeThreads / 32][kNB];  // each warp's counts while they are being added up
    unsigned long long sure[kMaxBeam];  // published: this CTA's keys above the bucket, unordered
    unsigned long long thr[kThrCap];    // published: this CTA's keys in the bucket, unordered
    unsigned long long all[kMaxBeam + kThrCap];  // the cluster's lists, gathered for ranking
    int warp_tot[32];
    int wcnt[2][kMergeThreads / 32];    // each warp's keys above the bucket / in it
    int n_sure, n_thr;                  // published: lengths of sure / thr (tie path: keys equal)
    int off_s[kMergeCTAs], off_t[kMergeCTAs], len_s[kMergeCTAs], len_t[kMergeCTAs];
    int digit, kk, dcount;
};

struct MergeOut {
    int32_t* parent;   // [k] beam of each survivor, best first
    int32_t* code;     // [k]
    float* key;        // [k]
    int32_t* n;        // number of survivors
};

// inclusive prefix sum over the block in thread order; returns the block total in `total`
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int kWarps = kMergeThreads / 32;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int tv = (lane < kWarps) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, tv, off);
            if (lane >= off) tv += y;
        }
        warp_tot[lane] = tv;
    }
    __syncthreads();
    const int add = (w > 0) ? warp_tot[w - 1] : 0;
    total = warp_tot[kWarps - 1];
    __syncthreads();
    return v + add;
}

constexpr int kMergeBatch = 8;  // keys per thread in flight when the range is read from global memory

__device__ __forceinline__ unsigned long long sel_entry(uint32_t u, int flat) {
    return ((unsigned long long)u << 32) | (unsigned)(0xFFFFFFFFu - (uint32_t)flat);
}

// explicit shared-memory operations (the merge's structures live in dynamic shared memory)
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void smem_add(int* p, int v) {
    asm volatile("red.shared.add.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
// address of the same shared-memory object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(const void* p, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ int peer_ld(uint32_t a) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long peer_ld64(uint32_t a) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
    return v;
}

// The top-min(k_want, #candidates) of N ordered keys (flat order, 0 = no candidate) of one
// request, in (key desc, flat asc) order.  Called by every CTA of a cluster of kC CTAs
// (kC <= kMergeCTAs) with the same arguments; `stage` is kMergeStage uint32 of shared memory.  range[0..1] =
// (~lower, upper) bound of the candidate keys and range[2] = ~(the smallest of the N / C rows'
// largest keys), all raised by stage 1 (gather_row); any bounds that contain every candidate
// and lie at or below that smallest maximum give the same result.  The merge sets the three
// words back to 0 for the next call once every CTA has read them.
template <int kC = kMergeCTAs>
__device__ __forceinline__ void merge_select(const uint32_t* __restrict__ keys, int N, int C, int k_want,
                                             uint32_t* __restrict__ range, const MergeOut out, uint32_t* stage,
                                             MergeSmem& sm) {
    static_assert(kNB == kMergeThreads, "one bucket per thread");
    cg::cluster_group cl = cg::this_cluster();
    const int cr = (int)cl.block_rank();
    const int tid = threadIdx.x;
    const int lo = (int)((int64_t)N * cr / kC);
    const int n = (int)((int64_t)N * (cr + 1) / kC) - lo;
    const uint32_t* g = keys + lo;
    const bool staged = n <= kMergeStage;
    // Every pass visits the CTA's keys; a range too long for shared memory is re-read from
    // global memory kMergeBatch keys per thread at a time.
    auto for_keys = [&](auto&& f) {
        if (staged) {
            // four independent shared loads per thread per step
            int i = tid;
            for (; i + 3 * kMergeThreads < n; i += 4 * kMergeThreads) {
                uint32_t v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = stage[i + u * kMergeThreads];
#pragma unroll
                for (int u = 0; u < 4; ++u) f(i + u * kMergeThreads, v[u]);
            }
            for (; i < n; i += kMergeThreads) f(i, stage[i]);
        } else {
            for (int base = 0; base < n; base += kMergeThreads * kMergeBatch) {
                uint32_t v[kMergeBatch];
#pragma unroll
                for (int u = 0; u < kMergeBatch; ++u) {
                    const int i = base + u * kMergeThreads + tid;
                    v[u] = i < n ? __ldcg(g + i) : 0u;
                }
#pragma unroll
                for (int u = 0; u < kMergeBatch; ++u) {
                    const int i = base + u * kMergeThreads + tid;
                    if (i < n) f(i, v[u]);
                }
            }
        }
    };

    // ---- stage the range with every load in flight (16-byte loads where aligned)
    const uint32_t r_lo = ~__ldcg(range), r_hi = __ldcg(range + 1);
    // With at least k_want rows, the rows' largest keys are k_want distinct candidates at or
    // above the smallest of them, so the k_want-th largest key is too: the keys below that
    // bound cannot be selected and no pass counts or collects them.
    const uint32_t a0 = max(r_lo, N / C >= k_want ? ~__ldcg(range + 2) : 0u);
    if (staged) {
        const int head = min(n, (int)((4 - ((reinterpret_cast<uintptr_t>(g) >> 2) & 3)) & 3));
        if (tid < head) stage[tid] = __ldcg(g + tid);
        const int n4 = (n - head) >> 2;
        const uint4* g4 = reinterpret_cast<const uint4*>(g + head);
        for (int base = 0; base < n4; base += kMergeThreads * kMergeBatch) {
            uint4 v[kMergeBatch];
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const int j = base + u * kMergeThreads + tid;
                if (j < n4) v[u] = __ldcg(g4 + j);
            }
#pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
                const int j = base + u * kMergeThreads + tid;
                if (j < n4) {
                    uint32_t* d = stage + head + 4 * j;
                    d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
                }
            }
        }
        for (int i = head + 4 * n4 + tid; i < n; i += kMergeThreads) stage[i] = __ldcg(g + i);
    }
    __syncthreads();

    // The threshold bucket [a, b] holding the W-th key and the number kk of its keys taken.
    // The first level's counts also give the number of candidates: when it is at most k_want
    // every candidate is taken (take_all: a = b = 2^32 - 1, no bucket).
    bool take_all = r_lo > r_hi;  // no candidate in this call
    int n_valid = 0;              // candidates at or above a0
    uint32_t a = a0, b = r_hi;
    int kk = k_want, c_d = 0;
    // Each warp counts into its own histogram, so that it also knows how many of its keys lie
    // above the final bucket (the sum, over the levels, of its counts above the chosen bucket)
    // and in it: the collect pass then needs no counting pass of its own.
    constexpr int kWarps = kMergeThreads / 32;
    const int lane = tid & 31, wid = tid >> 5;
    const int jb = kNB - 1 - tid;  // this thread's bucket in the cluster-wide counts
    int sure_w = 0, thr_w = 0;     // this warp's keys above the bucket and in it (warp-uniform)
    auto warp_count_from = [&](int j0) {
        int c = 0;
        for (int j = j0 + lane; j < kNB; j += 32) c += sm.hsub[wid][j];
        return (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
    };
    if (!take_all) {
        for (int level = 0; level < kLevels; ++level) {
            // buckets of 2^sh keys: the smallest power of two with (b - a) >> sh < kNB
            const uint32_t span = (b - a) >> kNBBits;
            const int sh = span == 0u ? 0 : 32 - __clz(span);
            const uint32_t width = 1u << sh;
            int* h = sm.hist[level & 1];  // its last readers passed the previous level's barrier
#pragma unroll
            for (int w = 0; w < kWarps; ++w) sm.hsub[w][tid] = 0;
            __syncthreads();
            int* hw = sm.hsub[wid];
            for_keys([&](int, uint32_t u) {
                if (u >= a && u <= b) smem_add(&hw[(u - a) >> sh], 1);
            });
            __syncthreads();
            {
                int cnt = 0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) cnt += sm.hsub[w][tid];
                h[tid] = cnt;  // published with a plain store
            }
            cl.sync();
            // the cluster's count of bucket tid, then the bucket of the kk-th key (thread order
            // is descending bucket order)
            int tsum = 0;
#pragma unroll
            for (int r = 0; r < kC; ++r) tsum += peer_ld(peer_addr(&h[jb], r));
            int total;
            const int incl = block_incl_scan(tsum, sm.warp_tot, total);
            if (level == 0) {
                n_valid = total;
                if (total <= k_want) {
                    take_all = true;
                    sure_w = warp_count_from(0);
                    break;
                }
            }
            if (incl - tsum < kk && kk <= incl) {
                sm.digit = jb;
                sm.kk = kk - (incl - tsum);
                sm.dcount = tsum;
            }
            __syncthreads();
            const int d = sm.digit;
            c_d = sm.dcount;
            sure_w += warp_count_from(d + 1);
            thr_w = sm.hsub[wid][d];
            const uint32_t na = a + (uint32_t)d * width;
            b = (b - na < width - 1u) ? b : na + (width - 1u);
            a = na;
            kk = sm.kk;
            __syncthreads();
            if (c_d <= kThrCap || a == b) break;
        }
    }
    if (take_all) {
        a = b = 0xFFFFFFFFu;
        kk = 0;
        c_d = 0;
    }
    const int n_take = take_all ? n_valid : k_want;
    const int n_sure = n_take - kk;          // keys above the bucket
    const bool ranked = c_d <= kThrCap;      // else: one key value, its first kk in flat order

    // ---- collect: this CTA's keys above the bucket into `sure`, the bucket's keys into `thr`
    // (tie path: only counted), in flat order within each warp's share, from the warp's offset
    // on (the warps' counts come from their histograms; a shared counter that every warp
    // appended to would serialise the warps).
    auto classify = [&](uint32_t u, bool& is_s, bool& is_t) {
        is_s = u >= a0 && (take_all || u > b);  // a0 >= 1: no 0 (no candidate) qualifies
        is_t = !take_all && !is_s && u >= a;    // then u <= b
    };
    // (the staged and the global loop are kept apart: a select between a shared and a global
    // load per key would put a global round trip on every iteration)
    auto for_keys_warp = [&](auto&& f) {
        if (staged) {
            for (int base = 0; base < n; base += 4 * kMergeThreads) {
                uint32_t v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = base + k * kMergeThreads + tid;
                    v[k] = i < n ? stage[i] : 0u;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) f(base + k * kMergeThreads + tid, v[k]);
            }
        } else {
            for (int base = 0; base < n; base += kMergeBatch * kMergeThreads) {
                uint32_t v[kMergeBatch];
#pragma unroll
                for (int k = 0; k < kMergeBatch; ++k) {
                    const int i = base + k * kMergeThreads + tid;
                    v[k] = i < n ? __ldcg(g + i) : 0u;
                }
#pragma unroll
                for (int k = 0; k < kMergeBatch; ++k) f(base + k * kMergeThreads + tid, v[k]);
            }
        }
    };
    {
        if (lane == 0) {
            sm.wcnt[0][wid] = sure_w;
            sm.wcnt[1][wid] = thr_w;
        }
        __syncthreads();
        int os = 0, ot = 0, ts = 0, tt = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            os += w < wid ? sm.wcnt[0][w] : 0;
            ot += w < wid ? sm.wcnt[1][w] : 0;
            ts += sm.wcnt[0][w];
            tt += sm.wcnt[1][w];
        }
        if (tid == 0) {
            sm.n_sure = ts;
            sm.n_thr = tt;
        }
        const unsigned lt = (1u << lane) - 1u;
        for_keys_warp([&](int i, uint32_t u) {
            bool is_s, is_t;
            classify(u, is_s, is_t);
            const unsigned bs = __ballot_sync(0xffffffffu, is_s), bt = __ballot_sync(0xffffffffu, is_t);
            if (is_s) sm.sure[os + __popc(bs & lt)] = sel_entry(u, lo + i);
            if (is_t && ranked) sm.thr[ot + __popc(bt & lt)] = sel_entry(u, lo + i);
            os += __popc(bs);
            ot += __popc(bt);
        });
    }
    cl.sync();
    // gather every CTA's lists (offsets in cluster rank order)
    if (tid < kC) {
        sm.len_s[tid] = peer_ld(peer_addr(&sm.n_sure, tid));
        sm.len_t[tid] = peer_ld(peer_addr(&sm.n_thr, tid));
    }
    __syncthreads();
    if (tid == 0) {
        int os = 0, ot = 0;
        for (int r = 0; r < kC; ++r) {
            sm.off_s[r] = os;
            sm.off_t[r] = ot;
            os += sm.len_s[r];
            ot += sm.len_t[r];
        }
    }
    __syncthreads();
    const int n_thr = ranked ? c_d : 0;
    unsigned long long* s_sure = sm.all;
    unsigned long long* s_thr = sm.all + n_sure;
    // every entry of every CTA's two lists at once: entry j of the concatenation (sure lists in
    // rank order, then bucket lists) comes from the CTA whose block holds it
    {
        const int tot_s = sm.off_s[kC - 1] + sm.len_s[kC - 1];
        const int tot = tot_s + (ranked ? n_thr : 0);
        for (int j = tid; j < tot; j += kMergeThreads) {
            const bool is_s = j < tot_s;
            const int jj = is_s ? j : j - tot_s;
            int r = 0;
#pragma unroll
            for (int k = 1; k < kC; ++k) r += jj >= (is_s ? sm.off_s[k] : sm.off_t[k]);
            const int i = jj - (is_s ? sm.off_s[r] : sm.off_t[r]);
            const uint32_t pa = peer_addr(is_s ? (const void*)(sm.sure + i) : (const void*)(sm.thr + i), r);
            (is_s ? s_sure : s_thr)[jj] = peer_ld64(pa);
        }
    }
    cl.sync();  // no CTA leaves while another still reads its lists
    if (cr == 0 && tid == 0) {
        range[0] = 0u;  // every CTA has read the bounds: clear them for the next call
        range[1] = 0u;
        range[2] = 0u;
    }

    auto emit = [&](int pos, unsigned long long e) {
        const uint32_t flat = 0xFFFFFFFFu - (uint32_t)(e & 0xFFFFFFFFull);
        out.parent[pos] = (int)(flat / (uint32_t)C);
        out.code[pos] = (int)(flat % (uint32_t)C);
        out.key[pos] = unorder_key((uint32_t)(e >> 32));
    };
    if (!ranked) {
        // a bucket of one key value a == b: its first kk keys in flat order follow the sure ones
        const int eq_before = sm.off_t[cr];
        const int ties_here = max(0, min(sm.len_t[cr], kk - eq_before));
        int seen = 0;
        for (int base = 0; base < n && seen < ties_here; base += kMergeThreads) {
            const int i = base + tid;
            const int e = (i < n && (staged ? stage[i] : __ldcg(g + i)) == a) ? 1 : 0;
            int chunk;
            const int incl = block_incl_scan(e, sm.warp_tot, chunk);
            const int rank = seen + incl - e;
            if (e && rank < ties_here) emit(n_sure + eq_before + rank, sel_entry(a, lo + i));
            seen += chunk;
        }
    }

    // ---- ranks: a sure entry's position is the number of sure entries above it; a bucket
    // entry's is n_sure + the number of bucket entries above it, and it is taken when below kk
    constexpr int kSplit = 8;  // threads counting for one entry
    auto rank_list = [&](const unsigned long long* list, int len, int pos0, int limit) {
        const int r0 = (int)((int64_t)len * cr / kC);
        const int r1 = (int)((int64_t)len * (cr + 1) / kC);
        for (int base = r0 * kSplit; base < r1 * kSplit; base += kMergeThreads) {
            const int idx = base + tid;
            const int e = idx / kSplit, part = idx % kSplit;
            const bool act = e < r1;
            const unsigned long long me = act ? list[e] : 0ull;
            int above = 0;
            if (act) {
#pragma unroll 4
                for (int j = part; j < len; j += kSplit) above += list[j] > me;
            }
#pragma unroll
            for (int off = kSplit / 2; off > 0; off >>= 1) above += __shfl_xor_sync(0xffffffffu, above, off);
            if (act && part == 0 && above < limit) emit(pos0 + above, me);
        }
    };
    rank_list(s_sure, n_sure, 0, n_sure);
    rank_list(s_thr, n_thr, n_sure, kk);
    if (cr == 0 && tid == 0) *out.n = n_take;
}

}  // namespace topk
}  // namespace grb
