// Log-softmax, item-constrained top-K, BeamPath advance and results.
//
// The output logits give the ranking (zhiding.cn recsys-examples article,
// section "语义ID：解决稀疏性与长尾问题"); the runtime keeps item-constrained
// top-K, dynamic beam width and BeamPath (section "语义ID生成式推荐专用推理框架");
// every surviving beam is returned ("Advancing Generative Recommendation
// Inference: our collaboration with NVIDIA on TensorRT LLM", section
// "Background: what inference a recommendation request needs").
//
// Kernels
//   k_logsoftmax_gather  one pass over each live logit row (a cluster of 4 CTAs
//                        per row): log-sum-exp of the full vocabulary, then the
//                        level's C code logits -> masked float32 keys
//                        key = S_b + (x - LSE_b), stored as order-preserving
//                        uint32 (0 = not a candidate).  HBM-bound.
//   k_topk_select        per request: radix select of the W-th largest key over
//                        n_live*C candidates (13/11/8-bit digits, the threshold
//                        digit compacted into shared memory), ties at the
//                        threshold taken in flat-index order, then a bitonic
//                        sort of the survivors by (key desc, flat asc).
//   k_advance            BeamPath commit: parent, token, trie node, score,
//                        ancestry row; sets the next step's live width.  No KV
//                        is moved: later steps reach a beam's BeamKV slots
//                        through its ancestry row.
//   k_results            code strings, item ids and scores of the final beams.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <limits.h>
#include <stdint.h>

#include "grbeam_internal.h"

namespace cg = cooperative_groups;

namespace grb {
namespace {

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

// a row takes part in the step when its request is still decoding (t_r < L_r) and the
// row holds one of the request's live beams
__device__ __forceinline__ bool row_live(const GrState& st, int row, int& r, int& b, int& t) {
    r = st.row_req[row];
    const GrReqDev& R = st.req[r];
    b = row - R.row_off;
    t = st.req_step[r];
    if (t >= R.n_levels) return false;
    return b < st.n_beams[r * (st.n_levels + 1) + t];
}

// ---------------------------------------------------------------------------
// K3: fused full-vocabulary log-softmax + level gather + trie mask
// ---------------------------------------------------------------------------
constexpr int kLsThreads = 256;

// Natural-log log-sum-exp of one logit row of V floats (16-byte aligned), split over the
// kLogitCluster CTAs of a cluster: each CTA reduces a quarter of the row with 16-byte
// loads into a running (max, sum), the cluster combines the four partials through
// distributed shared memory in a fixed order, and every CTA returns the same value.
__device__ __forceinline__ float cluster_row_lse(const float* __restrict__ x, int V, cg::cluster_group& cluster,
                                                 int part, float* red_m, float* red_s, float* part_ms) {
    const int n4 = V >> 2;
    const int b0 = (int)((int64_t)n4 * part / kLogitCluster);
    const int b1 = (int)((int64_t)n4 * (part + 1) / kLogitCluster);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float m = -CUDART_INF_F, s = 0.f;
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
            const float ml = m * CUDART_L2E_F;
            s += exp2f(fmaf(v[u].x, CUDART_L2E_F, -ml)) + exp2f(fmaf(v[u].y, CUDART_L2E_F, -ml)) +
                 exp2f(fmaf(v[u].z, CUDART_L2E_F, -ml)) + exp2f(fmaf(v[u].w, CUDART_L2E_F, -ml));
        }
    }
    for (; i < b1; i += kLsThreads) {
        float4 v = __ldcs(x4 + i);
        float cm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (cm > m) { s *= exp2f((m - cm) * CUDART_L2E_F); m = cm; }
        const float ml = m * CUDART_L2E_F;
        s += exp2f(fmaf(v.x, CUDART_L2E_F, -ml)) + exp2f(fmaf(v.y, CUDART_L2E_F, -ml)) +
             exp2f(fmaf(v.z, CUDART_L2E_F, -ml)) + exp2f(fmaf(v.w, CUDART_L2E_F, -ml));
    }
    if (part == kLogitCluster - 1) {  // ragged tail of a row whose length is not a multiple of 4
        for (int j = (n4 << 2) + threadIdx.x; j < V; j += kLsThreads) {
            float v = x[j];
            lse_merge(m, s, v, 1.f);
        }
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
    // every CTA combines the four partials in the same order
    float mm = -CUDART_INF_F, ss = 0.f;
    for (int k = 0; k < kLogitCluster; ++k) {
        const float* pk = cluster.map_shared_rank(part_ms, k);
        lse_merge(mm, ss, pk[0], pk[1]);
    }
    cluster.sync();  // keep every CTA's shared memory alive until all have read it
    return mm + logf(ss);
}


__global__ void __cluster_dims__(kLogitCluster, 1, 1) __launch_bounds__(kLsThreads)
k_logsoftmax_gather(GrState st, const float* __restrict__ logits, int64_t ld,
                    float* __restrict__ logprobs_out, float* __restrict__ lse_out,
                    const float* __restrict__ lse_in) {
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kLogitCluster;
    const int part = (int)cluster.block_rank();
    int r, b;
    int t;
    if (!row_live(st, row, r, b, t)) return;  // uniform over the cluster

    __shared__ float red_m[kLsThreads / 32], red_s[kLsThreads / 32];
    __shared__ float part_ms[2];

    const float* x = logits + (int64_t)row * ld;
    const int V = st.vocab;
    float lse;
    if (lse_in == nullptr) {
        lse = cluster_row_lse(x, V, cluster, part, red_m, red_s, part_ms);
    } else {
        lse = lse_in[row];
    }
    if (part == 0 && threadIdx.x == 0 && lse_out != nullptr) lse_out[row] = lse;

    // level gather of C codes, split over the cluster
    const GrReqDev& R = st.req[r];
    const int C = st.C;
    const int64_t node = (t == 0) ? 0 : st.node[(int64_t)(t - 1) * st.rows + row];
    const float S = (t == 0) ? 0.f : st.score[(int64_t)(t - 1) * st.rows + row];
    if (node < 0 || node >= R.n_nodes) {
        if (threadIdx.x == 0 && part == 0) atomicOr(st.status, kStatusBadNode);
        return;
    }
    const uint32_t* mk = R.mask + node * R.mask_words;
    const float* xc = x + st.code_base + (int64_t)t * C;
    uint32_t* out = st.cand + (int64_t)row * C;
    const int c0 = (int)((int64_t)C * part / kLogitCluster);
    const int c1 = (int)((int64_t)C * (part + 1) / kLogitCluster);
    for (int c = c0 + threadIdx.x; c < c1; c += kLsThreads) {
        const bool valid = (mk[c >> 5] >> (c & 31)) & 1u;
        const float xv = xc[c];
        const float lp = __fsub_rn(xv, lse);
        float key = __fadd_rn(S, lp);
        uint32_t u = 0;
        if (valid) {
            if (key != key) {
                atomicOr(st.status, kStatusNanKey);
            } else {
                if (key == 0.f) key = 0.f;  // -0.0 -> +0.0
                u = order_key(key);
            }
        }
        out[c] = u;
        if (logprobs_out != nullptr) logprobs_out[(int64_t)row * C + c] = valid ? lp : -CUDART_INF_F;
    }
}

// ---------------------------------------------------------------------------
// K4: cross-beam top-K of one request
// ---------------------------------------------------------------------------
// Keys are order-preserving uint32 (0 = not a candidate); the flat index of a
// candidate is its position b*C + c in the request's key array.  The k-th
// largest key tau is found digit by digit (13 bits, then 11, then 8):
//   A  one pass over all keys: histogram of the top 13 bits;
//   B  one pass: keys above the threshold digit go straight to the output
//      set, keys in the threshold digit are compacted into shared memory;
//   C  the remaining 19 bits are resolved on the compacted keys;
//   D  keys above tau are taken, keys equal to tau in flat-index order;
// then the survivors are sorted by (key desc, flat asc) with a bitonic network.
// If the threshold digit holds more than kSelCap keys, B-D run on global
// memory instead (three histogram passes over all keys).
constexpr int kSelThreads = 1024;
constexpr int kBinsA = 8192;    // top digit: sign, exponent, 4 mantissa bits
constexpr int kShiftA = 19;
constexpr int kSelCap = 4096;   // compacted threshold-digit keys kept in shared memory

struct SelSmem {
    int hist[kBinsA];
    uint32_t ck[kSelCap];       // compacted keys of the threshold digit
    uint32_t ci[kSelCap];       // their flat indices
    unsigned long long sel[kMaxBeam];
    int warp_tot[32];
    int digit, kk, count, n_sel, n_c;
};

// inclusive prefix sum over the block in thread order; returns the block total
__device__ __forceinline__ int block_incl_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int tv = (lane < (kSelThreads >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, tv, off);
            if (lane >= off) tv += y;
        }
        warp_tot[lane] = tv;  // inclusive warp prefix
    }
    __syncthreads();
    const int add = (w > 0) ? warp_tot[w - 1] : 0;
    total = warp_tot[(kSelThreads >> 5) - 1];
    __syncthreads();
    return v + add;
}

// digit d of the kk-th largest element given a histogram of nbins bins:
// sum(bins > d) < kk <= sum(bins >= d); writes sm.digit and sm.kk (kk within d)
__device__ __forceinline__ void find_digit(SelSmem& sm, int nbins, int kk) {
    const int tid = threadIdx.x;
    const int per = nbins > kSelThreads ? nbins / kSelThreads : 1;
    const bool owner = tid < nbins / per;
    const int hi = nbins - 1 - tid * per;  // thread order = descending bin order
    int v = 0;
    if (owner)
        for (int e = 0; e < per; ++e) v += sm.hist[hi - e];
    int total;
    const int incl = block_incl_scan(v, sm.warp_tot, total);
    const int excl = incl - v;
    if (owner && excl < kk && kk <= incl) {
        int acc = excl;
        for (int e = 0; e < per; ++e) {
            const int h = sm.hist[hi - e];
            if (acc + h >= kk) { sm.digit = hi - e; sm.kk = kk - acc; break; }
            acc += h;
        }
    }
    __syncthreads();
}

__device__ __forceinline__ unsigned long long sel_entry(uint32_t u, uint32_t flat) {
    return ((unsigned long long)u << 32) | (unsigned)(0xFFFFFFFFu - flat);
}

// warp-aggregated histogram add of `bin` for lanes with q set (all lanes call)
__device__ __forceinline__ void hist_add(int* hist, bool q, uint32_t bin) {
    if (__any_sync(0xffffffffu, q)) {
        const unsigned peers = __match_any_sync(0xffffffffu, q ? bin : 0xFFFFFFFFu);
        if (q && (__ffs(peers) - 1) == (int)(threadIdx.x & 31)) atomicAdd(&hist[bin], __popc(peers));
    }
}

// B-D on global memory, for a threshold digit too full for shared memory:
// two more histogram passes over all keys, then the gather
__device__ void select_global(SelSmem& sm, const uint32_t* keys, int N, uint32_t prefix, uint32_t pmask, int kk,
                              int k_want) {
    const int tid = threadIdx.x;
    const int shifts[2] = {8, 0};
    const int widths[2] = {11, 8};
    for (int pass = 0; pass < 2; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int i = tid; i < kBinsA; i += kSelThreads) sm.hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < N; base += kSelThreads) {
            const int i = base + tid;
            const uint32_t u = (i < N) ? keys[i] : 0u;
            const bool q = (u != 0) && ((u & pmask) == prefix);
            hist_add(sm.hist, q, (u >> sh) & dmask);
        }
        __syncthreads();
        find_digit(sm, 1 << widths[pass], kk);
        prefix |= (uint32_t)sm.digit << sh;
        pmask |= dmask << sh;
        kk = sm.kk;
    }
    const uint32_t tau = prefix;
    const int n_eq = sm.hist[sm.digit];
    __syncthreads();
    for (int i = tid; i < N; i += kSelThreads) {
        const uint32_t u = keys[i];
        if (u > tau || (n_eq == kk && u == tau)) sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(u, (uint32_t)i);
    }
    __syncthreads();
    if (n_eq != kk) {  // ties at the threshold: the kk smallest flat indices
        int base_rank = 0;
        for (int start = 0; start < N; start += kSelThreads) {
            const int i = start + tid;
            const int e = (i < N && keys[i] == tau) ? 1 : 0;
            int total;
            const int incl = block_incl_scan(e, sm.warp_tot, total);
            const int rank = base_rank + incl - e;
            if (e && rank < kk) sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(tau, (uint32_t)i);
            base_rank += total;
            if (base_rank >= kk) break;
        }
        __syncthreads();
    }
    (void)k_want;
}

__global__ void __launch_bounds__(kSelThreads) k_topk_select(GrState st) {
    extern __shared__ __align__(16) uint8_t sel_smem_raw[];
    SelSmem& sm = *reinterpret_cast<SelSmem*>(sel_smem_raw);
    const int r = blockIdx.x;
    const GrReqDev R = st.req[r];
    const int t = st.req_step[r];
    if (t >= R.n_levels) return;
    const int C = st.C;
    const int n_live = st.n_beams[r * (st.n_levels + 1) + t];
    const int N = n_live * C;
    const uint32_t* keys = st.cand + (int64_t)R.row_off * C;
    const int k_want = R.width;
    const int tid = threadIdx.x;

    // A: histogram of the top digit and the number of candidates
    for (int i = tid; i < kBinsA; i += kSelThreads) sm.hist[i] = 0;
    if (tid == 0) { sm.count = 0; sm.n_sel = 0; sm.n_c = 0; }
    __syncthreads();
    int my_valid = 0;
    for (int base = 0; base < N; base += 4 * kSelThreads) {
        uint32_t u[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = base + k * kSelThreads + tid;
            u[k] = (i < N) ? keys[i] : 0u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            my_valid += (u[k] != 0);
            hist_add(sm.hist, u[k] != 0, u[k] >> kShiftA);
        }
    }
    atomicAdd(&sm.count, my_valid);
    __syncthreads();
    const int n_valid = sm.count;
    int n_take;
    if (n_valid <= k_want) {
        // every candidate survives
        for (int i = tid; i < N; i += kSelThreads) {
            const uint32_t u = keys[i];
            if (u != 0) sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(u, (uint32_t)i);
        }
        n_take = n_valid;
    } else {
        find_digit(sm, kBinsA, k_want);
        const uint32_t dA = (uint32_t)sm.digit;
        int kk = sm.kk;
        const int cnt_a = sm.hist[dA];
        __syncthreads();
        n_take = k_want;
        if (cnt_a <= kSelCap) {
            // B: above the digit -> output set; the digit itself -> shared memory
            for (int i = tid; i < N; i += kSelThreads) {
                const uint32_t u = keys[i];
                if (u == 0) continue;
                const uint32_t d = u >> kShiftA;
                if (d > dA) {
                    sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(u, (uint32_t)i);
                } else if (d == dA) {
                    const int pos = atomicAdd(&sm.n_c, 1);
                    sm.ck[pos] = u;
                    sm.ci[pos] = (uint32_t)i;
                }
            }
            __syncthreads();
            const int n_c = sm.n_c;
            // C: the remaining 19 bits on the compacted keys
            uint32_t prefix = dA << kShiftA, pmask = ~((1u << kShiftA) - 1u);
            const int shifts[2] = {8, 0};
            const int widths[2] = {11, 8};
            for (int pass = 0; pass < 2; ++pass) {
                const int sh = shifts[pass];
                const uint32_t dmask = (1u << widths[pass]) - 1u;
                for (int i = tid; i < (1 << widths[pass]); i += kSelThreads) sm.hist[i] = 0;
                __syncthreads();
                for (int e = tid; e < n_c; e += kSelThreads) {
                    const uint32_t u = sm.ck[e];
                    if ((u & pmask) == prefix) atomicAdd(&sm.hist[(u >> sh) & dmask], 1);
                }
                __syncthreads();
                find_digit(sm, 1 << widths[pass], kk);
                prefix |= (uint32_t)sm.digit << sh;
                pmask |= dmask << sh;
                kk = sm.kk;
            }
            const uint32_t tau = prefix;
            const int n_eq = sm.hist[sm.digit];
            __syncthreads();
            // D: above tau, then ties at tau in flat-index order
            if (tid == 0) sm.count = 0;
            __syncthreads();
            for (int e = tid; e < n_c; e += kSelThreads) {
                const uint32_t u = sm.ck[e];
                if (u > tau || (n_eq == kk && u == tau)) {
                    sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(u, sm.ci[e]);
                } else if (u == tau) {
                    sm.hist[atomicAdd(&sm.count, 1)] = (int)sm.ci[e];  // tie indices
                }
            }
            __syncthreads();
            if (n_eq != kk) {
                int P = 1;
                while (P < n_eq) P <<= 1;
                for (int e = n_eq + tid; e < P; e += kSelThreads) sm.hist[e] = INT_MAX;
                __syncthreads();
                for (int k = 2; k <= P; k <<= 1) {  // ascending sort of the tie indices
                    for (int j = k >> 1; j > 0; j >>= 1) {
                        for (int e = tid; e < P; e += kSelThreads) {
                            const int ex = e ^ j;
                            if (ex > e) {
                                const int a = sm.hist[e], c = sm.hist[ex];
                                if (((e & k) == 0) ? (a > c) : (a < c)) { sm.hist[e] = c; sm.hist[ex] = a; }
                            }
                        }
                        __syncthreads();
                    }
                }
                for (int e = tid; e < kk; e += kSelThreads)
                    sm.sel[atomicAdd(&sm.n_sel, 1)] = sel_entry(tau, (uint32_t)sm.hist[e]);
                __syncthreads();
            }
        } else {
            select_global(sm, keys, N, dA << kShiftA, ~((1u << kShiftA) - 1u), kk, k_want);
        }
    }
    __syncthreads();
    // bitonic sort of n_take entries, descending
    int P = 1;
    while (P < n_take) P <<= 1;
    for (int i = n_take + tid; i < P; i += kSelThreads) sm.sel[i] = 0ull;
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += kSelThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = sm.sel[i], c = sm.sel[ixj];
                    const bool desc = ((i & k) == 0);
                    if (desc ? (a < c) : (a > c)) { sm.sel[i] = c; sm.sel[ixj] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < n_take; i += kSelThreads) {
        const unsigned long long e = sm.sel[i];
        const uint32_t flat = 0xFFFFFFFFu - (uint32_t)(e & 0xFFFFFFFFull);
        st.sel_parent[R.row_off + i] = (int)(flat / (uint32_t)C);
        st.sel_code[R.row_off + i] = (int)(flat % (uint32_t)C);
        st.sel_key[R.row_off + i] = unorder_key((uint32_t)(e >> 32));
    }
    if (tid == 0) st.n_sel[r] = n_take;
}

// ---------------------------------------------------------------------------
// K5: BeamPath advance (no KV copies)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxBeam) k_advance(GrState st) {
    const int r = blockIdx.x;
    const GrReqDev R = st.req[r];
    __shared__ int t_sh;
    if (threadIdx.x == 0) t_sh = st.req_step[r];
    __syncthreads();
    const int t = t_sh;
    if (t >= R.n_levels) return;
    const int L = st.n_levels;
    const int n = st.n_sel[r];
    if (threadIdx.x == 0) {
        st.n_beams[r * (L + 1) + t + 1] = n;
        st.req_step[r] = t + 1;  // every thread has its copy of t already
    }
    const int i = threadIdx.x;
    if (i >= n) return;
    const int row = R.row_off + i;
    const int p = st.sel_parent[row];
    const int c = st.sel_code[row];
    const int64_t prow = R.row_off + p;
    const int64_t pnode = (t == 0) ? 0 : st.node[(int64_t)(t - 1) * st.rows + prow];
    if (pnode < 0 || pnode >= R.n_nodes) { atomicOr(st.status, kStatusBadNode); return; }
    const uint32_t* mk = R.mask + pnode * R.mask_words;
    int rank = 0;
    for (int w = 0; w < (c >> 5); ++w) rank += __popc(mk[w]);
    rank += __popc(mk[c >> 5] & ((1u << (c & 31)) - 1u));
    const int64_t lvl = (int64_t)t * st.rows;
    st.parent[lvl + row] = p;
    st.token[lvl + row] = st.code_base + t * st.C + c;
    st.node[lvl + row] = R.child_base[pnode] + rank;
    st.score[lvl + row] = st.sel_key[row];
    int32_t* dst = st.path + (lvl + row) * L;
    if (t > 0) {
        const int32_t* src = st.path + ((int64_t)(t - 1) * st.rows + prow) * L;
        for (int j = 0; j < t; ++j) dst[j] = src[j];
    }
    dst[t] = i;
}

// ---------------------------------------------------------------------------
// K6: results of the final level
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kMaxBeam) k_results(GrState st) {
    const int r = blockIdx.x;
    const GrReqDev R = st.req[r];
    const int L = R.n_levels;
    const int n = st.n_beams[r * (st.n_levels + 1) + L];
    const int i = threadIdx.x;
    if (i >= n) return;
    const int row = R.row_off + i;
    const int64_t last = (int64_t)(L - 1) * st.rows + row;
    const int32_t* path = st.path + last * st.n_levels;
    for (int j = 0; j < L; ++j) {
        const int slot = path[j];
        const int tok = st.token[(int64_t)j * st.rows + R.row_off + slot];
        st.res_codes[(int64_t)row * st.n_levels + j] = tok - st.code_base - j * st.C;
    }
    const int64_t leaf = (int64_t)st.node[last] - R.leaf_base;
    st.res_items[row] = (leaf >= 0) ? R.leaf_item[leaf] : -1;
    st.res_scores[row] = st.score[last];
}

__global__ void k_init_state(GrState st) {
    const int L1 = st.n_levels + 1;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < st.n_req * L1; i += gridDim.x * blockDim.x)
        st.n_beams[i] = (i % L1 == 0) ? 1 : 0;
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < st.n_req; r += gridDim.x * blockDim.x) st.req_step[r] = 0;
    if (blockIdx.x == 0 && threadIdx.x < 4) st.status[threadIdx.x] = 0;
}

// a request (re)starts at level 0 with its single root beam
__global__ void k_init_request(GrState st, int r) {
    const int L1 = st.n_levels + 1;
    for (int i = threadIdx.x; i < L1; i += blockDim.x) st.n_beams[r * L1 + i] = (i == 0) ? 1 : 0;
    if (threadIdx.x == 0) st.req_step[r] = 0;
}

// every request past `step` goes back to it (its levels 0..step-1 stay committed)
__global__ void k_set_step(GrState st, int step) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < st.n_req; r += gridDim.x * blockDim.x)
        if (st.req_step[r] > step) st.req_step[r] = step;
}

// ---------------------------------------------------------------------------
// Multi-item scoring: label-token log-probabilities and the ranking
// ---------------------------------------------------------------------------
// One cluster per candidate row: log-sum-exp of the full vocabulary, then the label
// tokens' entries x[label] - LSE (each rounded once).
__global__ void __cluster_dims__(kLogitCluster, 1, 1) __launch_bounds__(kLsThreads)
k_label_logprobs(const float* __restrict__ logits, int64_t ld, int vocab, const int32_t* __restrict__ labels,
                 int n_labels, float* __restrict__ out, int32_t* __restrict__ status) {
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kLogitCluster;
    const int part = (int)cluster.block_rank();
    __shared__ float red_m[kLsThreads / 32], red_s[kLsThreads / 32];
    __shared__ float part_ms[2];
    const float* x = logits + (int64_t)row * ld;
    const float lse = cluster_row_lse(x, vocab, cluster, part, red_m, red_s, part_ms);
    if (part != 0) return;
    for (int k = threadIdx.x; k < n_labels; k += kLsThreads) {
        const float lp = __fsub_rn(x[labels[k]], lse);
        if (lp != lp) atomicOr(status, kStatusNanKey);
        out[(int64_t)row * n_labels + k] = lp;
    }
}

// One CTA per request: its candidates ordered by the first label's log-probability,
// highest first, ties by candidate index (bitonic sort of (key, ~index) pairs).
constexpr int kRankThreads = 1024;
__global__ void __launch_bounds__(kRankThreads) k_rank(const float* __restrict__ lp, int n_labels,
                                                      const int32_t* __restrict__ cand_off,
                                                      int32_t* __restrict__ rank_out, int32_t* __restrict__ status) {
    __shared__ unsigned long long e[kRankThreads];
    const int r = blockIdx.x;
    const int c0 = cand_off[r], n = cand_off[r + 1] - c0;
    const int tid = threadIdx.x;
    unsigned long long v = 0ull;  // padding sorts last
    if (tid < n) {
        float f = lp[(int64_t)(c0 + tid) * n_labels];
        uint32_t u = 0;
        if (f != f) atomicOr(status, kStatusNanKey);
        else u = order_key(f == 0.f ? 0.f : f);
        v = ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)tid);
    }
    e[tid] = v;
    __syncthreads();
    for (int k = 2; k <= kRankThreads; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int p = tid ^ j;
            if (p > tid) {
                const unsigned long long a = e[tid], b = e[p];
                if (((tid & k) == 0) ? (a < b) : (a > b)) { e[tid] = b; e[p] = a; }
            }
            __syncthreads();
        }
    }
    if (tid < n) rank_out[c0 + tid] = (int32_t)(0xFFFFFFFFu - (uint32_t)(e[tid] & 0xFFFFFFFFull));
}

}  // namespace

cudaError_t launch_label_logprobs(const float* logits, int64_t ld, int vocab, const int32_t* labels, int n_labels,
                                  int n_rows, float* out, int32_t* status, cudaStream_t s) {
    k_label_logprobs<<<n_rows * kLogitCluster, kLsThreads, 0, s>>>(logits, ld, vocab, labels, n_labels, out, status);
    return cudaGetLastError();
}

cudaError_t launch_rank(const float* lp, int n_labels, const int32_t* cand_off, int n_req, int32_t* rank_out,
                        int32_t* status, cudaStream_t s) {
    k_rank<<<n_req, kRankThreads, 0, s>>>(lp, n_labels, cand_off, rank_out, status);
    return cudaGetLastError();
}

cudaError_t launch_init_state(const GrState& st, cudaStream_t s) {
    k_init_state<<<1, 256, 0, s>>>(st);
    return cudaGetLastError();
}

cudaError_t launch_init_request(const GrState& st, int r, cudaStream_t s) {
    k_init_request<<<1, 32, 0, s>>>(st, r);
    return cudaGetLastError();
}

cudaError_t launch_set_step(const GrState& st, int step, cudaStream_t s) {
    k_set_step<<<1, 256, 0, s>>>(st, step);
    return cudaGetLastError();
}

cudaError_t launch_logsoftmax_gather(const GrState& st, const float* logits, int64_t ld,
                                     float* logprobs_out, float* lse_out, const float* lse_in,
                                     cudaStream_t s) {
    dim3 grid(st.rows * kLogitCluster);
    k_logsoftmax_gather<<<grid, kLsThreads, 0, s>>>(st, logits, ld, logprobs_out, lse_out, lse_in);
    return cudaGetLastError();
}

cudaError_t launch_topk_select(const GrState& st, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_topk_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(SelSmem));
        if (e != cudaSuccess) return e;
        attr = true;
    }
    k_topk_select<<<st.n_req, kSelThreads, sizeof(SelSmem), s>>>(st);
    return cudaGetLastError();
}

cudaError_t launch_advance(const GrState& st, cudaStream_t s) {
    k_advance<<<st.n_req, kMaxBeam, 0, s>>>(st);
    return cudaGetLastError();
}

cudaError_t launch_results(const GrState& st, cudaStream_t s) {
    k_results<<<st.n_req, kMaxBeam, 0, s>>>(st);
    return cudaGetLastError();
}

}  // namespace grb
