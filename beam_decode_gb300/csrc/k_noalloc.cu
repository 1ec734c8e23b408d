// Item-constrained top-K of one request without caller-provided scratch.
//
// gr_constrained_topk needs the workspace that the caller allocates for a
// gr_beam handle.  Some callers cannot allocate device memory: plugins of an
// inference server that are handed only their input and output tensors, or
// services whose device memory is budgeted once at start-up and must not
// grow per request.  gr_constrained_topk_noalloc serves them: the caller
// passes only inputs and outputs, and the candidate keys that pass from the
// first kernel to the second live in a fixed array of this library,
// g_noalloc_keys, which every GPU that loads the library keeps until the
// process exits.
//
// What it computes is the selection of gr_constrained_topk for one request:
// key(b, c) = S_b + (x[b][code_lo + c] - LSE_b) over the codes c whose bit is
// set in the row's mask, ordered by key descending then flat index b*C + c
// ascending, the first min(k, #candidates) kept.  The arithmetic (the
// four-CTA log-sum-exp of each row, the order-preserving key encoding, the
// radix select and the bitonic sort) is the same as in k_topk.cu, so both
// entry points return identical selections for identical inputs.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "grbeam_internal.h"

namespace cg = cooperative_groups;

namespace grb {
gr_status set_error(gr_status code, const char* fmt, ...);  // api.cu
}

namespace {

constexpr int kNaMaxCandidates = GR_NOALLOC_MAX_CANDIDATES;
constexpr int kNaCluster = 4;
constexpr int kNaThreads = 256;
constexpr int kNaSelThreads = 1024;
constexpr int kNaHistBins = 4096;
constexpr int kNaMaxDevices = 64;

// Scratch of the no-alloc path: ordered candidate keys [n_rows][n_codes].
// Host code must not use this name as an address (it is a host-side stand-in);
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint32_t g_noalloc_keys[kNaMaxCandidates];

__device__ __forceinline__ uint32_t na_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float na_unorder_key(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ void na_lse_merge(float& m, float& s, float m2, float s2) {
    if (m2 > m) {
        s = s * exp2f((m - m2) * CUDART_L2E_F) + s2;
        m = m2;
    } else if (m2 > -CUDART_INF_F) {
        s = s + s2 * exp2f((m2 - m) * CUDART_L2E_F);
    }
}

// one 4-CTA cluster per row: row log-sum-exp, then the masked keys of the codes
__global__ void __cluster_dims__(kNaCluster, 1, 1) __launch_bounds__(kNaThreads)
k_na_logsoftmax_gather(const float* __restrict__ logits, int64_t ld, int vocab, int code_lo, int n_codes,
                       const float* __restrict__ scores, const uint32_t* __restrict__ mask, int mask_words,
                       uint32_t* __restrict__ keys) {
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kNaCluster;
    const int part = (int)cluster.block_rank();
    __shared__ float red_m[kNaThreads / 32], red_s[kNaThreads / 32];
    __shared__ float part_ms[2];
    const float* x = logits + (int64_t)row * ld;
    const int n4 = vocab >> 2;
    const int b0 = (int)((int64_t)n4 * part / kNaCluster);
    const int b1 = (int)((int64_t)n4 * (part + 1) / kNaCluster);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float m = -CUDART_INF_F, s = 0.f;
    int i = b0 + threadIdx.x;
    for (; i + 3 * kNaThreads < b1; i += 4 * kNaThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(x4 + i + u * kNaThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float cm = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
            if (cm > m) { s *= exp2f((m - cm) * CUDART_L2E_F); m = cm; }
            const float ml = m * CUDART_L2E_F;
            s += exp2f(fmaf(v[u].x, CUDART_L2E_F, -ml)) + exp2f(fmaf(v[u].y, CUDART_L2E_F, -ml)) +
                 exp2f(fmaf(v[u].z, CUDART_L2E_F, -ml)) + exp2f(fmaf(v[u].w, CUDART_L2E_F, -ml));
        }
    }
    for (; i < b1; i += kNaThreads) {
        float4 v = __ldcs(x4 + i);
        float cm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        if (cm > m) { s *= exp2f((m - cm) * CUDART_L2E_F); m = cm; }
        const float ml = m * CUDART_L2E_F;
        s += exp2f(fmaf(v.x, CUDART_L2E_F, -ml)) + exp2f(fmaf(v.y, CUDART_L2E_F, -ml)) +
             exp2f(fmaf(v.z, CUDART_L2E_F, -ml)) + exp2f(fmaf(v.w, CUDART_L2E_F, -ml));
    }
    if (part == kNaCluster - 1)
        for (int j = (n4 << 2) + threadIdx.x; j < vocab; j += kNaThreads) na_lse_merge(m, s, x[j], 1.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        na_lse_merge(m, s, m2, s2);
    }
    if ((threadIdx.x & 31) == 0) { red_m[threadIdx.x >> 5] = m; red_s[threadIdx.x >> 5] = s; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float mm = red_m[0], ss = red_s[0];
        for (int k = 1; k < kNaThreads / 32; ++k) na_lse_merge(mm, ss, red_m[k], red_s[k]);
        part_ms[0] = mm;
        part_ms[1] = ss;
    }
    cluster.sync();
    float mm = -CUDART_INF_F, ss = 0.f;
    for (int k = 0; k < kNaCluster; ++k) {
        const float* pk = cluster.map_shared_rank(part_ms, k);
        na_lse_merge(mm, ss, pk[0], pk[1]);
    }
    const float lse = mm + logf(ss);
    cluster.sync();

    const float S = scores ? scores[row] : 0.f;
    const uint32_t* mk = mask + (int64_t)row * mask_words;
    const float* xc = x + code_lo;
    uint32_t* out = keys + (int64_t)row * n_codes;
    const int c0 = (int)((int64_t)n_codes * part / kNaCluster);
    const int c1 = (int)((int64_t)n_codes * (part + 1) / kNaCluster);
    for (int c = c0 + threadIdx.x; c < c1; c += kNaThreads) {
        const bool valid = (mk[c >> 5] >> (c & 31)) & 1u;
        float key = __fadd_rn(S, __fsub_rn(xc[c], lse));
        uint32_t u = 0;
        if (valid && key == key) {  // a NaN key is not a candidate
            if (key == 0.f) key = 0.f;
            u = na_order_key(key);
        }
        out[c] = u;  // every entry is written on every call: nothing left from the last call is read
    }
}

__device__ __forceinline__ int na_block_incl_scan(int v, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
    }
    if (lane == 31) warp_tot[w] = v;
    __syncthreads();
    if (w == 0) {
        int tv = (lane < (kNaSelThreads >> 5)) ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, tv, off);
            if (lane >= off) tv += y;
        }
        warp_tot[lane] = tv;
    }
    __syncthreads();
    const int add = (w > 0) ? warp_tot[w - 1] : 0;
    total = warp_tot[(kNaSelThreads >> 5) - 1];
    __syncthreads();
    return v + add;
}

// one CTA: radix select of the k-th largest key, ties at the threshold in flat
// order, bitonic sort of the survivors
__global__ void __launch_bounds__(kNaSelThreads)
k_na_select(const uint32_t* __restrict__ keys, int N, int n_codes, int k_want, int32_t* __restrict__ out_parent,
            int32_t* __restrict__ out_code, float* __restrict__ out_key, int32_t* __restrict__ out_n) {
    __shared__ int hist[kNaHistBins];
    __shared__ int warp_tot[32];
    __shared__ int sh_digit, sh_kk, sh_count, sh_gt, sh_eqcnt;
    __shared__ unsigned long long sel[grb::kMaxBeam];
    const int tid = threadIdx.x;
    uint32_t prefix = 0, pmask = 0;
    int kk = k_want, n_valid = 0;
    const int shifts[3] = {20, 8, 0};
    const int widths[3] = {12, 12, 8};
    bool take_all = false;
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int i = tid; i < kNaHistBins; i += kNaSelThreads) hist[i] = 0;
        if (tid == 0) sh_count = 0;
        __syncthreads();
        int my_valid = 0;
        for (int base = 0; base < N; base += kNaSelThreads) {
            const int i = base + tid;
            const uint32_t u = (i < N) ? keys[i] : 0u;
            const bool q = (u != 0) && ((u & pmask) == prefix);
            my_valid += (u != 0);
            const uint32_t bin = q ? ((u >> sh) & dmask) : 0xFFFFFFFFu;
            const unsigned peers = __match_any_sync(0xffffffffu, bin);
            if (q && (__ffs(peers) - 1) == (tid & 31)) atomicAdd(&hist[bin], __popc(peers));
        }
        if (pass == 0) {
            atomicAdd(&sh_count, my_valid);
            __syncthreads();
            n_valid = sh_count;
            if (n_valid <= k_want) { take_all = true; break; }
        }
        __syncthreads();
        const int nbins = 1 << widths[pass];
        const int per = nbins / kNaSelThreads > 0 ? nbins / kNaSelThreads : 1;
        const int owner_active = (tid < nbins / per);
        const int hi = nbins - 1 - tid * per;
        int v = 0;
        if (owner_active)
            for (int e = 0; e < per; ++e) v += hist[hi - e];
        int total;
        const int incl = na_block_incl_scan(v, warp_tot, total);
        const int excl = incl - v;
        if (owner_active && excl < kk && kk <= incl) {
            int acc = excl;
            for (int e = 0; e < per; ++e) {
                const int h = hist[hi - e];
                if (acc + h >= kk) { sh_digit = hi - e; sh_kk = kk - acc; break; }
                acc += h;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sh_digit << sh;
        pmask |= dmask << sh;
        kk = sh_kk;
        if (pass == 2 && tid == 0) sh_eqcnt = hist[sh_digit];
        __syncthreads();
    }
    const uint32_t tau = take_all ? 0u : prefix;
    if (tid == 0) sh_gt = 0;
    __syncthreads();
    const bool eq_all = take_all || (sh_eqcnt == kk);
    const int n_take = take_all ? n_valid : k_want;
    for (int i = tid; i < N; i += kNaSelThreads) {
        const uint32_t u = keys[i];
        const bool pick = take_all ? (u != 0) : (u > tau || (eq_all && u == tau));
        if (pick) {
            const int pos = atomicAdd(&sh_gt, 1);
            sel[pos] = ((unsigned long long)u << 32) | (unsigned)(0xFFFFFFFFu - (uint32_t)i);
        }
    }
    __syncthreads();
    if (!eq_all) {
        int base_rank = 0;
        for (int start = 0; start < N; start += kNaSelThreads) {
            const int i = start + tid;
            const int e = (i < N && keys[i] == tau) ? 1 : 0;
            int total;
            const int incl = na_block_incl_scan(e, warp_tot, total);
            const int rank = base_rank + incl - e;
            if (e && rank < kk) {
                const int pos = atomicAdd(&sh_gt, 1);
                sel[pos] = ((unsigned long long)tau << 32) | (unsigned)(0xFFFFFFFFu - (uint32_t)i);
            }
            base_rank += total;
            if (base_rank >= kk) break;
        }
        __syncthreads();
    }
    int P = 1;
    while (P < n_take) P <<= 1;
    for (int i = n_take + tid; i < P; i += kNaSelThreads) sel[i] = 0ull;
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += kNaSelThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = sel[i], c = sel[ixj];
                    const bool desc = ((i & k) == 0);
                    if (desc ? (a < c) : (a > c)) { sel[i] = c; sel[ixj] = a; }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < n_take; i += kNaSelThreads) {
        const unsigned long long e = sel[i];
        const uint32_t flat = 0xFFFFFFFFu - (uint32_t)(e & 0xFFFFFFFFull);
        out_parent[i] = (int)(flat / (uint32_t)n_codes);
        out_code[i] = (int)(flat % (uint32_t)n_codes);
        out_key[i] = na_unorder_key((uint32_t)(e >> 32));
    }
    if (tid == 0) *out_n = n_take;
}

std::mutex g_na_mutex;
void* g_na_addr[kNaMaxDevices] = {};

// device address of g_noalloc_keys on the current device (looked up once per device)
gr_status noalloc_scratch(uint32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return grb::set_error(GR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kNaMaxDevices) return grb::set_error(GR_ERR_UNSUPPORTED, "device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_na_mutex);
    if (g_na_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_keys);
        if (e != cudaSuccess || p == nullptr)
            return grb::set_error(GR_ERR_CUDA, "cudaGetSymbolAddress(g_noalloc_keys): %s", cudaGetErrorString(e));
        g_na_addr[dev] = p;
    }
    *out = static_cast<uint32_t*>(g_na_addr[dev]);
    return GR_OK;
}

}  // namespace

extern "C" gr_status gr_constrained_topk_noalloc(const float* logits, int64_t ld, int n_rows, int vocab, int code_lo,
                                                 int n_codes, const float* beam_scores, const uint32_t* valid_mask,
                                                 int k, int32_t* out_parent, int32_t* out_code, float* out_key,
                                                 int32_t* out_n, gr_stream_t stream) {
    if (logits == nullptr || valid_mask == nullptr || out_parent == nullptr || out_code == nullptr ||
        out_key == nullptr || out_n == nullptr)
        return grb::set_error(GR_ERR_INVALID_ARG, "NULL input or output pointer");
    if (n_rows < 1 || vocab < 1 || n_codes < 1 || k < 1)
        return grb::set_error(GR_ERR_INVALID_ARG, "n_rows, vocab, n_codes and k must be >= 1");
    if (n_codes > grb::kMaxCodes) return grb::set_error(GR_ERR_CAPACITY, "n_codes above %d", grb::kMaxCodes);
    if (k > grb::kMaxBeam) return grb::set_error(GR_ERR_CAPACITY, "k above %d", grb::kMaxBeam);
    if ((int64_t)n_rows * n_codes > kNaMaxCandidates)
        return grb::set_error(GR_ERR_CAPACITY, "n_rows * n_codes = %lld above the fixed scratch of %d candidates",
                              (long long)n_rows * n_codes, kNaMaxCandidates);
    if (code_lo < 0 || (int64_t)code_lo + n_codes > vocab)
        return grb::set_error(GR_ERR_INVALID_ARG, "codes [code_lo, code_lo + n_codes) outside the vocabulary");
    if (ld < vocab || ld % 4 != 0 || (reinterpret_cast<uintptr_t>(logits) & 15) != 0)
        return grb::set_error(GR_ERR_INVALID_ARG, "logits must be 16-byte aligned with ld >= vocab, ld % 4 == 0");
    uint32_t* keys = nullptr;
    gr_status s = noalloc_scratch(&keys);
    if (s != GR_OK) return s;
    cudaStream_t cs = (cudaStream_t)stream;
    const int mask_words = (n_codes + 31) / 32;
    k_na_logsoftmax_gather<<<n_rows * kNaCluster, kNaThreads, 0, cs>>>(logits, ld, vocab, code_lo, n_codes,
                                                                       beam_scores, valid_mask, mask_words, keys);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        k_na_select<<<1, kNaSelThreads, 0, cs>>>(keys, n_rows * n_codes, n_codes, k, out_parent, out_code, out_key,
                                                 out_n);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return grb::set_error(GR_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return GR_OK;
}
