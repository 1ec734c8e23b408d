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
//   k_logsoftmax_gather  one pass over each live logit row (a cluster of 2 CTAs
//                        per row): log-sum-exp of the full vocabulary, then the
//                        level's C code logits -> masked float32 keys
//                        key = S_b + (x - LSE_b), stored as order-preserving
//                        uint32 (0 = not a candidate); stage 1 of the top-K
//                        (each beam keeps its own top min(W, C) keys).
//                        HBM-bound.
//   k_topk_merge         stage 2, one cluster of 8 CTAs per request: radix
//                        select of the W-th largest key over the n_live*C
//                        candidates, ties at the threshold in flat-index order,
//                        each survivor written at its rank (key desc, flat asc).
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
#include "topk_dev.cuh"

namespace cg = cooperative_groups;

namespace grb {
namespace {

using topk::order_key;
using topk::unorder_key;

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
// K3: fused full-vocabulary log-softmax + level gather + trie mask + top-K stage 1
// ---------------------------------------------------------------------------
constexpr int kLsThreads = topk::kLsThreads;

__global__ void __cluster_dims__(kLogitCluster, 1, 1) __launch_bounds__(kLsThreads, 8)
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
    __shared__ uint32_t row_keys[kMaxCodes];

    const float* x = logits + (int64_t)row * ld;
    const int V = st.vocab;
    float lse;
    if (lse_in == nullptr) {
        lse = topk::cluster_row_lse(x, V, cluster, part, red_m, red_s, part_ms);
    } else {
        lse = lse_in[row];
    }
    if (part == 0 && threadIdx.x == 0 && lse_out != nullptr) lse_out[row] = lse;

    // level gather of the C codes (stage 1 of the top-K included), a part of the row per CTA
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
    const bool nan = topk::gather_row(xc, mk, S, lse, C, R.width, part, row_keys, st.cand + (int64_t)row * C,
                                      st.key_range + 4 * r, [&](int c, bool valid, float lp) {
                                          if (logprobs_out != nullptr)
                                              logprobs_out[(int64_t)row * C + c] = valid ? lp : -CUDART_INF_F;
                                      });
    if (nan) atomicOr(st.status, kStatusNanKey);
}

// ---------------------------------------------------------------------------
// K4: stage 2 of the top-K, the cross-beam merge of one request per cluster
// ---------------------------------------------------------------------------
constexpr size_t kMergeSmemBytes = sizeof(topk::MergeSmem) + 4ull * topk::kMergeStage;

template <int kC>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(topk::kMergeThreads)
k_topk_merge(GrState st) {
    extern __shared__ __align__(16) uint8_t merge_smem_raw[];
    topk::MergeSmem& sm = *reinterpret_cast<topk::MergeSmem*>(merge_smem_raw);
    uint32_t* stage = reinterpret_cast<uint32_t*>(merge_smem_raw + sizeof(topk::MergeSmem));
    const int r = blockIdx.x / kC;
    const GrReqDev& R = st.req[r];
    const int t = st.req_step[r];
    if (t >= R.n_levels) return;  // uniform over the cluster
    const int C = st.C;
    const int n_live = st.n_beams[r * (st.n_levels + 1) + t];
    const topk::MergeOut out{st.sel_parent + R.row_off, st.sel_code + R.row_off, st.sel_key + R.row_off,
                             st.n_sel + r};
    topk::merge_select<kC>(st.cand + (int64_t)R.row_off * C, n_live * C, C, R.width, st.key_range + 4 * r, out,
                           stage, sm);
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
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 4 * st.n_req; i += gridDim.x * blockDim.x)
        st.key_range[i] = 0u;
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
__global__ void __cluster_dims__(kLogitCluster, 1, 1) __launch_bounds__(kLsThreads, 8)
k_label_logprobs(const float* __restrict__ logits, int64_t ld, int vocab, const int32_t* __restrict__ labels,
                 int n_labels, float* __restrict__ out, int32_t* __restrict__ status) {
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kLogitCluster;
    const int part = (int)cluster.block_rank();
    __shared__ float red_m[kLsThreads / 32], red_s[kLsThreads / 32];
    __shared__ float part_ms[2];
    const float* x = logits + (int64_t)row * ld;
    const float lse = topk::cluster_row_lse(x, vocab, cluster, part, red_m, red_s, part_ms);
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

// Launch status of this launch only (cudaLaunchKernelEx's return value): a pending error of
// unrelated earlier work stays with the caller.  A kernel compiled with cluster dimensions keeps
// them.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

cudaError_t launch_label_logprobs(const float* logits, int64_t ld, int vocab, const int32_t* labels, int n_labels,
                                  int n_rows, float* out, int32_t* status, cudaStream_t s) {
    return launch(k_label_logprobs, dim3(n_rows * kLogitCluster), dim3(kLsThreads), 0, s, logits, ld, vocab, labels,
                  n_labels, out, status);
}

cudaError_t launch_rank(const float* lp, int n_labels, const int32_t* cand_off, int n_req, int32_t* rank_out,
                        int32_t* status, cudaStream_t s) {
    return launch(k_rank, dim3(n_req), dim3(kRankThreads), 0, s, lp, n_labels, cand_off, rank_out, status);
}

cudaError_t launch_init_state(const GrState& st, cudaStream_t s) {
    return launch(k_init_state, dim3(1), dim3(256), 0, s, st);
}

cudaError_t launch_init_request(const GrState& st, int r, cudaStream_t s) {
    return launch(k_init_request, dim3(1), dim3(32), 0, s, st, r);
}

cudaError_t launch_set_step(const GrState& st, int step, cudaStream_t s) {
    return launch(k_set_step, dim3(1), dim3(256), 0, s, st, step);
}

cudaError_t launch_logsoftmax_gather(const GrState& st, const float* logits, int64_t ld,
                                     float* logprobs_out, float* lse_out, const float* lse_in,
                                     cudaStream_t s) {
    return launch(k_logsoftmax_gather, dim3(st.rows * kLogitCluster), dim3(kLsThreads), 0, s, st, logits, ld,
                  logprobs_out, lse_out, lse_in);
}

// Clusters of 8 CTAs per request while every request's cluster fits the GPU at once (two merge
// CTAs per SM by shared memory), else of 4: with 64 requests (512 CTAs of 8-clusters, two
// waves) the 4-clusters measured 12.6 against 17.5 us.
template <int kC>
cudaError_t launch_merge(const GrState& st, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_topk_merge<kC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kMergeSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    return launch(k_topk_merge<kC>, dim3(st.n_req * kC), dim3(topk::kMergeThreads), kMergeSmemBytes, s, st);
}

cudaError_t launch_topk_select(const GrState& st, cudaStream_t s) {
    return st.n_req * topk::kMergeCTAs <= 2 * st.n_sm ? launch_merge<topk::kMergeCTAs>(st, s) : launch_merge<4>(st, s);
}

cudaError_t launch_advance(const GrState& st, cudaStream_t s) {
    return launch(k_advance, dim3(st.n_req), dim3(kMaxBeam), 0, s, st);
}

cudaError_t launch_results(const GrState& st, cudaStream_t s) {
    return launch(k_results, dim3(st.n_req), dim3(kMaxBeam), 0, s, st);
}

}  // namespace grb
