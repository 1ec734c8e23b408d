// Item-constrained top-K of one request without caller-provided scratch.
//
// gr_constrained_topk needs the workspace that the caller allocates for a
// gr_beam handle.  Some callers cannot allocate device memory: plugins of an
// inference server that are handed only their input and output tensors, or
// services whose device memory is budgeted once at start-up and must not
// grow per request.  gr_constrained_topk_noalloc serves them: the caller
// passes only inputs and outputs, and the candidate keys that pass from the
// first kernel to the second live in one fixed array of this library,
// g_noalloc_scratch, which every GPU that loads the library keeps until the
// process exits (the second kernel exchanges everything else through the
// shared memory of its cluster).
//
// What it computes is the selection of gr_constrained_topk for one request:
// key(b, c) = S_b + (x[b][code_lo + c] - LSE_b) over the codes c whose bit is
// set in the row's mask, ordered by key descending then flat index b*C + c
// ascending, the first min(k, #candidates) kept.  Both entry points run the
// same device code (topk_dev.cuh: the clustered log-sum-exp of each row, the
// key encoding, the per-beam stage 1 and the cross-beam merge), so they
// return identical selections and keys for identical inputs.
#include <cuda_runtime.h>
#include <stdint.h>

#include "grbeam_internal.h"
#include "topk_dev.cuh"

namespace grb {
gr_status set_error(gr_status code, const char* fmt, ...);  // api.cu
}

namespace {

using namespace grb;
namespace cg = cooperative_groups;

constexpr int kNaMaxCandidates = GR_NOALLOC_MAX_CANDIDATES;
constexpr size_t kNaKeysBytes = 4ull * kNaMaxCandidates;  // ordered candidate keys [n_rows][n_codes]

// Scratch of the no-alloc path: the candidate keys, then three bound words of them (~lower,
// upper, ~smallest row maximum) that the first kernel raises and the second reads and clears
// (zero at load).
// Host code must not use this name as an address (it is a host-side stand-in);
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNaKeysBytes + 256];

// one kLogitCluster-CTA cluster per row: row log-sum-exp, then the masked keys of the codes (stage 1
// keeps each row's own top `keep`)
__global__ void __cluster_dims__(kLogitCluster, 1, 1) __launch_bounds__(topk::kLsThreads, 8)
k_na_logsoftmax_gather(const float* __restrict__ logits, int64_t ld, int vocab, int code_lo, int n_codes,
                       const float* __restrict__ scores, const uint32_t* __restrict__ mask, int mask_words, int keep,
                       uint8_t* __restrict__ scratch) {
    cg::cluster_group cluster = cg::this_cluster();
    const int row = blockIdx.x / kLogitCluster;
    const int part = (int)cluster.block_rank();
    __shared__ float red_m[topk::kLsThreads / 32], red_s[topk::kLsThreads / 32];
    __shared__ float part_ms[2];
    __shared__ uint32_t row_keys[kMaxCodes];
    const float* x = logits + (int64_t)row * ld;
    const float lse = topk::cluster_row_lse(x, vocab, cluster, part, red_m, red_s, part_ms);
    const float S = scores ? scores[row] : 0.f;
    const uint32_t* mk = mask + (int64_t)row * mask_words;
    const float* xc = x + code_lo;
    // a NaN key is not a candidate (there is no status word here)
    topk::gather_row(xc, mk, S, lse, n_codes, keep, part, row_keys,
                     reinterpret_cast<uint32_t*>(scratch) + (int64_t)row * n_codes,
                     reinterpret_cast<uint32_t*>(scratch + kNaKeysBytes), [](int, bool, float) {});
}

constexpr size_t kNaMergeSmem = sizeof(topk::MergeSmem) + 4ull * topk::kMergeStage;

// one cluster: the cross-beam merge of the request's keys
__global__ void __cluster_dims__(topk::kMergeCTAs, 1, 1) __launch_bounds__(topk::kMergeThreads)
k_na_merge(int n_rows, int n_codes, int k, uint8_t* __restrict__ scratch, int32_t* __restrict__ out_parent,
           int32_t* __restrict__ out_code, float* __restrict__ out_key, int32_t* __restrict__ out_n) {
    extern __shared__ __align__(16) uint8_t na_smem_raw[];
    topk::MergeSmem& sm = *reinterpret_cast<topk::MergeSmem*>(na_smem_raw);
    uint32_t* stage = reinterpret_cast<uint32_t*>(na_smem_raw + sizeof(topk::MergeSmem));
    const topk::MergeOut out{out_parent, out_code, out_key, out_n};
    topk::merge_select(reinterpret_cast<const uint32_t*>(scratch), n_rows * n_codes, n_codes, k,
                       reinterpret_cast<uint32_t*>(scratch + kNaKeysBytes), out, stage, sm);
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
    // The array's device address on the current device and context, looked up on every call
    // (a host-side lookup; it does not synchronise), so that it is never stale.
    void* scratch = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || scratch == nullptr)
        return grb::set_error(GR_ERR_CUDA, "cudaGetSymbolAddress(g_noalloc_scratch): %s", cudaGetErrorString(e));
    e = cudaFuncSetAttribute(k_na_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNaMergeSmem);
    if (e != cudaSuccess) return grb::set_error(GR_ERR_CUDA, "merge kernel set-up: %s", cudaGetErrorString(e));
    cudaStream_t cs = (cudaStream_t)stream;
    uint8_t* sp = static_cast<uint8_t*>(scratch);
    // launch status of these two kernels only (an earlier, unrelated pending error is left alone)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_rows * kLogitCluster);
    cfg.blockDim = dim3(topk::kLsThreads);
    cfg.stream = cs;
    const int mask_words = (n_codes + 31) / 32;
    e = cudaLaunchKernelEx(&cfg, k_na_logsoftmax_gather, logits, ld, vocab, code_lo, n_codes, beam_scores, valid_mask,
                           mask_words, k, sp);
    if (e == cudaSuccess) {
        cfg.gridDim = dim3(topk::kMergeCTAs);
        cfg.blockDim = dim3(topk::kMergeThreads);
        cfg.dynamicSmemBytes = kNaMergeSmem;
        e = cudaLaunchKernelEx(&cfg, k_na_merge, n_rows, n_codes, k, sp, out_parent, out_code, out_key, out_n);
    }
    if (e != cudaSuccess) return grb::set_error(GR_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return GR_OK;
}
