// Internal layout shared by the host library and the kernels of libgrbeam.
//
// Everything here lives in the caller's workspace (device memory) and is
// described by GrState, which every kernel receives by value.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/grbeam.h"

namespace grb {

constexpr int kMaxBeam = 1024;        // W_r upper bound (one CTA of the selection kernel)
constexpr int kMaxCodes = 1024;       // C upper bound
constexpr int kMaxLevels = 8;         // L upper bound
constexpr int kMaxSegment = 16;       // tokens of one scored candidate (multi-item scoring)
constexpr int kMaxPriv = 16;          // private keys of one query row (BeamKV path or own segment)
constexpr int kTileRows = 128;        // query rows per tensor-core tile (TMEM lanes)
constexpr int kTileKeys = 128;        // context keys per tile
constexpr int kUnitRows = 256;        // query rows per attention unit (two tiles)
constexpr int kLogitCluster = 2;      // CTAs sharing one logit row
constexpr int kTmapsPerReq = 3;       // ContextKV tensor maps of a request: K, V, K in half tiles of 64 keys

// status word bits (device)
constexpr int kStatusNanKey = 1;      // a candidate key was NaN
constexpr int kStatusTimeout = 2;     // a pipeline wait gave up
constexpr int kStatusBadNode = 4;     // trie walk left the valid node range

// Per-request record (device copy).
struct GrReqDev {
    int row_off;        // first row of the request
    int width;          // W_r
    int ctx_len;        // T_r
    int n_levels;       // L_r (<= cfg.n_levels; the levels of the request's trie)
    int unit_off;       // first attention unit of the request
    int n_ub;           // units per KV head: ceil(W_r * G / kUnitRows)
    int mask_words;     // 32-bit words per trie node mask
    int pad0;
    int64_t ctx_off;    // first token in the ContextKV pool
    int64_t leaf_base;  // node id of the first leaf
    int64_t n_nodes;    // inner nodes
    const uint32_t* mask;      // [n_inner][mask_words]
    const int32_t* child_base; // [n_inner]
    const int64_t* leaf_item;  // [n_items]
};

// A unit: up to two 128-row query tiles of one (request, KV head).
struct GrAttnUnit {
    int req;
    int head;           // KV head
    int beam0;          // first beam of the unit
    int nqt;            // query tiles (1 or 2)
    int first_slot;     // jobs of the unit are slots [first_slot, first_slot + n_slots)
    int n_slots;
    int n_tiles;        // ceil(T_r / kTileKeys)
    // the request's fixed fields, so that a job needs no request lookup
    int row_off;        // first row of the request
    int width;          // W_r
    int ctx_len;        // T_r
    int n_levels;       // L_r
    int pad;
};

// One piece of attention work: key tiles [t0, t1) of one unit.  It carries a copy of its
// unit, so that starting a job takes one table read.
struct GrAttnJob {
    int unit;
    int t0, t1;
    int slot;           // partial-result slot (== job index)
    GrAttnUnit u;
};

struct GrState {
    GrReqDev* req;
    int n_req;
    int rows;           // sum of W_r
    int n_levels;       // L
    int C;              // codes per level
    int code_base;
    int vocab;
    int n_layers, n_q_heads, n_kv_heads, head_dim;
    int64_t pool_tokens;

    int32_t* row_req;   // [rows] request of each row
    int32_t* req_step;  // [n_req] t_r: the level each request decodes next (t_r == L_r: finished);
                        // kernels read it, k_advance moves it, so steps replay without the host
    int32_t* n_beams;   // [n_req][L+1] live beams entering step t
    int32_t* parent;    // [L][rows] BeamPath: parent slot at level t-1
    int32_t* token;     // [L][rows]
    int32_t* node;      // [L][rows] trie node after consuming the level's code
    float* score;       // [L][rows]
    int32_t* path;      // [L][rows][L] slots on the path, levels 0..t
    uint32_t* cand;     // [rows][C] ordered candidate keys (0 = not a candidate)
    int32_t* sel_parent;// [rows] selection of the current step (request-relative rank)
    int32_t* sel_code;  // [rows]
    float* sel_key;     // [rows]
    int32_t* n_sel;     // [n_req]
    int32_t* status;    // [4]
    uint32_t* key_range;// [n_req][4] (~lower, upper, ~smallest row maximum, unused) of the step's candidate keys (top-K)

    // attention
    CUtensorMap* tmaps; // [n_req][kTmapsPerReq] (K, V, K half tiles) of the ContextKV pool
    GrAttnJob* jobs;    // [n_jobs]
    int2* cta_jobs;     // [n_cta] job range of each CTA
    GrAttnUnit* units;  // [n_units]
    int n_units, n_jobs, n_cta;  // n_cta: CTAs, or CTA pairs when attn_pair
    int attn_pair;      // the decode attention runs on CTA pairs (k_pair_attn)
    int attn_one;       // every unit has one query tile: the single-CTA kernel double-buffers S
    int n_sm;           // SMs of the device (the top-K merge sizes its clusters by it)
    float* o_part;      // [n_jobs][D][kUnitRows] pieces of split units (later key ranges), column-major
    float* lse_part;    // [n_jobs][kUnitRows]
    uint32_t* piece_flag; // [n_jobs][kUnitRows] 1 = piece row published and not yet merged
    const uint16_t* beam_k; // bf16 [NL][L-1][rows][Hkv][D]; scoring: the candidates' own tokens [NL][rows][Hkv][D]
    const uint16_t* beam_v;
    // multi-item scoring: row -> first row of its candidate, and its position in the candidate
    const int32_t* seg_first;
    const int32_t* seg_pos;

    // results staging
    int32_t* res_codes; // [rows][L]
    int64_t* res_items; // [rows]
    float* res_scores;  // [rows]
};

// ---- launchers (k_topk.cu) ----
cudaError_t launch_init_state(const GrState& st, cudaStream_t s);
cudaError_t launch_init_request(const GrState& st, int r, cudaStream_t s);
cudaError_t launch_set_step(const GrState& st, int step, cudaStream_t s);
cudaError_t launch_logsoftmax_gather(const GrState& st, const float* logits, int64_t ld,
                                     float* logprobs_out, float* lse_out, const float* lse_in,
                                     cudaStream_t s);
cudaError_t launch_topk_select(const GrState& st, cudaStream_t s);
cudaError_t launch_advance(const GrState& st, cudaStream_t s);
cudaError_t launch_results(const GrState& st, cudaStream_t s);
constexpr int kMaxCandidates = 1024;  // candidates of one scored request (one CTA ranks them)
cudaError_t launch_label_logprobs(const float* logits, int64_t ld, int vocab, const int32_t* labels, int n_labels,
                                  int n_rows, float* out, int32_t* status, cudaStream_t s);
cudaError_t launch_rank(const float* lp, int n_labels, const int32_t* cand_off, int n_req, int32_t* rank_out,
                        int32_t* status, cudaStream_t s);

// ---- launchers (k_attn.cu) ----
cudaError_t ctx_attn_smem_bytes(int head_dim, size_t* bytes);
cudaError_t launch_ctx_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                            int64_t wait_limit_ns, cudaStream_t s);
// ---- launchers (k_attn_pair.cu) ----
cudaError_t pair_attn_smem_bytes(size_t* bytes);
cudaError_t launch_pair_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                             int64_t wait_limit_ns, cudaStream_t s);
cudaError_t launch_score_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                              int64_t wait_limit_ns, cudaStream_t s);

}  // namespace grb
