/*
 * grbeam.h -- C ABI of the GB300 wide-beam semantic-ID decode step.
 *
 * One decode step of semantic-ID generative recommendation with a split KV
 * layout, as described in the zhiding.cn article on NVIDIA recsys-examples,
 * section "语义ID生成式推荐专用推理框架" (semantic-ID GR inference framework):
 *   - ContextKV: the long request context, stored once per request and shared
 *     by all of its beams;
 *   - BeamKV:    the short history of tokens each beam decoded itself;
 *   - BeamPath:  the beams' ancestry, so no beam is stored as an independent
 *                long sequence;
 *   - dynamic beam width and item-constrained top-K.
 * Beam search returns every surviving beam, not only the best ("Advancing
 * Generative Recommendation Inference: our collaboration with NVIDIA on
 * TensorRT LLM", section "Background: what inference a recommendation request
 * needs").
 *
 * Each request r decodes its own step t_r = 0 .. L_r-1 (L_r = the semantic-ID
 * length of its catalogue, at most gr_config.n_levels).  One batch step is, in
 * call order:
 *   for every layer: the caller writes the K/V of the token each request with
 *            t_r >= 1 chose at level t_r-1 into its BeamKV slot
 *            (gr_beam_kv_slot_request / gr_beam_kv_slot), then calls
 *            gr_decode_attn();
 *   gr_constrained_topk() on the step's logit rows (for a request at t_r = 0:
 *            its prefill logits, one live row);
 *   gr_beam_advance(), which moves every request that is still decoding to
 *            t_r + 1.
 * Requests therefore need not be in step: requests of different lengths share
 * a batch, and a finished request's slot can take a new request
 * (gr_beam_admit) while the others keep decoding (GR-native continuous
 * batching, same article and section).  When t_r reaches L_r,
 * gr_beam_results() returns all beams of request r.
 *
 * The step state lives on the device (every kernel reads t_r there and
 * gr_beam_advance moves it), so a whole captured step replays as a CUDA graph
 * without the host (direct-pool-view CUDA-graph replay, same section): see
 * gr_beam_set_graph_mode.
 *
 * Conventions
 *   - Memory: the caller allocates and owns every device buffer (ContextKV
 *     pool, BeamKV pool, workspace, trie buffer, inputs, outputs).  The library
 *     never allocates device memory; a handle owns host metadata only.
 *   - Streams: gr_stream_t is a cudaStream_t (NULL = legacy default stream).
 *     Every call that takes a stream only enqueues work on it, except
 *     gr_beam_results / gr_beam_path / gr_beam_status, which synchronise it.
 *   - Rows: request r owns the contiguous rows [row_off[r], row_off[r] + W_r)
 *     of every per-row tensor (queries, attention output, logits, BeamKV
 *     slots); W_r is the request's maximum beam width.  Row b of request r is
 *     beam slot b.  Rows of beams that are not live at this step are ignored
 *     on input and written as zeros (attention) or left untouched (top-K).
 *   - Errors: argument, state and capacity errors are returned synchronously
 *     and leave the handle unchanged.  Errors that only the device can see
 *     (a NaN key, a timed-out wait) set a status word that gr_beam_status(),
 *     gr_beam_results() and gr_beam_path() report as GR_ERR_DEVICE /
 *     GR_ERR_TIMEOUT.  gr_last_error() gives a message for the calling thread.
 *     No C++ exception crosses this interface.
 *   - Threads: a handle may be used by one thread at a time.
 */
#ifndef GRBEAM_H_
#define GRBEAM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int gr_status;
#define GR_OK               0
#define GR_ERR_INVALID_ARG (-1)  /* bad pointer, size, alignment or value      */
#define GR_ERR_UNSUPPORTED (-2)  /* valid but not supported by this build      */
#define GR_ERR_CAPACITY    (-3)  /* buffer too small / size above a maximum    */
#define GR_ERR_STATE       (-4)  /* call out of order for the current step     */
#define GR_ERR_CUDA        (-5)  /* a CUDA runtime call failed                 */
#define GR_ERR_TIMEOUT     (-6)  /* a device-side wait gave up                 */
#define GR_ERR_DEVICE      (-7)  /* a kernel flagged invalid data (NaN key...) */

typedef void* gr_stream_t;          /* cudaStream_t */
typedef struct gr_trie gr_trie;     /* item catalogue on the device */
typedef struct gr_beam gr_beam;     /* one batch of requests being decoded */

/* Model geometry and code layout of a batch. */
typedef struct {
    int n_layers;          /* attention layers                                  */
    int n_q_heads;         /* Hq                                                */
    int n_kv_heads;        /* Hkv; Hq % Hkv == 0; query head q reads KV head q / (Hq/Hkv) */
    int head_dim;          /* D: 64 or 128                                      */
    int vocab;             /* V: length of a logit row                          */
    int code_base;         /* token id of (level 0, code 0)                     */
    int n_levels;          /* L: codes per item (1..8)                          */
    int codes_per_level;   /* C: codes per level (1..1024)                      */
    int64_t pool_tokens;   /* tokens per (layer, KV head) in the ContextKV pool */
} gr_config;
/* Level-t code c is vocabulary token code_base + t*C + c; the L*C code tokens
 * must lie inside [0, vocab). */

/* One request of the batch. */
typedef struct {
    int64_t ctx_offset;    /* first token of this request in the ContextKV pool */
    int ctx_len;           /* T_r >= 1; ctx_offset + T_r <= pool_tokens         */
    int beam_width;        /* W_r: maximum beams, 1..1024                       */
    const gr_trie* trie;   /* catalogue: C must match gr_config, its n_levels   */
                           /* (= L_r) may be 1..gr_config.n_levels              */
} gr_request;

/* Device buffers of a batch (all owned by the caller). */
typedef struct {
    const void* ctx_k;     /* bf16 [n_layers][n_kv_heads][pool_tokens][head_dim] */
    const void* ctx_v;     /* same layout as ctx_k                               */
    void* beam_k;          /* bf16 [n_layers][n_levels-1][rows][n_kv_heads][head_dim],
                              gr_beam_kv_bytes() bytes; NULL allowed when n_levels == 1 */
    void* beam_v;          /* same layout as beam_k                              */
    void* workspace;       /* gr_beam_workspace_bytes() bytes, 256-byte aligned  */
    size_t workspace_bytes;
} gr_buffers;

/* ------------------------------------------------------------------------ */
/* Item catalogue (item-constrained generation)                             */
/* ------------------------------------------------------------------------ */

/* Device bytes needed by gr_trie_create for these items.
 * codes: host int32 [n_items][n_levels], each in [0, codes_per_level). */
gr_status gr_trie_device_bytes(const int32_t* codes, int64_t n_items, int n_levels,
                               int codes_per_level, size_t* bytes);

/* Build the prefix trie of the items on the host and upload it into dev_buf
 * (caller-owned device memory of at least gr_trie_device_bytes(), 256-byte
 * aligned) with one asynchronous copy on `stream`; the host staging copy is
 * released once the copy completes (the call waits for it).
 * item_ids: host int64 [n_items] returned by gr_beam_results, or NULL for
 * 0..n_items-1.  Duplicate code tuples -> GR_ERR_INVALID_ARG.
 * Each inner node stores a bitmask of its valid child codes and the index of
 * its first child; a child is found by the rank of its code in the mask. */
gr_status gr_trie_create(const int32_t* codes, const int64_t* item_ids, int64_t n_items,
                         int n_levels, int codes_per_level, void* dev_buf, size_t dev_bytes,
                         gr_stream_t stream, gr_trie** out);
gr_status gr_trie_destroy(gr_trie* trie);   /* host object only; dev_buf stays the caller's */

/* ------------------------------------------------------------------------ */
/* Batch handle                                                              */
/* ------------------------------------------------------------------------ */

/* Workspace bytes for this batch (schedule, attention partials, candidate
 * keys, selection, BeamPath, results staging, status word). */
gr_status gr_beam_workspace_bytes(const gr_config* cfg, const gr_request* reqs, int n_requests,
                                  size_t* bytes);
/* Bytes of ONE BeamKV tensor (K or V) for this batch. */
gr_status gr_beam_kv_bytes(const gr_config* cfg, const gr_request* reqs, int n_requests,
                           size_t* bytes);

/* The attention schedule gr_beam_create builds for requests of these context
 * lengths (ctx_len[r] >= 1) and beam widths (beam_width[r] in 1..1024) on a
 * GPU with n_sm SMs, for the decode-attention kernel attn_kernel (0 the
 * automatic choice, which is the single-CTA kernel; 1 the single-CTA kernel;
 * 2 the CTA-pair kernel, head_dim 128 only; see gr_beam_set_attn_kernel).
 * Host only: no device, no trie, nothing allocated.  Only the head counts and
 * head_dim of cfg are read.  The decode attention kernel works through this
 * table, so it is the place to check its invariants without a GPU.
 *
 * A unit is up to 256 query rows (two 128-row tiles) of one (request, KV
 * head).  Its key tiles of 128 keys are cut into contiguous ranges, the jobs,
 * spread over CTAs in order.  A unit's jobs own the consecutive piece slots
 * [first slot, first slot + slots); the job of the first range merges.  For
 * the CTA-pair kernel (each pair of CTAs computes a whole 256-row unit, one
 * 128-row tile per CTA) the schedule is over n_sm / 2 pairs and "ctas" below
 * are pairs.
 *   units [max_units][7] int32: request, KV head, first beam, query tiles,
 *                               first slot, slots, key tiles
 *   jobs  [max_jobs][4]  int32: unit, first key tile, end key tile, slot
 *   ctas  [max_ctas][2]  int32: first job, end job of each CTA
 * *n_units, *n_jobs and *n_ctas are always written.  The arrays (caller-owned
 * host memory) are filled only when all three are large enough; otherwise
 * GR_ERR_CAPACITY is returned.  Errors: GR_ERR_INVALID_ARG (NULL pointer,
 * n_requests < 1, n_sm < 1, attn_kernel outside 0..2, bad lengths or widths),
 * GR_ERR_UNSUPPORTED (query heads per KV head not 1, 2, 4, 8 or 16; the pair
 * kernel with head_dim other than 128). */
gr_status gr_attn_schedule(const gr_config* cfg, const int* ctx_len, const int* beam_width,
                           int n_requests, int n_sm, int attn_kernel, int* n_units, int* n_jobs,
                           int* n_ctas, int32_t* units, int max_units, int32_t* jobs, int max_jobs,
                           int32_t* ctas, int max_ctas);

/* Validate the batch, carve the workspace, upload the request table, the
 * attention schedule and the TMA descriptors of the ContextKV pool, and put
 * every request at step 0 with one root beam of score 0 (enqueued on
 * `stream`).  The handle stays valid until gr_beam_destroy. */
gr_status gr_beam_create(const gr_config* cfg, const gr_request* reqs, int n_requests,
                         const gr_buffers* bufs, gr_stream_t stream, gr_beam** out);
gr_status gr_beam_destroy(gr_beam* beam);

/* rows_total = sum of W_r; row_offsets (optional, n_requests+1 ints) gets the
 * first row of each request and rows_total last. */
gr_status gr_beam_rows(const gr_beam* beam, int* rows_total, int* row_offsets);
/* Batch steps (gr_beam_advance calls) since create or the last rewind; for a
 * batch whose requests started together this is every request's t_r. */
gr_status gr_beam_step(const gr_beam* beam, int* step);
/* Step t_r of one request (t_r == L_r: finished) and its length L_r; either
 * output may be NULL.  After graph-mode replays call gr_beam_sync first. */
gr_status gr_beam_request_step(const gr_beam* beam, int request, int* step, int* n_levels);

/* Zero-copy view of BeamKV for the token chosen at level t-1, when every
 * request with a BeamKV level open is at the same step t >= 1 (GR_ERR_STATE
 * otherwise): bf16 [rows][n_kv_heads][head_dim] for `layer`.  The caller writes
 * each live beam's new K and V there (slot b = row b) before gr_decode_attn. */
gr_status gr_beam_kv_slot(gr_beam* beam, int layer, void** k_new, void** v_new);
/* The same view for one request at its own step t_r >= 1: bf16
 * [W_r][n_kv_heads][head_dim] (rows row_off[r] ..), level t_r-1 of `layer`. */
gr_status gr_beam_kv_slot_request(gr_beam* beam, int layer, int request, void** k_new, void** v_new);

/* ------------------------------------------------------------------------ */
/* Hot path                                                                  */
/* ------------------------------------------------------------------------ */

/* GQA decode attention, layer `layer`, of every live beam of every request at
 * a step 1 <= t_r < L_r: beam b of request r attends to its request's T_r
 * context tokens followed by the t_r BeamKV tokens on its path (levels
 * 0..t_r-1, slots from BeamPath), scale 1/sqrt(D).  This is the attention
 * backend that works directly on the ContextKV / BeamKV / BeamPath layout
 * (gr-decode_atten in the zhiding.cn recsys-examples article, section
 * "语义ID生成式推荐专用推理框架").
 *   q   bf16 [rows][n_q_heads][head_dim], 16-byte aligned
 *   out bf16 [rows][n_q_heads][head_dim]; rows of dead beams of those requests
 *       are written as zeros, rows of other requests (t_r == 0 or finished)
 *       are not written
 * The context part runs on the tensor cores (tcgen05, TMA-fed), the BeamKV
 * part from rows staged in shared memory by asynchronous copies, merged by a
 * log-sum-exp combine.  Each layer may be called once per step. */
gr_status gr_decode_attn(gr_beam* beam, int layer, const void* q, void* out, gr_stream_t stream);

/* Full-vocabulary log-softmax of every live row, then the item-constrained
 * top-K of each request across (beam, code) candidates of level t (the beam
 * scores come from the output logits: same article, section
 * "语义ID：解决稀疏性与长尾问题"; the item-constrained top-K and the dynamic
 * beam width: section "语义ID生成式推荐专用推理框架"):
 *   key(b, c) = S_b + (x[b][code_base + t*C + c] - LSE_b)   (float32, each
 *   operation rounded once), over codes c valid after beam b's prefix;
 *   order: key descending, then flat index b*C + c ascending;
 *   the first min(W_r, #candidates) survive (dynamic width).
 *   logits        fp32 [rows][ld], ld >= vocab, ld % 4 == 0, 16-byte aligned;
 *                 for t = 0 only row row_off[r] of each request is read
 *   logprobs_out  optional fp32 [rows][C]: x - LSE of the level's codes,
 *                 -inf for invalid codes (live rows only)
 *   lse_out       optional fp32 [rows]: LSE_b (live rows only)
 *   lse_in        optional fp32 [rows]: use these LSE_b instead of computing
 *                 them (for bit-exact comparison with a reference)
 * The selection is kept in the workspace until gr_beam_advance. */
gr_status gr_constrained_topk(gr_beam* beam, const float* logits, int64_t ld, float* logprobs_out,
                              float* lse_out, const float* lse_in, gr_stream_t stream);

/* Commit each decoding request's selection of its step t_r to BeamPath
 * (parent slot, token, trie node, score, ancestry) and set the live width of
 * step t_r+1; no KV is moved: beams are tracked through their ancestry
 * instead of being kept as independent long sequences (BeamPath, same
 * article, section "语义ID生成式推荐专用推理框架").  Every decoding request
 * moves to t_r+1. */
gr_status gr_beam_advance(gr_beam* beam, gr_stream_t stream);

/* Every request past step `step` goes back to it, so that it can be decoded
 * again from the BeamPath levels before it; step 0 starts again from the root
 * beam.  0 <= step <= gr_beam_step() (GR_ERR_STATE otherwise; not checked in
 * graph mode).  Enqueued on `stream` (one kernel and nothing else, so it can be
 * part of a captured graph). */
gr_status gr_beam_rewind(gr_beam* beam, int step, gr_stream_t stream);

/* GR-native continuous batching: slot `request` (finished, t_r == L_r, or not
 * started, t_r == 0) takes a new request between two batch steps.  Its
 * beam_width must fit the slot's rows (the slot's W_r at create); context
 * and catalogue are free.  The attention schedule is rebuilt on the host and
 * its tables (a few KB) are copied into the workspace on `stream`, after the
 * work already queued there; the new request starts at t_r = 0 with one root
 * beam.  GR_ERR_STATE in the middle of a step or in graph mode. */
gr_status gr_beam_admit(gr_beam* beam, int request, const gr_request* req, gr_stream_t stream);

/* Graph mode (enable != 0, between steps): gr_decode_attn, gr_constrained_topk,
 * gr_beam_advance and gr_beam_rewind only enqueue their kernels, taking every
 * decision from the device-resident step state, so the calls of a step can be
 * captured once (cudaStreamBeginCapture or a framework's graph capture) and
 * the graph replayed for later steps.  The host's copy of the step state is
 * not updated meanwhile: gr_beam_sync reloads it.  Timing events are off. */
gr_status gr_beam_set_graph_mode(gr_beam* beam, int enable);
/* Reload the host's copy of every request's step from the device (synchronises
 * `stream`) and report the device status word. */
gr_status gr_beam_sync(gr_beam* beam, gr_stream_t stream);

/* All surviving beams of request `request` once it finished (t_r == L_r),
 * best first (beam search returns every surviving beam, not only the best:
 * "Advancing Generative Recommendation Inference: our collaboration with
 * NVIDIA on TensorRT LLM", section "Background: what inference a
 * recommendation request needs"); synchronises `stream`.  A beam's parents
 * at every level are read with gr_beam_path.
 *   codes     int32 [W_r][L_r]        code of each level
 *   item_ids  int64 [W_r]             item of the code string
 *   scores    fp32  [W_r]             sum of the code log-probabilities
 *   n_out     number of beams written
 * Reports a device status error if a kernel flagged one. */
gr_status gr_beam_results(gr_beam* beam, int request, int32_t* codes, int64_t* item_ids,
                          float* scores, int* n_out, gr_stream_t stream);

/* BeamPath of one level (synchronises `stream`): for the n_out beams that
 * level t produced, parent slot at level t-1, token id, trie node id, score.
 * Any output pointer may be NULL. */
gr_status gr_beam_path(gr_beam* beam, int request, int level, int32_t* parents, int32_t* tokens,
                       int32_t* nodes, float* scores, int* n_out, gr_stream_t stream);

/* Synchronise `stream` and report the device status word (GR_OK,
 * GR_ERR_DEVICE or GR_ERR_TIMEOUT); clear_flag != 0 clears it afterwards. */
gr_status gr_beam_status(gr_beam* beam, int clear_flag, gr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Multi-item candidate scoring                                              */
/* ------------------------------------------------------------------------ */
/* "Advancing Generative Recommendation Inference: our collaboration with
 * NVIDIA on TensorRT LLM", sections "Background: what inference a
 * recommendation request needs" and "Scoring many candidates at once": the
 * user prefix and all candidates form one sequence in which each candidate
 * sees only the prefix and itself; the log-probabilities of label tokens
 * ("yes" / "no") read at each candidate's last token rank the candidates.
 * Here the prefix is the request's context in the ContextKV pool (read once
 * per request on the tensor cores, as in decode) and each candidate token's
 * other keys are its own candidate's tokens up to itself. */
typedef struct gr_score gr_score;

typedef struct {
    int n_layers, n_q_heads, n_kv_heads, head_dim, vocab;   /* as in gr_config */
    int64_t pool_tokens;       /* tokens per (layer, KV head) in the ContextKV pool */
    int n_labels;              /* 1..16 label tokens                              */
    const int32_t* label_ids;  /* host [n_labels], each in [0, vocab); label 0 ranks */
} gr_score_config;

typedef struct {
    int64_t ctx_offset;        /* the user prefix in the ContextKV pool           */
    int ctx_len;               /* >= 1                                            */
    int n_candidates;          /* 1..1024                                         */
    const int32_t* seg_lens;   /* host [n_candidates]: tokens of each candidate, 1..16 */
} gr_score_request;

typedef struct {
    const void* ctx_k;         /* as in gr_buffers                                */
    const void* ctx_v;
    void* seg_k;               /* bf16 [n_layers][rows][n_kv_heads][head_dim]: K of every
                                  candidate token (row order below); the caller writes it */
    void* seg_v;               /* same layout                                     */
    void* workspace;           /* gr_score_workspace_bytes() bytes, 256-byte aligned */
    size_t workspace_bytes;
} gr_score_buffers;

/* Rows: the candidate tokens of request 0 (candidate 0's tokens first, in order),
 * then request 1's, ...; q, out, seg_k and seg_v use this row order.  Candidates
 * are numbered globally in the same order. */
gr_status gr_score_workspace_bytes(const gr_score_config* cfg, const gr_score_request* reqs, int n_requests,
                                   size_t* bytes);
gr_status gr_score_create(const gr_score_config* cfg, const gr_score_request* reqs, int n_requests,
                          const gr_score_buffers* bufs, gr_stream_t stream, gr_score** out);
gr_status gr_score_destroy(gr_score* score);
/* rows_total = all candidate tokens; row_offsets / cand_offsets (optional,
 * n_requests+1 ints): first row / first candidate of each request, then the totals. */
gr_status gr_score_rows(const gr_score* score, int* rows_total, int* row_offsets, int* cand_offsets);
/* Masked attention of every candidate token at `layer`: each row attends to its
 * request's prefix and to its own candidate's tokens up to itself.
 *   q, out  bf16 [rows][n_q_heads][head_dim], 16-byte aligned */
gr_status gr_score_attn(gr_score* score, int layer, const void* q, void* out, gr_stream_t stream);
/* Label log-probabilities and the ranking:
 *   logits    fp32 [n_candidates_total][ld]: row c = the logits at candidate c's
 *             last token; ld >= vocab, ld % 4 == 0, 16-byte aligned
 *   logprobs  fp32 [n_candidates_total][n_labels]: x[label] - LSE over the vocabulary
 *   ranking   int32 [n_candidates_total] (optional): per request, its candidates'
 *             indices within the request by label 0's log-probability, highest first,
 *             ties by index */
gr_status gr_score_labels(gr_score* score, const float* logits, int64_t ld, float* logprobs, int32_t* ranking,
                          gr_stream_t stream);
/* Synchronise `stream` and report the device status word (a NaN log-probability
 * or a timed-out wait); clear_flag != 0 clears it. */
gr_status gr_score_status(gr_score* score, int clear_flag, gr_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Measurement                                                               */
/* ------------------------------------------------------------------------ */

/* Kernel kinds, for gr_beam_kernel_stats. */
#define GR_KERNEL_ATTN        0  /* decode attention: shared context on the tensor cores,
                                    BeamKV part and log-sum-exp combine in its epilogue */
#define GR_KERNEL_LOGSOFTMAX  1  /* full-vocab log-softmax + level gather + mask    */
#define GR_KERNEL_TOPK        2  /* cross-beam top-K selection per request          */
#define GR_KERNEL_ADVANCE     3  /* BeamPath advance                                */
#define GR_KERNEL_RESULTS     4  /* result gather                                    */
#define GR_KERNEL_INIT        5  /* state initialisation                             */
#define GR_KERNEL_KINDS       6

/* enable != 0: bracket every kernel launch with CUDA events on its stream
 * (host-side event objects; no device memory). */
gr_status gr_beam_set_timing(gr_beam* beam, int enable);
/* Launch count of a kernel kind since the last reset and, if timing was on,
 * the summed device time in milliseconds (synchronises the timed events).
 * reset != 0 clears the counters after reading. */
gr_status gr_beam_kernel_stats(gr_beam* beam, int kind, int64_t* launches, double* total_ms, int reset);

/* Test hook: limit (in nanoseconds) of every pipeline wait inside the
 * attention kernel (a thread waiting for data, for a tensor-core result or
 * for another warp); 0 restores the default of 2 s.  A wait that exceeds it
 * makes the kernel stop: it sets GR_ERR_TIMEOUT in the status word, drains
 * the copies and tensor-core operations it already issued (with a fixed
 * limit that this hook does not change), frees its tensor memory and
 * returns; the CUDA context stays usable.  A negative value makes every
 * pipeline wait give up on its first check, for fault-path tests. */
gr_status gr_beam_set_wait_limit(gr_beam* beam, int64_t nanoseconds);

/* Test hook: which decode-attention kernel the batch runs (between steps, not
 * in graph mode): 0 the automatic choice (the single-CTA kernel), 1 the
 * single-CTA kernel (two 128-row query tiles per CTA sharing whole K/V
 * tiles), 2 the CTA-pair kernel (cta_group::2 MMAs, each CTA holding half of
 * every K/V tile; head_dim 128 only, GR_ERR_UNSUPPORTED otherwise).  Both
 * compute the same attention.  The schedule is rebuilt and its tables copied
 * into the workspace on `stream`. */
gr_status gr_beam_set_attn_kernel(gr_beam* beam, int mode, gr_stream_t stream);
/* *pair = 1 when the batch runs the CTA-pair kernel, 0 for the single-CTA one. */
gr_status gr_beam_attn_kernel(const gr_beam* beam, int* pair);

/* ------------------------------------------------------------------------ */
/* Constrained top-K without caller-provided scratch                         */
/* ------------------------------------------------------------------------ */

/* The pages have no counterpart to this entry point; it serves callers that
 * cannot allocate device memory -- plugins of an inference server that are
 * handed only their input and output tensors, or services whose device
 * memory is budgeted once at start-up and must not grow per request.  They
 * cannot create a gr_beam handle, whose workspace the caller allocates.
 *
 * It computes, for ONE request, what gr_constrained_topk computes: the
 * full-vocabulary log-sum-exp LSE_b of each row, key(b, c) = S_b +
 * (x[b][code_lo + c] - LSE_b) (float32, each operation rounded once) over the
 * codes c whose bit is set in the row's mask, ordered by key descending then
 * flat index b*n_codes + c ascending; the first min(k, #candidates) are
 * written.  NaN keys are not candidates.  Identical inputs give the same
 * selection and keys as gr_constrained_topk.
 *   logits       device fp32 [n_rows][ld], ld >= vocab, ld % 4 == 0, 16-byte aligned
 *   beam_scores  device fp32 [n_rows] (S_b), or NULL for all zero
 *   valid_mask   device uint32 [n_rows][ceil(n_codes/32)]: bit c of row b set
 *                when code c may follow beam b's prefix
 *   out_parent, out_code  device int32 [k]; out_key device fp32 [k];
 *   out_n        device int32 [1]: number written
 * Limits: n_rows * n_codes <= GR_NOALLOC_MAX_CANDIDATES, n_codes <= 1024,
 * k <= 1024; larger sizes return GR_ERR_CAPACITY and launch nothing.
 * Scratch: the candidate keys and three words of bounds on them (their
 * key range and the smallest of the rows' largest keys) live in one
 * fixed device array of the library (GR_NOALLOC_MAX_CANDIDATES x 4 bytes =
 * 1 MiB, plus 256 bytes) that every GPU which loads the library holds until
 * the process exits.  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.  The bound words must start at
 * zero: they do when the library is loaded, and every call's last kernel
 * clears them again.  Every call on a device shares that one array and
 * overwrites it, so calls that overlap on the GPU (concurrent streams, or
 * several host threads) race and must be serialised by the caller; calls
 * queued on one stream are fine.  Each call looks the array's device address
 * up (cudaGetSymbolAddress, with the current device).  Enqueues two kernels
 * on `stream` and returns without synchronising. */
#define GR_NOALLOC_MAX_CANDIDATES (256 * 1024)
gr_status gr_constrained_topk_noalloc(const float* logits, int64_t ld, int n_rows, int vocab, int code_lo,
                                      int n_codes, const float* beam_scores, const uint32_t* valid_mask, int k,
                                      int32_t* out_parent, int32_t* out_code, float* out_key, int32_t* out_n,
                                      gr_stream_t stream);

const char* gr_status_str(gr_status status);
const char* gr_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* GRBEAM_H_ */
