// Host side of libgrbeam: the C ABI declared in include/grbeam.h.
//
// The split KV layout (ContextKV shared per request, BeamKV per beam, BeamPath
// ancestry), dynamic beam width and item-constrained top-K follow the zhiding.cn
// recsys-examples article, section "语义ID生成式推荐专用推理框架"; returning
// every beam follows "Advancing Generative Recommendation Inference: our
// collaboration with NVIDIA on TensorRT LLM", section "Background: what
// inference a recommendation request needs".  Beam search lives entirely on
// the device: no call between create and results synchronises the host
// (vLLM's out-of-engine, CPU-scheduled beam search is what the same page,
// section "Why beam search could not saturate the GPU in vLLM", names as the
// bottleneck).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <new>
#include <string>
#include <vector>

#include "grbeam_internal.h"

using namespace grb;

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
namespace {
thread_local std::string g_last_error;

gr_status fail(gr_status code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

gr_status cuda_fail(cudaError_t e, const char* what) {
    return fail(GR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define GR_CUDA(call, what)                            \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 3-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds
gr_status make_tmap_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                       uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    EncodeTiledFn fn = encode_tiled();
    if (fn == nullptr) return fail(GR_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GR_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GR_OK;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}
}  // namespace

namespace grb {
// error reporting for entry points defined in other translation units
gr_status set_error(gr_status code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}
}  // namespace grb

// ---------------------------------------------------------------------------
// trie
// ---------------------------------------------------------------------------
struct gr_trie {
    int n_levels = 0, C = 0, mask_words = 0;
    int64_t n_items = 0, n_inner = 0, leaf_base = 0;
    const uint32_t* mask = nullptr;
    const int32_t* child_base = nullptr;
    const int64_t* leaf_item = nullptr;
};

namespace {
struct TrieLayout {
    int64_t n_inner = 0, n_items = 0;
    int mask_words = 0;
    size_t off_mask = 0, off_child = 0, off_leaf = 0, total = 0;
};

gr_status check_items(const int32_t* codes, int64_t n_items, int n_levels, int C) {
    if (codes == nullptr && n_items > 0) return fail(GR_ERR_INVALID_ARG, "codes is NULL");
    if (n_items < 1) return fail(GR_ERR_INVALID_ARG, "n_items must be >= 1");
    if (n_levels < 1 || n_levels > kMaxLevels) return fail(GR_ERR_UNSUPPORTED, "n_levels must be in 1..%d", kMaxLevels);
    if (C < 1 || C > kMaxCodes) return fail(GR_ERR_UNSUPPORTED, "codes_per_level must be in 1..%d", kMaxCodes);
    for (int64_t i = 0; i < n_items * n_levels; ++i)
        if (codes[i] < 0 || codes[i] >= C)
            return fail(GR_ERR_INVALID_ARG, "code %d of item %lld out of range", codes[i], (long long)(i / n_levels));
    return GR_OK;
}

// sort item indices lexicographically by code tuple; count prefix nodes
gr_status trie_order(const int32_t* codes, int64_t n, int L, std::vector<int64_t>& order,
                     std::vector<int64_t>& level_nodes) {
    order.resize(n);
    for (int64_t i = 0; i < n; ++i) order[i] = i;
    std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
        return std::lexicographical_compare(codes + a * L, codes + a * L + L, codes + b * L, codes + b * L + L);
    });
    for (int64_t i = 1; i < n; ++i)
        if (std::equal(codes + order[i] * L, codes + order[i] * L + L, codes + order[i - 1] * L))
            return fail(GR_ERR_INVALID_ARG, "duplicate item (items %lld and %lld have the same codes)",
                        (long long)order[i - 1], (long long)order[i]);
    // nodes at depth d (d = 0 root .. L leaves): distinct prefixes of length d
    level_nodes.assign(L + 1, 0);
    level_nodes[0] = 1;
    for (int d = 1; d <= L; ++d) {
        int64_t cnt = 0;
        for (int64_t i = 0; i < n; ++i)
            if (i == 0 || !std::equal(codes + order[i] * L, codes + order[i] * L + d, codes + order[i - 1] * L))
                ++cnt;
        level_nodes[d] = cnt;
    }
    return GR_OK;
}

TrieLayout trie_layout(const std::vector<int64_t>& level_nodes, int L, int C) {
    TrieLayout t;
    t.mask_words = (C + 31) / 32;
    for (int d = 0; d < L; ++d) t.n_inner += level_nodes[d];
    t.n_items = level_nodes[L];
    t.off_mask = 0;
    t.off_child = align_up(t.off_mask + (size_t)t.n_inner * t.mask_words * 4, 256);
    t.off_leaf = align_up(t.off_child + (size_t)t.n_inner * 4, 256);
    t.total = align_up(t.off_leaf + (size_t)t.n_items * 8, 256);
    return t;
}
}  // namespace

extern "C" gr_status gr_trie_device_bytes(const int32_t* codes, int64_t n_items, int n_levels, int codes_per_level,
                                          size_t* bytes) {
    if (bytes == nullptr) return fail(GR_ERR_INVALID_ARG, "bytes is NULL");
    gr_status s = check_items(codes, n_items, n_levels, codes_per_level);
    if (s != GR_OK) return s;
    std::vector<int64_t> order, level_nodes;
    try {
        if ((s = trie_order(codes, n_items, n_levels, order, level_nodes)) != GR_OK) return s;
    } catch (const std::bad_alloc&) {
        return fail(GR_ERR_CAPACITY, "host allocation failed");
    }
    *bytes = trie_layout(level_nodes, n_levels, codes_per_level).total;
    return GR_OK;
}

extern "C" gr_status gr_trie_create(const int32_t* codes, const int64_t* item_ids, int64_t n_items, int n_levels,
                                    int codes_per_level, void* dev_buf, size_t dev_bytes, gr_stream_t stream,
                                    gr_trie** out) {
    if (out == nullptr) return fail(GR_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    gr_status s = check_items(codes, n_items, n_levels, codes_per_level);
    if (s != GR_OK) return s;
    if (dev_buf == nullptr || (reinterpret_cast<uintptr_t>(dev_buf) & 255) != 0)
        return fail(GR_ERR_INVALID_ARG, "dev_buf must be non-NULL and 256-byte aligned");
    const int L = n_levels, C = codes_per_level;
    try {
        std::vector<int64_t> order, level_nodes;
        if ((s = trie_order(codes, n_items, L, order, level_nodes)) != GR_OK) return s;
        const TrieLayout lay = trie_layout(level_nodes, L, C);
        if (dev_bytes < lay.total)
            return fail(GR_ERR_CAPACITY, "trie needs %zu device bytes, got %zu", lay.total, dev_bytes);
        std::vector<uint8_t> host(lay.total, 0);
        uint32_t* mask = reinterpret_cast<uint32_t*>(host.data() + lay.off_mask);
        int32_t* child = reinterpret_cast<int32_t*>(host.data() + lay.off_child);
        int64_t* leaf = reinterpret_cast<int64_t*>(host.data() + lay.off_leaf);
        // node ids: depth 0 (root) first, then depth 1, ..., leaves last
        std::vector<int64_t> level_base(L + 1, 0);
        for (int d = 1; d <= L; ++d) level_base[d] = level_base[d - 1] + level_nodes[d - 1];
        if (level_base[L] + level_nodes[L] > INT32_MAX) return fail(GR_ERR_CAPACITY, "too many trie nodes");
        // walk the sorted items once per depth: node id of each item's prefix.
        // Children of one parent are contiguous in sorted order, numbered in
        // code order, so child(node, c) = child_base[node] + rank of c in mask.
        std::vector<int64_t> cur(n_items, 0), next(n_items, 0);
        for (int d = 0; d < L; ++d) {
            int64_t child_id = level_base[d + 1] - 1;
            int64_t last_parent = -1;
            for (int64_t k = 0; k < n_items; ++k) {
                const int32_t* it = codes + order[k] * L;
                const bool new_child = (k == 0) || !std::equal(it, it + d + 1, codes + order[k - 1] * L);
                if (new_child) {
                    ++child_id;
                    const int64_t parent = cur[k];
                    if (parent != last_parent) {
                        child[parent] = (int32_t)child_id;
                        last_parent = parent;
                    }
                    mask[(size_t)parent * lay.mask_words + (it[d] >> 5)] |= 1u << (it[d] & 31);
                }
                next[k] = child_id;
            }
            std::swap(cur, next);
        }
        for (int64_t k = 0; k < n_items; ++k)
            leaf[cur[k] - level_base[L]] = item_ids ? item_ids[order[k]] : order[k];
        GR_CUDA(cudaMemcpyAsync(dev_buf, host.data(), lay.total, cudaMemcpyHostToDevice, (cudaStream_t)stream),
                "trie upload");
        GR_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "trie upload sync");
        gr_trie* t = new gr_trie;
        t->n_levels = L;
        t->C = C;
        t->mask_words = lay.mask_words;
        t->n_items = n_items;
        t->n_inner = lay.n_inner;
        t->leaf_base = level_base[L];
        uint8_t* db = static_cast<uint8_t*>(dev_buf);
        t->mask = reinterpret_cast<const uint32_t*>(db + lay.off_mask);
        t->child_base = reinterpret_cast<const int32_t*>(db + lay.off_child);
        t->leaf_item = reinterpret_cast<const int64_t*>(db + lay.off_leaf);
        *out = t;
    } catch (const std::bad_alloc&) {
        return fail(GR_ERR_CAPACITY, "host allocation failed");
    }
    return GR_OK;
}

extern "C" gr_status gr_trie_destroy(gr_trie* trie) {
    delete trie;
    return GR_OK;
}

// ---------------------------------------------------------------------------
// batch handle
// ---------------------------------------------------------------------------
namespace {
struct Schedule {
    std::vector<GrAttnUnit> units;
    std::vector<GrAttnJob> jobs;
    std::vector<int2> cta_jobs;
};

struct Caps {
    size_t units = 0, jobs = 0, ctas = 0;
};

struct WsLayout {
    size_t req, row_req, req_step, n_beams, parent, token, node, score, path, cand, sel_parent, sel_code, sel_key, n_sel,
        status, key_range, tmaps, jobs, cta_jobs, units, tables_end, o_part, lse_part, piece_flag, res_codes, res_items, res_scores,
        total;
};

gr_status check_config(const gr_config* c, const gr_request* reqs, int n) {
    if (c == nullptr || (reqs == nullptr && n > 0)) return fail(GR_ERR_INVALID_ARG, "NULL config or requests");
    if (n < 1) return fail(GR_ERR_INVALID_ARG, "n_requests must be >= 1");
    if (c->n_layers < 1) return fail(GR_ERR_INVALID_ARG, "n_layers must be >= 1");
    if (c->n_kv_heads < 1 || c->n_q_heads < c->n_kv_heads || c->n_q_heads % c->n_kv_heads != 0)
        return fail(GR_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
    const int G = c->n_q_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
        return fail(GR_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4, 8 or 16 (got %d)", G);
    if (c->head_dim != 64 && c->head_dim != 128) return fail(GR_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c->n_levels < 1 || c->n_levels > kMaxLevels)
        return fail(GR_ERR_UNSUPPORTED, "n_levels must be in 1..%d", kMaxLevels);
    if (c->codes_per_level < 1 || c->codes_per_level > kMaxCodes)
        return fail(GR_ERR_UNSUPPORTED, "codes_per_level must be in 1..%d", kMaxCodes);
    if (c->vocab < 1 || c->code_base < 0 ||
        (int64_t)c->code_base + (int64_t)c->n_levels * c->codes_per_level > c->vocab)
        return fail(GR_ERR_INVALID_ARG, "code tokens [code_base, code_base + L*C) must lie inside the vocabulary");
    if (c->pool_tokens < 1) return fail(GR_ERR_INVALID_ARG, "pool_tokens must be >= 1");
    for (int r = 0; r < n; ++r) {
        const gr_request& q = reqs[r];
        if (q.ctx_len < 1 || q.ctx_offset < 0 || q.ctx_offset + q.ctx_len > c->pool_tokens)
            return fail(GR_ERR_INVALID_ARG, "request %d: context [%lld, %lld) outside the pool", r,
                        (long long)q.ctx_offset, (long long)(q.ctx_offset + q.ctx_len));
        if (q.beam_width < 1 || q.beam_width > kMaxBeam)
            return fail(GR_ERR_CAPACITY, "request %d: beam_width must be in 1..%d", r, kMaxBeam);
        if (q.trie == nullptr) return fail(GR_ERR_INVALID_ARG, "request %d: trie is NULL", r);
        if (q.trie->n_levels < 1 || q.trie->n_levels > c->n_levels || q.trie->C != c->codes_per_level)
            return fail(GR_ERR_INVALID_ARG, "request %d: the trie needs 1..%d levels of %d codes", r, c->n_levels,
                        c->codes_per_level);
    }
    return GR_OK;
}

// Attention schedule: units of <= 256 query rows per (request, KV head);
// their key tiles are cut into ~equal contiguous ranges, one per CTA.
Schedule build_schedule(const gr_config* c, const gr_request* reqs, int n, int n_sm,
                        std::vector<int>& unit_off, std::vector<int>& n_ub, bool pair = false) {
    Schedule s;
    const int G = c->n_q_heads / c->n_kv_heads;
    const int bpu = kUnitRows / G;
    unit_off.resize(n);
    n_ub.resize(n);
    int64_t total = 0;
    for (int r = 0; r < n; ++r) {
        unit_off[r] = (int)s.units.size();
        n_ub[r] = (reqs[r].beam_width + bpu - 1) / bpu;
        const int tiles = (reqs[r].ctx_len + kTileKeys - 1) / kTileKeys;
        for (int h = 0; h < c->n_kv_heads; ++h)
            for (int ub = 0; ub < n_ub[r]; ++ub) {
                GrAttnUnit u{};
                u.req = r;
                u.head = h;
                u.beam0 = ub * bpu;
                const int rows = std::min(bpu, reqs[r].beam_width - u.beam0) * G;  // query rows of this unit
                u.nqt = (rows + kTileRows - 1) / kTileRows;
                u.n_tiles = tiles;
                s.units.push_back(u);
                total += (int64_t)tiles * u.nqt;
            }
    }
    int64_t tiles_all = 0;
    for (auto& u : s.units) tiles_all += u.n_tiles;
    // the pair kernel runs one unit on a CTA pair: its "CTAs" below are pairs
    const int n_cta = (int)std::min<int64_t>(std::max(pair ? n_sm / 2 : n_sm, 1), tiles_all);
    // Cost model of a CTA's time (measured on the attention kernel at ctx 5000, in units of
    // ~83 ns): a key tile costs 20 with two query tiles (they ping-pong) and 17 with one;
    // every job after a CTA's first costs kSwitch more (publish, the next job's Q, pipeline
    // refill); a unit's first key range, the merger, costs kMerge more (pieces, BeamKV keys,
    // output).  kMerge = 75 came from a sweep over the long, short, mixed and page1 workloads
    // (75 against 105: page1 -3 %, mixed -1 %, the others unchanged).  The makespan bound T is the smallest for which a greedy walk fits every
    // unit into n_cta CTAs: units and key tiles in order (so the units of a KV head stay on
    // neighbouring CTAs), a unit cut where a CTA's budget runs out.  A cut unit's first range
    // is then the last job of its CTA and its later ranges are the first jobs of the next
    // CTAs, which publish them before they wait for anything.
    // The pair kernel (cost in the same units): a key tile costs a pair 7 with one or two
    // query tiles (each CTA computes its 128 rows of an M = 256 MMA), a job switch 30, a
    // merge 100.
    // A schedule that cuts units runs past its bound by more than one that keeps them whole (the
    // mergers wait for their pieces and read them at the end of the launch): 48 more at long,
    // 82 more at short, measured on the single-CTA kernel.  Units are kept whole when the
    // smallest bound without cuts is within kSplit of the smallest with them: short then runs
    // 2 whole units per CTA (54.4 us against 59.5 with cuts), while long (bounds 791 / 875),
    // page1 and mixed keep their cuts.
    const int64_t kSwitch = pair ? 30 : 36, kMerge = pair ? 100 : 75, kSplit = pair ? 0 : 60;
    auto tile_cost = [pair](const GrAttnUnit& u) -> int64_t { return pair ? 7 : (u.nqt == 2 ? 20 : 17); };
    // returns the CTAs used (n_cta + 1: does not fit); with emit, writes jobs and ranges; with
    // cut == false a unit that does not fit the rest of a CTA's budget moves whole to the next
    bool cut = true;
    auto walk = [&](int64_t T, bool emit) -> int {
        int cta = 0, njobs = 0, job_begin = 0;
        int64_t load = 0;
        if (emit) s.jobs.clear();
        auto next_cta = [&]() {
            if (emit && cta < n_cta) s.cta_jobs[cta] = make_int2(job_begin, (int)s.jobs.size());
            job_begin = (int)s.jobs.size();
            ++cta;
            load = 0;
            njobs = 0;
        };
        for (int ui = 0; ui < (int)s.units.size(); ++ui) {
            GrAttnUnit& u = s.units[ui];
            if (emit) u.first_slot = (int)s.jobs.size();
            const int64_t tc = tile_cost(u);
            int t0 = 0;
            while (t0 < u.n_tiles) {
                if (cta >= n_cta) return n_cta + 1;
                const int64_t sw = njobs > 0 ? kSwitch : 0;
                const int64_t merge = t0 == 0 ? kMerge : 0;
                const int rem = u.n_tiles - t0;
                int take = rem;
                if (load + sw + merge + rem * tc > T) {
                    const int64_t fit = cut ? (T - load - sw - merge) / tc : 0;
                    if (fit < 1) {
                        if (njobs == 0) return n_cta + 1;  // not even one tile in an empty CTA
                        next_cta();
                        continue;
                    }
                    take = (int)std::min<int64_t>(fit, rem);
                }
                if (emit) s.jobs.push_back(GrAttnJob{ui, t0, t0 + take, (int)s.jobs.size()});
                load += sw + merge + take * tc;
                ++njobs;
                t0 += take;
                if (t0 < u.n_tiles) next_cta();  // the rest of the unit opens the next CTA
            }
            if (emit) u.n_slots = (int)s.jobs.size() - u.first_slot;
        }
        const int used = cta + (njobs > 0 ? 1 : 0);
        if (emit) {
            next_cta();
            for (int k = cta; k < n_cta; ++k) s.cta_jobs[k] = make_int2((int)s.jobs.size(), (int)s.jobs.size());
        }
        return used;
    };
    int64_t all = 0;
    for (auto& u : s.units) all += kMerge + kSwitch + u.n_tiles * tile_cost(u);
    auto smallest_bound = [&]() {
        int64_t lo = 1, hi = all;  // hi: one CTA takes everything, which always fits
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (walk(mid, false) <= n_cta) hi = mid;
            else lo = mid + 1;
        }
        return lo;
    };
    const int64_t t_cut = smallest_bound();
    cut = false;
    const int64_t t_whole = kSplit > 0 ? smallest_bound() : t_cut + 1;
    cut = !(t_whole <= t_cut + kSplit);
    s.cta_jobs.assign(n_cta, make_int2(0, 0));
    walk(cut ? t_cut : t_whole, true);
    (void)total;
    return s;
}

// Which decode-attention kernel a batch runs: mode 2 the CTA-pair kernel (head_dim 128),
// otherwise the single-CTA kernel.  The automatic choice (mode 0) is the single-CTA kernel:
// on the measured workloads (contexts 1000..5000, beams 30..256) it is the faster of the two.
bool choose_pair(const gr_config* c, int mode) { return c->head_dim == 128 && mode == 2; }

// Each unit gets its request's fixed fields, and each job a copy of its unit: starting a
// job on the device then takes one table read.
void finalize_jobs(Schedule& s, const GrReqDev* rq) {
    for (auto& u : s.units) {
        u.row_off = rq[u.req].row_off;
        u.width = rq[u.req].width;
        u.ctx_len = rq[u.req].ctx_len;
        u.n_levels = rq[u.req].n_levels;
    }
    for (auto& j : s.jobs) j.u = s.units[j.unit];
}

WsLayout ws_layout(const gr_config* c, int n, int rows, const Caps& k) {
    WsLayout w{};
    size_t o = 0;
    auto take = [&](size_t bytes, size_t align = 256) {
        o = align_up(o, align);
        size_t r = o;
        o += bytes;
        return r;
    };
    const int L = c->n_levels;
    // tables (uploaded at create and at every admission) come first
    w.req = take(sizeof(GrReqDev) * n);
    w.row_req = take(4ull * rows);
    w.tmaps = take(sizeof(CUtensorMap) * kTmapsPerReq * n, 128);
    w.jobs = take(sizeof(GrAttnJob) * k.jobs);
    w.cta_jobs = take(sizeof(int2) * k.ctas);
    w.units = take(sizeof(GrAttnUnit) * k.units);
    w.tables_end = align_up(o, 256);
    // device state
    w.req_step = take(4ull * n);
    w.n_beams = take(4ull * n * (L + 1));
    w.parent = take(4ull * L * rows);
    w.token = take(4ull * L * rows);
    w.node = take(4ull * L * rows);
    w.score = take(4ull * L * rows);
    w.path = take(4ull * L * rows * L);
    w.cand = take(4ull * rows * c->codes_per_level);
    w.sel_parent = take(4ull * rows);
    w.sel_code = take(4ull * rows);
    w.sel_key = take(4ull * rows);
    w.n_sel = take(4ull * n);
    w.status = take(16);
    w.key_range = take(16ull * n);
    w.o_part = take(4ull * k.jobs * kUnitRows * c->head_dim);
    w.lse_part = take(4ull * k.jobs * kUnitRows);
    w.piece_flag = take(4ull * k.jobs * kUnitRows);
    w.res_codes = take(4ull * rows * L);
    w.res_items = take(8ull * rows);
    w.res_scores = take(4ull * rows);
    w.total = align_up(o, 256);
    return w;
}

// Capacities of the schedule tables: admissions rebuild the schedule, and a request
// admitted into a slot never has more beams than the slot's rows, so the units never
// outnumber those at create; every cut of a unit adds one job, at most one per CTA.
Caps caps_of(const Schedule& s, int n_sm) {
    Caps k;
    k.units = s.units.size();
    k.ctas = (size_t)std::max(n_sm, 1);
    k.jobs = k.units + k.ctas;
    return k;
}

int rows_of(const gr_request* reqs, int n) {
    int rows = 0;
    for (int r = 0; r < n; ++r) rows += reqs[r].beam_width;
    return rows;
}
}  // namespace

struct gr_beam {
    gr_config cfg{};
    int n_req = 0, rows = 0;
    std::vector<int> row_off;     // [n_req + 1] rows of each request slot (fixed at create)
    std::vector<gr_request> reqs; // the request each slot holds now
    gr_buffers bufs{};
    GrState st{};
    Schedule sched;
    WsLayout w{};
    Caps caps{};
    std::vector<uint8_t> img;     // host image of the device tables
    int n_sm = 0;
    // host mirror of the device step state (call-order checks); graph mode leaves it alone
    int step = 0;                 // advances since create or the last rewind
    std::vector<int> req_step;    // t_r of each request
    std::vector<uint8_t> attn_done;
    bool topk_done = false;
    bool graph_mode = false;
    // measurement
    bool timing = false;
    int64_t launches[GR_KERNEL_KINDS] = {};
    struct Ev { cudaEvent_t a, b; };
    std::vector<Ev> events[GR_KERNEL_KINDS];
    std::vector<Ev> event_pool;
    int64_t wait_limit_ns = 2000000000ll;
    int attn_mode = 0;            // 0 automatic, 1 single-CTA kernel, 2 CTA-pair kernel

    int levels(int r) const { return reqs[r].trie->n_levels; }
    bool decoding(int r) const { return req_step[r] < levels(r); }
    bool attending(int r) const { return req_step[r] >= 1 && req_step[r] < levels(r); }

    ~gr_beam() {
        for (int k = 0; k < GR_KERNEL_KINDS; ++k)
            for (auto& e : events[k]) event_pool.push_back(e);
        for (auto& e : event_pool) {
            cudaEventDestroy(e.a);
            cudaEventDestroy(e.b);
        }
    }
};

namespace {
// wrap one launch: count it, bracket it with events when timing is on
template <typename F>
gr_status run_kernel(gr_beam* h, int kind, cudaStream_t s, F&& launch) {
    gr_beam::Ev ev{nullptr, nullptr};
    const bool timed = h->timing && !h->graph_mode;
    if (timed) {
        if (!h->event_pool.empty()) {
            ev = h->event_pool.back();
            h->event_pool.pop_back();
        } else {
            GR_CUDA(cudaEventCreate(&ev.a), "event create");
            GR_CUDA(cudaEventCreate(&ev.b), "event create");
        }
        GR_CUDA(cudaEventRecord(ev.a, s), "event record");
    }
    cudaError_t e = launch();
    if (e != cudaSuccess) {
        if (ev.a) h->event_pool.push_back(ev);
        return cuda_fail(e, "kernel launch");
    }
    ++h->launches[kind];
    if (timed) {
        GR_CUDA(cudaEventRecord(ev.b, s), "event record");
        h->events[kind].push_back(ev);
    }
    return GR_OK;
}

gr_status status_from_word(int w) {
    if (w & kStatusTimeout) return fail(GR_ERR_TIMEOUT, "a device-side wait timed out (status 0x%x)", w);
    if (w & (kStatusNanKey | kStatusBadNode)) return fail(GR_ERR_DEVICE, "a kernel flagged invalid data (status 0x%x)", w);
    return GR_OK;
}

// (Re)build the attention schedule for the requests the slots hold now and write the
// host image of every device table; the caller uploads it with one copy.
gr_status build_tables(gr_beam* h) {
    const gr_config* cfg = &h->cfg;
    std::vector<int> unit_off, n_ub;
    const bool pair = choose_pair(cfg, h->attn_mode);
    Schedule sc = build_schedule(cfg, h->reqs.data(), h->n_req, h->n_sm, unit_off, n_ub, pair);
    if (sc.units.size() > h->caps.units || sc.jobs.size() > h->caps.jobs || sc.cta_jobs.size() > h->caps.ctas)
        return fail(GR_ERR_CAPACITY, "attention schedule exceeds the workspace's tables");
    h->sched = std::move(sc);
    const WsLayout& w = h->w;
    h->img.assign(w.tables_end, 0);
    uint8_t* img = h->img.data();
    GrReqDev* rq = reinterpret_cast<GrReqDev*>(img + w.req);
    int32_t* rr = reinterpret_cast<int32_t*>(img + w.row_req);
    for (int r = 0; r < h->n_req; ++r) {
        const gr_request& q = h->reqs[r];
        const gr_trie* t = q.trie;
        GrReqDev d{};
        d.row_off = h->row_off[r];
        d.width = q.beam_width;
        d.ctx_len = q.ctx_len;
        d.n_levels = t->n_levels;
        d.unit_off = unit_off[r];
        d.n_ub = n_ub[r];
        d.mask_words = t->mask_words;
        d.ctx_off = q.ctx_offset;
        d.leaf_base = t->leaf_base;
        d.n_nodes = t->n_inner;
        d.mask = t->mask;
        d.child_base = t->child_base;
        d.leaf_item = t->leaf_item;
        rq[r] = d;
        for (int b = h->row_off[r]; b < h->row_off[r + 1]; ++b) rr[b] = r;
    }
    CUtensorMap* tm = reinterpret_cast<CUtensorMap*>(img + w.tmaps);
    const int D = cfg->head_dim;
    const uint64_t zdim = (uint64_t)cfg->n_layers * cfg->n_kv_heads;
    for (int r = 0; r < h->n_req; ++r) {
        const gr_request& q = h->reqs[r];
        const uint64_t off = (uint64_t)q.ctx_offset * D * 2;
        const uint64_t s1 = (uint64_t)D * 2, s2 = (uint64_t)cfg->pool_tokens * D * 2;
        gr_status s;
        CUtensorMap* m = tm + kTmapsPerReq * r;
        const uint8_t* kb = static_cast<const uint8_t*>(h->bufs.ctx_k) + off;
        if ((s = make_tmap_3d(&m[0], kb, D, q.ctx_len, zdim, s1, s2, 64, kTileKeys, 1)) != GR_OK ||
            (s = make_tmap_3d(&m[1], static_cast<const uint8_t*>(h->bufs.ctx_v) + off, D, q.ctx_len, zdim, s1, s2, 64,
                              kTileKeys, 1)) != GR_OK ||
            (s = make_tmap_3d(&m[2], kb, D, q.ctx_len, zdim, s1, s2, 64, kTileKeys / 2, 1)) != GR_OK)
            return s;
    }
    h->st.attn_pair = pair ? 1 : 0;
    // the single-CTA kernel double-buffers S when no unit has a second query tile
    bool one = !pair;
    for (const auto& u : h->sched.units) one = one && u.nqt == 1;
    h->st.attn_one = one ? 1 : 0;
    finalize_jobs(h->sched, rq);
    memcpy(img + w.jobs, h->sched.jobs.data(), sizeof(GrAttnJob) * h->sched.jobs.size());
    memcpy(img + w.cta_jobs, h->sched.cta_jobs.data(), sizeof(int2) * h->sched.cta_jobs.size());
    memcpy(img + w.units, h->sched.units.data(), sizeof(GrAttnUnit) * h->sched.units.size());
    h->st.n_units = (int)h->sched.units.size();
    h->st.n_jobs = (int)h->sched.jobs.size();
    h->st.n_cta = (int)h->sched.cta_jobs.size();
    h->st.n_sm = h->n_sm;
    return GR_OK;
}
}  // namespace

extern "C" gr_status gr_beam_workspace_bytes(const gr_config* cfg, const gr_request* reqs, int n_requests,
                                             size_t* bytes) {
    if (bytes == nullptr) return fail(GR_ERR_INVALID_ARG, "bytes is NULL");
    gr_status s = check_config(cfg, reqs, n_requests);
    if (s != GR_OK) return s;
    int n_sm = device_sm_count();
    if (n_sm <= 0) n_sm = 148;
    std::vector<int> uo, nu;
    Schedule sc = build_schedule(cfg, reqs, n_requests, n_sm, uo, nu);
    *bytes = ws_layout(cfg, n_requests, rows_of(reqs, n_requests), caps_of(sc, n_sm)).total;
    return GR_OK;
}

extern "C" gr_status gr_attn_schedule(const gr_config* cfg, const int* ctx_len, const int* beam_width,
                                      int n_requests, int n_sm, int attn_kernel, int* n_units, int* n_jobs, int* n_ctas,
                                      int32_t* units, int max_units, int32_t* jobs, int max_jobs, int32_t* ctas,
                                      int max_ctas) {
    if (cfg == nullptr || ctx_len == nullptr || beam_width == nullptr || n_units == nullptr || n_jobs == nullptr ||
        n_ctas == nullptr)
        return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (n_requests < 1 || n_sm < 1) return fail(GR_ERR_INVALID_ARG, "n_requests and n_sm must be >= 1");
    if (attn_kernel < 0 || attn_kernel > 2) return fail(GR_ERR_INVALID_ARG, "attn_kernel must be 0, 1 or 2");
    if (attn_kernel == 2 && cfg->head_dim != 128)
        return fail(GR_ERR_UNSUPPORTED, "the CTA-pair kernel needs head_dim 128 (got %d)", cfg->head_dim);
    if (cfg->n_kv_heads < 1 || cfg->n_q_heads < cfg->n_kv_heads || cfg->n_q_heads % cfg->n_kv_heads != 0)
        return fail(GR_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
    const int G = cfg->n_q_heads / cfg->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
        return fail(GR_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4, 8 or 16 (got %d)", G);
    std::vector<gr_request> reqs(n_requests);
    for (int r = 0; r < n_requests; ++r) {
        if (ctx_len[r] < 1 || beam_width[r] < 1 || beam_width[r] > kMaxBeam)
            return fail(GR_ERR_INVALID_ARG, "request %d: ctx_len >= 1 and beam_width in 1..%d", r, kMaxBeam);
        reqs[r] = gr_request{};
        reqs[r].ctx_len = ctx_len[r];
        reqs[r].beam_width = beam_width[r];
    }
    std::vector<int> uo, nu;
    const Schedule sc = build_schedule(cfg, reqs.data(), n_requests, n_sm, uo, nu, choose_pair(cfg, attn_kernel));
    *n_units = (int)sc.units.size();
    *n_jobs = (int)sc.jobs.size();
    *n_ctas = (int)sc.cta_jobs.size();
    if (*n_units > max_units || *n_jobs > max_jobs || *n_ctas > max_ctas || units == nullptr || jobs == nullptr ||
        ctas == nullptr)
        return fail(GR_ERR_CAPACITY, "schedule needs %d units, %d jobs, %d CTAs", *n_units, *n_jobs, *n_ctas);
    for (int k = 0; k < *n_units; ++k) {
        const GrAttnUnit& u = sc.units[k];
        const int32_t v[7] = {u.req, u.head, u.beam0, u.nqt, u.first_slot, u.n_slots, u.n_tiles};
        for (int e = 0; e < 7; ++e) units[7 * k + e] = v[e];
    }
    for (int k = 0; k < *n_jobs; ++k) {
        const GrAttnJob& j = sc.jobs[k];
        jobs[4 * k + 0] = j.unit;
        jobs[4 * k + 1] = j.t0;
        jobs[4 * k + 2] = j.t1;
        jobs[4 * k + 3] = j.slot;
    }
    for (int k = 0; k < *n_ctas; ++k) {
        ctas[2 * k + 0] = sc.cta_jobs[k].x;
        ctas[2 * k + 1] = sc.cta_jobs[k].y;
    }
    return GR_OK;
}

extern "C" gr_status gr_beam_kv_bytes(const gr_config* cfg, const gr_request* reqs, int n_requests, size_t* bytes) {
    if (bytes == nullptr) return fail(GR_ERR_INVALID_ARG, "bytes is NULL");
    gr_status s = check_config(cfg, reqs, n_requests);
    if (s != GR_OK) return s;
    const int rows = rows_of(reqs, n_requests);
    *bytes = (size_t)cfg->n_layers * std::max(cfg->n_levels - 1, 0) * rows * cfg->n_kv_heads * cfg->head_dim * 2;
    return GR_OK;
}

extern "C" gr_status gr_beam_create(const gr_config* cfg, const gr_request* reqs, int n_requests,
                                    const gr_buffers* bufs, gr_stream_t stream, gr_beam** out) {
    if (out == nullptr || bufs == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL out or buffers");
    *out = nullptr;
    gr_status s = check_config(cfg, reqs, n_requests);
    if (s != GR_OK) return s;
    if (bufs->ctx_k == nullptr || bufs->ctx_v == nullptr || bufs->workspace == nullptr)
        return fail(GR_ERR_INVALID_ARG, "ctx_k, ctx_v and workspace must be device pointers");
    if (cfg->n_levels > 1 && (bufs->beam_k == nullptr || bufs->beam_v == nullptr))
        return fail(GR_ERR_INVALID_ARG, "beam_k / beam_v are required when n_levels > 1");
    if ((reinterpret_cast<uintptr_t>(bufs->workspace) & 255) != 0)
        return fail(GR_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if ((reinterpret_cast<uintptr_t>(bufs->ctx_k) & 15) != 0 || (reinterpret_cast<uintptr_t>(bufs->ctx_v) & 15) != 0)
        return fail(GR_ERR_INVALID_ARG, "ctx_k / ctx_v must be 16-byte aligned");
    const int n_sm = device_sm_count();
    if (n_sm <= 0) return fail(GR_ERR_CUDA, "no CUDA device");
    cudaStream_t cs = (cudaStream_t)stream;
    gr_beam* h = nullptr;
    try {
        h = new gr_beam;
        h->cfg = *cfg;
        h->n_req = n_requests;
        h->reqs.assign(reqs, reqs + n_requests);
        h->bufs = *bufs;
        h->n_sm = n_sm;
        h->rows = rows_of(reqs, n_requests);
        h->row_off.resize(n_requests + 1);
        h->row_off[0] = 0;
        for (int r = 0; r < n_requests; ++r) h->row_off[r + 1] = h->row_off[r] + reqs[r].beam_width;
        std::vector<int> unit_off, n_ub;
        h->caps = caps_of(build_schedule(cfg, reqs, n_requests, n_sm, unit_off, n_ub), n_sm);
        h->w = ws_layout(cfg, n_requests, h->rows, h->caps);
        const WsLayout& w = h->w;
        if (bufs->workspace_bytes < w.total) {
            gr_status e = fail(GR_ERR_CAPACITY, "workspace needs %zu bytes, got %zu", w.total, bufs->workspace_bytes);
            delete h;
            return e;
        }
        uint8_t* ws = static_cast<uint8_t*>(bufs->workspace);
        GrState& st = h->st;
        st.req = reinterpret_cast<GrReqDev*>(ws + w.req);
        st.n_req = n_requests;
        st.rows = h->rows;
        st.n_levels = cfg->n_levels;
        st.C = cfg->codes_per_level;
        st.code_base = cfg->code_base;
        st.vocab = cfg->vocab;
        st.n_layers = cfg->n_layers;
        st.n_q_heads = cfg->n_q_heads;
        st.n_kv_heads = cfg->n_kv_heads;
        st.head_dim = cfg->head_dim;
        st.pool_tokens = cfg->pool_tokens;
        st.row_req = reinterpret_cast<int32_t*>(ws + w.row_req);
        st.req_step = reinterpret_cast<int32_t*>(ws + w.req_step);
        st.n_beams = reinterpret_cast<int32_t*>(ws + w.n_beams);
        st.parent = reinterpret_cast<int32_t*>(ws + w.parent);
        st.token = reinterpret_cast<int32_t*>(ws + w.token);
        st.node = reinterpret_cast<int32_t*>(ws + w.node);
        st.score = reinterpret_cast<float*>(ws + w.score);
        st.path = reinterpret_cast<int32_t*>(ws + w.path);
        st.cand = reinterpret_cast<uint32_t*>(ws + w.cand);
        st.sel_parent = reinterpret_cast<int32_t*>(ws + w.sel_parent);
        st.sel_code = reinterpret_cast<int32_t*>(ws + w.sel_code);
        st.sel_key = reinterpret_cast<float*>(ws + w.sel_key);
        st.n_sel = reinterpret_cast<int32_t*>(ws + w.n_sel);
        st.status = reinterpret_cast<int32_t*>(ws + w.status);
        st.key_range = reinterpret_cast<uint32_t*>(ws + w.key_range);
        st.tmaps = reinterpret_cast<CUtensorMap*>(ws + w.tmaps);
        st.jobs = reinterpret_cast<GrAttnJob*>(ws + w.jobs);
        st.cta_jobs = reinterpret_cast<int2*>(ws + w.cta_jobs);
        st.units = reinterpret_cast<GrAttnUnit*>(ws + w.units);
        st.piece_flag = reinterpret_cast<uint32_t*>(ws + w.piece_flag);
        st.o_part = reinterpret_cast<float*>(ws + w.o_part);
        st.lse_part = reinterpret_cast<float*>(ws + w.lse_part);
        st.beam_k = static_cast<const uint16_t*>(bufs->beam_k);
        st.beam_v = static_cast<const uint16_t*>(bufs->beam_v);
        st.res_codes = reinterpret_cast<int32_t*>(ws + w.res_codes);
        st.res_items = reinterpret_cast<int64_t*>(ws + w.res_items);
        st.res_scores = reinterpret_cast<float*>(ws + w.res_scores);
        if ((s = build_tables(h)) != GR_OK) {
            delete h;
            return s;
        }
        cudaError_t e = cudaMemcpyAsync(ws, h->img.data(), h->img.size(), cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(st.piece_flag, 0, 4ull * h->caps.jobs * kUnitRows, cs);
        if (e == cudaSuccess) e = launch_init_state(st, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
        if (e != cudaSuccess) {
            delete h;
            return cuda_fail(e, "workspace upload");
        }
        h->launches[GR_KERNEL_INIT] += 1;
        h->req_step.assign(n_requests, 0);
        h->attn_done.assign(cfg->n_layers, 0);
    } catch (const std::bad_alloc&) {
        delete h;
        return fail(GR_ERR_CAPACITY, "host allocation failed");
    }
    *out = h;
    return GR_OK;
}

extern "C" gr_status gr_beam_destroy(gr_beam* beam) {
    delete beam;
    return GR_OK;
}

extern "C" gr_status gr_beam_rows(const gr_beam* h, int* rows_total, int* row_offsets) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (rows_total) *rows_total = h->rows;
    if (row_offsets)
        for (int r = 0; r <= h->n_req; ++r) row_offsets[r] = h->row_off[r];
    return GR_OK;
}

extern "C" gr_status gr_beam_step(const gr_beam* h, int* step) {
    if (h == nullptr || step == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    *step = h->step;
    return GR_OK;
}

extern "C" gr_status gr_beam_request_step(const gr_beam* h, int request, int* step, int* n_levels) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (request < 0 || request >= h->n_req) return fail(GR_ERR_INVALID_ARG, "request %d out of range", request);
    if (step) *step = h->req_step[request];
    if (n_levels) *n_levels = h->levels(request);
    return GR_OK;
}

namespace {
// BeamKV rows [row0, row0 + n) of `layer` at `level`
void kv_view(const gr_beam* h, int layer, int level, int row0, void** k, void** v) {
    const gr_config& c = h->cfg;
    const size_t off =
        ((((size_t)layer * (c.n_levels - 1) + level) * h->rows) + row0) * c.n_kv_heads * c.head_dim * 2;
    *k = static_cast<uint8_t*>(h->bufs.beam_k) + off;
    *v = static_cast<uint8_t*>(h->bufs.beam_v) + off;
}
}  // namespace

extern "C" gr_status gr_beam_kv_slot(gr_beam* h, int layer, void** k_new, void** v_new) {
    if (h == nullptr || k_new == nullptr || v_new == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(GR_ERR_INVALID_ARG, "layer %d out of range", layer);
    int t = -1;
    for (int r = 0; r < h->n_req; ++r) {
        if (!h->attending(r)) continue;
        if (t >= 0 && h->req_step[r] != t)
            return fail(GR_ERR_STATE, "requests decode different levels: use gr_beam_kv_slot_request");
        t = h->req_step[r];
    }
    if (t < 1) return fail(GR_ERR_STATE, "no request has a BeamKV level open");
    kv_view(h, layer, t - 1, 0, k_new, v_new);
    return GR_OK;
}

extern "C" gr_status gr_beam_kv_slot_request(gr_beam* h, int layer, int request, void** k_new, void** v_new) {
    if (h == nullptr || k_new == nullptr || v_new == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(GR_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (request < 0 || request >= h->n_req) return fail(GR_ERR_INVALID_ARG, "request %d out of range", request);
    if (!h->attending(request))
        return fail(GR_ERR_STATE, "request %d has no BeamKV level open (step %d of %d)", request, h->req_step[request],
                    h->levels(request));
    kv_view(h, layer, h->req_step[request] - 1, h->row_off[request], k_new, v_new);
    return GR_OK;
}

extern "C" gr_status gr_decode_attn(gr_beam* h, int layer, const void* q, void* out, gr_stream_t stream) {
    if (h == nullptr || q == nullptr || out == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(GR_ERR_INVALID_ARG, "layer %d out of range", layer);
    if ((reinterpret_cast<uintptr_t>(q) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0)
        return fail(GR_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    if (!h->graph_mode) {
        bool any = false;
        for (int r = 0; r < h->n_req; ++r) any = any || h->attending(r);
        if (!any) return fail(GR_ERR_STATE, "no request is at a decode step 1..L-1 (step %d)", h->step);
        if (h->topk_done) return fail(GR_ERR_STATE, "top-K of this step already ran; call gr_beam_advance");
        if (h->attn_done[layer]) return fail(GR_ERR_STATE, "layer %d already ran at step %d", layer, h->step);
    }
    const gr_config& c = h->cfg;
    const int G = c.n_q_heads / c.n_kv_heads;
    CUtensorMap qmap;  // 128 query rows per box: 128/G beams x G heads x 64 dimensions
    gr_status s = make_tmap_3d(&qmap, q, c.head_dim, c.n_q_heads, h->rows, (uint64_t)c.head_dim * 2,
                               (uint64_t)c.n_q_heads * c.head_dim * 2, 64, G, kTileRows / G);
    if (s != GR_OK) return s;
    cudaStream_t cs = (cudaStream_t)stream;
    const int64_t lim = h->wait_limit_ns;
    if ((s = run_kernel(h, GR_KERNEL_ATTN, cs, [&] {
             const uint16_t* qq = static_cast<const uint16_t*>(q);
             uint16_t* oo = static_cast<uint16_t*>(out);
             return h->st.attn_pair ? launch_pair_attn(h->st, qmap, layer, qq, oo, lim, cs)
                                    : launch_ctx_attn(h->st, qmap, layer, qq, oo, lim, cs);
         })) != GR_OK)
        return s;
    if (!h->graph_mode) h->attn_done[layer] = 1;
    return GR_OK;
}

extern "C" gr_status gr_constrained_topk(gr_beam* h, const float* logits, int64_t ld, float* logprobs_out,
                                         float* lse_out, const float* lse_in, gr_stream_t stream) {
    if (h == nullptr || logits == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (ld < h->cfg.vocab || ld % 4 != 0) return fail(GR_ERR_INVALID_ARG, "ld must be >= vocab and a multiple of 4");
    if ((reinterpret_cast<uintptr_t>(logits) & 15) != 0) return fail(GR_ERR_INVALID_ARG, "logits must be 16-byte aligned");
    if (!h->graph_mode) {
        bool any = false;
        for (int r = 0; r < h->n_req; ++r) any = any || h->decoding(r);
        if (!any) return fail(GR_ERR_STATE, "decoding is finished for every request");
        if (h->topk_done) return fail(GR_ERR_STATE, "top-K already ran at step %d; call gr_beam_advance", h->step);
    }
    cudaStream_t cs = (cudaStream_t)stream;
    gr_status s;
    if ((s = run_kernel(h, GR_KERNEL_LOGSOFTMAX, cs, [&] {
             return launch_logsoftmax_gather(h->st, logits, ld, logprobs_out, lse_out, lse_in, cs);
         })) != GR_OK)
        return s;
    if ((s = run_kernel(h, GR_KERNEL_TOPK, cs, [&] { return launch_topk_select(h->st, cs); })) != GR_OK) return s;
    if (!h->graph_mode) h->topk_done = true;
    return GR_OK;
}

extern "C" gr_status gr_beam_advance(gr_beam* h, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (!h->graph_mode && !h->topk_done)
        return fail(GR_ERR_STATE, "gr_constrained_topk has not run at step %d", h->step);
    cudaStream_t cs = (cudaStream_t)stream;
    gr_status s = run_kernel(h, GR_KERNEL_ADVANCE, cs, [&] { return launch_advance(h->st, cs); });
    if (s != GR_OK) return s;
    if (!h->graph_mode) {
        for (int r = 0; r < h->n_req; ++r)
            if (h->decoding(r)) ++h->req_step[r];
        h->step += 1;
        h->topk_done = false;
        std::fill(h->attn_done.begin(), h->attn_done.end(), 0);
    }
    return GR_OK;
}

extern "C" gr_status gr_beam_rewind(gr_beam* h, int step, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (step < 0) return fail(GR_ERR_INVALID_ARG, "step must be >= 0");
    if (!h->graph_mode && step > h->step)
        return fail(GR_ERR_STATE, "can rewind only to a decoded step 0..%d (asked %d)", h->step, step);
    cudaStream_t cs = (cudaStream_t)stream;
    gr_status s = run_kernel(h, GR_KERNEL_INIT, cs, [&] { return launch_set_step(h->st, step, cs); });
    if (s != GR_OK) return s;
    if (!h->graph_mode) {
        for (int r = 0; r < h->n_req; ++r) h->req_step[r] = std::min(h->req_step[r], step);
        h->step = std::min(h->step, step);
        h->topk_done = false;
        std::fill(h->attn_done.begin(), h->attn_done.end(), 0);
    }
    return GR_OK;
}

extern "C" gr_status gr_beam_admit(gr_beam* h, int request, const gr_request* req, gr_stream_t stream) {
    if (h == nullptr || req == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (h->graph_mode) return fail(GR_ERR_STATE, "admission needs the host step state: leave graph mode first");
    if (request < 0 || request >= h->n_req) return fail(GR_ERR_INVALID_ARG, "request %d out of range", request);
    if (h->topk_done || std::any_of(h->attn_done.begin(), h->attn_done.end(), [](uint8_t d) { return d != 0; }))
        return fail(GR_ERR_STATE, "admission happens between steps");
    if (h->req_step[request] != 0 && h->decoding(request))
        return fail(GR_ERR_STATE, "slot %d still decodes (step %d of %d)", request, h->req_step[request],
                    h->levels(request));
    const int slot_rows = h->row_off[request + 1] - h->row_off[request];
    if (req->beam_width < 1 || req->beam_width > slot_rows)
        return fail(GR_ERR_CAPACITY, "beam_width %d does not fit slot %d (%d rows)", req->beam_width, request, slot_rows);
    gr_status s = check_config(&h->cfg, req, 1);
    if (s != GR_OK) return s;
    const gr_request keep = h->reqs[request];
    h->reqs[request] = *req;
    if ((s = build_tables(h)) != GR_OK) {
        h->reqs[request] = keep;
        build_tables(h);
        return s;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    // the tables are small: one copy of the whole image, ordered after the work already
    // queued on the stream (which still reads the old tables)
    GR_CUDA(cudaMemcpyAsync(h->bufs.workspace, h->img.data(), h->img.size(), cudaMemcpyHostToDevice, cs), "admit");
    if ((s = run_kernel(h, GR_KERNEL_INIT, cs, [&] { return launch_init_request(h->st, request, cs); })) != GR_OK)
        return s;
    h->req_step[request] = 0;
    return GR_OK;
}

extern "C" gr_status gr_beam_set_graph_mode(gr_beam* h, int enable) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (enable && (h->topk_done || std::any_of(h->attn_done.begin(), h->attn_done.end(), [](uint8_t d) { return d; })))
        return fail(GR_ERR_STATE, "graph mode starts between steps");
    h->graph_mode = enable != 0;
    return GR_OK;
}

extern "C" gr_status gr_beam_set_attn_kernel(gr_beam* h, int mode, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (mode < 0 || mode > 2) return fail(GR_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
    if (mode == 2 && h->cfg.head_dim != 128) return fail(GR_ERR_UNSUPPORTED, "the CTA-pair kernel needs head_dim 128");
    if (h->graph_mode) return fail(GR_ERR_STATE, "the attention kernel changes outside graph mode");
    if (h->topk_done || std::any_of(h->attn_done.begin(), h->attn_done.end(), [](uint8_t d) { return d != 0; }))
        return fail(GR_ERR_STATE, "the attention kernel changes between steps");
    const int keep = h->attn_mode;
    h->attn_mode = mode;
    gr_status s = build_tables(h);
    if (s != GR_OK) {
        h->attn_mode = keep;
        build_tables(h);
        return s;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    GR_CUDA(cudaMemcpyAsync(h->bufs.workspace, h->img.data(), h->img.size(), cudaMemcpyHostToDevice, cs),
            "attention kernel tables");
    return GR_OK;
}

extern "C" gr_status gr_beam_attn_kernel(const gr_beam* h, int* pair) {
    if (h == nullptr || pair == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    *pair = h->st.attn_pair;
    return GR_OK;
}

extern "C" gr_status gr_beam_sync(gr_beam* h, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    cudaStream_t cs = (cudaStream_t)stream;
    std::vector<int32_t> t(h->n_req);
    int w = 0;
    GR_CUDA(cudaMemcpyAsync(t.data(), h->st.req_step, 4ull * h->n_req, cudaMemcpyDeviceToHost, cs), "sync");
    GR_CUDA(cudaMemcpyAsync(&w, h->st.status, 4, cudaMemcpyDeviceToHost, cs), "status read");
    GR_CUDA(cudaStreamSynchronize(cs), "sync");
    int steps = 0;
    for (int r = 0; r < h->n_req; ++r) {
        steps = std::max(steps, t[r] - h->req_step[r]);
        h->req_step[r] = t[r];
    }
    h->step += steps;
    h->topk_done = false;
    std::fill(h->attn_done.begin(), h->attn_done.end(), 0);
    return status_from_word(w);
}

extern "C" gr_status gr_beam_status(gr_beam* h, int clear_flag, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    cudaStream_t cs = (cudaStream_t)stream;
    int w = 0;
    GR_CUDA(cudaMemcpyAsync(&w, h->st.status, 4, cudaMemcpyDeviceToHost, cs), "status read");
    GR_CUDA(cudaStreamSynchronize(cs), "status sync");
    if (clear_flag && w != 0) {
        // a kernel that gave up may have left piece flags set: clear them with the status
        GR_CUDA(cudaMemsetAsync(h->st.status, 0, 16, cs), "status clear");
        GR_CUDA(cudaMemsetAsync(h->st.piece_flag, 0, 4ull * h->caps.jobs * kUnitRows, cs), "flag clear");
        GR_CUDA(cudaStreamSynchronize(cs), "status clear sync");
    }
    return status_from_word(w);
}

extern "C" gr_status gr_beam_results(gr_beam* h, int request, int32_t* codes, int64_t* item_ids, float* scores,
                                     int* n_out, gr_stream_t stream) {
    if (h == nullptr || n_out == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (request < 0 || request >= h->n_req) return fail(GR_ERR_INVALID_ARG, "request %d out of range", request);
    const int Lr = h->levels(request);
    if (h->req_step[request] < Lr)
        return fail(GR_ERR_STATE, "request %d is not finished (step %d of %d)", request, h->req_step[request], Lr);
    cudaStream_t cs = (cudaStream_t)stream;
    gr_status s = run_kernel(h, GR_KERNEL_RESULTS, cs, [&] { return launch_results(h->st, cs); });
    if (s != GR_OK) return s;
    const int L = h->cfg.n_levels;
    int n = 0, w = 0;
    GR_CUDA(cudaMemcpyAsync(&n, h->st.n_beams + request * (L + 1) + Lr, 4, cudaMemcpyDeviceToHost, cs), "results");
    GR_CUDA(cudaMemcpyAsync(&w, h->st.status, 4, cudaMemcpyDeviceToHost, cs), "status read");
    GR_CUDA(cudaStreamSynchronize(cs), "results sync");
    if ((s = status_from_word(w)) != GR_OK) return s;
    const int row0 = h->row_off[request];
    if (n > 0) {
        if (codes)  // rows of L_r codes, packed
            GR_CUDA(cudaMemcpy2DAsync(codes, 4ull * Lr, h->st.res_codes + (size_t)row0 * L, 4ull * L, 4ull * Lr, n,
                                      cudaMemcpyDeviceToHost, cs),
                    "results");
        if (item_ids)
            GR_CUDA(cudaMemcpyAsync(item_ids, h->st.res_items + row0, 8ull * n, cudaMemcpyDeviceToHost, cs), "results");
        if (scores)
            GR_CUDA(cudaMemcpyAsync(scores, h->st.res_scores + row0, 4ull * n, cudaMemcpyDeviceToHost, cs), "results");
        GR_CUDA(cudaStreamSynchronize(cs), "results sync");
    }
    *n_out = n;
    return GR_OK;
}

extern "C" gr_status gr_beam_path(gr_beam* h, int request, int level, int32_t* parents, int32_t* tokens,
                                  int32_t* nodes, float* scores, int* n_out, gr_stream_t stream) {
    if (h == nullptr || n_out == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (request < 0 || request >= h->n_req) return fail(GR_ERR_INVALID_ARG, "request %d out of range", request);
    if (level < 0 || level >= h->req_step[request])
        return fail(GR_ERR_STATE, "level %d of request %d is not committed (step %d)", level, request,
                    h->req_step[request]);
    cudaStream_t cs = (cudaStream_t)stream;
    const int L = h->cfg.n_levels;
    int n = 0, w = 0;
    GR_CUDA(cudaMemcpyAsync(&n, h->st.n_beams + request * (L + 1) + level + 1, 4, cudaMemcpyDeviceToHost, cs), "path");
    GR_CUDA(cudaMemcpyAsync(&w, h->st.status, 4, cudaMemcpyDeviceToHost, cs), "status read");
    GR_CUDA(cudaStreamSynchronize(cs), "path sync");
    gr_status s = status_from_word(w);
    if (s != GR_OK) return s;
    const size_t base = (size_t)level * h->rows + h->row_off[request];
    if (n > 0) {
        if (parents) GR_CUDA(cudaMemcpyAsync(parents, h->st.parent + base, 4ull * n, cudaMemcpyDeviceToHost, cs), "path");
        if (tokens) GR_CUDA(cudaMemcpyAsync(tokens, h->st.token + base, 4ull * n, cudaMemcpyDeviceToHost, cs), "path");
        if (nodes) GR_CUDA(cudaMemcpyAsync(nodes, h->st.node + base, 4ull * n, cudaMemcpyDeviceToHost, cs), "path");
        if (scores) GR_CUDA(cudaMemcpyAsync(scores, h->st.score + base, 4ull * n, cudaMemcpyDeviceToHost, cs), "path");
        GR_CUDA(cudaStreamSynchronize(cs), "path sync");
    }
    *n_out = n;
    return GR_OK;
}

extern "C" gr_status gr_beam_set_timing(gr_beam* h, int enable) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    h->timing = enable != 0;
    return GR_OK;
}

extern "C" gr_status gr_beam_kernel_stats(gr_beam* h, int kind, int64_t* launches, double* total_ms, int reset) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (kind < 0 || kind >= GR_KERNEL_KINDS) return fail(GR_ERR_INVALID_ARG, "kernel kind %d out of range", kind);
    if (launches) *launches = h->launches[kind];
    double ms = 0.0;
    for (auto& e : h->events[kind]) {
        GR_CUDA(cudaEventSynchronize(e.b), "event sync");
        float f = 0.f;
        GR_CUDA(cudaEventElapsedTime(&f, e.a, e.b), "event elapsed");
        ms += f;
    }
    if (total_ms) *total_ms = ms;
    if (reset) {
        h->launches[kind] = 0;
        for (auto& e : h->events[kind]) h->event_pool.push_back(e);
        h->events[kind].clear();
    }
    return GR_OK;
}

extern "C" gr_status gr_beam_set_wait_limit(gr_beam* h, int64_t nanoseconds) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    h->wait_limit_ns = (nanoseconds == 0) ? 2000000000ll : nanoseconds;
    return GR_OK;
}

// ---------------------------------------------------------------------------
// multi-item candidate scoring
// ---------------------------------------------------------------------------
namespace {
struct ScoreLayout {
    size_t req, tmaps, jobs, cta_jobs, units, seg_first, seg_pos, cand_off, labels, tables_end, status, o_part,
        lse_part, piece_flag, total;
};

gr_status check_score(const gr_score_config* c, const gr_score_request* reqs, int n) {
    if (c == nullptr || (reqs == nullptr && n > 0)) return fail(GR_ERR_INVALID_ARG, "NULL config or requests");
    if (n < 1) return fail(GR_ERR_INVALID_ARG, "n_requests must be >= 1");
    if (c->n_layers < 1) return fail(GR_ERR_INVALID_ARG, "n_layers must be >= 1");
    if (c->n_kv_heads < 1 || c->n_q_heads < c->n_kv_heads || c->n_q_heads % c->n_kv_heads != 0)
        return fail(GR_ERR_INVALID_ARG, "n_q_heads must be a positive multiple of n_kv_heads");
    const int G = c->n_q_heads / c->n_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
        return fail(GR_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4, 8 or 16 (got %d)", G);
    if (c->head_dim != 64 && c->head_dim != 128) return fail(GR_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c->vocab < 1 || c->pool_tokens < 1) return fail(GR_ERR_INVALID_ARG, "vocab and pool_tokens must be >= 1");
    if (c->n_labels < 1 || c->n_labels > 16 || c->label_ids == nullptr)
        return fail(GR_ERR_INVALID_ARG, "n_labels must be 1..16 with label_ids given");
    for (int k = 0; k < c->n_labels; ++k)
        if (c->label_ids[k] < 0 || c->label_ids[k] >= c->vocab)
            return fail(GR_ERR_INVALID_ARG, "label %d: token %d outside the vocabulary", k, c->label_ids[k]);
    for (int r = 0; r < n; ++r) {
        const gr_score_request& q = reqs[r];
        if (q.ctx_len < 1 || q.ctx_offset < 0 || q.ctx_offset + q.ctx_len > c->pool_tokens)
            return fail(GR_ERR_INVALID_ARG, "request %d: prefix outside the pool", r);
        if (q.n_candidates < 1 || q.n_candidates > kMaxCandidates)
            return fail(GR_ERR_CAPACITY, "request %d: n_candidates must be in 1..%d", r, kMaxCandidates);
        if (q.seg_lens == nullptr) return fail(GR_ERR_INVALID_ARG, "request %d: seg_lens is NULL", r);
        for (int k = 0; k < q.n_candidates; ++k)
            if (q.seg_lens[k] < 1 || q.seg_lens[k] > kMaxSegment)
                return fail(GR_ERR_CAPACITY, "request %d, candidate %d: %d tokens (1..%d)", r, k, q.seg_lens[k],
                            kMaxSegment);
    }
    return GR_OK;
}

// the decode schedule's view of a scoring batch: one "beam" per candidate token
void score_as_decode(const gr_score_config* c, const gr_score_request* reqs, int n, gr_config* dc,
                     std::vector<gr_request>& dr, int* rows) {
    *dc = gr_config{};
    dc->n_layers = c->n_layers;
    dc->n_q_heads = c->n_q_heads;
    dc->n_kv_heads = c->n_kv_heads;
    dc->head_dim = c->head_dim;
    dc->vocab = c->vocab;
    dc->n_levels = 1;
    dc->codes_per_level = 1;
    dc->pool_tokens = c->pool_tokens;
    dr.assign(n, gr_request{});
    *rows = 0;
    for (int r = 0; r < n; ++r) {
        int w = 0;
        for (int k = 0; k < reqs[r].n_candidates; ++k) w += reqs[r].seg_lens[k];
        dr[r].ctx_offset = reqs[r].ctx_offset;
        dr[r].ctx_len = reqs[r].ctx_len;
        dr[r].beam_width = w;
        *rows += w;
    }
}

ScoreLayout score_layout(int n, int rows, int n_cand, int n_labels, int head_dim, const Caps& k) {
    ScoreLayout w{};
    size_t o = 0;
    auto take = [&](size_t bytes, size_t align = 256) {
        o = align_up(o, align);
        size_t r = o;
        o += bytes;
        return r;
    };
    w.req = take(sizeof(GrReqDev) * n);
    w.tmaps = take(sizeof(CUtensorMap) * kTmapsPerReq * n, 128);
    w.jobs = take(sizeof(GrAttnJob) * k.jobs);
    w.cta_jobs = take(sizeof(int2) * k.ctas);
    w.units = take(sizeof(GrAttnUnit) * k.units);
    w.seg_first = take(4ull * rows);
    w.seg_pos = take(4ull * rows);
    w.cand_off = take(4ull * (n + 1));
    w.labels = take(4ull * n_labels);
    w.tables_end = align_up(o, 256);
    w.status = take(16);
    w.o_part = take(4ull * k.jobs * kUnitRows * head_dim);
    w.lse_part = take(4ull * k.jobs * kUnitRows);
    w.piece_flag = take(4ull * k.jobs * kUnitRows);
    w.total = align_up(o, 256);
    return w;
}
}  // namespace

struct gr_score {
    gr_score_config cfg{};
    std::vector<int32_t> labels;
    int n_req = 0, rows = 0, n_cand = 0;
    std::vector<int> row_off, cand_off;
    GrState st{};
    Caps caps{};
    ScoreLayout w{};
    int64_t wait_limit_ns = 2000000000ll;
};

extern "C" gr_status gr_score_workspace_bytes(const gr_score_config* cfg, const gr_score_request* reqs, int n,
                                              size_t* bytes) {
    if (bytes == nullptr) return fail(GR_ERR_INVALID_ARG, "bytes is NULL");
    gr_status s = check_score(cfg, reqs, n);
    if (s != GR_OK) return s;
    int n_sm = device_sm_count();
    if (n_sm <= 0) n_sm = 148;
    gr_config dc;
    std::vector<gr_request> dr;
    int rows = 0, n_cand = 0;
    score_as_decode(cfg, reqs, n, &dc, dr, &rows);
    for (int r = 0; r < n; ++r) n_cand += reqs[r].n_candidates;
    std::vector<int> uo, nu;
    Schedule sc = build_schedule(&dc, dr.data(), n, n_sm, uo, nu);
    *bytes = score_layout(n, rows, n_cand, cfg->n_labels, cfg->head_dim, caps_of(sc, n_sm)).total;
    return GR_OK;
}

extern "C" gr_status gr_score_create(const gr_score_config* cfg, const gr_score_request* reqs, int n,
                                     const gr_score_buffers* bufs, gr_stream_t stream, gr_score** out) {
    if (out == nullptr || bufs == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL out or buffers");
    *out = nullptr;
    gr_status s = check_score(cfg, reqs, n);
    if (s != GR_OK) return s;
    if (!bufs->ctx_k || !bufs->ctx_v || !bufs->seg_k || !bufs->seg_v || !bufs->workspace)
        return fail(GR_ERR_INVALID_ARG, "ctx_k, ctx_v, seg_k, seg_v and workspace must be device pointers");
    if ((reinterpret_cast<uintptr_t>(bufs->workspace) & 255) != 0)
        return fail(GR_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if ((reinterpret_cast<uintptr_t>(bufs->ctx_k) & 15) != 0 || (reinterpret_cast<uintptr_t>(bufs->ctx_v) & 15) != 0)
        return fail(GR_ERR_INVALID_ARG, "ctx_k / ctx_v must be 16-byte aligned");
    const int n_sm = device_sm_count();
    if (n_sm <= 0) return fail(GR_ERR_CUDA, "no CUDA device");
    cudaStream_t cs = (cudaStream_t)stream;
    gr_score* h = nullptr;
    try {
        h = new gr_score;
        h->cfg = *cfg;
        h->labels.assign(cfg->label_ids, cfg->label_ids + cfg->n_labels);
        h->cfg.label_ids = h->labels.data();
        h->n_req = n;
        gr_config dc;
        std::vector<gr_request> dr;
        score_as_decode(cfg, reqs, n, &dc, dr, &h->rows);
        h->row_off.assign(n + 1, 0);
        h->cand_off.assign(n + 1, 0);
        for (int r = 0; r < n; ++r) {
            h->row_off[r + 1] = h->row_off[r] + dr[r].beam_width;
            h->cand_off[r + 1] = h->cand_off[r] + reqs[r].n_candidates;
        }
        h->n_cand = h->cand_off[n];
        std::vector<int> unit_off, n_ub;
        Schedule sc = build_schedule(&dc, dr.data(), n, n_sm, unit_off, n_ub);
        h->caps = caps_of(sc, n_sm);
        h->w = score_layout(n, h->rows, h->n_cand, cfg->n_labels, cfg->head_dim, h->caps);
        const ScoreLayout& w = h->w;
        if (bufs->workspace_bytes < w.total) {
            gr_status e = fail(GR_ERR_CAPACITY, "workspace needs %zu bytes, got %zu", w.total, bufs->workspace_bytes);
            delete h;
            return e;
        }
        uint8_t* ws = static_cast<uint8_t*>(bufs->workspace);
        GrState& st = h->st;
        st.req = reinterpret_cast<GrReqDev*>(ws + w.req);
        st.n_req = n;
        st.rows = h->rows;
        st.n_levels = 1;
        st.vocab = cfg->vocab;
        st.n_layers = cfg->n_layers;
        st.n_q_heads = cfg->n_q_heads;
        st.n_kv_heads = cfg->n_kv_heads;
        st.head_dim = cfg->head_dim;
        st.pool_tokens = cfg->pool_tokens;
        st.status = reinterpret_cast<int32_t*>(ws + w.status);
        st.tmaps = reinterpret_cast<CUtensorMap*>(ws + w.tmaps);
        st.jobs = reinterpret_cast<GrAttnJob*>(ws + w.jobs);
        st.cta_jobs = reinterpret_cast<int2*>(ws + w.cta_jobs);
        st.units = reinterpret_cast<GrAttnUnit*>(ws + w.units);
        st.o_part = reinterpret_cast<float*>(ws + w.o_part);
        st.lse_part = reinterpret_cast<float*>(ws + w.lse_part);
        st.piece_flag = reinterpret_cast<uint32_t*>(ws + w.piece_flag);
        st.beam_k = static_cast<const uint16_t*>(bufs->seg_k);
        st.beam_v = static_cast<const uint16_t*>(bufs->seg_v);
        st.seg_first = reinterpret_cast<const int32_t*>(ws + w.seg_first);
        st.seg_pos = reinterpret_cast<const int32_t*>(ws + w.seg_pos);
        st.n_units = (int)sc.units.size();
        st.n_jobs = (int)sc.jobs.size();
        st.n_cta = (int)sc.cta_jobs.size();
        // host image of the tables
        std::vector<uint8_t> img(w.tables_end, 0);
        GrReqDev* rq = reinterpret_cast<GrReqDev*>(img.data() + w.req);
        CUtensorMap* tm = reinterpret_cast<CUtensorMap*>(img.data() + w.tmaps);
        int32_t* sf = reinterpret_cast<int32_t*>(img.data() + w.seg_first);
        int32_t* sp = reinterpret_cast<int32_t*>(img.data() + w.seg_pos);
        const int D = cfg->head_dim;
        const uint64_t zdim = (uint64_t)cfg->n_layers * cfg->n_kv_heads;
        for (int r = 0; r < n; ++r) {
            GrReqDev d{};
            d.row_off = h->row_off[r];
            d.width = dr[r].beam_width;
            d.ctx_len = reqs[r].ctx_len;
            d.n_levels = 1;
            d.unit_off = unit_off[r];
            d.n_ub = n_ub[r];
            d.ctx_off = reqs[r].ctx_offset;
            rq[r] = d;
            int row = h->row_off[r];
            for (int k = 0; k < reqs[r].n_candidates; ++k)
                for (int p = 0; p < reqs[r].seg_lens[k]; ++p, ++row) {
                    sf[row] = row - p;
                    sp[row] = p;
                }
            const uint64_t off = (uint64_t)reqs[r].ctx_offset * D * 2;
            const uint64_t s1 = (uint64_t)D * 2, s2 = (uint64_t)cfg->pool_tokens * D * 2;
            // the scoring pass runs the single-CTA kernel, which reads the first two maps
            if ((s = make_tmap_3d(&tm[kTmapsPerReq * r], static_cast<const uint8_t*>(bufs->ctx_k) + off, D,
                                  reqs[r].ctx_len, zdim, s1, s2, 64, kTileKeys, 1)) != GR_OK ||
                (s = make_tmap_3d(&tm[kTmapsPerReq * r + 1], static_cast<const uint8_t*>(bufs->ctx_v) + off, D,
                                  reqs[r].ctx_len, zdim, s1, s2, 64, kTileKeys, 1)) != GR_OK) {
                delete h;
                return s;
            }
        }
        finalize_jobs(sc, rq);
        memcpy(img.data() + w.jobs, sc.jobs.data(), sizeof(GrAttnJob) * sc.jobs.size());
        memcpy(img.data() + w.cta_jobs, sc.cta_jobs.data(), sizeof(int2) * sc.cta_jobs.size());
        memcpy(img.data() + w.units, sc.units.data(), sizeof(GrAttnUnit) * sc.units.size());
        memcpy(img.data() + w.cand_off, h->cand_off.data(), 4ull * (n + 1));
        memcpy(img.data() + w.labels, h->labels.data(), 4ull * h->labels.size());
        cudaError_t e = cudaMemcpyAsync(ws, img.data(), img.size(), cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(ws + w.status, 0, 16, cs);
        if (e == cudaSuccess) e = cudaMemsetAsync(st.piece_flag, 0, 4ull * h->caps.jobs * kUnitRows, cs);
        if (e == cudaSuccess) e = cudaStreamSynchronize(cs);  // img is released on return
        if (e != cudaSuccess) {
            delete h;
            return cuda_fail(e, "workspace upload");
        }
    } catch (const std::bad_alloc&) {
        delete h;
        return fail(GR_ERR_CAPACITY, "host allocation failed");
    }
    *out = h;
    return GR_OK;
}

extern "C" gr_status gr_score_destroy(gr_score* h) {
    delete h;
    return GR_OK;
}

extern "C" gr_status gr_score_rows(const gr_score* h, int* rows_total, int* row_offsets, int* cand_offsets) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    if (rows_total) *rows_total = h->rows;
    for (int r = 0; r <= h->n_req; ++r) {
        if (row_offsets) row_offsets[r] = h->row_off[r];
        if (cand_offsets) cand_offsets[r] = h->cand_off[r];
    }
    return GR_OK;
}

extern "C" gr_status gr_score_attn(gr_score* h, int layer, const void* q, void* out, gr_stream_t stream) {
    if (h == nullptr || q == nullptr || out == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (layer < 0 || layer >= h->cfg.n_layers) return fail(GR_ERR_INVALID_ARG, "layer %d out of range", layer);
    if ((reinterpret_cast<uintptr_t>(q) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0)
        return fail(GR_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    const gr_score_config& c = h->cfg;
    const int G = c.n_q_heads / c.n_kv_heads;
    CUtensorMap qmap;
    gr_status s = make_tmap_3d(&qmap, q, c.head_dim, c.n_q_heads, h->rows, (uint64_t)c.head_dim * 2,
                               (uint64_t)c.n_q_heads * c.head_dim * 2, 64, G, kTileRows / G);
    if (s != GR_OK) return s;
    cudaError_t e = launch_score_attn(h->st, qmap, layer, static_cast<const uint16_t*>(q), static_cast<uint16_t*>(out),
                                      h->wait_limit_ns, (cudaStream_t)stream);
    return e == cudaSuccess ? GR_OK : cuda_fail(e, "kernel launch");
}

extern "C" gr_status gr_score_labels(gr_score* h, const float* logits, int64_t ld, float* logprobs, int32_t* ranking,
                                     gr_stream_t stream) {
    if (h == nullptr || logits == nullptr || logprobs == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL argument");
    if (ld < h->cfg.vocab || ld % 4 != 0) return fail(GR_ERR_INVALID_ARG, "ld must be >= vocab and a multiple of 4");
    if ((reinterpret_cast<uintptr_t>(logits) & 15) != 0) return fail(GR_ERR_INVALID_ARG, "logits must be 16-byte aligned");
    cudaStream_t cs = (cudaStream_t)stream;
    const uint8_t* ws = reinterpret_cast<const uint8_t*>(h->st.req);
    const int32_t* labels = reinterpret_cast<const int32_t*>(ws + h->w.labels);
    cudaError_t e = launch_label_logprobs(logits, ld, h->cfg.vocab, labels, h->cfg.n_labels, h->n_cand, logprobs,
                                          h->st.status, cs);
    if (e == cudaSuccess && ranking != nullptr)
        e = launch_rank(logprobs, h->cfg.n_labels, reinterpret_cast<const int32_t*>(ws + h->w.cand_off), h->n_req,
                        ranking, h->st.status, cs);
    return e == cudaSuccess ? GR_OK : cuda_fail(e, "kernel launch");
}

extern "C" gr_status gr_score_status(gr_score* h, int clear_flag, gr_stream_t stream) {
    if (h == nullptr) return fail(GR_ERR_INVALID_ARG, "NULL handle");
    cudaStream_t cs = (cudaStream_t)stream;
    int w = 0;
    GR_CUDA(cudaMemcpyAsync(&w, h->st.status, 4, cudaMemcpyDeviceToHost, cs), "status read");
    GR_CUDA(cudaStreamSynchronize(cs), "status sync");
    if (clear_flag && w != 0) {
        GR_CUDA(cudaMemsetAsync(h->st.status, 0, 16, cs), "status clear");
        GR_CUDA(cudaMemsetAsync(h->st.piece_flag, 0, 4ull * h->caps.jobs * kUnitRows, cs), "flag clear");
        GR_CUDA(cudaStreamSynchronize(cs), "status clear sync");
    }
    return status_from_word(w);
}

extern "C" const char* gr_status_str(gr_status s) {
    switch (s) {
        case GR_OK: return "GR_OK";
        case GR_ERR_INVALID_ARG: return "GR_ERR_INVALID_ARG";
        case GR_ERR_UNSUPPORTED: return "GR_ERR_UNSUPPORTED";
        case GR_ERR_CAPACITY: return "GR_ERR_CAPACITY";
        case GR_ERR_STATE: return "GR_ERR_STATE";
        case GR_ERR_CUDA: return "GR_ERR_CUDA";
        case GR_ERR_TIMEOUT: return "GR_ERR_TIMEOUT";
        case GR_ERR_DEVICE: return "GR_ERR_DEVICE";
        default: return "unknown gr_status";
    }
}

extern "C" const char* gr_last_error(void) { return g_last_error.c_str(); }
