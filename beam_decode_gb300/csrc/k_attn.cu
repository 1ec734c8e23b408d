// GQA decode attention of every beam over the split KV layout.
//
// zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架"
// (semantic-ID GR inference framework): the long request context is kept once
// per request (ContextKV) and shared by all beams, each beam keeps only the
// short history of its own decoded tokens (BeamKV), and beam ancestry lives in
// BeamPath; the attention backend works directly on that layout.
//
// Because every beam of a request -- and every query head of a GQA group --
// reads the same ContextKV, the context part is a dense contraction: for one
// (request, KV head) the query block is n_beams*G rows x D, and
//     S = Q K^T / sqrt(D),  O = softmax(S) V
// over the request's T context keys.  That part runs on the tensor cores:
//
// k_ctx_attn (per CTA: a list of jobs = key-tile ranges of 256-row units)
//   warp 0     TMA producer: Q tiles once per job, then K and V tiles of 128
//              keys through a two-stage shared-memory ring (128-byte swizzle).
//   warps 1, 3 MMA issuers (one thread each): warp 3 issues S_i = Q_i K^T into
//              TMEM (M=128, N=128, K=16 per instruction), warp 1 issues
//              O_i += P_i V with P_i read from TMEM.
//   warp 2     TMEM allocation (512 columns: S0, S1, O0, O1).
//   warps 4-7  softmax of query tile 0; warps 8-11 softmax of query tile 1:
//              one thread per row (TMEM lane), online max/sum with a lazy
//              rescale of O (only when the running max grows by more than
//              2^8), P written back to TMEM as bf16 in place of S.
//   The two query tiles ping-pong: while one warpgroup exponentiates, the
//   tensor core runs the other tile's MMAs.
// Units of one (request, KV head) are scheduled on neighbouring CTAs so the
// second read of a K/V tile is served by L2; each context byte comes from HBM
// once per request.
//
// Epilogue: a unit whose key tiles were cut over several CTAs is finished by
// its first key range, which by construction of the schedule is the last job
// of its CTA; the later ranges run at the start of the next CTAs and publish
// their normalised fp32 piece, its log-sum-exp and a per-row ready flag,
// which the merger clears once it has read the row.  The first range merges,
// by a log-sum-exp combine, its own O (from TMEM), the pieces, and the beam
// part -- the t BeamKV keys found through the beam's ancestry row (levels
// 0..t-1), folded in one key at a time per row, from K/V rows bulk-copied into
// the freed shared-memory rings -- and writes the bf16 output row.  Rows of
// dead beams are written as zeros.  The launch is cooperative, so every CTA a
// merger waits for is resident.

// Every wait inside k_ctx_attn is bounded: past the limit the kernel flags
// GR_ERR_TIMEOUT, drains the copies and MMAs it issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "grbeam_internal.h"

namespace grb {
namespace {

// ---------------------------------------------------------------------------
// PTX wrappers (mbarrier, TMA, tcgen05)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(dst),
        "l"(tmap), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// untiled bulk copy global -> shared, completion counted on an mbarrier (16-byte aligned
// addresses, size a multiple of 16 bytes)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
// a store whose line L2 should keep (evict_last policy): a published piece waits there
// for its merger
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void st_keep(float4* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w), "l"(pol)
                 : "memory");
}
// untiled bulk copy shared -> global (bulk async-group completion)
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_read() {
    asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmap_acquire(const void* tmap) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

#define GRB_R8(i) "=r"(v[i + 0]), "=r"(v[i + 1]), "=r"(v[i + 2]), "=r"(v[i + 3]), "=r"(v[i + 4]), "=r"(v[i + 5]), \
                  "=r"(v[i + 6]), "=r"(v[i + 7])
#define GRB_W8(i) "r"(v[i + 0]), "r"(v[i + 1]), "r"(v[i + 2]), "r"(v[i + 3]), "r"(v[i + 4]), "r"(v[i + 5]), \
                  "r"(v[i + 6]), "r"(v[i + 7])

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers per
// thread; the wait is inside the same statement so no register is read early.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GRB_R8(0), GRB_R8(8), GRB_R8(16), GRB_R8(24)
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        GRB_W8(0), GRB_W8(8), GRB_W8(16), GRB_W8(24)
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// all 128 columns of this warp's 32 lanes in one round trip (128 registers per thread)
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GRB_R8(0), GRB_R8(8), GRB_R8(16), GRB_R8(24), GRB_R8(32), GRB_R8(40), GRB_R8(48), GRB_R8(56),
          GRB_R8(64), GRB_R8(72), GRB_R8(80), GRB_R8(88), GRB_R8(96), GRB_R8(104), GRB_R8(112), GRB_R8(120)
        : "r"(taddr)
        : "memory");
}

// packed fp32 pairs (Blackwell f32x2 ALU)
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// CTA-wide named barrier (all 384 threads), usable from separate code regions
__device__ __forceinline__ void named_bar_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(384) : "memory");
}

// register split between warpgroups (sums to the launch's 384 x 168)
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// Shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: bf16 x bf16 -> fp32, A K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// bounded waits
// ---------------------------------------------------------------------------
constexpr int64_t kDrainLimitNs = 1000000000ll;  // 1 s for draining issued work

struct Waiter {
    int64_t limit;          // ns; < 0: give up at the first failed check
    volatile int* abort;    // shared flag: some thread gave up
    int* status;            // global status word
};

// one thread
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const Waiter w) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (w.limit < 0 || ((++spins) & 31) == 0) {
            if (*w.abort) return false;
            if (w.limit < 0 || (int64_t)(global_timer() - t0) > w.limit) {
                *w.abort = 1;
                atomicOr(w.status, kStatusTimeout);
                return false;
            }
        }
    }
    return true;
}

// whole warp (convergent): returns the same value on every lane
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Waiter w) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    uint32_t spins = 0;
    for (;;) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        int give_up = 0;
        if (lane == 0) {
            if (t0 == 0) t0 = global_timer();
            if (w.limit < 0 || ((++spins) & 31) == 0) {
                if (*w.abort) give_up = 1;
                else if (w.limit < 0 || (int64_t)(global_timer() - t0) > w.limit) {
                    *w.abort = 1;
                    atomicOr(w.status, kStatusTimeout);
                    give_up = 1;
                }
            }
        }
        if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
}

// drain: fixed limit, no abort check
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    uint64_t t0 = global_timer();
    while (!mbar_try_wait(bar, parity)) {
        if ((int64_t)(global_timer() - t0) > kDrainLimitNs) return;
    }
}

// one thread waits for a flag written by another CTA of the same (cooperative) launch
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t value, const Waiter w) {
    const volatile uint32_t* f = reinterpret_cast<const volatile uint32_t*>(flag);
    if (*f == value) return true;
    const uint64_t t0 = global_timer();
    uint32_t spins = 0;
    while (*f != value) {
        if (w.limit < 0 || ((++spins) & 31) == 0) {
            if (*w.abort) return false;
            if (w.limit < 0 || (int64_t)(global_timer() - t0) > w.limit) {
                *w.abort = 1;
                atomicOr(w.status, kStatusTimeout);
                return false;
            }
        }
        __nanosleep(64);
    }
    return true;
}

// a unit takes part in a launch when its request is at a decode step 1 <= t_r < L_r
// (level 0 has no BeamKV and needs no attention; t_r == L_r is finished).  Every role of
// the CTA reads the same device-resident step, so they skip the same jobs.
template <bool kScore>
__device__ __forceinline__ bool decoding(const GrState& st, const GrAttnUnit& U) {
    if constexpr (kScore) return true;  // multi-item scoring: one pass, every unit takes part
    const int t = st.req_step[U.req];
    return t >= 1 && t < U.n_levels;
}

// ---------------------------------------------------------------------------
// one query row of a unit, as a softmax thread (TMEM lane) sees it
// ---------------------------------------------------------------------------
struct RowInfo {
    int b;                 // beam (decode) / candidate-token row (scoring) within the request
    bool row_ok;           // the row exists (b < W_r)
    bool live;             // and takes part: an alive beam / a scored token
    int n_priv;            // private keys: decode t (levels 0..t-1 of BeamKV), scoring pos + 1
    int pool0;             // scoring: pool row of the segment's first token
    int64_t orow_idx;      // query / output row (row x query head)
    const int32_t* path;   // decode: the beam's ancestry row at level t-1
};

template <bool kScore>
__device__ __forceinline__ RowInfo row_info(const GrState& st, const GrAttnUnit& U, int i, int row_t, int G) {
    RowInfo ri;
    const int t = kScore ? 0 : st.req_step[U.req];
    ri.b = U.beam0 + i * (kTileRows / G) + row_t / G;
    const int g = row_t % G;
    ri.row_ok = ri.b < U.width;
    ri.live = ri.row_ok && (kScore || ri.b < st.n_beams[U.req * (st.n_levels + 1) + t]);
    ri.orow_idx = (int64_t)(U.row_off + ri.b) * st.n_q_heads + U.head * G + g;
    ri.pool0 = 0;
    ri.path = nullptr;
    ri.n_priv = 0;
    if constexpr (kScore) {
        if (ri.live) {
            ri.n_priv = st.seg_pos[U.row_off + ri.b] + 1;
            ri.pool0 = st.seg_first[U.row_off + ri.b];
        }
    } else {
        ri.n_priv = ri.live ? t : 0;
        ri.path = st.path + ((int64_t)(t - 1) * st.rows + U.row_off + ri.b) * st.n_levels;
    }
    return ri;
}

// bf16 pair -> two floats
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// shared-memory plan
// ---------------------------------------------------------------------------
template <int D>
struct Plan {
    static constexpr int kBoxes = D / 64;               // 128-byte column boxes per row
    static constexpr int kBoxBytes = 128 * 128;         // 128 rows x 128 bytes
    static constexpr int kQTile = kBoxes * kBoxBytes;   // one 128-row query tile
    static constexpr int kKVTile = kBoxes * kBoxBytes;  // one 128-key K or V tile
    static constexpr int kStages = 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + 2 * kQTile;
    static constexpr int kVOff = kKOff + kStages * kKVTile;
    static constexpr int kBarOff = kVOff + kStages * kKVTile;
    static constexpr int kBytes = kBarOff + 512 + 1024;  // barriers, TMEM address, abort flag, alignment
    // TMEM columns
    static constexpr int kTmemCols = 512;
    static __device__ __forceinline__ int s_col(int i) { return i * 128; }
    static __device__ __forceinline__ int p_col(int i) { return i * 128; }  // bf16 P overwrites S in place
    static __device__ __forceinline__ int o_col(int i) { return 256 + i * D; }
};

enum Bar {
    B_Q_FULL = 0, B_Q_EMPTY = 1, B_K_FULL = 2, B_K_EMPTY = 4, B_V_FULL = 6, B_V_EMPTY = 8,
    B_S_FULL = 10, B_P_FULL = 12, B_O_FULL = 14, B_O_EMPTY = 16, B_DRAIN = 18, B_PVD = 20,
    B_BEAM = 22,  // one per softmax warp: its BeamKV rows copied into the freed rings
    B_MERGED = 30,  // a merging job that is not the CTA's last has finished with the rings and Q
    B_COUNT = 31
};

constexpr int kAttnThreads = 384;

template <int D, bool kScore>
__global__ void __launch_bounds__(kAttnThreads, 1)
k_ctx_attn(const __grid_constant__ CUtensorMap qmap, GrState st, int layer, const uint16_t* __restrict__ q,
           uint16_t* __restrict__ out, float scale_log2, float scale, int64_t wait_limit_ns) {
    using P = Plan<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + P::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kBarOff + 8 * B_COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::kBarOff + 8 * B_COUNT + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = st.n_q_heads / st.n_kv_heads;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        mbar_init(bar(B_Q_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_K_FULL + s), 1);
            mbar_init(bar(B_K_EMPTY + s), 1);
            mbar_init(bar(B_V_FULL + s), 1);
            mbar_init(bar(B_V_EMPTY + s), 1);
            mbar_init(bar(B_S_FULL + s), 1);
            mbar_init(bar(B_P_FULL + s), 128);
            mbar_init(bar(B_O_FULL + s), 1);
            mbar_init(bar(B_O_EMPTY + s), 128);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(bar(B_DRAIN + k), 1);
            mbar_init(bar(B_PVD + k), 1);
        }
        for (int k = 0; k < 8; ++k) mbar_init(bar(B_BEAM + k), 1);
        mbar_init(bar(B_MERGED), 8);  // one arrival per softmax warp (see the merge's end)
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), P::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int2 jr = st.cta_jobs[blockIdx.x];
    const Waiter wt{wait_limit_ns, abort_flag, st.status};

    // The producer / MMA / allocator warpgroup gives registers to the two softmax
    // warpgroups (128 x 56 + 2 x 128 x 224 = 384 x 168).  The two register
    // regions never rejoin: each side runs its own teardown and returns.
    if (warp < 4) {
        regs_dec<56>();
        // producer state (kept for the drain)
        uint32_t p_kit = 0, p_vit = 0, p_qcnt = 0, p_mcnt = 0;
    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                const GrAttnJob J = st.jobs[jb];
                const GrAttnUnit& U = J.u;
                if (!decoding<kScore>(st, U)) continue;
                const CUtensorMap* km = st.tmaps + 2 * U.req;
                const CUtensorMap* vm = km + 1;
                if (jb == jr.x || st.jobs[jb - 1].unit != J.unit) {
                    tmap_acquire(km);
                    tmap_acquire(vm);
                }
                if (p_qcnt > 0 && !(ok = wait1(bar(B_Q_EMPTY), (p_qcnt - 1) & 1, wt))) break;
                mbar_expect_tx(bar(B_Q_FULL), (uint32_t)(U.nqt * P::kQTile));
                for (int i = 0; i < U.nqt; ++i)
                    for (int kb = 0; kb < P::kBoxes; ++kb)
                        tma_load_3d(sb + P::kQOff + i * P::kQTile + kb * P::kBoxBytes, &qmap, bar(B_Q_FULL), kb * 64,
                                    U.head * G, U.row_off + U.beam0 + i * (kTileRows / G));
                ++p_qcnt;
                const int z = layer * st.n_kv_heads + U.head;
                for (int j = J.t0; j < J.t1; ++j) {
                    int s = p_kit & 1;
                    if (!(ok = wait1(bar(B_K_EMPTY + s), ((p_kit >> 1) & 1) ^ 1, wt))) break;
                    mbar_expect_tx(bar(B_K_FULL + s), P::kKVTile);
                    for (int kb = 0; kb < P::kBoxes; ++kb)
                        tma_load_3d(sb + P::kKOff + s * P::kKVTile + kb * P::kBoxBytes, km, bar(B_K_FULL + s),
                                    kb * 64, j * kTileKeys, z);
                    ++p_kit;
                    s = p_vit & 1;
                    if (!(ok = wait1(bar(B_V_EMPTY + s), ((p_vit >> 1) & 1) ^ 1, wt))) break;
                    mbar_expect_tx(bar(B_V_FULL + s), P::kKVTile);
                    for (int kb = 0; kb < P::kBoxes; ++kb)
                        tma_load_3d(sb + P::kVOff + s * P::kKVTile + kb * P::kBoxBytes, vm, bar(B_V_FULL + s),
                                    kb * 64, j * kTileKeys, z);
                    ++p_vit;
                }
                // A merging job stages its BeamKV keys in the rings and reads q from its Q tile:
                // the next job's loads wait until its merge is done.
                if (ok && J.slot == U.first_slot && jb < jr.y - 1) {
                    if (!(ok = wait1(bar(B_MERGED), p_mcnt & 1, wt))) break;
                    ++p_mcnt;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // Two MMA issuers (one thread each): warp 3 issues S_i = Q_i K^T, warp 1 issues
        // O_i += P_i V.  S_i of key tile j overwrites P_i of tile j-1, so it waits until
        // that PV has completed (B_PVD + i).  Each thread's waits and commits then overlap
        // the other's MMAs, which keeps the tensor pipe fed.
        if (lane == 0) {
            bool mma_issued = false;
            bool ok = true;
            if (warp == 3) {
                constexpr uint32_t idesc_s = idesc_bf16(128, kTileKeys, false);
                uint32_t kit = 0, qcnt = 0, s_i[2] = {0, 0};
                for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                    const GrAttnJob J = st.jobs[jb];
                    const GrAttnUnit& U = J.u;
                    if (!decoding<kScore>(st, U)) continue;
                    const int nqt = U.nqt;
                    const int n = J.t1 - J.t0;
                    if (!(ok = wait1(bar(B_Q_FULL), qcnt & 1, wt))) break;
                    ++qcnt;
                    for (int jj = 0; jj < n && ok; ++jj) {
                        const int ks = kit & 1;
                        if (!(ok = wait1(bar(B_K_FULL + ks), (kit >> 1) & 1, wt))) break;
                        for (int i = 0; i < nqt; ++i) {
                            if (s_i[i] > 0 && !(ok = wait1(bar(B_PVD + i), (s_i[i] - 1) & 1, wt))) break;
                            tc_fence_after();
                            const uint32_t d = tmem + P::s_col(i);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = (kk >> 2) * P::kBoxBytes + (kk & 3) * 32;
                                const uint64_t a = smem_desc(sb + P::kQOff + i * P::kQTile + off, 16, 1024);
                                const uint64_t b = smem_desc(sb + P::kKOff + ks * P::kKVTile + off, 16, 1024);
                                mma_ss(d, a, b, idesc_s, kk > 0 ? 1u : 0u);
                            }
                            mma_issued = true;
                            tc_commit(bar(B_S_FULL + i));
                            ++s_i[i];
                        }
                        if (!ok) break;
                        tc_commit(bar(B_K_EMPTY + ks));
                        ++kit;
                        if (jj == n - 1) tc_commit(bar(B_Q_EMPTY));
                    }
                }
            } else {
                constexpr uint32_t idesc_o = idesc_bf16(128, D, true);
                uint32_t vit = 0, pv_i[2] = {0, 0}, jobs_i[2] = {0, 0};
                for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                    const GrAttnJob J = st.jobs[jb];
                    const GrAttnUnit& U = J.u;
                    if (!decoding<kScore>(st, U)) continue;
                    const int nqt = U.nqt;
                    const int n = J.t1 - J.t0;
                    for (int jj = 0; jj < n && ok; ++jj) {
                        const int vs = vit & 1;
                        if (!(ok = wait1(bar(B_V_FULL + vs), (vit >> 1) & 1, wt))) break;
                        for (int i = 0; i < nqt; ++i) {
                            if (!(ok = wait1(bar(B_P_FULL + i), pv_i[i] & 1, wt))) break;
                            if (jj == 0 && jobs_i[i] > 0 && !(ok = wait1(bar(B_O_EMPTY + i), (jobs_i[i] - 1) & 1, wt)))
                                break;
                            tc_fence_after();
                            const uint32_t d = tmem + P::o_col(i);
#pragma unroll
                            for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                                const uint32_t a = tmem + P::p_col(i) + kk * 8;
                                const uint64_t b =
                                    smem_desc(sb + P::kVOff + vs * P::kKVTile + kk * 16 * 128, P::kBoxBytes, 1024);
                                mma_ts(d, a, b, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_issued = true;
                            tc_commit(bar(B_PVD + i));  // S_i of the next tile may overwrite P_i
                            ++pv_i[i];
                            if (jj == n - 1) tc_commit(bar(B_O_FULL + i));
                        }
                        if (!ok) break;
                        tc_commit(bar(B_V_EMPTY + vs));
                        ++vit;
                    }
                    for (int i = 0; i < nqt; ++i) ++jobs_i[i];
                }
            }
            // all issued tensor-core work (and its commits) completes before TMEM is freed
            if (mma_issued) {
                const int dr = B_DRAIN + (warp == 3 ? 1 : 0);
                tc_commit(bar(dr));
                wait_drain(bar(dr), 0);
            }
        }
        __syncwarp();
    }
        tc_fence_before();
        named_bar_sync(1);
        // after an abort, every copy the producer issued must land before the CTA exits
        if (warp == 0 && lane == 0 && *abort_flag) {
            if (p_qcnt > 0) wait_drain(bar(B_Q_FULL), (p_qcnt - 1) & 1);
            for (int s = 0; s < 2; ++s) {
                const uint32_t nk = (p_kit + 1 - s) / 2;  // issues into stage s
                if (nk > 0) wait_drain(bar(B_K_FULL + s), (nk - 1) & 1);
                const uint32_t nv = (p_vit + 1 - s) / 2;
                if (nv > 0) wait_drain(bar(B_V_FULL + s), (nv - 1) & 1);
            }
        }
        __syncwarp();
        named_bar_sync(2);
        tc_fence_after();
        if (warp == 2) tmem_dealloc(tmem, P::kTmemCols);
        return;
    }

    regs_inc<224>();
    {
        // softmax warpgroups
        const int i = (warp - 4) >> 2;           // query tile of this warpgroup
        const int quarter = warp & 3;            // TMEM lane quarter
        const int row_t = quarter * 32 + lane;   // row within the tile
        const int prow = i * kTileRows + row_t;  // row within the unit
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t tiles = 0, jobs = 0, ktiles = 0, bcnt = 0;
        bool ok = true;
        // A published piece's ready flag is raised once the next job's first key tile is done
        // (or when a job skips this warpgroup, or at the end): by then the piece's stores have
        // drained and the release fence costs little.  Its merger reads it only at the end of
        // its own job.
        uint32_t* pend_flag = nullptr;
        auto raise_flag = [&]() {
            if (pend_flag != nullptr) {
                __threadfence();
                *reinterpret_cast<volatile uint32_t*>(pend_flag) = 1u;
                pend_flag = nullptr;
            }
        };
        for (int jb = jr.x; jb < jr.y && ok; ++jb) {
            const GrAttnJob J = st.jobs[jb];
            const GrAttnUnit& U = J.u;
            if (!decoding<kScore>(st, U)) continue;
            const int n = J.t1 - J.t0;
            ktiles += n;  // key tiles the S issuer has taken through the K ring so far
            if (i >= U.nqt) {
                raise_flag();
                continue;
            }
            const RowInfo ri = row_info<kScore>(st, U, i, row_t, G);
            const int ctx_len = U.ctx_len;
            const bool merger = (J.slot == U.first_slot);
            float m_used = -CUDART_INF_F, l = 0.f;
            for (int jj = 0; jj < n; ++jj) {
                if (!(ok = wait_warp(bar(B_S_FULL + i), tiles & 1, wt))) break;
                tc_fence_after();
                uint32_t sv[128];
                tmem_ld128(tmem + lane_base + P::s_col(i), sv);
                const int valid = ctx_len - (J.t0 + jj) * kTileKeys;
                if (valid < kTileKeys) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= valid) sv[c] = __float_as_uint(-CUDART_INF_F);
                }
                // row maximum: four independent 3-input max chains
                float a0 = -CUDART_INF_F, a1 = -CUDART_INF_F, a2 = -CUDART_INF_F, a3 = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    a0 = fmax3(a0, __uint_as_float(sv[c + 0]), __uint_as_float(sv[c + 1]));
                    a1 = fmax3(a1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
                    a2 = fmax3(a2, __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
                    a3 = fmax3(a3, __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
                }
                const float mx = fmax3(fmaxf(a0, a1), a2, a3);
                if (jj == 0) {
                    m_used = mx;
                } else {
                    const bool need = (mx - m_used) * scale_log2 > 8.f;
                    if (__any_sync(0xffffffffu, need)) {
                        const float m_new = need ? mx : m_used;
                        const float alpha = exp2f((m_used - m_new) * scale_log2);
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t ov[32];
                            const uint32_t ta = tmem + lane_base + P::o_col(i) + 32 * c;
                            tmem_ld32(ta, ov);
#pragma unroll
                            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st32(ta, ov);
                        }
                        tmem_st_wait();
                        l *= alpha;
                        m_used = m_new;
                    }
                }
                // p = 2^(s*scale_log2 - m*scale_log2), two columns per packed FMA
                const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
                const uint64_t mb2 = f2_pack(-m_used * scale_log2, -m_used * scale_log2);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sc2, mb2),
                              x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
                    sv[c] = pack_bf16x2(p0, p1);
                }
                float s0, s1, s2, s3, s4, s5, s6, s7;
                f2_unpack(acc[0], s0, s1);
                f2_unpack(acc[1], s2, s3);
                f2_unpack(acc[2], s4, s5);
                f2_unpack(acc[3], s6, s7);
                l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
                tmem_st32(tmem + lane_base + P::p_col(i), sv);
                tmem_st32(tmem + lane_base + P::p_col(i) + 32, sv + 32);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(B_P_FULL + i));
                ++tiles;
                raise_flag();
            }
            if (!ok) break;
            const float lse_own = m_used * scale + logf(l);
            const float inv_l = 1.f / l;
            // A merging job reads its pieces' ready flags and log-sum-exps while its last PV
            // MMAs are still running: the weights of the parts are known when O arrives.
            constexpr int kPieceRegs = 4;
            const int n_other = merger ? U.n_slots - 1 : 0;
            const float* lse_col = st.lse_part + (int64_t)U.first_slot * kUnitRows + prow;
            float wp[kPieceRegs];
            float M = lse_own, w_own = 1.f, den = 1.f;
            if (merger) {
                bool have = true;
                if (ri.live)
                    for (int pp = 1; pp <= n_other && have; ++pp)
                        have = wait_flag(st.piece_flag + (int64_t)(U.first_slot + pp) * kUnitRows + prow, 1u, wt);
                if (__any_sync(0xffffffffu, !have)) { ok = false; break; }
                __threadfence();
                // the context part: own O and the published pieces, relative to the max M of
                // their log-sum-exps; a and den stay unnormalised until the end
#pragma unroll
                for (int pp = 0; pp < kPieceRegs; ++pp)
                    wp[pp] = (ri.live && pp < n_other) ? __ldcg(lse_col + (int64_t)(pp + 1) * kUnitRows) : -CUDART_INF_F;
#pragma unroll
                for (int pp = 0; pp < kPieceRegs; ++pp) M = fmaxf(M, wp[pp]);
                for (int pp = kPieceRegs + 1; ri.live && pp <= n_other; ++pp)
                    M = fmaxf(M, __ldcg(lse_col + (int64_t)pp * kUnitRows));
                w_own = __expf(lse_own - M);
                den = w_own;
#pragma unroll
                for (int pp = 0; pp < kPieceRegs; ++pp) {
                    wp[pp] = pp < n_other ? __expf(wp[pp] - M) : 0.f;
                    den += wp[pp];
                }
            }
            // The merge copies its rows' BeamKV keys into the freed rings (the producer holds
            // the next job's loads until the merge is done).  Keys are numbered warp-wide and
            // staged kSlots at a time.  Decode:
            // key (level j, beam bl of the warp's beams) is j * nbw + bl.  Scoring: a key is a
            // pool row, numbered from the warp's first one (its rows' segments are consecutive
            // pool rows).  The first batch's ancestry lookups are done here, before O arrives.
            constexpr int kSlotBytes = 4 * D + 16;       // a key's K row, V row, one chunk of padding
            constexpr int kArea = P::kKVTile / 2;        // each softmax warp's share of the two rings
            constexpr int kSlots = kArea / kSlotBytes;   // keys staged at a time
            const int L = st.n_levels;
            const int row_off = U.row_off;
            const int nbw = G >= 32 ? 1 : 32 / G;        // beams the warp's rows belong to
            const int bl = G >= 32 ? 0 : lane / G;       // this row's beam among them
            const int b_first = U.beam0 + i * (kTileRows / G) + (quarter * 32) / G;
            auto key_row = [&](int j, int pool) -> int64_t {
                return kScore ? ((int64_t)layer * st.rows + pool) * st.n_kv_heads + U.head
                              : (((int64_t)layer * (L - 1) + j) * st.rows + pool) * st.n_kv_heads + U.head;
            };
            int lo = 0, total = 0;
            auto key_of = [&](int p0) -> int64_t {  // the key lane l stages in batch p0 (-1: none)
                const int idx = p0 + lane;
                if (lane >= kSlots || idx >= total) return -1;
                if constexpr (kScore) {
                    return key_row(0, lo + idx);
                } else {
                    const int t = st.req_step[U.req];
                    const int j = idx / nbw, b = b_first + (idx - j * nbw);
                    if (b >= U.width || b >= st.n_beams[U.req * (L + 1) + t]) return -1;
                    return key_row(j, row_off + __ldg(st.path + ((int64_t)(t - 1) * st.rows + row_off + b) * L + j));
                }
            };
            int64_t key0 = -1;
            if (merger) {
                if constexpr (kScore) {
                    lo = (int)__reduce_min_sync(0xffffffffu, (unsigned)(ri.live ? ri.pool0 : 0x7fffffff));
                    const int hi = __reduce_max_sync(0xffffffffu, ri.live ? ri.pool0 + ri.n_priv - 1 : -1);
                    total = hi >= lo ? hi - lo + 1 : 0;
                } else {
                    total = __reduce_max_sync(0xffffffffu, ri.n_priv) * nbw;
                }
                key0 = key_of(0);
            }
            // epilogue
            if (!(ok = wait_warp(bar(B_O_FULL + i), jobs & 1, wt))) break;
            tc_fence_after();
            uint32_t ov[D];  // this piece's unnormalised O row
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_base + P::o_col(i) + 32 * c, ov + 32 * c);
            tc_fence_before();
            mbar_arrive(bar(B_O_EMPTY + i));  // TMEM O is free for the next job
            ++jobs;
            if (!merger) {
                // a later key range of a split unit: publish the normalised piece and its
                // log-sum-exp; the ready flag follows (see pend_flag).  The merger clears the
                // flag once it has read the row, so flags need no per-launch tag and a
                // captured step replays.  Only live rows are published (the merger reads no
                // other row).  Layout [slot][D/4][256 rows][4]: a warp stores 32 consecutive
                // rows' 16-byte chunks of one column group per instruction (512 bytes).
                if (ri.live) {
                    float4* dst = reinterpret_cast<float4*>(st.o_part) + (int64_t)J.slot * (D / 4) * kUnitRows + prow;
                    const uint64_t keep = l2_evict_last();
#pragma unroll
                    for (int c = 0; c < D / 4; ++c)
                        st_keep(dst + (int64_t)c * kUnitRows,
                                make_float4(__uint_as_float(ov[4 * c]) * inv_l, __uint_as_float(ov[4 * c + 1]) * inv_l,
                                           __uint_as_float(ov[4 * c + 2]) * inv_l, __uint_as_float(ov[4 * c + 3]) * inv_l),
                                keep);
                    __stcg(st.lse_part + (int64_t)J.slot * kUnitRows + prow, lse_own);
                    pend_flag = st.piece_flag + (int64_t)J.slot * kUnitRows + prow;
                }
                continue;
            }
            // The first key range merges, by a log-sum-exp combine: its own O (registers),
            // the other pieces (finished earlier, at the start of their CTAs' ranges) and the
            // beam part -- the row's private keys (decode: the t BeamKV tokens on its beam's
            // ancestry path; scoring: its own candidate up to itself), folded in one key at a
            // time with an online max.  Each thread works on its own row.  The K and V rings are
            // free once the job's last key tile's MMAs have completed (the producer holds the
            // next job's loads until this merge is done): each warp copies the private keys' K
            // and V rows of its 32 rows there (bulk copies, 31 key slots at a time), reads q
            // from the job's Q tile, and finally passes its bf16 output rows through the same
            // space, one bulk store per row.
            float* a = reinterpret_cast<float*>(ov);  // the row accumulates in place of O
            {
                const float c_own = ri.live ? w_own * inv_l : 0.f;
#pragma unroll
                for (int c = 0; c < D; ++c) a[c] = ri.live ? __uint_as_float(ov[c]) * c_own : 0.f;
            }
            // ---- the beam part's set-up: the row's private keys are folded in one at a time
            constexpr int kKC = D / 8;                   // 16-byte chunks of a bf16 row
            uint8_t* area = smem + P::kKOff + (warp - 4) * kArea;
            const uint8_t* qs = smem + P::kQOff + i * P::kQTile + row_t * 128;  // this row in the Q tile
            // fold one key (its K and V rows) into (M, den, a)
            auto fold = [&](const uint4* kp, const uint4* vp) {
                float d0 = 0.f, d1 = 0.f;
#pragma unroll 4
                for (int c = 0; c < kKC; ++c) {
                    const uint4 qa = *reinterpret_cast<const uint4*>(qs + (c >> 3) * P::kBoxBytes +
                                                                     (((c & 7) ^ (row_t & 7)) << 4));
                    const uint4 ka = kp[c];
                    const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w}, kw[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        d0 = fmaf(bf_lo(qw[h2]), bf_lo(kw[h2]), d0);
                        d1 = fmaf(bf_hi(qw[h2]), bf_hi(kw[h2]), d1);
                    }
                }
                const float s = (d0 + d1) * scale;
                if (s > M) {
                    const float r = __expf(M - s);
                    den *= r;
#pragma unroll
                    for (int c = 0; c < D; ++c) a[c] *= r;
                    M = s;
                }
                const float pw = __expf(s - M);
                den += pw;
#pragma unroll
                for (int c = 0; c < kKC; ++c) {
                    const uint4 v = vp[c];
                    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        a[8 * c + 2 * h2] = fmaf(pw, bf_lo(vw[h2]), a[8 * c + 2 * h2]);
                        a[8 * c + 2 * h2 + 1] = fmaf(pw, bf_hi(vw[h2]), a[8 * c + 2 * h2 + 1]);
                    }
                }
            };
            const uint32_t bbar = bar(B_BEAM + warp - 4);
            const uint32_t area_s = smem_u32(area);
            auto copy = [&](int64_t key) {  // lane l stages one key (or none: key < 0) in slot l
                const unsigned copies = __ballot_sync(0xffffffffu, key >= 0);
                if (lane == 0) mbar_expect_tx(bbar, (uint32_t)__popc(copies) * (uint32_t)(4 * D));
                __syncwarp();
                if (key >= 0) {
                    bulk_load(area_s + lane * kSlotBytes, st.beam_k + key * D, 2 * D, bbar);
                    bulk_load(area_s + lane * kSlotBytes + 2 * D, st.beam_v + key * D, 2 * D, bbar);
                }
            };
            {
                // Query tile 0's warps stage in the K ring, free once the last key tile's S
                // MMAs (both tiles') have completed; tile 1's warps in the V ring, free once the
                // last PV MMAs have (its own is done: O arrived).  No more tiles are loaded.
                // The first batch of copies goes out before the pieces are read, so that the
                // two overlap.
                const uint32_t kl = ktiles - 1;  // the CTA's last key tile
                if (!(ok = wait_warp(bar((i == 0 ? B_K_EMPTY : B_V_EMPTY) + (kl & 1)), (kl >> 1) & 1, wt))) break;
                if (total > 0) copy(key0);
            }
            // ---- the published pieces
#pragma unroll 1
            for (int pp = 1; ri.live && pp <= n_other; ++pp) {
                float w = 0.f;
#pragma unroll
                for (int k = 0; k < kPieceRegs; ++k) w = (k == pp - 1) ? wp[k] : w;
                if (pp > kPieceRegs) {
                    w = __expf(__ldcg(lse_col + (int64_t)pp * kUnitRows) - M);
                    den += w;
                }
                const float4* src =
                    reinterpret_cast<const float4*>(st.o_part) + (int64_t)(U.first_slot + pp) * (D / 4) * kUnitRows + prow;
                constexpr int kBatch = D / 8;  // chunks per batch of loads
#pragma unroll
                for (int c0 = 0; c0 < D / 4; c0 += kBatch) {
                    float4 x[kBatch];
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) x[u] = __ldcg(src + (int64_t)(c0 + u) * kUnitRows);
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        float* ac = a + 4 * (c0 + u);
                        ac[0] = fmaf(w, x[u].x, ac[0]);
                        ac[1] = fmaf(w, x[u].y, ac[1]);
                        ac[2] = fmaf(w, x[u].z, ac[2]);
                        ac[3] = fmaf(w, x[u].w, ac[3]);
                    }
                }
                st.piece_flag[(int64_t)(U.first_slot + pp) * kUnitRows + prow] = 0u;  // consumed
            }
            // ---- the beam part, one key at a time
            {
#pragma unroll 1
                for (int p0 = 0; p0 < total; p0 += kSlots) {
                    if (p0 > 0) copy(key_of(p0));
                    const uint32_t par = bcnt & 1;
                    ++bcnt;
                    if (!(ok = wait_warp(bbar, par, wt))) {
                        wait_drain(bbar, par);  // no copy may land after the CTA has gone
                        break;
                    }
                    for (int j = 0; j < ri.n_priv; ++j) {
                        const int kidx = kScore ? ri.pool0 + j - lo : j * nbw + bl;
                        if (kidx < p0 || kidx >= p0 + kSlots) continue;
                        const uint8_t* sl = area + (kidx - p0) * kSlotBytes;
                        fold(reinterpret_cast<const uint4*>(sl), reinterpret_cast<const uint4*>(sl + 2 * D));
                    }
                    __syncwarp();  // every row is done with these slots before they are refilled
                }
                if (!ok) break;
            }
            {
                // dead beams come out as exact zeros: none of their (unwritten) inputs is used
                const float inv_den = ri.live ? 1.f / den : 0.f;
#pragma unroll
                for (int c = 0; c < D; ++c) a[c] = ri.live ? a[c] * inv_den : 0.f;
            }
            // ---- bf16 output rows (rows beyond the request are another request's: not written)
            constexpr int kChunks = D * 2 / 16;  // 16-byte chunks per bf16 row
            {
                // each row through the warp's own share of the rings (free again; rows padded by
                // one chunk against bank conflicts), then one bulk store per row
                constexpr int kRowStride = 2 * D + 16;
                uint8_t* stg = area + lane * kRowStride;
#pragma unroll
                for (int c = 0; c < kChunks; ++c)
                    *reinterpret_cast<uint4*>(stg + c * 16) =
                        make_uint4(pack_bf16x2(a[8 * c], a[8 * c + 1]), pack_bf16x2(a[8 * c + 2], a[8 * c + 3]),
                                   pack_bf16x2(a[8 * c + 4], a[8 * c + 5]), pack_bf16x2(a[8 * c + 6], a[8 * c + 7]));
                fence_proxy_async_smem();  // the row's generic writes, then the bulk copy reads them
                if (ri.row_ok) bulk_store(out + ri.orow_idx * D, smem_u32(stg), 2 * D);
                bulk_commit_and_wait_read();  // the shared rows have been read
            }
            // The producer may refill the rings and the Q tile.  Each merging warp arrives once
            // its rows are done; with one query tile the first warpgroup's warps arrive for the
            // second as well (a warpgroup without rows must not arrive on its own: it would run
            // ahead to the next job's phase).
            __syncwarp();
            if (lane == 0 && jb < jr.y - 1) mbar_arrive_n(bar(B_MERGED), U.nqt == 1 ? 2u : 1u);
        }
        raise_flag();
    }
    tc_fence_before();
    named_bar_sync(1);
    named_bar_sync(2);
}

}  // namespace

cudaError_t ctx_attn_smem_bytes(int head_dim, size_t* bytes) {
    if (head_dim == 128) *bytes = Plan<128>::kBytes;
    else if (head_dim == 64) *bytes = Plan<64>::kBytes;
    else return cudaErrorInvalidValue;
    return cudaSuccess;
}

template <int D, bool kScore>
cudaError_t launch_ctx_attn_d(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q,
                              uint16_t* out, float scale_log2, float scale, int64_t wait_limit_ns, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_ctx_attn<D, kScore>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Plan<D>::kBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    // cooperative: every CTA is resident at once, so a merging CTA may wait for the
    // flags of the pieces other CTAs publish
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(st.n_cta);
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = Plan<D>::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_ctx_attn<D, kScore>, qmap, st, layer, q, out, scale_log2, scale,
                              wait_limit_ns);
}

template <bool kScore>
cudaError_t launch_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                        int64_t wait_limit_ns, cudaStream_t s) {
    const float scale = 1.f / sqrtf((float)st.head_dim);
    const float scale_log2 = scale * 1.4426950408889634f;
    if (st.head_dim != 128 && st.head_dim != 64) return cudaErrorInvalidValue;
    if (st.head_dim == 128)
        return launch_ctx_attn_d<128, kScore>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
    return launch_ctx_attn_d<64, kScore>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
}

cudaError_t launch_ctx_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q,
                            uint16_t* out, int64_t wait_limit_ns, cudaStream_t s) {
    return launch_attn<false>(st, qmap, layer, q, out, wait_limit_ns, s);
}

cudaError_t launch_score_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q,
                              uint16_t* out, int64_t wait_limit_ns, cudaStream_t s) {
    return launch_attn<true>(st, qmap, layer, q, out, wait_limit_ns, s);
}

}  // namespace grb
