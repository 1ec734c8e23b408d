// Device code shared by the two decode-attention kernels of libgrbeam (k_attn.cu):
// PTX wrappers for mbarriers, TMA and tcgen05, the bounded waits, the view of one
// query row, and the end of a job for one row (the piece it publishes, or the merge
// of the pieces, the BeamKV part and the bf16 output).
//
// Every wait is bounded: past the limit the waiter sets GR_ERR_TIMEOUT in the
// status word and the kernel drains what it issued, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "grbeam_internal.h"

namespace grb {
namespace attn {

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
// 16-byte asynchronous copy global -> shared (through L2), completed by cp_async_wait_all
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// the thread's copies have landed (they read valid global memory, so this always ends)
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
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

// one thread waits for a flag written by another CTA of the same (cooperative) launch; the
// acquire load orders the thread's later reads of what the writer published before it
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t value, const Waiter w) {
    if (ld_acquire_gpu(flag) == value) return true;
    const uint64_t t0 = global_timer();
    uint32_t spins = 0;
    while (ld_acquire_gpu(flag) != value) {
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
// the end of a job for one query row
// ---------------------------------------------------------------------------
// A merging warp stages its rows' private keys (BeamKV K and V rows) in its staging area,
// kEpiSlots keys at a time: slot k holds a key's K row, its V row and one 16-byte chunk of
// padding (against bank conflicts when the lanes read different slots).
template <int D>
struct EpiArea {
    static constexpr int kSlotBytes = 4 * D + 16;
    static constexpr int kSlots = 32;
    static constexpr int kBytes = kSlots * kSlotBytes;  // a warp's staging area
};

// The private keys a merging warp folds in, located when its job starts: the lookups along the
// beams' ancestry (dependent global loads) then overlap the job's key tiles instead of
// delaying its end.  Keys are numbered warp-wide.  Decode: key (level j, beam bl of the warp's
// beams) is j * nbw + bl.  Scoring: a key is a pool row, numbered from the warp's first one
// (its rows' segments are consecutive pool rows).  Lane l stages key p0 + l of a batch.
struct EpiKeys {
    int lo;         // scoring: the warp's first pool row
    int total;      // keys the warp stages (0: none, or the job does not merge)
    int64_t key0;   // the BeamKV / pool row lane l stages in the first batch (-1: none)
    int64_t key1;   // in the second batch
};

template <bool kScore>
__device__ __forceinline__ int64_t epi_key_row(const GrState& st, const GrAttnUnit& U, int layer, int lo, int total,
                                               int b_first, int G, int lane, int p0) {
    const int idx = p0 + lane;
    if (idx >= total) return -1;
    const int L = st.n_levels;
    if constexpr (kScore) {
        return ((int64_t)layer * st.rows + lo + idx) * st.n_kv_heads + U.head;
    } else {
        const int nbw = G >= 32 ? 1 : 32 / G;  // beams the warp's rows belong to
        const int t = st.req_step[U.req];
        const int j = idx / nbw, b = b_first + (idx - j * nbw);
        if (b >= U.width || b >= st.n_beams[U.req * (L + 1) + t]) return -1;
        const int pool = U.row_off + __ldg(st.path + ((int64_t)(t - 1) * st.rows + U.row_off + b) * L + j);
        return (((int64_t)layer * (L - 1) + j) * st.rows + pool) * st.n_kv_heads + U.head;
    }
}

// b_first: the beam of the warp's first row (decode)
template <int D, bool kScore>
__device__ __forceinline__ EpiKeys epi_keys(const GrState& st, const GrAttnUnit& U, const GrAttnJob& J,
                                            const RowInfo& ri, int layer, int b_first, int G, int lane) {
    EpiKeys k{0, 0, -1, -1};
    if (J.slot != U.first_slot) return k;  // a later key range publishes; it stages nothing
    if constexpr (kScore) {
        k.lo = (int)__reduce_min_sync(0xffffffffu, (unsigned)(ri.live ? ri.pool0 : 0x7fffffff));
        const int hi = __reduce_max_sync(0xffffffffu, ri.live ? ri.pool0 + ri.n_priv - 1 : -1);
        k.total = hi >= k.lo ? hi - k.lo + 1 : 0;
    } else {
        const int nbw = G >= 32 ? 1 : 32 / G;
        k.total = __reduce_max_sync(0xffffffffu, ri.n_priv) * nbw;
    }
    constexpr int kS = EpiArea<D>::kSlots;
    k.key0 = epi_key_row<kScore>(st, U, layer, k.lo, k.total, b_first, G, lane, 0);
    if (k.total > kS) k.key1 = epi_key_row<kScore>(st, U, layer, k.lo, k.total, b_first, G, lane, kS);
    return k;
}

// One row's end of a job (each softmax thread of the kernel works on its own row, all 32
// lanes of a warp together): the row's unnormalised O over the job's key tiles, its running
// max m_used (in score units) and sum l are
//   - published as a normalised fp32 piece + log-sum-exp when the job is a later key range of
//     a unit cut over several jobs (the ready flag is raised by the caller, see pend_flag);
//   - merged otherwise (the unit's first range): the context part from its own O and the
//     published pieces by a log-sum-exp combine, then the row's private keys folded in one at
//     a time (decode: the t BeamKV keys on its beam's ancestry path; scoring: its own
//     candidate up to itself), then the bf16 output row.
// ek are the warp's keys (epi_keys at the job's start); qs is the row in the job's Q tile
// (128-byte rows, 64-dimension boxes of 128 rows), area the warp's EpiArea<D>::kBytes of
// staging space, free once wait_area() returns true.  wait_o(ov) waits for the job's last PV,
// reads the row's O into ov and frees the TMEM accumulator; merged() runs once a merging warp
// is done with area and the Q tile.  Returns false when a wait gave up.
template <int D, bool kScore, class WaitO, class WaitArea, class Merged>
__device__ __forceinline__ bool job_epilogue(const GrState& st, const GrAttnUnit& U, const GrAttnJob& J,
                                             const RowInfo& ri, const EpiKeys& ek, int row_t, int lane, int b_first,
                                             int prow, int layer, float scale, float m_used, float l,
                                             const uint8_t* qs, uint8_t* area, uint32_t*& pend_flag, uint16_t* __restrict__ out, const Waiter& wt,
                                             WaitO&& wait_o, WaitArea&& wait_area, Merged&& merged) {
    constexpr int kQBox = 128 * 128;  // bytes between the 64-dimension boxes of a query tile
    constexpr int kSlotBytes = EpiArea<D>::kSlotBytes;
    constexpr int kSlots = EpiArea<D>::kSlots;
    const int G = st.n_q_heads / st.n_kv_heads;
    const bool merger = (J.slot == U.first_slot);
    const float lse_own = m_used * scale + logf(l);
    const float inv_l = 1.f / l;
    const int nbw = G >= 32 ? 1 : 32 / G;  // beams the warp's rows belong to
    const int bl = G >= 32 ? 0 : lane / G;  // this row's beam among them
    const uint32_t area_s = smem_u32(area);
    // Stage a batch: lane l's key (or none: key < 0) into slot l.  The warp copies one key per
    // instruction (two for D = 64), each lane 16 bytes of its K or V row, so the reads of a key
    // are contiguous.
    auto stage = [&](int64_t key) {
        constexpr int kCh = D / 4;          // 16-byte chunks of a key's K and V rows
        constexpr int kPer = 32 / kCh;      // keys per instruction
        const int sub = lane / kCh, ch = lane % kCh;
        const uint16_t* src = (ch < D / 8 ? st.beam_k : st.beam_v) + (ch % (D / 8)) * 8;
#pragma unroll 4
        for (int k = 0; k < 32; k += kPer) {
            const int64_t kk = __shfl_sync(0xffffffffu, key, k + sub);
            if (kk >= 0) cp_async16(area_s + (k + sub) * kSlotBytes + ch * 16, src + kk * D);
        }
        cp_async_commit();
    };
    // A merging warp's first batch of keys goes out as soon as the staging area is free (the
    // job's last key tile has been used), before its pieces and its O: the copies overlap them.
    // A warp that gives up waits for its copies: none may land after the CTA has gone.
    if (merger && ek.total > 0) {
        if (!wait_area()) return false;
        stage(ek.key0);
    }
    auto give_up = [&]() {
        cp_async_wait_all();
        return false;
    };
    // A merging job reads its pieces' ready flags and log-sum-exps while its last PV MMAs are
    // still running: the weights of the parts are known when O arrives.
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
        if (__any_sync(0xffffffffu, !have)) return give_up();
        // the context part: own O and the published pieces, relative to the max M of their
        // log-sum-exps; a and den stay unnormalised until the end
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
    uint32_t ov[D];  // this piece's unnormalised O row
    if (!wait_o(ov)) return give_up();
    if (!merger) {
        // a later key range of a split unit: publish the normalised piece and its log-sum-exp;
        // the ready flag follows (see pend_flag).  The merger clears the flag once it has read
        // the row, so flags need no per-launch tag and a captured step replays.  Only live rows
        // are published (the merger reads no other row).  Layout [slot][D/4][256 rows][4]: a
        // warp stores 32 consecutive rows' 16-byte chunks of one column group per instruction.
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
        return true;
    }
    // The first key range merges, by a log-sum-exp combine: its own O (registers), the other
    // pieces (finished earlier, at the start of their CTAs' ranges) and the beam part -- the
    // row's private keys, folded in one key at a time with an online max, from the staging
    // area; q comes from the job's Q tile.
    float* a = reinterpret_cast<float*>(ov);  // the row accumulates in place of O
    {
        const float c_own = ri.live ? w_own * inv_l : 0.f;
#pragma unroll
        for (int c = 0; c < D; ++c) a[c] = ri.live ? __uint_as_float(ov[c]) * c_own : 0.f;
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
    constexpr int kKC = D / 8;  // 16-byte chunks of a bf16 row
    // fold one key (its K and V rows) into (M, den, a)
    auto fold = [&](const uint4* kp, const uint4* vp) {
        float d0 = 0.f, d1 = 0.f;
#pragma unroll 4
        for (int c = 0; c < kKC; ++c) {
            const uint4 qa = *reinterpret_cast<const uint4*>(qs + (c >> 3) * kQBox + (((c & 7) ^ (row_t & 7)) << 4));
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
#pragma unroll 1
    for (int p0 = 0; p0 < ek.total; p0 += kSlots) {
        if (p0 > 0) stage(p0 == kSlots ? ek.key1 : epi_key_row<kScore>(st, U, layer, ek.lo, ek.total, b_first, G, lane, p0));
        cp_async_wait_all();
        __syncwarp();  // every lane's copies have landed
        for (int j = 0; j < ri.n_priv; ++j) {
            const int kidx = kScore ? ri.pool0 + j - ek.lo : j * nbw + bl;
            if (kidx < p0 || kidx >= p0 + kSlots) continue;
            const uint8_t* sl = area + (kidx - p0) * kSlotBytes;
            fold(reinterpret_cast<const uint4*>(sl), reinterpret_cast<const uint4*>(sl + 2 * D));
        }
        __syncwarp();  // every row is done with these slots before they are refilled
    }
    // ---- the bf16 output rows (rows beyond the request are another request's: not written);
    // dead beams come out as exact zeros (none of their unwritten inputs is used).  The rows
    // pass through the staging area (one padding chunk per row against bank conflicts) so that
    // each store instruction writes whole rows: lanes 0..kCpr-1 one row, the next kCpr lanes
    // the next, and so on.
    const float inv_den = ri.live ? 1.f / den : 0.f;
    constexpr int kRowStride = 2 * D + 16;
    constexpr int kCpr = D / 8;             // 16-byte chunks per bf16 row
    constexpr int kRowsPer = 32 / kCpr;     // rows per store instruction
    {
        uint8_t* stg = area + lane * kRowStride;
#pragma unroll
        for (int c = 0; c < kCpr; ++c)
            *reinterpret_cast<uint4*>(stg + c * 16) =
                make_uint4(pack_bf16x2(a[8 * c] * inv_den, a[8 * c + 1] * inv_den),
                           pack_bf16x2(a[8 * c + 2] * inv_den, a[8 * c + 3] * inv_den),
                           pack_bf16x2(a[8 * c + 4] * inv_den, a[8 * c + 5] * inv_den),
                           pack_bf16x2(a[8 * c + 6] * inv_den, a[8 * c + 7] * inv_den));
    }
    const int64_t orow = ri.row_ok ? ri.orow_idx : -1;
    __syncwarp();
    {
        const int sub = lane / kCpr, ch = lane % kCpr;
#pragma unroll 4
        for (int r0 = 0; r0 < 32; r0 += kRowsPer) {
            const int r = r0 + sub;
            const int64_t o = __shfl_sync(0xffffffffu, orow, r);
            const uint4 v = *reinterpret_cast<const uint4*>(area + r * kRowStride + ch * 16);
            if (o >= 0) reinterpret_cast<uint4*>(out + o * D)[ch] = v;
        }
    }
    __syncwarp();
    // the staging area and the Q tile are no longer needed: the next job's loads may start
    merged();
    return true;
}

}  // namespace attn
}  // namespace grb
