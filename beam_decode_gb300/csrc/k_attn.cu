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
//   warp 1     MMA issuer (one thread): S_i = Q_i K^T into TMEM (M=128, N=128,
//              K=16 per instruction), O_i += P_i V with P_i read from TMEM.
//   warp 2     TMEM allocation (512 columns: S0, S1, O0, O1).
//   warps 4-7  softmax of query tile 0; warps 8-11 softmax of query tile 1:
//              one thread per row (TMEM lane), online max/sum with a lazy
//              rescale of O (only when the running max grows by more than
//              2^8), P written back to TMEM as bf16 in place of S.
//   The two query tiles ping-pong: while one warpgroup exponentiates, the
//   tensor core runs the other tile's MMAs.  Each job writes its normalised
//   partial O (fp32) and log-sum-exp to a slot of the workspace.
// Units of one (request, KV head) are scheduled on neighbouring CTAs so the
// second read of a K/V tile is served by L2; each context byte comes from HBM
// once per request.
//
// k_beam_attn: one warp per (row, KV head).  The t BeamKV keys of the beam are
// found through its ancestry row (levels 0..t-1) and read with vector loads;
// scores are warp reductions; the context partials and the beam part are
// merged with a log-sum-exp combine and written as bf16.
//
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
    static constexpr int kBytes = kBarOff + 256 + 1024;  // barriers, TMEM address, abort flag, alignment
    // TMEM columns
    static constexpr int kTmemCols = 512;
    static __device__ __forceinline__ int s_col(int i) { return i * 128; }
    static __device__ __forceinline__ int p_col(int i) { return i * 128; }  // bf16 P overwrites S in place
    static __device__ __forceinline__ int o_col(int i) { return 256 + i * D; }
};

enum Bar {
    B_Q_FULL = 0, B_Q_EMPTY = 1, B_K_FULL = 2, B_K_EMPTY = 4, B_V_FULL = 6, B_V_EMPTY = 8,
    B_S_FULL = 10, B_P_FULL = 12, B_O_FULL = 14, B_O_EMPTY = 16, B_DRAIN = 18, B_COUNT = 19
};

constexpr int kAttnThreads = 384;

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
k_ctx_attn(const __grid_constant__ CUtensorMap qmap, GrState st, int layer, float scale_log2, float scale,
           int64_t wait_limit_ns) {
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
        mbar_init(bar(B_DRAIN), 1);
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
        uint32_t p_kit = 0, p_vit = 0, p_qcnt = 0;
    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                const GrAttnJob J = st.jobs[jb];
                const GrAttnUnit U = st.units[J.unit];
                const GrReqDev& R = st.req[U.req];
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
                                    U.head * G, R.row_off + U.beam0 + i * (kTileRows / G));
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
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            bool mma_issued = false;
            constexpr uint32_t idesc_s = idesc_bf16(128, kTileKeys, false);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, true);
            uint32_t kit = 0, vit = 0, qcnt = 0;
            uint32_t tiles[2] = {0, 0}, jobs_i[2] = {0, 0};
            bool ok = true;
            auto issue_s = [&](int i, int ks) {
                const uint32_t d = tmem + P::s_col(i);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * P::kBoxBytes + (kk & 3) * 32;
                    const uint64_t a = smem_desc(sb + P::kQOff + i * P::kQTile + off, 16, 1024);
                    const uint64_t b = smem_desc(sb + P::kKOff + ks * P::kKVTile + off, 16, 1024);
                    mma_ss(d, a, b, idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int i, int vs, bool acc) {
                const uint32_t d = tmem + P::o_col(i);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                    const uint32_t a = tmem + P::p_col(i) + kk * 8;
                    const uint64_t b = smem_desc(sb + P::kVOff + vs * P::kKVTile + kk * 16 * 128, P::kBoxBytes, 1024);
                    mma_ts(d, a, b, idesc_o, (acc || kk > 0) ? 1u : 0u);
                }
            };
            for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                const GrAttnJob J = st.jobs[jb];
                const GrAttnUnit U = st.units[J.unit];
                const int nqt = U.nqt;
                const int n = J.t1 - J.t0;
                if (!(ok = wait1(bar(B_Q_FULL), qcnt & 1, wt))) break;
                ++qcnt;
                int ks = kit & 1;
                if (!(ok = wait1(bar(B_K_FULL + ks), (kit >> 1) & 1, wt))) break;
                tc_fence_after();
                for (int i = 0; i < nqt; ++i) {
                    issue_s(i, ks);
                    tc_commit(bar(B_S_FULL + i));
                }
                mma_issued = true;
                tc_commit(bar(B_K_EMPTY + ks));
                ++kit;
                if (n == 1) tc_commit(bar(B_Q_EMPTY));
                for (int jj = 0; jj < n && ok; ++jj) {
                    const int vs = vit & 1;
                    if (!(ok = wait1(bar(B_V_FULL + vs), (vit >> 1) & 1, wt))) break;
                    for (int i = 0; i < nqt; ++i) {
                        if (!(ok = wait1(bar(B_P_FULL + i), tiles[i] & 1, wt))) break;
                        tc_fence_after();
                        if (jj == 0 && jobs_i[i] > 0) {
                            if (!(ok = wait1(bar(B_O_EMPTY + i), (jobs_i[i] - 1) & 1, wt))) break;
                            tc_fence_after();
                        }
                        issue_pv(i, vs, jj > 0);
                        ++tiles[i];
                        if (jj == n - 1) {
                            tc_commit(bar(B_O_FULL + i));
                        } else {
                            if (i == 0) {
                                ks = kit & 1;
                                if (!(ok = wait1(bar(B_K_FULL + ks), (kit >> 1) & 1, wt))) break;
                                tc_fence_after();
                            }
                            issue_s(i, ks);
                            tc_commit(bar(B_S_FULL + i));
                            if (i == nqt - 1) {
                                tc_commit(bar(B_K_EMPTY + ks));
                                ++kit;
                                if (jj + 1 == n - 1) tc_commit(bar(B_Q_EMPTY));
                            }
                        }
                    }
                    if (!ok) break;
                    tc_commit(bar(B_V_EMPTY + vs));
                    ++vit;
                }
                for (int i = 0; i < nqt; ++i) ++jobs_i[i];
            }
            // all issued tensor-core work (and its commits) completes before TMEM is freed
            if (mma_issued) {
                tc_commit(bar(B_DRAIN));
                wait_drain(bar(B_DRAIN), 0);
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
        const int i = (warp - 4) >> 2;          // query tile of this warpgroup
        const int quarter = warp & 3;           // TMEM lane quarter
        const int row_t = quarter * 32 + lane;  // row within the tile
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t tiles = 0, jobs = 0;
        bool ok = true;
        for (int jb = jr.x; jb < jr.y && ok; ++jb) {
            const GrAttnJob J = st.jobs[jb];
            const GrAttnUnit U = st.units[J.unit];
            if (i >= U.nqt) continue;
            const int ctx_len = st.req[U.req].ctx_len;
            const int n = J.t1 - J.t0;
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
            }
            if (!ok) break;
            // epilogue: normalised partial O and its log-sum-exp
            if (!(ok = wait_warp(bar(B_O_FULL + i), jobs & 1, wt))) break;
            tc_fence_after();
            const float inv_l = 1.f / l;
            const int prow = i * kTileRows + row_t;
            float* orow = st.o_part + ((int64_t)J.slot * kUnitRows + prow) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_base + P::o_col(i) + 32 * c, ov);
                float4* dst = reinterpret_cast<float4*>(orow + 32 * c);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    dst[e] = make_float4(__uint_as_float(ov[4 * e]) * inv_l, __uint_as_float(ov[4 * e + 1]) * inv_l,
                                         __uint_as_float(ov[4 * e + 2]) * inv_l, __uint_as_float(ov[4 * e + 3]) * inv_l);
            }
            st.lse_part[(int64_t)J.slot * kUnitRows + prow] = m_used * scale + logf(l);
            tc_fence_before();
            mbar_arrive(bar(B_O_EMPTY + i));
            ++jobs;
        }
    }
    tc_fence_before();
    named_bar_sync(1);
    named_bar_sync(2);
}

// ---------------------------------------------------------------------------
// K2: BeamKV part + log-sum-exp combine with the context partials
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

template <int D, int G, int TMAX>
__global__ void __launch_bounds__(256) k_beam_attn(GrState st, int t, int layer, const uint16_t* __restrict__ q,
                                                   uint16_t* __restrict__ out, float scale) {
    constexpr int E = D / 32;  // elements per lane
    constexpr int kPieces = 3;  // context pieces held in registers (more are streamed)
    const int gw = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int Hkv = st.n_kv_heads, Hq = st.n_q_heads, L = st.n_levels;
    if (gw >= st.rows * Hkv) return;
    const int row = gw / Hkv, h = gw % Hkv;
    // round 1: everything that depends only on (row, head)
    const int4 meta = st.combine_meta[gw];  // first slot, slots << 16 | local row, beam, request width
    const int r = st.row_req[row];
    const uint16_t* qp = q + ((int64_t)row * Hq + h * G) * D + lane * E;
    uint16_t* o = out + ((int64_t)row * Hq + h * G) * D + lane * E;
    float qv[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if constexpr (E == 4) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(qp + g * D));
            qv[g][0] = __uint_as_float(u.x << 16); qv[g][1] = __uint_as_float(u.x & 0xFFFF0000u);
            qv[g][2] = __uint_as_float(u.y << 16); qv[g][3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
            const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(qp + g * D));
            qv[g][0] = __uint_as_float(u << 16); qv[g][1] = __uint_as_float(u & 0xFFFF0000u);
        }
    }
    // ancestry row: only written for live beams, so every slot is clamped into the
    // request's rows before it forms an address (a dead row's result is discarded)
    const int32_t* path = st.path + ((int64_t)(t - 1) * st.rows + row) * L;
    const int width = meta.w;
    int slot[TMAX];
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
        const int v = (j < t) ? __ldg(path + j) : 0;
        slot[j] = ((unsigned)v < (unsigned)width) ? v : 0;
    }
    // round 2: live width, context pieces, BeamKV rows
    const int n_live = st.n_beams[r * (L + 1) + t];
    const int b = meta.z, lr = meta.y & 0xFFFF, first = meta.x, n_slots = meta.y >> 16;
    float plse[kPieces][G], pv[kPieces][G][E];
#pragma unroll
    for (int p = 0; p < kPieces; ++p) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (p < n_slots) {
                const int64_t pr = (int64_t)(first + p) * kUnitRows + lr + g;
                plse[p][g] = __ldg(st.lse_part + pr);
                const float* op = st.o_part + pr * D + lane * E;
                if constexpr (E == 4) {
                    const float4 v4 = __ldg(reinterpret_cast<const float4*>(op));
                    pv[p][g][0] = v4.x; pv[p][g][1] = v4.y; pv[p][g][2] = v4.z; pv[p][g][3] = v4.w;
                } else {
                    const float2 v2 = __ldg(reinterpret_cast<const float2*>(op));
                    pv[p][g][0] = v2.x; pv[p][g][1] = v2.y;
                }
            } else {
                plse[p][g] = -CUDART_INF_F;
#pragma unroll
                for (int e = 0; e < E; ++e) pv[p][g][e] = 0.f;
            }
        }
    }
    float kf[TMAX][E], vf[TMAX][E];
#pragma unroll
    for (int j = 0; j < TMAX; ++j) {
        if (j < t) {
            const int64_t kv = (((int64_t)layer * (L - 1) + j) * st.rows + (row - b) + slot[j]) * Hkv + h;
            const uint16_t* kp = st.beam_k + kv * D + lane * E;
            const uint16_t* vp = st.beam_v + kv * D + lane * E;
            if constexpr (E == 4) {
                const uint2 ku = __ldg(reinterpret_cast<const uint2*>(kp)), vu = __ldg(reinterpret_cast<const uint2*>(vp));
                kf[j][0] = __uint_as_float(ku.x << 16); kf[j][1] = __uint_as_float(ku.x & 0xFFFF0000u);
                kf[j][2] = __uint_as_float(ku.y << 16); kf[j][3] = __uint_as_float(ku.y & 0xFFFF0000u);
                vf[j][0] = __uint_as_float(vu.x << 16); vf[j][1] = __uint_as_float(vu.x & 0xFFFF0000u);
                vf[j][2] = __uint_as_float(vu.y << 16); vf[j][3] = __uint_as_float(vu.y & 0xFFFF0000u);
            } else {
                const uint32_t ku = __ldg(reinterpret_cast<const uint32_t*>(kp));
                const uint32_t vu = __ldg(reinterpret_cast<const uint32_t*>(vp));
                kf[j][0] = __uint_as_float(ku << 16); kf[j][1] = __uint_as_float(ku & 0xFFFF0000u);
                vf[j][0] = __uint_as_float(vu << 16); vf[j][1] = __uint_as_float(vu & 0xFFFF0000u);
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) { kf[j][e] = 0.f; vf[j][e] = 0.f; }
        }
    }
    if (t >= st.req[r].n_levels || b >= n_live) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < E; e += 2) *reinterpret_cast<uint32_t*>(o + g * D + e) = 0u;
        return;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        // beam scores
        float sj[TMAX];
        float M = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < TMAX; ++j) {
            float d = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) d = fmaf(qv[g][e], kf[j][e], d);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            sj[j] = (j < t) ? d * scale : -CUDART_INF_F;
            M = fmaxf(M, sj[j]);
        }
#pragma unroll
        for (int p = 0; p < kPieces; ++p) M = fmaxf(M, plse[p][g]);
        for (int p = kPieces; p < n_slots; ++p)
            M = fmaxf(M, __ldg(st.lse_part + (int64_t)(first + p) * kUnitRows + lr + g));
        float acc[E], den = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
        for (int p = 0; p < kPieces; ++p) {
            const float w = __expf(plse[p][g] - M);  // 0 for absent pieces
            den += w;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w, pv[p][g][e], acc[e]);
        }
        for (int p = kPieces; p < n_slots; ++p) {  // rare: units cut into more than kPieces
            const int64_t pr = (int64_t)(first + p) * kUnitRows + lr + g;
            const float w = __expf(__ldg(st.lse_part + pr) - M);
            den += w;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w, __ldg(st.o_part + pr * D + lane * E + e), acc[e]);
        }
#pragma unroll
        for (int j = 0; j < TMAX; ++j) {
            const float w = __expf(sj[j] - M);  // 0 beyond level t
            den += w;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = fmaf(w, vf[j][e], acc[e]);
        }
        const float inv = 1.f / den;
#pragma unroll
        for (int e = 0; e < E; e += 2)
            *reinterpret_cast<__nv_bfloat162*>(o + g * D + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
    }
}

template <int D, int TMAX>
cudaError_t launch_beam_attn_t(const GrState& st, int t, int layer, const uint16_t* q, uint16_t* out,
                               cudaStream_t s, int blocks, float scale) {
    switch (st.n_q_heads / st.n_kv_heads) {
        case 1: k_beam_attn<D, 1, TMAX><<<blocks, 256, 0, s>>>(st, t, layer, q, out, scale); break;
        case 2: k_beam_attn<D, 2, TMAX><<<blocks, 256, 0, s>>>(st, t, layer, q, out, scale); break;
        case 4: k_beam_attn<D, 4, TMAX><<<blocks, 256, 0, s>>>(st, t, layer, q, out, scale); break;
        case 8: k_beam_attn<D, 8, TMAX><<<blocks, 256, 0, s>>>(st, t, layer, q, out, scale); break;
        case 16: k_beam_attn<D, 16, TMAX><<<blocks, 256, 0, s>>>(st, t, layer, q, out, scale); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// BeamKV depth buckets keep the per-level registers small for the usual t = 1, 2
template <int D>
cudaError_t launch_beam_attn_d(const GrState& st, int t, int layer, const uint16_t* q, uint16_t* out,
                               cudaStream_t s, int blocks, float scale) {
    if (t <= 2) return launch_beam_attn_t<D, 2>(st, t, layer, q, out, s, blocks, scale);
    if (t <= 4) return launch_beam_attn_t<D, 4>(st, t, layer, q, out, s, blocks, scale);
    return launch_beam_attn_t<D, kMaxLevels>(st, t, layer, q, out, s, blocks, scale);
}

}  // namespace

cudaError_t ctx_attn_smem_bytes(int head_dim, size_t* bytes) {
    if (head_dim == 128) *bytes = Plan<128>::kBytes;
    else if (head_dim == 64) *bytes = Plan<64>::kBytes;
    else return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t launch_ctx_attn(const GrState& st, const CUtensorMap& qmap, int layer, int64_t wait_limit_ns,
                            cudaStream_t s) {
    const float scale = 1.f / sqrtf((float)st.head_dim);
    const float scale_log2 = scale * 1.4426950408889634f;
    if (st.head_dim == 128) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(k_ctx_attn<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Plan<128>::kBytes);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        k_ctx_attn<128><<<st.n_cta, kAttnThreads, Plan<128>::kBytes, s>>>(qmap, st, layer, scale_log2, scale,
                                                                           wait_limit_ns);
    } else if (st.head_dim == 64) {
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(k_ctx_attn<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 Plan<64>::kBytes);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        k_ctx_attn<64><<<st.n_cta, kAttnThreads, Plan<64>::kBytes, s>>>(qmap, st, layer, scale_log2, scale,
                                                                         wait_limit_ns);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_beam_attn(const GrState& st, int t, int layer, const uint16_t* q, uint16_t* out,
                             cudaStream_t s) {
    const float scale = 1.f / sqrtf((float)st.head_dim);
    const int64_t warps = (int64_t)st.rows * st.n_kv_heads;
    const int blocks = (int)((warps * 32 + 255) / 256);
    if (st.head_dim == 128) return launch_beam_attn_d<128>(st, t, layer, q, out, s, blocks, scale);
    if (st.head_dim == 64) return launch_beam_attn_d<64>(st, t, layer, q, out, s, blocks, scale);
    return cudaErrorInvalidValue;
}

}  // namespace grb
