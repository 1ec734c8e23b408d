// GQA decode attention of every beam over the split KV layout, on CTA pairs.
//
// zhiding.cn recsys-examples article, section "语义ID生成式推荐专用推理框架"
// (semantic-ID GR inference framework): the long request context is kept once
// per request (ContextKV) and shared by all beams, each beam keeps only the
// short history of its own decoded tokens (BeamKV), and beam ancestry lives in
// BeamPath; the attention backend works directly on that layout.
//
// The context part of a 256-row unit (beams x query heads of one request and
// KV head) is one dense contraction per 128-key tile:
//     S = Q K^T / sqrt(D)   (M = 256 rows, N = 128 keys, K = D = 128)
//     O += softmax(S) V     (M = 256 rows, N = D, K = 128 keys)
// issued as tcgen05 MMAs of a CTA pair (cta_group::2): each CTA of the pair
// holds 128 of the unit's query rows and HALF of every K and V tile (keys
// 0-63 / 64-127 of K, dimensions 0-63 / 64-127 of V), and the pair's two
// tensor cores each compute their 128 rows from both halves.  Per SM this is
// half the shared-memory footprint and fill traffic of a CTA that holds whole
// tiles, which leaves room in TMEM for two S buffers, two P buffers and O:
//     columns   0-255  S0, S1 (fp32)      256-383  P0, P1 (bf16 pairs)
//              384-511 O  (fp32)
// so the S of a tile is computed two tiles ahead of its PV and an S buffer is
// free as soon as its softmax has loaded it.  Per CTA:
//   warps 0, 2  TMA producers: warp 0 its half of the Q tile (128 rows) once
//               per job and its halves of K, warp 2 its halves of V, through
//               4-stage rings (128-byte swizzle).  Loads complete on the leader
//               CTA's barriers (cta_group::2).
//   warps 1, 3  (leader CTA only) the MMA issuers, one thread each: warp 3
//               issues S up to two tiles ahead, warp 1 issues PV as each P
//               arrives; commits are multicast to both CTAs' barriers.
//   warp 2      also the TMEM allocation (both CTAs, collective).
//   warps 4-11  softmax, one thread per row: warps 4-7 take the even key
//               tiles, warps 8-11 the odd ones (a warp of each on every SMSP,
//               on the same rows), passing the running max from tile to tile
//               through shared memory.  Lazy rescale of O (only when the running
//               max grows by more than 2^8), P written to TMEM as bf16.  Warps
//               4-7 then end each job for their rows: publish the piece of a cut
//               unit, or merge the pieces, the BeamKV part and the bf16 output
//               (attn_dev.cuh).
// Both units of a (request, KV head) run on neighbouring pairs, so the second
// read of a K/V tile is served by L2: each context byte comes from HBM once
// per request.  The launch is cooperative, so every CTA a merger waits for is
// resident.
//
// Every wait is bounded: past the limit the kernel flags GR_ERR_TIMEOUT,
// settles and drains the copies and MMAs it issued, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "attn_dev.cuh"
#include "grbeam_internal.h"

namespace grb {
namespace {

using namespace attn;

// ---------------------------------------------------------------------------
// CTA-pair PTX (cta_group::2, distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the same shared-memory address in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
// arrive on a barrier of the pair (possibly the peer's); the tensor-memory accesses it
// publishes are ordered by the tcgen05 fences around it
__device__ __forceinline__ void arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
__device__ __forceinline__ void complete_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool try_wait_cl(uint32_t bar, uint32_t parity) {
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
// one thread, a barrier that other CTAs of the pair signal
__device__ __forceinline__ bool wait1_cl(uint32_t bar, uint32_t parity, const Waiter w) {
    if (try_wait_cl(bar, parity)) return true;
    uint64_t t0 = global_timer();
    uint32_t spins = 0;
    while (!try_wait_cl(bar, parity)) {
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
// whole warp (convergent), a barrier that the pair signals
__device__ __forceinline__ bool wait_warp_cl(uint32_t bar, uint32_t parity, const Waiter w) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    uint32_t spins = 0;
    for (;;) {
        const bool ok = try_wait_cl(bar, parity);
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
__device__ __forceinline__ void wait_drain_cl(uint32_t bar, uint32_t parity) {
    uint64_t t0 = global_timer();
    while (!try_wait_cl(bar, parity)) {
        if ((int64_t)(global_timer() - t0) > kDrainLimitNs) return;
    }
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// TMA tile load into this CTA's shared memory, completion counted on a barrier of the pair
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* tmap, uint32_t bar_cluster, int c0, int c1,
                                                 int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, "
        "%5}], [%2];" ::"r"(dst),
        "l"(tmap), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T over the pair (M = 256)
__device__ __forceinline__ void mma_ss_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem] over the pair (M = 256)
__device__ __forceinline__ void mma_ts_pair(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
// arrive on the barrier at this address in both CTAs once the issued MMAs have completed
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}
// the same, this CTA's barrier only
__device__ __forceinline__ void commit_own(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// ---------------------------------------------------------------------------
// shared-memory plan (head_dim 128)
// ---------------------------------------------------------------------------
struct PairPlan {
    static constexpr int kD = 128;
    static constexpr int kQBox = 128 * 128;         // 128 rows x 64 dimensions
    static constexpr int kQTile = 2 * kQBox;        // this CTA's 128 query rows
    static constexpr int kKBox = 64 * 128;          // 64 keys x 64 dimensions
    static constexpr int kKHalf = 2 * kKBox;        // 64 keys x 128 dimensions
    static constexpr int kVHalf = 128 * 128;        // 128 keys x 64 dimensions
    static constexpr int kStages = 4;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQOff + kQTile;
    // the epilogue stages in the K ring and the 2 KB after it
    static constexpr int kEpiArea = EpiArea<kD>::kBytes;  // each epilogue warp's staging space
    static constexpr int kEpiPad = 4 * kEpiArea - kStages * kKHalf;
    static constexpr int kVOff = kKOff + kStages * kKHalf + kEpiPad;
    static constexpr int kMxOff = kVOff + kStages * kVHalf;  // m of a tile [parity][128], set 1's m [128]
    static constexpr int kLOff = kMxOff + 2 * 2 * 128 * 4;    // set 1's row sums [128]
    static constexpr int kCntOff = kLOff + 128 * 4;           // producer's fill counts (teardown)
    static constexpr int kBarOff = kCntOff + 64;
    static constexpr int kBytes = kBarOff + 512 + 1024;       // barriers, TMEM address, abort flag, alignment
    static constexpr int kTmemCols = 512;
    static __device__ __forceinline__ int s_col(int b) { return b * 128; }
    static __device__ __forceinline__ int p_col(int b) { return 256 + b * 64; }
    static constexpr int kOCol = 384;
    static_assert(kEpiPad >= 0 && kEpiPad % 1024 == 0, "the V ring stays 1024-byte aligned");
};

enum PairBar {
    PB_Q_FULL = 0, PB_Q_EMPTY = 1,
    PB_K_FULL = 2, PB_K_EMPTY = 6, PB_V_FULL = 10, PB_V_EMPTY = 14,  // kStages each
    PB_S_FULL = 18, PB_S_EMPTY = 20, PB_P_FULL = 22, PB_PVD = 24,     // two each
    PB_O_FULL = 26, PB_O_EMPTY = 27, PB_DRAIN = 28,  // two: one per MMA issuer
    PB_MERGED = 30,  // a merging job that is not the pair's last has finished with the K ring and Q
    PB_MX = 31,      // [quarter][tile parity]: the m a tile used is published
    PB_LX = 39,      // [quarter]: set 1's row sums are written (job end)
    PB_LXE = 43,     // [quarter]: set 0 has read them
    PB_COUNT = 47
};

constexpr int kPairThreads = 384;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
k_pair_attn(const __grid_constant__ CUtensorMap qmap, GrState st, int layer, const uint16_t* __restrict__ q,
            uint16_t* __restrict__ out, float scale_log2, float scale, int64_t wait_limit_ns) {
    using P = PairPlan;
    constexpr int D = P::kD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + P::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kBarOff + 8 * PB_COUNT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::kBarOff + 8 * PB_COUNT + 8);
    uint32_t* fills = reinterpret_cast<uint32_t*>(smem + P::kCntOff);  // [0] Q, [1] K, [2] V loads issued

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int G = st.n_q_heads / st.n_kv_heads;

    if (threadIdx.x == 0) {
        mbar_init(bar(PB_Q_FULL), 1);
        mbar_init(bar(PB_Q_EMPTY), 1);
        for (int s = 0; s < P::kStages; ++s) {
            mbar_init(bar(PB_K_FULL + s), 1);
            mbar_init(bar(PB_K_EMPTY + s), 1);
            mbar_init(bar(PB_V_FULL + s), 1);
            mbar_init(bar(PB_V_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(PB_S_FULL + b), 1);
            mbar_init(bar(PB_S_EMPTY + b), 8);  // the 4 softmax warps of a tile x 2 CTAs
            mbar_init(bar(PB_P_FULL + b), 8);
            mbar_init(bar(PB_PVD + b), 1);
        }
        mbar_init(bar(PB_O_FULL), 1);
        mbar_init(bar(PB_O_EMPTY), 8);  // 4 epilogue warps x 2 CTAs
        mbar_init(bar(PB_DRAIN), 1);
        mbar_init(bar(PB_DRAIN + 1), 1);
        mbar_init(bar(PB_MERGED), 4);
        for (int k = 0; k < 8; ++k) mbar_init(bar(PB_MX + k), 1);  // the warp of the tile
        for (int k = 0; k < 4; ++k) mbar_init(bar(PB_LX + k), 1);   // the warp of set 1
        for (int k = 0; k < 4; ++k) mbar_init(bar(PB_LXE + k), 1);  // the warp of set 0
        *abort_flag = 0;
        fills[0] = fills[1] = fills[2] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        tmem_alloc_pair(smem_u32(tmem_slot), P::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before either signals the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int2 jr = st.cta_jobs[pair];
    const Waiter wt{wait_limit_ns, abort_flag, st.status};
    // the leader's barriers, as addresses of the pair
    auto lbar = [&](int i) -> uint32_t { return mapa(bar(i), 0); };

    if (warp < 4) {
        regs_dec<56>();
        uint32_t p_qcnt = 0, p_kit = 0, p_vit = 0, p_mcnt = 0;
        if (warp == 0 || warp == 2) {
            if (lane == 0) {
                // ---- TMA producers (both CTAs): warp 0 loads Q and K, warp 2 loads V, so that
                // each ring refills as soon as its own stage is consumed (V lags K by the
                // softmax)
                const bool kq = warp == 0;
                bool ok = true;
                for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                    const GrAttnJob J = st.jobs[jb];
                    const GrAttnUnit& U = J.u;
                    if (!decoding<false>(st, U)) continue;
                    const CUtensorMap* vm = st.tmaps + 3 * U.req + 1;
                    const CUtensorMap* km = st.tmaps + 3 * U.req + 2;  // half tiles of 64 keys
                    if (jb == jr.x || st.jobs[jb - 1].unit != J.unit) tmap_acquire(kq ? km : vm);
                    const int z = layer * st.n_kv_heads + U.head;
                    if (kq) {
                        if (p_qcnt > 0 && !(ok = wait1_cl(bar(PB_Q_EMPTY), (p_qcnt - 1) & 1, wt))) break;
                        if (leader) mbar_expect_tx(bar(PB_Q_FULL), 2u * P::kQTile);
                        for (int kb = 0; kb < 2; ++kb)
                            tma_load_3d_pair(sb + P::kQOff + kb * P::kQBox, &qmap, lbar(PB_Q_FULL), kb * 64, U.head * G,
                                             U.row_off + U.beam0 + (int)rank * (kTileRows / G));
                        fills[0] = ++p_qcnt;
                        for (int j = J.t0; j < J.t1; ++j) {
                            const int s = p_kit % P::kStages;
                            if (!(ok = wait1_cl(bar(PB_K_EMPTY + s), ((p_kit / P::kStages) & 1) ^ 1, wt))) break;
                            if (leader) mbar_expect_tx(bar(PB_K_FULL + s), 2u * P::kKHalf);
                            for (int kb = 0; kb < 2; ++kb)
                                tma_load_3d_pair(sb + P::kKOff + s * P::kKHalf + kb * P::kKBox, km, lbar(PB_K_FULL + s),
                                                 kb * 64, j * kTileKeys + (int)rank * 64, z);
                            fills[1] = ++p_kit;
                        }
                        // a merging job stages its BeamKV keys in the K ring and reads q from its Q
                        // tile: the next job's loads wait until its merge is done
                        if (ok && J.slot == U.first_slot && jb < jr.y - 1) {
                            if (!(ok = wait1(bar(PB_MERGED), p_mcnt & 1, wt))) break;
                            ++p_mcnt;
                        }
                    } else {
                        for (int j = J.t0; j < J.t1; ++j) {
                            const int s = p_vit % P::kStages;
                            if (!(ok = wait1_cl(bar(PB_V_EMPTY + s), ((p_vit / P::kStages) & 1) ^ 1, wt))) break;
                            if (leader) mbar_expect_tx(bar(PB_V_FULL + s), 2u * P::kVHalf);
                            tma_load_3d_pair(sb + P::kVOff + s * P::kVHalf, vm, lbar(PB_V_FULL + s), (int)rank * 64,
                                             j * kTileKeys, z);
                            fills[2] = ++p_vit;
                        }
                    }
                }
            }
            __syncwarp();
        } else if (warp == 1 || warp == 3) {
            // ---- MMA issuers (leader CTA, one thread each): warp 3 issues S = Q K^T up to two
            // tiles ahead (an S buffer is free once its softmax has loaded it), warp 1 issues
            // O += P V as each P arrives.  With two issuers one thread's waits and commits overlap
            // the other's MMAs, which keeps the tensor pipe fed.
            if (lane == 0 && leader) {
                bool mma_issued = false, ok = true;
                uint32_t g = 0;  // key tiles of the pair so far (S and P buffers alternate)
                if (warp == 3) {
                    constexpr uint32_t idesc_s = idesc_bf16(256, kTileKeys, false);
                    uint32_t kit = 0, qcnt = 0;
                    for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                        const GrAttnJob J = st.jobs[jb];
                        const GrAttnUnit& U = J.u;
                        if (!decoding<false>(st, U)) continue;
                        const int n = J.t1 - J.t0;
                        if (!(ok = wait1_cl(bar(PB_Q_FULL), qcnt & 1, wt))) break;
                        ++qcnt;
                        for (int jj = 0; jj < n; ++jj, ++g) {
                            const uint32_t b = g & 1;
                            // the softmax of tile g - 2 has loaded its S from this buffer
                            if (g >= 2 && !(ok = wait1_cl(bar(PB_S_EMPTY + b), ((g >> 1) - 1) & 1, wt))) break;
                            const int ks = kit % P::kStages;
                            if (!(ok = wait1_cl(bar(PB_K_FULL + ks), (kit / P::kStages) & 1, wt))) break;
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t a = smem_desc(sb + P::kQOff + (kk >> 2) * P::kQBox + (kk & 3) * 32, 16, 1024);
                                const uint64_t bd = smem_desc(
                                    sb + P::kKOff + ks * P::kKHalf + (kk >> 2) * P::kKBox + (kk & 3) * 32, 16, 1024);
                                mma_ss_pair(tmem + P::s_col(b), a, bd, idesc_s, kk > 0 ? 1u : 0u);
                            }
                            mma_issued = true;
                            commit_pair(bar(PB_S_FULL + b));
                            commit_pair(bar(PB_K_EMPTY + ks));
                            if (jj == n - 1) commit_pair(bar(PB_Q_EMPTY));
                            ++kit;
                        }
                    }
                } else {
                    constexpr uint32_t idesc_o = idesc_bf16(256, D, true);
                    uint32_t vit = 0, jobs = 0;
                    for (int jb = jr.x; jb < jr.y && ok; ++jb) {
                        const GrAttnJob J = st.jobs[jb];
                        const GrAttnUnit& U = J.u;
                        if (!decoding<false>(st, U)) continue;
                        const int n = J.t1 - J.t0;
                        for (int jj = 0; jj < n; ++jj, ++g) {
                            const uint32_t b = g & 1;
                            if (!(ok = wait1_cl(bar(PB_P_FULL + b), (g >> 1) & 1, wt))) break;
                            const int vs = vit % P::kStages;
                            if (!(ok = wait1_cl(bar(PB_V_FULL + vs), (vit / P::kStages) & 1, wt))) break;
                            if (jj == 0 && jobs > 0 && !(ok = wait1_cl(bar(PB_O_EMPTY), (jobs - 1) & 1, wt))) break;
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                                const uint64_t bd =
                                    smem_desc(sb + P::kVOff + vs * P::kVHalf + kk * 16 * 128, P::kVHalf, 1024);
                                mma_ts_pair(tmem + P::kOCol, tmem + P::p_col(b) + kk * 8, bd, idesc_o,
                                            (jj > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_issued = true;
                            commit_pair(bar(PB_PVD + b));
                            commit_pair(bar(PB_V_EMPTY + vs));
                            if (jj == n - 1) commit_pair(bar(PB_O_FULL));
                            ++vit;
                        }
                        ++jobs;
                    }
                }
                // all issued tensor-core work (and its commits) completes before TMEM is freed
                if (mma_issued) {
                    const int dr = PB_DRAIN + (warp == 3 ? 1 : 0);
                    commit_own(bar(dr));
                    wait_drain_cl(bar(dr), 0);
                }
            }
            __syncwarp();
        }
        tc_fence_before();
        named_bar_sync(1);
        cluster_sync_all();
        // After an abort, every copy of the pair must have landed before either CTA leaves.  The
        // copies of both CTAs complete on the leader's barriers, so the leader's producer settles
        // each phase it or the peer left unmatched (its own expected bytes of a copy the peer
        // never issued, or the peer's copy it never armed for), then waits for all of them.
        if (leader && warp == 0 && lane == 0 &&
            (*abort_flag != 0 || ld_peer_u32(mapa(smem_u32(const_cast<int*>(abort_flag)), 1)) != 0)) {
            const uint32_t peer_fills[3] = {ld_peer_u32(mapa(smem_u32(fills), 1)), ld_peer_u32(mapa(smem_u32(fills + 1), 1)),
                                            ld_peer_u32(mapa(smem_u32(fills + 2), 1))};
            const uint32_t own[3] = {fills[0], fills[1], fills[2]};  // both producers of this CTA
            const int first[3] = {PB_Q_FULL, PB_K_FULL, PB_V_FULL};
            const int stages[3] = {1, P::kStages, P::kStages};
            const uint32_t half[3] = {P::kQTile, P::kKHalf, P::kVHalf};
            for (int k = 0; k < 3; ++k)
                for (int s = 0; s < stages[k]; ++s) {
                    // the n-th copy of a ring goes to stage n % stages; a CTA issues copy n of stage s
                    // only once copy n - 1 of it was consumed, so at most the last phase is unmatched
                    const uint32_t nl = own[k] > (uint32_t)s ? (own[k] - 1 - s) / stages[k] + 1 : 0;
                    const uint32_t np = peer_fills[k] > (uint32_t)s ? (peer_fills[k] - 1 - s) / stages[k] + 1 : 0;
                    const uint32_t nmax = nl > np ? nl : np;
                    if (nmax == 0) continue;
                    if (nl < nmax) mbar_expect_tx(bar(first[k] + s), half[k]);  // the peer's copy, never armed
                    else if (np < nmax) complete_tx(bar(first[k] + s), half[k]);  // armed, the peer never copied
                    wait_drain_cl(bar(first[k] + s), (nmax - 1) & 1);
                }
        }
        __syncwarp();
        cluster_sync_all();
        tc_fence_after();
        if (warp == 2) tmem_dealloc_pair(tmem, P::kTmemCols);
        return;
    }

    regs_inc<224>();
    {
        // ---- softmax: warps 4-7 (set 0) take the even key tiles of the pair, warps 8-11
        // (set 1) the odd ones; warp 4 + q and warp 8 + q share TMEM lanes 32q..32q+31 (the
        // same 32 rows) and sit on the same SMSP, so one's waits overlap the other's work.
        // The running max m passes from tile to tile: a tile's warp publishes the m it uses
        // (the previous tile's, raised only when its own max exceeds it by more than 2^8 in
        // exp2 units) as soon as it has its row max, and the next tile's warp waits for it.
        // Each set keeps its own row sum, relative to the last m it used; the two are combined
        // at the end of the job.  The tile whose m rises rescales O (after the previous
        // tile's PV has completed).
        const int set = (warp - 4) >> 2;
        const int quarter = warp & 3;
        const int row_t = quarter * 32 + lane;            // row within this CTA's 128 (TMEM lane)
        const int prow = (int)rank * kTileRows + row_t;   // row within the unit
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        float* m_ex = reinterpret_cast<float*>(smem + P::kMxOff);  // [tile parity][128] the m a tile used
        float* l_ex = reinterpret_cast<float*>(smem + P::kLOff);   // set 1's row sums at the job end
        float* lm_ex = m_ex + 256;                                 // set 1's m at the job end
        const uint32_t s_empty0 = mapa(bar(PB_S_EMPTY), 0), p_full0 = mapa(bar(PB_P_FULL), 0);
        const uint32_t o_empty0 = mapa(bar(PB_O_EMPTY), 0);
        uint32_t g = 0, jobs = 0, jdone = 0, ktiles = 0;
        bool ok = true;
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
            if (!decoding<false>(st, U)) continue;
            const int n = J.t1 - J.t0;
            ktiles += n;  // key tiles the pair has taken through the K ring so far
            const RowInfo ri = row_info<false>(st, U, (int)rank, row_t, G);
            const int b_first = U.beam0 + (int)rank * (kTileRows / G) + (quarter * 32) / G;
            // set 0 ends the job: it looks up the private keys it will stage now
            const EpiKeys ek = set == 0 ? epi_keys<D, false>(st, U, J, ri, layer, b_first, G, lane) : EpiKeys{0, 0, -1, -1};
            const int ctx_len = U.ctx_len;
            float m_mine = -CUDART_INF_F, l = 0.f;  // this set's m and row sum
            for (int jj = 0; jj < n; ++jj, ++g) {
                if ((int)(g & 1) != set) continue;
                const uint32_t b = g & 1;
                if (!(ok = wait_warp_cl(bar(PB_S_FULL + b), (g >> 1) & 1, wt))) break;
                tc_fence_after();
                uint32_t sv[128];
                tmem_ld128(tmem + lane_base + P::s_col(b), sv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_cluster(s_empty0 + 8u * b);  // the S buffer may be overwritten
                const int valid = ctx_len - (J.t0 + jj) * kTileKeys;
                if (valid < kTileKeys) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= valid) sv[c] = __float_as_uint(-CUDART_INF_F);
                }
                float a0 = -CUDART_INF_F, a1 = -CUDART_INF_F, a2 = -CUDART_INF_F, a3 = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    a0 = fmax3(a0, __uint_as_float(sv[c + 0]), __uint_as_float(sv[c + 1]));
                    a1 = fmax3(a1, __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
                    a2 = fmax3(a2, __uint_as_float(sv[c + 4]), __uint_as_float(sv[c + 5]));
                    a3 = fmax3(a3, __uint_as_float(sv[c + 6]), __uint_as_float(sv[c + 7]));
                }
                const float mx = fmax3(fmaxf(a0, a1), a2, a3);
                // the m of the previous tile (its warp published it).  Its slot is the one this tile
                // writes next, so the wait comes first even at a job's first tile, whose m is its own.
                float m_prev = -CUDART_INF_F;
                if (g > 0) {
                    const uint32_t gq = g - 1;
                    if (!(ok = wait_warp(bar(PB_MX + quarter * 2 + (gq & 1)), (gq >> 1) & 1, wt))) break;
                    if (jj > 0) m_prev = m_ex[(gq & 1) * 128 + row_t];
                }
                const bool need = jj == 0 || (mx - m_prev) * scale_log2 > 8.f;
                const float m_new = need ? mx : m_prev;
                m_ex[b * 128 + row_t] = m_new;
                __syncwarp();  // the warp's stores, then one arrival that releases them
                if (lane == 0) mbar_arrive(bar(PB_MX + quarter * 2 + b));
                // this set's sum follows m (its previous tiles were summed relative to m_mine)
                if (m_mine != m_new) l *= exp2f((m_mine - m_new) * scale_log2);
                m_mine = m_new;
                if (jj > 0 && __any_sync(0xffffffffu, need)) {
                    // O holds the previous tiles (relative to m_prev) once that tile's PV has completed
                    const float alpha = exp2f((m_prev - m_new) * scale_log2);
                    const uint32_t gq = g - 1;
                    if (!(ok = wait_warp_cl(bar(PB_PVD + (gq & 1)), (gq >> 1) & 1, wt))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        const uint32_t ta = tmem + lane_base + P::kOCol + 32 * c;
                        tmem_ld32(ta, ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(ta, ov);
                    }
                    tmem_st_wait();
                }
                // p = 2^(s*scale_log2 - m*scale_log2), two columns per packed FMA
                const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
                const uint64_t mb2 = f2_pack(-m_new * scale_log2, -m_new * scale_log2);
                uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sc2, mb2), x0,
                              x1);
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
                // the P buffer of tile g - 2 is free once that tile's PV has completed
                if (g >= 2 && !(ok = wait_warp_cl(bar(PB_PVD + b), ((g >> 1) - 1) & 1, wt))) break;
                tc_fence_after();
                tmem_st32(tmem + lane_base + P::p_col(b), sv);
                tmem_st32(tmem + lane_base + P::p_col(b) + 32, sv + 32);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_cluster(p_full0 + 8u * b);
                raise_flag();
            }
            if (!ok) break;
            // the row's sum over both sets, relative to the job's final m (the larger of theirs)
            if (set == 1) {
                // the slot is free once set 0 has read the previous job's sums
                if (jdone > 0 && !(ok = wait_warp(bar(PB_LXE + quarter), (jdone - 1) & 1, wt))) break;
                l_ex[row_t] = l;
                lm_ex[row_t] = m_mine;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(PB_LX + quarter));
                ++jdone;
                continue;  // warps 4-7 end the job for their rows
            }
            if (!(ok = wait_warp(bar(PB_LX + quarter), jdone & 1, wt))) break;
            ++jdone;
            {
                const float m1 = lm_ex[row_t], l1 = l_ex[row_t];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(PB_LXE + quarter));
                const float mf = fmaxf(m_mine, m1);
                l = (m_mine == mf ? l : l * exp2f((m_mine - mf) * scale_log2)) +
                    (m1 == mf ? l1 : l1 * exp2f((m1 - mf) * scale_log2));
                m_mine = mf;
            }
            const uint8_t* qs = smem + P::kQOff + row_t * 128;  // this row in the Q tile
            uint8_t* area = smem + P::kKOff + quarter * P::kEpiArea;
            ok = job_epilogue<D, false>(
                st, U, J, ri, ek, row_t, lane, b_first, prow, layer, scale, m_mine, l, qs, area, pend_flag, out, wt,
                [&](uint32_t* ov) {
                    if (!wait_warp_cl(bar(PB_O_FULL), jobs & 1, wt)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_base + P::kOCol + 32 * c, ov + 32 * c);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) arrive_cluster(o_empty0);  // TMEM O is free for the next job
                    ++jobs;
                    return true;
                },
                [&]() {
                    // the K ring is free once the S MMAs of the pair's last key tile have completed
                    const uint32_t kl = ktiles - 1;
                    return wait_warp_cl(bar(PB_K_EMPTY + kl % P::kStages), (kl / P::kStages) & 1, wt);
                },
                [&]() {
                    if (lane == 0 && jb < jr.y - 1) mbar_arrive(bar(PB_MERGED));
                });
            if (!ok) break;
        }
        raise_flag();
    }
    tc_fence_before();
    named_bar_sync(1);
    cluster_sync_all();
    cluster_sync_all();
}

}  // namespace

cudaError_t pair_attn_smem_bytes(size_t* bytes) {
    *bytes = PairPlan::kBytes;
    return cudaSuccess;
}

cudaError_t launch_pair_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                             int64_t wait_limit_ns, cudaStream_t s) {
    if (st.head_dim != PairPlan::kD) return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e =
            cudaFuncSetAttribute(k_pair_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, PairPlan::kBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const float scale = 1.f / sqrtf((float)st.head_dim);
    const float scale_log2 = scale * 1.4426950408889634f;
    // cooperative: every CTA is resident at once, so a merging pair may wait for the flags
    // of the pieces other pairs publish; the pairs are clusters of two CTAs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * st.n_cta);
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = PairPlan::kBytes;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_pair_attn, qmap, st, layer, q, out, scale_log2, scale, wait_limit_ns);
}

}  // namespace grb
