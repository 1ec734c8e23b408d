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

#include "attn_dev.cuh"
#include "grbeam_internal.h"

namespace grb {
namespace {

using namespace attn;


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
    // the epilogue stages in the rings: query tile 0's four warps in the K ring and the pad
    // after it, tile 1's in the V ring and the pad after that
    static constexpr int kEpiArea = EpiArea<D>::kBytes;  // each softmax warp's staging space
    static constexpr int kEpiPad = 4 * kEpiArea - kStages * kKVTile;
    static constexpr int kVOff = kKOff + kStages * kKVTile + kEpiPad;
    static constexpr int kBarOff = kVOff + kStages * kKVTile + kEpiPad;
    static constexpr int kBytes = kBarOff + 512 + 1024;  // barriers, TMEM address, abort flag, alignment
    static_assert(kEpiPad >= 0 && kEpiPad % 1024 == 0, "the V ring stays 1024-byte aligned");
    // TMEM columns
    static constexpr int kTmemCols = 512;
    static __device__ __forceinline__ int s_col(int i) { return i * 128; }
    static __device__ __forceinline__ int p_col(int i) { return i * 128; }  // bf16 P overwrites S in place
    static __device__ __forceinline__ int o_col(int i) { return 256 + i * D; }
};

enum Bar {
    B_Q_FULL = 0, B_Q_EMPTY = 1, B_K_FULL = 2, B_K_EMPTY = 4, B_V_FULL = 6, B_V_EMPTY = 8,
    B_S_FULL = 10, B_P_FULL = 12, B_O_FULL = 14, B_O_EMPTY = 16, B_DRAIN = 18, B_PVD = 20,
    B_MERGED = 22,  // a merging job that is not the CTA's last has finished with the rings and Q
    B_COUNT = 23
};

constexpr int kAttnThreads = 384;

// kOne: every unit of the launch has a single query tile (at most 128 rows).  Query tile 1's
// TMEM columns then serve as a second S buffer for tile 0: S^g goes to buffer g & 1, so S of
// the next key tile is computed while the softmax of this one runs, and only S^(g+2) waits for
// PV^g (which reads P^g from the same buffer).  Warps 8-11 have no rows and idle.
template <int D, bool kScore, bool kOne = false>
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
                const CUtensorMap* km = st.tmaps + kTmapsPerReq * U.req;
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
                            const int bi = kOne ? (int)(kit & 1) : i;  // the S buffer
                            if (s_i[bi] > 0 && !(ok = wait1(bar(B_PVD + bi), (s_i[bi] - 1) & 1, wt))) break;
                            tc_fence_after();
                            const uint32_t d = tmem + P::s_col(bi);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = (kk >> 2) * P::kBoxBytes + (kk & 3) * 32;
                                const uint64_t a = smem_desc(sb + P::kQOff + i * P::kQTile + off, 16, 1024);
                                const uint64_t b = smem_desc(sb + P::kKOff + ks * P::kKVTile + off, 16, 1024);
                                mma_ss(d, a, b, idesc_s, kk > 0 ? 1u : 0u);
                            }
                            mma_issued = true;
                            tc_commit(bar(B_S_FULL + bi));
                            ++s_i[bi];
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
                            const int bi = kOne ? (int)(vit & 1) : i;  // the P buffer
                            if (!(ok = wait1(bar(B_P_FULL + bi), pv_i[bi] & 1, wt))) break;
                            if (jj == 0 && jobs_i[i] > 0 && !(ok = wait1(bar(B_O_EMPTY + i), (jobs_i[i] - 1) & 1, wt)))
                                break;
                            tc_fence_after();
                            const uint32_t d = tmem + P::o_col(i);
#pragma unroll
                            for (int kk = 0; kk < kTileKeys / 16; ++kk) {
                                const uint32_t a = tmem + P::p_col(bi) + kk * 8;
                                const uint64_t b =
                                    smem_desc(sb + P::kVOff + vs * P::kKVTile + kk * 16 * 128, P::kBoxBytes, 1024);
                                mma_ts(d, a, b, idesc_o, (jj > 0 || kk > 0) ? 1u : 0u);
                            }
                            mma_issued = true;
                            tc_commit(bar(B_PVD + bi));  // the next S of this buffer may overwrite P
                            ++pv_i[bi];
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
        uint32_t tiles = 0, jobs = 0, ktiles = 0;
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
            const int b_first = U.beam0 + i * (kTileRows / G) + (quarter * 32) / G;
            const EpiKeys ek = epi_keys<D, kScore>(st, U, J, ri, layer, b_first, G, lane);  // looked up now
            const int ctx_len = U.ctx_len;
            float m_used = -CUDART_INF_F, l = 0.f;
            for (int jj = 0; jj < n; ++jj) {
                const int bs = kOne ? (int)(tiles & 1) : i;  // the S / P buffer of this key tile
                if (!(ok = wait_warp(bar(B_S_FULL + bs), (kOne ? tiles >> 1 : tiles) & 1, wt))) break;
                tc_fence_after();
                uint32_t sv[128];
                tmem_ld128(tmem + lane_base + P::s_col(bs), sv);
                const int valid = ctx_len - (J.t0 + jj) * kTileKeys;
                auto mask = [&]() {  // keys past the context
                    if (valid < kTileKeys) {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (c >= valid) sv[c] = __float_as_uint(-CUDART_INF_F);
                    }
                };
                mask();
                if constexpr (kOne) {
                    // The exponentials are taken relative to a reference max known before the tile: the
                    // running max m_used (a job's first tile: the max of its first 8 columns).  The row
                    // max comes out of the same pass.  Only when it exceeds the reference by more than
                    // 2^8 (in exp2 units) is the tile redone relative to it (S reloaded from TMEM, O and
                    // l rescaled): the max is off the tile's critical chain, and every p is <= 2^8.
                    float m_ref = m_used;
                    if (jj == 0) {
                        m_ref = fmax3(fmax3(__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2])),
                                      fmax3(__uint_as_float(sv[3]), __uint_as_float(sv[4]), __uint_as_float(sv[5])),
                                      fmaxf(__uint_as_float(sv[6]), __uint_as_float(sv[7])));
                    }
                    uint64_t acc[4];
                    for (;;) {
                        // p = 2^(s*scale_log2 - m*scale_log2), two columns per packed FMA; the row max
                        // in four independent 3-input max chains
                        const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
                        const uint64_t mb2 = f2_pack(-m_ref * scale_log2, -m_ref * scale_log2);
                        float mc[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
    #pragma unroll
                        for (int c = 0; c < 4; ++c) acc[c] = 0ull;
    #pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const float s0 = __uint_as_float(sv[2 * c]), s1 = __uint_as_float(sv[2 * c + 1]);
                            mc[c & 3] = fmax3(mc[c & 3], s0, s1);
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(s0, s1), sc2, mb2), x0, x1);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            acc[c & 3] = f2_add(acc[c & 3], f2_pack(p0, p1));
                            sv[c] = pack_bf16x2(p0, p1);
                        }
                        const float mx = fmax3(fmaxf(mc[0], mc[1]), mc[2], mc[3]);
                        const bool need = (mx - m_ref) * scale_log2 > 8.f;
                        if (!__any_sync(0xffffffffu, need)) break;
                        // rare: some row's max grew past the reference
                        const float m_new = need ? mx : m_ref;
                        if (jj > 0) {
                            // O holds the previous key tiles once the last PV has completed (with one
                            // S buffer per query tile this S waited for it; with kOne it did not)
                            if (kOne && !(ok = wait_warp(bar(B_PVD + ((tiles - 1) & 1)), ((tiles - 1) >> 1) & 1, wt)))
                                break;
                            tc_fence_after();
                            const float alpha = exp2f((m_ref - m_new) * scale_log2);
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
                        }
                        m_ref = m_new;
                        tmem_ld128(tmem + lane_base + P::s_col(bs), sv);  // S is still there: P is stored below
                        mask();
                    }
                    if (!ok) break;
                    m_used = m_ref;
                    float t0, t1, t2, t3, t4, t5, t6, t7;
                    f2_unpack(acc[0], t0, t1);
                    f2_unpack(acc[1], t2, t3);
                    f2_unpack(acc[2], t4, t5);
                    f2_unpack(acc[3], t6, t7);
                    l += ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7));
                } else {
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
                            // O holds the previous key tiles once the last PV has completed (with one
                            // S buffer per query tile this S waited for it; with kOne it did not)
                            if (kOne && !(ok = wait_warp(bar(B_PVD + ((tiles - 1) & 1)), ((tiles - 1) >> 1) & 1, wt)))
                                break;
                            tc_fence_after();
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
                }
                tmem_st32(tmem + lane_base + P::p_col(bs), sv);
                tmem_st32(tmem + lane_base + P::p_col(bs) + 32, sv + 32);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(B_P_FULL + bs));
                ++tiles;
                raise_flag();
            }
            if (!ok) break;
            const uint8_t* qs = smem + P::kQOff + i * P::kQTile + row_t * 128;  // this row in the Q tile
            uint8_t* area = smem + P::kKOff + (warp - 4) * P::kEpiArea;
            ok = job_epilogue<D, kScore>(
                st, U, J, ri, ek, row_t, lane, b_first, prow, layer, scale, m_used, l, qs, area, pend_flag, out, wt,
                [&](uint32_t* ov) {
                    if (!wait_warp(bar(B_O_FULL + i), jobs & 1, wt)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(tmem + lane_base + P::o_col(i) + 32 * c, ov + 32 * c);
                    tc_fence_before();
                    mbar_arrive(bar(B_O_EMPTY + i));  // TMEM O is free for the next job
                    ++jobs;
                    return true;
                },
                [&]() {
                    // Query tile 0's warps stage in the K ring, free once the last key tile's S MMAs
                    // (both tiles') have completed; tile 1's warps in the V ring, free once the last
                    // PV MMAs have (its own is done: O arrived).
                    const uint32_t kl = ktiles - 1;  // the CTA's last key tile
                    return wait_warp(bar((i == 0 ? B_K_EMPTY : B_V_EMPTY) + (kl & 1)), (kl >> 1) & 1, wt);
                },
                [&]() {
                    // The producer may refill the rings and the Q tile.  Each merging warp arrives once
                    // its rows are done; with one query tile the first warpgroup's warps arrive for the
                    // second as well (a warpgroup without rows must not arrive on its own: it would run
                    // ahead to the next job's phase).
                    if (lane == 0 && jb < jr.y - 1) mbar_arrive_n(bar(B_MERGED), U.nqt == 1 ? 2u : 1u);
                });
            if (!ok) break;
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

template <int D, bool kScore, bool kOne>
cudaError_t launch_ctx_attn_d(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q,
                              uint16_t* out, float scale_log2, float scale, int64_t wait_limit_ns, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(k_ctx_attn<D, kScore, kOne>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    return cudaLaunchKernelEx(&cfg, k_ctx_attn<D, kScore, kOne>, qmap, st, layer, q, out, scale_log2, scale,
                              wait_limit_ns);
}

template <bool kScore>
cudaError_t launch_attn(const GrState& st, const CUtensorMap& qmap, int layer, const uint16_t* q, uint16_t* out,
                        int64_t wait_limit_ns, cudaStream_t s) {
    const float scale = 1.f / sqrtf((float)st.head_dim);
    const float scale_log2 = scale * 1.4426950408889634f;
    if (st.head_dim != 128 && st.head_dim != 64) return cudaErrorInvalidValue;
    if (!kScore && st.attn_one) {  // every unit one query tile wide: two S buffers for it
        if (st.head_dim == 128)
            return launch_ctx_attn_d<128, false, true>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
        return launch_ctx_attn_d<64, false, true>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
    }
    if (st.head_dim == 128)
        return launch_ctx_attn_d<128, kScore, false>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
    return launch_ctx_attn_d<64, kScore, false>(st, qmap, layer, q, out, scale_log2, scale, wait_limit_ns, s);
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
