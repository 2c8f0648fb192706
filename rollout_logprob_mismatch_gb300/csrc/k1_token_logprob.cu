// k1_token_logprob.cu -- fused selected-token logprob for sm_103a.
//
// l_t = z_t[a_t] - log sum_v exp(z_t[v]),  z_t = h_t W^T   (icarus "RL: Training
// Inference Mismatch", section "log p"; LoongSage "Train-Inference Consistency"
// section 3, FP32 LM head: here bf16 operands with fp32 accumulation).
//
// Persistent CTA pairs (one CTA per SM) walk work units (two m-tiles of 128
// tokens, one per CTA, and a vocabulary chunk of 1024 ids).  Per unit and
// 256-column tile:
//   warp 0     TMA: the CTA's own h tile [128 x 64] and its own half of the W
//              tile [128 x 64], 128-byte swizzle, into a 6-stage shared-memory
//              ring; the bytes of both CTAs complete on the even CTA's barrier,
//              and a stage is refilled when the pair UMMA has released it;
//   warp 1     (even CTA) one thread issues the 2-SM tcgen05.mma (M = 256 over
//              the pair, N = 256, K = 16, bf16 -> fp32): each CTA's TMEM gets
//              its own 128 rows x 256 columns, from both CTAs' halves of W, so
//              every W byte leaves L2 once per pair; two accumulators (2 x 256
//              columns), k ascending;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, one TMEM lane (= one
//              token row) per thread, an online max / sum-of-exp over the columns
//              in ascending order, and the target logit picked from the exact
//              accumulator value.  The [N, V] logits never leave the SM.
// A batch of one m-tile runs in single CTAs (1-SM UMMA, M = 128, both halves
// of each W tile loaded by the CTA itself; same k order, same bits).
// Each unit writes its chunk's (max, sum) per row; a second small kernel folds
// the chunks of a row in a fixed order.  The split is a function of V alone and
// every row is reduced in the same order whatever the batch holds, so a row's
// outputs are bit-identical across batch sizes and compositions (llm-infra-atlas
// "训推一致性与 determinism", sections 1.2 and 6: batch-invariant GEMM with a
// fixed reduction order).
#include <algorithm>
#include <cstdlib>

#include <cuda_bf16.h>

#include "k1_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "unit_ring.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

constexpr uint32_t TMEM_COLS = 2 * K1_BN;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int SUBCOLS = 32;

struct Unit {
    int mt, ch;
};

// Units run m-tile fastest inside a band of `band` m-tiles, so the CTAs that are
// resident together share the same W chunk (read once from HBM, then from L2)
// while the band's h rows stay in L2.  The order affects speed only.
// Returns the unit's m-group (a.cluster consecutive m-tiles, one per CTA of
// the cluster) in .mt and its vocabulary chunk in .ch.
__device__ __forceinline__ Unit unit_of(int u, const K1Args &a)
{
    const int per_band = a.band * a.num_chunks;
    const int b = u / per_band;
    const int rem = u - b * per_band;
    const int m0 = b * a.band;
    const int mb = min(a.band, a.num_m_groups - m0);
    Unit r;
    r.ch = rem / mb;
    r.mt = m0 + (rem - r.ch * mb);
    return r;
}

__device__ __forceinline__ int tiles_in_chunk(int ch, int V)
{
    const int lo = ch * K1_VCHUNK;
    const int hi = min(V, lo + K1_VCHUNK);
    return (hi - lo + K1_BN - 1) / K1_BN;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&b);
}

// MODE 0: the forward (per-chunk max / sum and the target logit).  MODE 1: the
// backward's logit gradient dz = g (onehot(a) - p) / tau, p = softmax(z / tau)
// from the forward's lse, written as bf16 rows of length a.dz_ld.
template <int MODE, int CL>
__global__ void __launch_bounds__(K1_THREADS, 1)
    k1_main_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_h_tail, const K1Args a)
{
    constexpr bool PAIR = CL == 2;
    constexpr int STAGES = k1_stages(CL);
    constexpr uint32_t B_BYTES = k1_b_bytes(CL);
    constexpr uint32_t STAGE_TX = K1_A_BYTES + B_BYTES;   // bytes this CTA loads per stage
    constexpr uint32_t IDESC = idesc_bf16_f32(K1_BM * CL, K1_BN);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + STAGES * K1_A_BYTES;
    uint8_t *tail_area = smem + STAGES * (K1_A_BYTES + B_BYTES);
    // units claimed in order (unit_ring.cuh); its users: the UMMA issuer, the
    // epilogue warps of both CTAs, the odd CTA's producer
    UnitRing<CL, 1 + 4 * CL + (CL - 1)> ring(tail_area);
    uint64_t *bars = reinterpret_cast<uint64_t *>(tail_area + UNIT_RING_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);    // in a pair the even CTA's, expecting the bytes of both CTAs
            mbar_init(empty(s), 1);   // released by the (pair) UMMA
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 4 * CL);   // in a pair the even CTA's: the epilogue warps of both
        }
        mbar_init(drain, 1);
        ring.init();
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_h);
        if (a.tail_mt >= 0)
            tma_prefetch_desc(&tmap_h_tail);
        tma_prefetch_desc(&tmap_w);
    }
    pdl_wait();                // h, W, targets, the unit counter may be written by earlier work
    pdl_launch_dependents();   // the combine kernel may start launching
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();   // every CTA's barriers exist before the other CTA's TMA, UMMA or threads reach them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t rank = cluster_ctarank();
    const int KBH = (a.D + K1_BK - 1) / K1_BK;   // k-tiles of h
    const int KB = KBH * a.w_segments;          // k-tiles of W: 1 or 3 bf16 parts of each weight
    const uint64_t budget = a.wait_budget_ns;
    // shared::cluster addresses of the barriers both CTAs of a pair signal (the even CTA's)
    auto full_pair = [&](int s) { return PAIR ? mapa_shared(full(s), 0) : full(s); };
    auto tempty_pair = [&](int b) { return PAIR ? mapa_shared(tempty(b), 0) : tempty(b); };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (every CTA)
            const uint64_t pol_h = l2_policy_evict_last();
            const uint64_t pol_w = l2_policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            int ahead = -1;   // the even CTA claims one unit ahead of its loads
            bool ok = rank != 0 || ring.claim(a.sched, a.units, ahead, abort_flag, budget);
            while (ok) {
                int u = -1;
                if (!(rank == 0 ? ring.next(a.sched, a.units, u, ahead, abort_flag, budget)
                                : ring.take(u, true, rank, abort_flag, budget)))
                    break;
                if (u < 0)
                    break;
                TIM_DCHECK(u < a.units, a.status, TIM_CHECK_UNIT, u, a.units);
                const Unit w = unit_of(u, a);
                const int mt = w.mt * CL + static_cast<int>(rank);
                // the last m-tile of a batch whose size is not a multiple of 16 rows
                // reads a zero-padded copy of its rows (same values, fast loads); an
                // m-tile past the batch (the pair peer of a last odd m-tile) reads
                // past the end of that copy: zeros, again through a map of 16k rows
                const bool tail = a.tail_mt >= 0 && mt >= a.tail_mt;
                const CUtensorMap *hmap = tail ? &tmap_h_tail : &tmap_h;
                const int hrow = tail ? (mt - a.tail_mt) * K1_BM : mt * K1_BM;
                const int nt = tiles_in_chunk(w.ch, a.V);
                for (int j = 0; ok && j < nt; ++j) {
                    const int v0 = w.ch * K1_VCHUNK + j * K1_BN;
                    int kh = 0;   // kb mod KBH: the h tile meets each part of W in turn
                    for (int kb = 0; kb < KB; ++kb) {
                        // the stage is free once the UMMA that read it has completed
                        if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag, budget)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = full_pair(stage);
                        // innermost coordinates are whole 16 bytes (8 bf16), rows not negative
                        TIM_DCHECK((((kh | kb) * K1_BK) & 7) == 0 && hrow >= 0 && v0 >= 0, a.status,
                                   TIM_CHECK_TMA_COORD, hrow,
                                   (static_cast<uint64_t>(kb) << 32) | static_cast<uint32_t>(kh * K1_BK));
                        if (PAIR) {
                            // own h tile + own half of the W tile; both CTAs' bytes complete
                            // on the even CTA's barrier, whose one arrival expects them all
                            // (the other CTA's bytes may land first: the count goes below zero
                            // and the phase still cannot complete before that arrival)
                            if (rank == 0)
                                mbar_arrive_expect_tx(full(stage), 2 * STAGE_TX);
                            tma_load_2d_pair(sA + stage * K1_A_BYTES, hmap, fb, kh * K1_BK, hrow, pol_h);
                            tma_load_2d_pair(sB + stage * B_BYTES, &tmap_w, fb, kb * K1_BK,
                                             v0 + static_cast<int>(rank) * K1_W_BOX_ROWS, pol_w);
                        } else {   // h tile + both halves of the W tile
                            mbar_arrive_expect_tx(fb, STAGE_TX);
                            tma_load_2d(sA + stage * K1_A_BYTES, hmap, fb, kh * K1_BK, hrow, pol_h);
                            tma_load_2d(sB + stage * B_BYTES, &tmap_w, fb, kb * K1_BK, v0, pol_w);
                            tma_load_2d(sB + stage * B_BYTES + B_BYTES / 2, &tmap_w, fb, kb * K1_BK,
                                        v0 + K1_W_BOX_ROWS, pol_w);
                        }
                        if (++kh == KBH)
                            kh = 0;
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // no TMA write may still be landing in shared memory when the CTA
            // exits: a stage's last fill has landed once the UMMA released it
            // (after an abort the bounded wait lets it land anyway)
            for (int s = 0; s < STAGES; ++s)
                if (issued & (1u << s))
                    drain_wait(empty(s), (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ UMMA issuer (the even CTA of a pair)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            // a commit arrives on this CTA's barrier and, in a pair, on the peer's
            auto commit_both = [&](uint32_t bar) {
                if (PAIR) {
                    umma_commit_pair(bar);
                    umma_commit_pair(mapa_shared(bar, 1));
                } else {
                    umma_commit(bar);
                }
            };
            while (ok) {
                int u = -1;
                if (!ring.take(u, true, rank, abort_flag, budget) || u < 0)
                    break;
                const Unit w = unit_of(u, a);
                const int nt = tiles_in_chunk(w.ch, a.V);
                for (int j = 0; ok && j < nt; ++j) {
                    if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag, budget)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(acc * K1_BN);
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!mbar_wait(full(stage), phase, abort_flag, budget)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = sdesc_kmajor_sw128(sA + stage * K1_A_BYTES);
                        const uint64_t bd = sdesc_kmajor_sw128(sB + stage * B_BYTES);
#pragma unroll
                        for (int k = 0; k < K1_BK / 16; ++k) {   // +32 bytes along K per step
                            if (PAIR)
                                umma_bf16_pair(d, ad + 2u * k, bd + 2u * k, IDESC, (kb | k) != 0);
                            else
                                umma_bf16(d, ad + 2u * k, bd + 2u * k, IDESC, (kb | k) != 0);
                        }
                        commit_both(empty(stage));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok)
                        break;
                    commit_both(tfull(acc));
                    acc ^= 1;
                    if (acc == 0)
                        acc_phase ^= 1u;
                }
            }
            // every UMMA issued has finished (in both CTAs' TMEM) before TMEM is released
            if (PAIR)
                umma_commit_pair(drain);
            else
                umma_commit(drain);
            drain_wait(drain, 0);
        }
    } else if (MODE == 1) {
        // ---------------------------------------------------- backward epilogue, warps 2..5
        const int q = warp & 3;
        const int r_in_tile = q * 32 + lane;
        const float zscale = LOG2E * a.inv_temp;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        while (ok) {
            int u = -1;
            if (!ring.take(u, lane == 0, rank, abort_flag, budget) || u < 0)
                break;
            const Unit w = unit_of(u, a);
            const int nt = tiles_in_chunk(w.ch, a.V);
            const int row = (w.mt * CL + static_cast<int>(rank)) * K1_BM + r_in_tile;
            const bool live = row < a.N;
            const int tgt = live ? __ldg(a.targets + row) : -1;
            const float gs = live ? __ldg(a.grad + row) * a.inv_temp : 0.f;   // g / tau
            const float l2 = live ? __ldg(a.lse_in + row) * LOG2E : 0.f;     // p = 2^(z zscale - l2)
            TIM_DCHECK(!live || (isfinite(gs) && isfinite(l2)), a.status, TIM_CHECK_BACKWARD_INPUT, row,
                       __float_as_uint(isfinite(gs) ? l2 : gs));
            uint16_t *dzrow = a.dz + static_cast<size_t>(live ? row : 0) * static_cast<size_t>(a.dz_ld);
            for (int j = 0; j < nt; ++j) {
                if (!mbar_wait(tfull(acc), acc_phase, abort_flag, budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int c0 = w.ch * K1_VCHUNK + j * K1_BN;
                const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * K1_BN);
#pragma unroll 1
                for (int sc = 0; sc < K1_BN / SUBCOLS; ++sc) {
                    const int col0 = c0 + sc * SUBCOLS;
                    if (col0 >= a.V)
                        break;
                    float v[SUBCOLS];
                    __syncwarp();
                    tmem_load32(tb + static_cast<uint32_t>(sc * SUBCOLS), v);
                    uint32_t pk[SUBCOLS / 2];
#pragma unroll
                    for (int jj = 0; jj < SUBCOLS; jj += 2) {
                        const float p0 = ex2(fmaf(v[jj], zscale, -l2));
                        const float p1 = ex2(fmaf(v[jj + 1], zscale, -l2));
                        const float d0 = gs * ((col0 + jj == tgt ? 1.f : 0.f) - p0);
                        const float d1 = gs * ((col0 + jj + 1 == tgt ? 1.f : 0.f) - p1);
                        pk[jj / 2] = pack_bf16x2(d0, d1);
                    }
                    TIM_DCHECK(!live || (row < a.N && col0 < a.dz_ld), a.status, TIM_CHECK_STORE, row, col0);
                    if (live) {
                        if (col0 + SUBCOLS <= a.V) {   // 64 bytes at a 64-byte offset of a 16-byte aligned row
                            uint4 *dst = reinterpret_cast<uint4 *>(dzrow + col0);
#pragma unroll
                            for (int k = 0; k < SUBCOLS / 8; ++k)
                                dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                        } else {
#pragma unroll
                            for (int jj = 0; jj < SUBCOLS; ++jj)
                                if (col0 + jj < a.V)
                                    dzrow[col0 + jj] = static_cast<uint16_t>(pk[jj / 2] >> (16 * (jj & 1)));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        mbar_arrive_remote_cta(tempty_pair(acc));
                    else
                        mbar_arrive(tempty(acc));
                }
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
        }
    } else {
        // ---------------------------------------------------- epilogue, warps 2..5
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        const int r_in_tile = q * 32 + lane;
        const float zscale = LOG2E * a.inv_temp;   // e^(z / tau) = 2^(z zscale)
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        while (ok) {
            int u = -1;
            if (!ring.take(u, lane == 0, rank, abort_flag, budget) || u < 0)
                break;
            const Unit w = unit_of(u, a);
            const int nt = tiles_in_chunk(w.ch, a.V);
            const int row = (w.mt * CL + static_cast<int>(rank)) * K1_BM + r_in_tile;
            const int tgt = row < a.N ? __ldg(a.targets + row) : -1;
            float run_m = -INFINITY, run_s = 0.f, zt = 0.f;
            bool found = false;
            for (int j = 0; j < nt; ++j) {
                if (!mbar_wait(tfull(acc), acc_phase, abort_flag, budget)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int c0 = w.ch * K1_VCHUNK + j * K1_BN;
                const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * K1_BN);
#pragma unroll 1
                for (int sc = 0; sc < K1_BN / SUBCOLS; ++sc) {
                    const int col0 = c0 + sc * SUBCOLS;
                    if (col0 >= a.V)
                        break;
                    float v[SUBCOLS];
                    __syncwarp();   // tcgen05.ld is .sync.aligned: the warp must be converged
                    tmem_load32(tb + static_cast<uint32_t>(sc * SUBCOLS), v);
                    if (col0 + SUBCOLS > a.V) {
#pragma unroll
                        for (int jj = 0; jj < SUBCOLS; ++jj)
                            if (col0 + jj >= a.V)
                                v[jj] = -INFINITY;
                    }
#ifdef TIM_DEBUG
                    if (row < a.N) {   // a logit of a real column is finite unless h or W is not
                        int badc = -1;
#pragma unroll
                        for (int jj = 0; jj < SUBCOLS; ++jj)
                            if (col0 + jj < a.V && !isfinite(v[jj]) && badc < 0)
                                badc = jj;
                        TIM_DCHECK(badc < 0, a.status, TIM_CHECK_LOGIT, row,
                                   (static_cast<uint64_t>(col0 + badc) << 32) | __float_as_uint(v[badc < 0 ? 0 : badc]));
                    }
#endif
                    float m0 = v[0], m1 = v[1], m2 = v[2], m3 = v[3];
#pragma unroll
                    for (int jj = 4; jj < SUBCOLS; jj += 4) {
                        m0 = fmaxf(m0, v[jj]);
                        m1 = fmaxf(m1, v[jj + 1]);
                        m2 = fmaxf(m2, v[jj + 2]);
                        m3 = fmaxf(m3, v[jj + 3]);
                    }
                    const float new_m = fmaxf(run_m, fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
                    const float nm = new_m * zscale;
                    const float rescale = ex2(fmaf(run_m, zscale, -nm));
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
                    for (int jj = 0; jj < SUBCOLS; jj += 4) {
                        s0 += ex2(fmaf(v[jj], zscale, -nm));
                        s1 += ex2(fmaf(v[jj + 1], zscale, -nm));
                        s2 += ex2(fmaf(v[jj + 2], zscale, -nm));
                        s3 += ex2(fmaf(v[jj + 3], zscale, -nm));
                    }
                    run_s = fmaf(run_s, rescale, (s0 + s1) + (s2 + s3));
                    run_m = new_m;
                    const unsigned off = static_cast<unsigned>(tgt - col0);
                    if (off < static_cast<unsigned>(SUBCOLS)) {
#pragma unroll
                        for (int jj = 0; jj < SUBCOLS; ++jj)
                            if (off == static_cast<unsigned>(jj))
                                zt = v[jj];
                        found = true;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        mbar_arrive_remote_cta(tempty_pair(acc));
                    else
                        mbar_arrive(tempty(acc));
                }
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
            if (!ok)
                break;
            TIM_DCHECK(w.ch < a.num_chunks, a.status, TIM_CHECK_STORE, row, w.ch);
            if (row < a.N) {
                a.part[static_cast<size_t>(row) * a.num_chunks + w.ch] = make_float2(run_m, run_s);
                if (found)
                    a.za[row] = zt;
            }
        }
    }

    tc_fence_before();
    // no CTA leaves while the other CTA of its pair may still load into the
    // pair's stages, arrive on its barriers or have UMMA write its TMEM
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem, TMEM_COLS);
        else
            tmem_dealloc(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
}

// Folds the per-chunk (max, sum) pairs of a row (m_c is a max of raw logits,
// s_c a sum of e^((z - m_c) / tau)): M = max_c m_c, S = sum_c s_c e^((m_c - M) / tau),
// lse = M / tau + ln S, l = z_a / tau - lse.  One warp per row:
// lane i takes chunks i, i + 32, ... in order, then a fixed xor-shuffle tree sums
// the lanes and lane 0's value is used.  The order depends on the number of
// chunks (a function of V) only.
__global__ void __launch_bounds__(256)
    k1_combine_kernel(const float2 *__restrict__ part, const float *__restrict__ za,
                      const int32_t *__restrict__ targets, int32_t N, int32_t V, int32_t num_chunks,
                      float inv_temp, float *__restrict__ out_logp, float *__restrict__ out_lse, int *status)
{
    pdl_wait();   // the partials come from k1_main_kernel
    pdl_launch_dependents();
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= N)
        return;   // uniform over the warp
    const float2 *p = part + t * num_chunks;
    float M = -INFINITY;
    for (int c = lane; c < num_chunks; c += 32)
        M = fmaxf(M, p[c].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float S = 0.f;
    for (int c = lane; c < num_chunks; c += 32) {
        const float2 q = p[c];
        S = fmaf(q.y, expf((q.x - M) * inv_temp), S);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        S += __shfl_xor_sync(0xffffffffu, S, o);
    if (lane == 0) {
        const float lse = M * inv_temp + logf(S);
        out_lse[t] = lse;
        const int a = targets[t];
        TIM_DCHECK(a < V, status, TIM_CHECK_TARGET, t, static_cast<uint32_t>(a));   // negative: ignore label
        out_logp[t] = (a >= 0 && a < V) ? za[t] * inv_temp - lse : __int_as_float(0x7fc00000);
    }
}

} // namespace

int64_t k1_band_bytes()
{
    static const int64_t v = [] {
        const char *e = std::getenv("TIM_K1_BAND_MB");
        const long long mb = e ? std::atoll(e) : 0;
        return mb > 0 ? static_cast<int64_t>(mb) << 20 : K1_BAND_BYTES;
    }();
    return v;
}

cudaError_t k1_prepare_device()
{
    cudaError_t e = cudaSuccess;
    for (auto kernel : {k1_main_kernel<0, K1_CLUSTER>, k1_main_kernel<1, K1_CLUSTER>, k1_main_kernel<0, 1>,
                        k1_main_kernel<1, 1>})
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(K1_SMEM_BYTES));
    return e;
}

cudaError_t k1_launch_main(const CUtensorMap &tmap_h, const CUtensorMap &tmap_w, const CUtensorMap &tmap_h_tail,
                           const K1Args &a,
                           cudaStream_t stream, int mode)
{
    static int max_clusters[2][2][64] = {};   // per cluster size, mode and device, found once
    const int cl = a.cluster == 1 ? 1 : K1_CLUSTER;
    const int ci = cl == 1 ? 1 : 0;
    auto kernel = cl == 1 ? (mode == 1 ? k1_main_kernel<1, 1> : k1_main_kernel<0, 1>)
                          : (mode == 1 ? k1_main_kernel<1, K1_CLUSTER> : k1_main_kernel<0, K1_CLUSTER>);
    const int md = mode == 1 ? 1 : 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.blockDim = dim3(K1_THREADS, 1, 1);
    cfg.dynamicSmemBytes = K1_SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev >= 0 && dev < 64 && max_clusters[ci][md][dev] == 0) {
        int n = 0;
        cfg.gridDim = dim3(cl * 1024, 1, 1);
        e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
        if (e != cudaSuccess)
            return e;
        max_clusters[ci][md][dev] = n > 0 ? n : 1;
    }
    const int clusters =
        static_cast<int>(std::min<int64_t>(a.units, dev >= 0 && dev < 64 ? max_clusters[ci][md][dev] : 1));
    cfg.gridDim = dim3(cl * clusters, 1, 1);
    cfg.numAttrs = 2;
    if ((e = cudaMemsetAsync(a.sched, 0, sizeof(int), stream)) != cudaSuccess)   // units are claimed from 0
        return e;
    return cudaLaunchKernelEx(&cfg, kernel, tmap_h, tmap_w, tmap_h_tail, a);
}

// The padded last m-tile: rows [0, rows) of src copied, rows [rows, K1_BM) zero,
// in 16-byte units (rows of D bf16, D % 8 == 0).
__global__ void __launch_bounds__(256) k1_pad_tail_kernel(const uint4 *__restrict__ src, int64_t rows, int64_t D,
                                                         uint4 *__restrict__ dst)
{
    const int64_t per_row = D / 8, total = static_cast<int64_t>(K1_BM) * per_row;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        dst[i] = i < rows * per_row ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t k1_launch_pad_tail(const void *src, int64_t rows, int64_t D, void *dst, cudaStream_t stream)
{
    const int64_t total = static_cast<int64_t>(K1_BM) * (D / 8);
    const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 1024));
    k1_pad_tail_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src), rows, D,
                                                   static_cast<uint4 *>(dst));
    return cudaGetLastError();
}

cudaError_t k1_launch_combine(const float2 *part, const float *za, const int32_t *targets,
                              int32_t N, int32_t V, int32_t num_chunks, float inv_temp, float *out_logp,
                              float *out_lse, int *status, cudaStream_t stream)
{
    const int threads = 256;   // 8 rows per CTA, one warp each
    const int blocks = static_cast<int>((static_cast<int64_t>(N) * 32 + threads - 1) / threads);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k1_combine_kernel, part, za, targets, N, V, num_chunks, inv_temp, out_logp,
                              out_lse, status);
}

} // namespace tim
