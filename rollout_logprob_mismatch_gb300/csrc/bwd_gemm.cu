// bwd_gemm.cu -- the backward's two contractions as 2-SM tcgen05 GEMMs (sm_103a).
//
// The gradient of l_t = log softmax(h_t W^T / tau)[a_t], weighted by g_t, is
// dz = (g / tau)(onehot(a) - softmax(z / tau)) per logit (the fused kernel in
// k1_token_logprob.cu writes it in bf16), then
//   dh = dz W        [rows, D] = [rows, V] [V, D]     A = dz   (K-major), B = W (MN-major)
//   dW (+)= dz^T h   [V, D]    = [V, rows] [rows, D]  A = dz^T (MN-major), B = h (MN-major)
// (HN page "Train-infer mismatch for Open-weight MoE RL", the unclipped
// importance-sampling gradient, which weights the gradient of each token's log
// probability; icarus "RL: Training Inference Mismatch", the trainer's
// recompute of log p).
//
// C[m, n] = sum_k A[m, k] B[n, k]: one persistent launch computes both (dh's
// tiles, long in k, claimed first, then dW's short ones, so pairs never idle
// through a last partial wave of dh).  CTA pairs claim 256 x 256 tiles of C in
// order (unit_ring.cuh; n fastest), and per tile
//   warp 0     TMA: the CTA's 128 rows of A and its half (128) of the B tile,
//              64 k per stage, 128-byte swizzle, into a 7-stage ring; both
//              CTAs' bytes complete on the even CTA's barrier;
//   warp 1     (even CTA) tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16,
//              bf16 -> fp32, k ascending, into one of two TMEM accumulators;
//   warps 2-5  epilogue: tcgen05.ld, one row of C per thread, 128-byte
//              streaming stores (C += when accumulating).
// Each element of C sums its products in one order fixed by K alone (64-wide
// k steps ascending, the tensor core's fixed order inside a step): a row of dh
// depends on its own dz row, W and V only, whatever else the batch holds.
#include <algorithm>
#include <type_traits>

#include <cuda_bf16.h>

#include "bwd_internal.h"
#include "tim_internal.h"
#include "tim_ptx.cuh"
#include "unit_ring.cuh"
#include "../../include/tim.h"

namespace tim {
namespace {

constexpr uint32_t TMEM_COLS = 2 * G_BN;
constexpr uint32_t MN_BLOCK_BYTES = G_MNMAJOR_BOX_ROWS * 128;   // 64 k rows of 64 m/n elements
static_assert(UNIT_RING_BYTES + 8 * (2 * G_STAGES + 5) + 8 <= G_TAIL_BYTES, "tail area too small");
static_assert(G_A_BYTES == 2 * MN_BLOCK_BYTES && G_B_BYTES == 2 * MN_BLOCK_BYTES, "two MN blocks per operand tile");

// Problem 0's A is K-major, problem 1's MN-major; B is MN-major in both.
__global__ void __launch_bounds__(G_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a0, const __grid_constant__ CUtensorMap tmap_b0,
                     const __grid_constant__ CUtensorMap tmap_a1, const __grid_constant__ CUtensorMap tmap_b1,
                     const __grid_constant__ GemmArgs a)
{
    constexpr uint32_t STAGE_TX = G_A_BYTES + G_B_BYTES;   // bytes each CTA loads per stage
    constexpr uint32_t B_KSTEP = 128u;   // MN-major B: 16 rows of 128 bytes per K = 16 (16-byte units)
    using AKmajor = std::integral_constant<bool, false>;
    using AMNmajor = std::integral_constant<bool, true>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + G_STAGES * G_A_BYTES;
    uint8_t *tail_area = smem + G_STAGES * (G_A_BYTES + G_B_BYTES);
    // users of a unit: the UMMA issuer, 4 epilogue warps per CTA, the odd CTA's producer
    UnitRing<2, 1 + 8 + 1> ring(tail_area);
    uint64_t *bars = reinterpret_cast<uint64_t *>(tail_area + UNIT_RING_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (G_STAGES + s); };
    auto tfull = [&](int b) { return bar0 + 8u * (2 * G_STAGES + b); };
    auto tempty = [&](int b) { return bar0 + 8u * (2 * G_STAGES + 2 + b); };
    const uint32_t drain = bar0 + 8u * (2 * G_STAGES + 4);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * G_STAGES + 5);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(full(s), 1);    // the even CTA's counts: one arrival expecting both CTAs' bytes
            mbar_init(empty(s), 1);   // released by the pair UMMA
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull(b), 1);
            mbar_init(tempty(b), 8);   // the even CTA's counts: the epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        ring.init();
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a0);
        tma_prefetch_desc(&tmap_b0);
        if (a.p[1].units > 0) {
            tma_prefetch_desc(&tmap_a1);
            tma_prefetch_desc(&tmap_b1);
        }
    }
    pdl_wait();   // the operands and the unit counter are written by earlier work
    pdl_launch_dependents();
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();   // both CTAs' barriers exist before the other CTA's TMA, UMMA or threads reach them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t rank = cluster_ctarank();
    const uint64_t budget = a.wait_budget_ns;
    const int units0 = a.p[0].units, units = a.p[0].units + a.p[1].units;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint64_t pol = l2_policy_evict_normal(), pol_keep = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            // the k loop of one tile of problem P (A K-major or MN-major)
            auto produce = [&](auto a_mn, const GemmProblem &P, const CUtensorMap *ma, const CUtensorMap *mbm,
                               int lu) -> bool {
                constexpr bool A_MN = decltype(a_mn)::value;
                const uint64_t pol_b = P.b_keep ? pol_keep : pol;
                const int mb = lu / P.n_blocks, nb = lu - (lu / P.n_blocks) * P.n_blocks;
                const int m0 = mb * (2 * G_BM) + static_cast<int>(rank) * G_BM;     // this CTA's rows of C
                const int n0 = nb * G_BN + static_cast<int>(rank) * (G_BN / 2);    // this CTA's half of B
                const int KT = (P.K + G_BK - 1) / G_BK;
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait(empty(stage), phase ^ 1u, abort_flag, budget))
                        return false;
                    const uint32_t f = mapa_shared(full(stage), 0);   // the even CTA's barrier
                    if (rank == 0)
                        mbar_arrive_expect_tx(full(stage), 2 * STAGE_TX);
                    const int k0 = kb * G_BK;
                    // innermost coordinates are whole 16 bytes (8 bf16) and none is negative
                    TIM_DCHECK(((m0 | n0 | k0) & 7) == 0 && m0 >= 0 && n0 >= 0, a.status, TIM_CHECK_TMA_COORD, k0,
                               static_cast<uint64_t>(m0) << 32 | static_cast<uint32_t>(n0));
                    const uint32_t dA = sA + stage * G_A_BYTES, dB = sB + stage * G_B_BYTES;
                    if (A_MN) {
                        tma_load_2d_pair(dA, ma, f, m0, k0, pol);
                        tma_load_2d_pair(dA + MN_BLOCK_BYTES, ma, f, m0 + 64, k0, pol);
                    } else {
                        tma_load_2d_pair(dA, ma, f, k0, m0, pol);
                    }
                    tma_load_2d_pair(dB, mbm, f, n0, k0, pol_b);
                    tma_load_2d_pair(dB + MN_BLOCK_BYTES, mbm, f, n0 + 64, k0, pol_b);
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return true;
            };
            int ahead = -1;   // the even CTA claims one unit ahead of its loads
            bool ok = rank != 0 || ring.claim(a.sched, units, ahead, abort_flag, budget);
            while (ok) {
                int u = -1;
                if (!(rank == 0 ? ring.next(a.sched, units, u, ahead, abort_flag, budget)
                                : ring.take(u, true, rank, abort_flag, budget)))
                    break;
                if (u < 0)
                    break;
                TIM_DCHECK(u < units, a.status, TIM_CHECK_UNIT, u, units);
                ok = u < units0 ? produce(AKmajor{}, a.p[0], &tmap_a0, &tmap_b0, u)
                                : produce(AMNmajor{}, a.p[1], &tmap_a1, &tmap_b1, u - units0);
            }
            // a stage's last fill has landed once the UMMA released it
            for (int s = 0; s < G_STAGES; ++s)
                if (issued & (1u << s))
                    drain_wait(empty(s), (last_par >> s) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ UMMA issuer (the even CTA)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            auto commit_both = [&](uint32_t bar) {
                umma_commit_pair(bar);
                umma_commit_pair(mapa_shared(bar, 1));
            };
            // the k loop of one tile into accumulator d
            auto mma = [&](auto a_mn, const GemmProblem &P, uint32_t d) -> bool {
                constexpr bool A_MN = decltype(a_mn)::value;
                constexpr uint32_t IDESC = idesc_bf16_f32(2 * G_BM, G_BN, A_MN, true);
                // descriptor start-address step (16-byte units) per K = 16: 32 bytes
                // along a K-major row, or 16 rows of 128 bytes in an MN-major tile
                constexpr uint32_t A_KSTEP = A_MN ? 128u : 2u;
                const int KT = (P.K + G_BK - 1) / G_BK;
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait(full(stage), phase, abort_flag, budget))
                        return false;
                    tc_fence_after();
                    const uint32_t aa = sA + stage * G_A_BYTES, ba = sB + stage * G_B_BYTES;
                    const uint64_t ad = A_MN ? sdesc_mnmajor_sw128(aa, MN_BLOCK_BYTES) : sdesc_kmajor_sw128(aa);
                    const uint64_t bd = sdesc_mnmajor_sw128(ba, MN_BLOCK_BYTES);
#pragma unroll
                    for (int k = 0; k < G_BK / 16; ++k)
                        umma_bf16_pair(d, ad + A_KSTEP * k, bd + B_KSTEP * k, IDESC, (kb | k) != 0);
                    commit_both(empty(stage));
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return true;
            };
            while (true) {
                int u = -1;
                if (!ring.take(u, true, rank, abort_flag, budget) || u < 0)
                    break;
                if (!mbar_wait(tempty(acc), acc_phase ^ 1u, abort_flag, budget))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * G_BN);
                if (!(u < units0 ? mma(AKmajor{}, a.p[0], d) : mma(AMNmajor{}, a.p[1], d)))
                    break;
                commit_both(tfull(acc));
                acc ^= 1;
                if (acc == 0)
                    acc_phase ^= 1u;
            }
            umma_commit_pair(drain);
            drain_wait(drain, 0);
        }
    } else {
        // ---------------------------------------------------- epilogue, warps 2..5
        const int q = warp & 3;   // TMEM lane quarter this warp may read
        int acc = 0;
        uint32_t acc_phase = 0;
        while (true) {
            int u = -1;
            if (!ring.take(u, lane == 0, rank, abort_flag, budget) || u < 0)
                break;
            const GemmProblem &P = u < units0 ? a.p[0] : a.p[1];
            const int lu = u < units0 ? u : u - units0;
            const int mb = lu / P.n_blocks, nb = lu - (lu / P.n_blocks) * P.n_blocks;
            const int M = P.M, N = P.N;
            const bool accumulate = P.accumulate != 0;
            const int row = mb * (2 * G_BM) + static_cast<int>(rank) * G_BM + q * 32 + lane;
            float *crow = P.C + static_cast<size_t>(row < M ? row : 0) * static_cast<size_t>(P.ldc);
            if (!mbar_wait(tfull(acc), acc_phase, abort_flag, budget))
                break;
            tc_fence_after();
            const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * G_BN);
#pragma unroll 1
            for (int sc = 0; sc < G_BN / 32; ++sc) {
                const int c0 = nb * G_BN + sc * 32;
                if (c0 >= N)
                    break;   // uniform over the warp
                float v[32];
                __syncwarp();
                tmem_load32(tb + static_cast<uint32_t>(sc * 32), v);
                TIM_DCHECK(row >= M || c0 + 32 <= P.ldc || c0 + 4 * ((N - c0 + 3) / 4) <= P.ldc, a.status,
                           TIM_CHECK_STORE, row, c0);
                if (row < M) {
                    float4 *dst = reinterpret_cast<float4 *>(crow + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (c0 + 4 * j < N) {   // N % 4 == 0: a group of four is all in or all out
                            float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                            if (accumulate) {
                                const float4 p = __ldcs(dst + j);
                                o.x += p.x;
                                o.y += p.y;
                                o.z += p.z;
                                o.w += p.w;
                            }
                            __stcs(dst + j, o);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_remote_cta(mapa_shared(tempty(acc), 0));
            acc ^= 1;
            if (acc == 0)
                acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    // no CTA leaves while the other CTA may still load into the pair's stages,
    // arrive on its barriers or have UMMA write its TMEM
    __syncwarp();
    cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag)
        atomicCAS(a.status, 0, static_cast<int>(TIM_ERR_TIMEOUT));
}

} // namespace

cudaError_t gemm_prepare_device()
{
    return cudaFuncSetAttribute(gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(G_SMEM_BYTES));
}

cudaError_t gemm_launch(const CUtensorMap (&tmap_a)[2], const CUtensorMap (&tmap_b)[2], const GemmArgs &a,
                        cudaStream_t stream)
{
    static int max_pairs[64] = {};   // per device, found once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.blockDim = dim3(G_THREADS, 1, 1);
    cfg.dynamicSmemBytes = G_SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dev >= 0 && dev < 64 && max_pairs[dev] == 0) {
        int n = 0;
        cfg.gridDim = dim3(2 * 1024, 1, 1);
        if ((e = cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel, &cfg)) != cudaSuccess)
            return e;
        max_pairs[dev] = n > 0 ? n : 1;
    }
    const int64_t units = static_cast<int64_t>(a.p[0].units) + a.p[1].units;
    const int pairs = static_cast<int>(std::min<int64_t>(units, dev >= 0 && dev < 64 ? max_pairs[dev] : 1));
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.numAttrs = 2;
    if ((e = cudaMemsetAsync(a.sched, 0, sizeof(int), stream)) != cudaSuccess)
        return e;
    return cudaLaunchKernelEx(&cfg, gemm_pair_kernel, tmap_a[0], tmap_b[0], tmap_a[1], tmap_b[1], a);
}

} // namespace tim
