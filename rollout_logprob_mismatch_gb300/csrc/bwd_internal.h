// bwd_internal.h -- the backward's two contractions (dh = dz W, dW = dz^T h):
// tile shapes, arguments and launcher of the pair-UMMA GEMM.  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tim {

// C[m, n] (+)= sum_k A[m, k] B[n, k]: a CTA pair computes a 256 x 256 tile of C
// (128 rows of it per CTA, TMEM lane = row), k ascending in 64-wide steps.
constexpr int G_BM = 128;      // rows of C per CTA
constexpr int G_BN = 256;      // columns of C per tile (UMMA N)
constexpr int G_BK = 64;       // k per pipeline stage (one 128-byte swizzled row)
constexpr int G_STAGES = 7;
constexpr int G_THREADS = 192; // warp 0 TMA, warp 1 UMMA + TMEM, warps 2-5 epilogue
constexpr uint32_t G_A_BYTES = G_BM * G_BK * 2;          // per CTA and stage
constexpr uint32_t G_B_BYTES = (G_BN / 2) * G_BK * 2;    // the CTA's half of the B tile
constexpr uint32_t G_TAIL_BYTES = 512;                   // unit ring, mbarriers, TMEM address, abort flag
constexpr uint32_t G_SMEM_BYTES = G_STAGES * (G_A_BYTES + G_B_BYTES) + G_TAIL_BYTES + 1024;
// TMA boxes: K-major operands [128 rows x 64 k]; MN-major ones [64 k rows x 64
// m/n] (128 bytes of m/n per k), two per CTA and stage.
constexpr int G_KMAJOR_BOX_ROWS = 128;
constexpr int G_MNMAJOR_BOX_ROWS = 64;

struct GemmArgs {
    float *C;           // row-major [M][ldc] fp32, 16-byte aligned, ldc % 4 == 0
    int64_t ldc;
    int32_t M, N, K;    // N % 4 == 0
    int32_t n_blocks;   // ceil(N / 256)
    int32_t units;      // ceil(M / 256) * n_blocks, n fastest
    int32_t accumulate; // 1: C += A B^T; 0: C = A B^T
    int32_t b_keep;     // B is small and read by every tile: loaded with an L2 evict-last hint
    int *sched;         // unit counter, zeroed by the launcher
    int *status;        // device status word
    uint64_t wait_budget_ns;
};

cudaError_t gemm_prepare_device();

// a_mn / b_mn: A (resp. B) is stored MN-major (the m (n) index contiguous, a
// [K][M] ([K][N]) matrix); else K-major ([M][K], [N][K]); B must be MN-major.
// tmap_a / tmap_b use the box shapes above.  Zeroes a.sched on the stream,
// then launches at most as many pairs as fit on the device at once.
cudaError_t gemm_launch(const CUtensorMap &tmap_a, const CUtensorMap &tmap_b, bool a_mn, bool b_mn,
                        const GemmArgs &a, cudaStream_t stream);

} // namespace tim
