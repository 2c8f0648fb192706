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

// One GEMM of a launch.
struct GemmProblem {
    float *C;           // row-major [M][ldc] fp32, 16-byte aligned, ldc % 4 == 0
    int64_t ldc;
    int32_t M, N, K;    // N % 4 == 0
    int32_t n_blocks;   // ceil(N / 256)
    int32_t units;      // ceil(M / 256) * n_blocks, n fastest
    int32_t accumulate; // 1: C += A B^T; 0: C = A B^T
    int32_t b_keep;     // B is small and read by every tile: loaded with an L2 evict-last hint
};

// Two independent GEMMs in one persistent launch: problem 0 with A K-major,
// problem 1 with A MN-major (the m index contiguous: a [K][M] matrix), both
// with B MN-major ([K][N]).  The pairs claim problem 0's tiles first, then
// problem 1's, so a pair done with a long tile of the first takes short tiles
// of the second instead of idling through a last partial wave.
struct GemmArgs {
    GemmProblem p[2];   // p[1].units may be 0
    int *sched;         // unit counter, zeroed by the launcher
    int *status;        // device status word
    uint64_t wait_budget_ns;
};

cudaError_t gemm_prepare_device();

// tmap_a[i] / tmap_b[i]: the operands of problem i with the box shapes above
// (A of problem 0: K-major box; the others: MN-major boxes).  Zeroes a.sched on
// the stream, then launches at most as many pairs as fit on the device at once.
cudaError_t gemm_launch(const CUtensorMap (&tmap_a)[2], const CUtensorMap (&tmap_b)[2], const GemmArgs &a,
                        cudaStream_t stream);

} // namespace tim
