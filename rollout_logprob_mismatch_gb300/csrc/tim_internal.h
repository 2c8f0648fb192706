// tim_internal.h -- declarations shared by the library's own translation units
// (kernels and the C-ABI layer).  Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tim {

// ---------------------------------------------------------------- token logprob (K1)
// Tile shape of the fused LM head.  These, and the vocabulary chunk, are
// compile-time constants: the reduction order of a row depends on D and V only.
constexpr int K1_BM = 128;        // rows (tokens) per tile = TMEM lanes
constexpr int K1_BN = 256;        // vocabulary columns per tile = UMMA N
constexpr int K1_BK = 64;         // bf16 elements per 128-byte swizzled row
constexpr int K1_STAGES = 4;      // TMA -> UMMA pipeline depth
constexpr int K1_VCHUNK = 1024;   // vocabulary columns per split-V partial
constexpr int K1_THREADS = 192;   // warp 0 TMA, warp 1 UMMA + TMEM, warps 2-5 epilogue

constexpr uint32_t K1_A_BYTES = K1_BM * K1_BK * 2;
constexpr uint32_t K1_B_BYTES = K1_BN * K1_BK * 2;
constexpr uint32_t K1_STAGE_BYTES = K1_A_BYTES + K1_B_BYTES;
constexpr uint32_t K1_BAR_BYTES = 256;
constexpr uint32_t K1_SMEM_BYTES = K1_STAGES * K1_STAGE_BYTES + K1_BAR_BYTES + 1024;

inline int64_t k1_num_chunks(int64_t V) { return (V + K1_VCHUNK - 1) / K1_VCHUNK; }

struct K1Args {
    const int32_t *targets;   // [N]
    float2 *part;             // [num_chunks][N]: per-chunk (max, sum of exp(z - max))
    float *za;                // [N]: the target's logit, written by the chunk holding it
    int *status;              // device status word
    int32_t N, D, V;
    int32_t num_m_tiles, num_chunks, band, units;
    uint64_t wait_budget_ns;
};

cudaError_t k1_launch_main(const CUtensorMap &tmap_h, const CUtensorMap &tmap_w, const K1Args &a,
                           int grid, cudaStream_t stream);
cudaError_t k1_launch_combine(const float2 *part, const float *za, const int32_t *targets,
                              int32_t N, int32_t V, int32_t num_chunks, float *out_logp,
                              float *out_lse, cudaStream_t stream);
cudaError_t k1_prepare_device();   // per-device function attributes

// ---------------------------------------------------------------- mismatch stats (K2)
constexpr int K2_THREADS = 256;        // tokens per round of one sequence
constexpr int K2_GROUP = 16;           // rounds summed plainly before the compensated fold
constexpr int K2_BATCH_THREADS = 512;
constexpr int K2_REC = 16;             // doubles per sequence record in the workspace

struct K2Args {
    const float *l_tr, *l_ro;
    const uint8_t *mask;
    const int32_t *off;
    int32_t S;
    int64_t N;
    float C;
    float log_c_down;      // largest float <= ln C: delta > this  <=>  r > C
    double tau;            // rejection threshold (already defaulted)
    int32_t estimator;     // 3 or 1
    float *token_weight;   // optional
    float *seq_stats;      // [S][12]
    int32_t *seq_flags;    // [S]
    double *batch;         // [20]
    double *rec;           // workspace [S][K2_REC]
    int *status;
};

cudaError_t k2_launch(const K2Args &a, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- shared by the C-ABI files
cudaError_t status_word_address(int **out);   // the library's device status word
int record_error(int code, const char *msg);  // message for tim_last_error()

} // namespace tim
