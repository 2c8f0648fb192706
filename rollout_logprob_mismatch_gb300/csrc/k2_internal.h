// k2_internal.h -- the mismatch pass's launch shape, workspace and arguments.
// Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace tim {

// ---------------------------------------------------------------- mismatch stats (K2)
constexpr int K2_WARPS = 8;                        // warps per CTA (three CTAs per SM)
constexpr int K2_CTAS_PER_SM = 3;
constexpr int K2_THREADS = K2_WARPS * 32;
constexpr int K2_CHUNK = 448;                      // tokens per staged chunk (a multiple of 64)
constexpr int K2_STAGES = 2;                       // staged chunks per warp (double buffer)
constexpr int K2_F_BYTES = K2_CHUNK * 4 + 32;      // one fp32 array's chunk + 16-byte alignment slack
constexpr int K2_M_BYTES = K2_CHUNK + 32;          // the mask's chunk + slack
constexpr int K2_STAGE_BYTES = 2 * K2_F_BYTES + K2_M_BYTES;
constexpr int K2_BAR_BYTES = K2_WARPS * K2_STAGES * 8;
constexpr int K2_SMEM_BYTES = K2_BAR_BYTES + K2_WARPS * K2_STAGES * K2_STAGE_BYTES;
constexpr int64_t K2_LONG = 8192;                  // longer sequences are reduced by a whole CTA
constexpr int K2_CLAIM_BLOCK = 4;                  // sequences per ticket in the bulk of a large batch
constexpr int K2_FOLD_THREADS = 256;               // fold CTA
constexpr int K2_FOLD_SEQS = 4 * K2_FOLD_THREADS;  // sequences per fold CTA
constexpr int K2_REC_WORDS = 16;                   // 4-byte words per sequence record (64 bytes a sequence)
constexpr int K2_PART_WORDS = 40;                  // 4-byte words per fold partial
static_assert(K2_STAGE_BYTES % 16 == 0 && K2_BAR_BYTES % 16 == 0, "bulk-copy destinations stay 16-byte aligned");

// Workspace: the sequence counter and the fold's ticket (256 bytes, zeroed per
// call), the records (16 words per sequence), the fold partials.
inline int64_t k2_blocks(int64_t S) { return (S + K2_FOLD_SEQS - 1) / K2_FOLD_SEQS; }
inline size_t k2_workspace_bytes(int64_t S)
{
    return 256 + static_cast<size_t>(S) * K2_REC_WORDS * 4 + static_cast<size_t>(k2_blocks(S)) * K2_PART_WORDS * 4;
}

struct K2Args {
    const float *l_tr, *l_ro;
    const uint8_t *mask;
    const int32_t *off;
    int32_t S;
    int64_t N;
    float C;
    float log_c_down;      // largest float <= ln C: delta > this  <=>  r > C
    float tau;             // rejection threshold (already defaulted)
    uint64_t wait_budget_ns;
    int32_t estimator;     // 3 or 1
    float *token_weight;   // optional
    float *seq_stats;      // [S][12]
    int32_t *seq_flags;    // [S]
    double *batch;         // [20]
    int *claim;            // workspace: sequence counter ...
    int *blk_done;         // ... and the fold CTAs' ticket (zeroed by k2_launch)
    uint32_t *rec;         // workspace: sequence records, [S][K2_REC_WORDS]
    uint32_t *part;        // workspace: block partials, [ceil(S / K2_FOLD_SEQS)][K2_PART_WORDS]
    int32_t stats_vec;     // seq_stats is 16-byte aligned (rows written as float4)
    int *status;
};

// The fold alone, over a.rec (a.S records): 256 bytes (the ticket, zeroed
// here) then the fold partials.
inline size_t k2_fold_workspace_bytes(int64_t S) { return 256 + static_cast<size_t>(k2_blocks(S)) * K2_PART_WORDS * 4; }

cudaError_t k2_launch(const K2Args &a, int num_sms, cudaStream_t stream);
cudaError_t k2_launch_fold(const K2Args &a, cudaStream_t stream);
cudaError_t k2_prepare_device();   // per-device function attributes

} // namespace tim
