// ppo_internal.h -- launch parameters of the TIS-weighted PPO surrogate kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tim {

constexpr int PPO_WARPS = 8;
constexpr int PPO_THREADS = PPO_WARPS * 32;
constexpr int PPO_CTAS_PER_SM = 3;
constexpr int PPO_CHUNK = 256;                      // tokens per warp step: 8 per lane, loaded before use
constexpr int64_t PPO_LONG = 8192;                  // longer sequences are reduced by a whole CTA
constexpr int PPO_CLAIM_BLOCK = 4;                  // sequences per ticket in the bulk of a large batch
constexpr int PPO_FOLD_THREADS = 256;
constexpr int PPO_FOLD_SEQS = 4 * PPO_FOLD_THREADS; // sequences per fold CTA
constexpr int PPO_REC_WORDS = 6;                    // 4-byte words per sequence record (structure of arrays)
constexpr int PPO_PART_WORDS = 16;                  // 4-byte words per fold partial
static_assert(PPO_CHUNK % 64 == 0, "a chunk is whole 64-token lane groups");

inline size_t ppo_workspace_bytes(int64_t S)
{
    const int64_t parts = (S + PPO_FOLD_SEQS - 1) / PPO_FOLD_SEQS;
    return static_cast<size_t>(S) * PPO_REC_WORDS * 4 + static_cast<size_t>(parts) * PPO_PART_WORDS * 4 + 1024;
}

struct PpoArgs {
    const float *l_th, *l_old, *l_ro, *adv;
    const uint8_t *mask;
    const int32_t *off;
    int32_t S;
    int64_t N;
    float C;
    float log_c_down;      // largest float <= ln C:              l_old - l_ro > this  <=>  w capped
    float log_hi_down;     // largest float <= ln(1 + eps_high):  l_th - l_old > this  <=>  r > 1 + eps_high
    float log_lo_up;       // smallest float >= ln(1 - eps_low):  l_th - l_old < this  <=>  r < 1 - eps_low
    float r_hi, r_lo;      // 1 + eps_high, 1 - eps_low
    float *token_loss;     // optional
    float *token_grad;     // optional
    float *seq_loss;       // [S]
    double *batch;         // [TIM_PPO_FIELDS]
    uint32_t *rec;         // workspace: sequence records, [PPO_REC_WORDS][S]
    uint32_t *part;        // workspace: fold partials, [ceil(S / PPO_FOLD_SEQS)][PPO_PART_WORDS]
    unsigned *ticket;      // workspace: fold CTAs finished (zeroed by ppo_seq_kernel)
    int *claim;            // workspace: the sequences' ticket counter (zeroed before ppo_seq_kernel)
    int *status;
};

cudaError_t ppo_launch(const PpoArgs &a, int num_sms, cudaStream_t stream);

} // namespace tim
