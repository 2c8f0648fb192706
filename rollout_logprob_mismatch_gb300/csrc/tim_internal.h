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
constexpr int K1_CLUSTER = 2;     // CTAs per cluster: m-tiles sharing (multicasting) one W tile
constexpr int K1_W_BOX_ROWS = K1_BN / K1_CLUSTER;   // W rows each CTA of a cluster loads
// Units walk the vocabulary in bands of m-tiles whose h rows (at most this many
// bytes) stay in L2 while the band's clusters stream each W chunk from HBM once.
// (TIM_K1_BAND_MB overrides it; the band changes the order of work, never a result.)
constexpr int64_t K1_BAND_BYTES = int64_t(32) << 20;   // measured best on the 8192 x 4096 x 151936 head
int64_t k1_band_bytes();

constexpr uint32_t K1_A_BYTES = K1_BM * K1_BK * 2;
constexpr uint32_t K1_B_BYTES = K1_BN * K1_BK * 2;
constexpr uint32_t K1_STAGE_BYTES = K1_A_BYTES + K1_B_BYTES;
constexpr uint32_t K1_BAR_BYTES = 256;
constexpr uint32_t K1_SMEM_BYTES = K1_STAGES * K1_STAGE_BYTES + K1_BAR_BYTES + 1024;

inline int64_t k1_num_chunks(int64_t V) { return (V + K1_VCHUNK - 1) / K1_VCHUNK; }

struct K1Args {
    const int32_t *targets;   // [N]
    float2 *part;             // [N][num_chunks]: per-chunk (max, sum of exp(z - max))
    float *za;                // [N]: the target's logit, written by the chunk holding it
    int *status;              // device status word
    float inv_temp;           // 1 / temperature (1 for raw logits)
    int32_t N, D, V;
    int32_t w_segments;       // 1: W bf16 [V, D]; 3: fp32 W split into three bf16 parts, [V][3][Dp]
    int32_t num_m_tiles, num_chunks;
    int32_t num_m_groups;     // ceil(num_m_tiles / K1_CLUSTER): m-tiles of one cluster
    int32_t band, units;      // units = num_m_groups * num_chunks, one per cluster
    uint64_t wait_budget_ns;
    // backward (mode 1) only
    const float *grad;        // [N] upstream gradient of each l_t
    const float *lse_in;      // [N] the forward's lse
    uint16_t *dz;             // [N][dz_ld] bf16 gradient of the logits
    int64_t dz_ld;
};

// Launches one cluster of K1_CLUSTER CTAs per unit, at most as many clusters
// as fit on the device at once (persistent).  mode 0: forward; 1: backward dz.
cudaError_t k1_launch_main(const CUtensorMap &tmap_h, const CUtensorMap &tmap_w, const K1Args &a,
                           cudaStream_t stream, int mode = 0);
cudaError_t k1_launch_combine(const float2 *part, const float *za, const int32_t *targets,
                              int32_t N, int32_t V, int32_t num_chunks, float inv_temp, float *out_logp,
                              float *out_lse, cudaStream_t stream);
cudaError_t k1_prepare_device();   // per-device function attributes

// FP32 LM head: W fp32 [V, D] -> three bf16 parts [V][3][Dp], Dp = D rounded up
// to K1_BK, padding zero; w = part0 + part1 + part2 exactly.
inline int64_t k1_split_cols(int64_t D) { return (D + K1_BK - 1) / K1_BK * K1_BK; }
cudaError_t k1_launch_split(const float *W, int64_t V, int64_t D, void *W_split, int num_sms, cudaStream_t stream);

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
constexpr int K2_FOLD_THREADS = 256;               // fold CTA
constexpr int K2_FOLD_SEQS = 4 * K2_FOLD_THREADS;  // sequences per fold CTA
constexpr int K2_REC_WORDS = 16;                   // 4-byte words per sequence record (structure of arrays)
constexpr int K2_PART_WORDS = 40;                  // 4-byte words per fold partial
static_assert(K2_STAGE_BYTES % 16 == 0 && K2_BAR_BYTES % 16 == 0, "bulk-copy destinations stay 16-byte aligned");

inline size_t k2_workspace_bytes(int64_t S)
{
    const int64_t parts = (S + K2_FOLD_SEQS - 1) / K2_FOLD_SEQS;
    return static_cast<size_t>(S) * K2_REC_WORDS * 4 + static_cast<size_t>(parts) * K2_PART_WORDS * 4 + 256;
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
    uint32_t *rec;         // workspace: sequence records, [K2_REC_WORDS][S]
    uint32_t *part;        // workspace: fold partials, [ceil(S / K2_FOLD_SEQS)][K2_PART_WORDS]
    int *status;
};

cudaError_t k2_launch(const K2Args &a, int num_sms, cudaStream_t stream);
cudaError_t k2_prepare_device();   // per-device function attributes

// Launch attribute list that makes a launch a programmatic dependent of the
// previous kernel in its stream (its kernel calls pdl_wait() before reading).
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

// ---------------------------------------------------------------- shared by the C-ABI files
cudaError_t status_word_address(int **out);   // the library's device status word
int record_error(int code, const char *msg);  // message for tim_last_error()

} // namespace tim
