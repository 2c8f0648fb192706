// k1_internal.h -- the fused token logprob's tile shapes, arguments and launchers
// (forward, backward dz mode, FP32-head weight split).  Not part of the ABI.
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
constexpr int K1_W_BOX_ROWS = K1_BN / K1_CLUSTER;   // W rows of one TMA box (a CTA of a 2-CTA cluster loads one)
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

// TMA loads of an h tile run markedly slower (measured: 1.4x the whole call at
// N = 1) when the tensor map's row count is not a multiple of 16, so the last
// m-tile of such a batch is read from a zero-padded copy of K1_BM rows.
constexpr int64_t K1_TAIL_ROWS_ALIGN = 16;
inline bool k1_needs_tail_pad(int64_t N) { return N % K1_TAIL_ROWS_ALIGN != 0; }

struct K1Args {
    const int32_t *targets;   // [N]
    float2 *part;             // [N][num_chunks]: per-chunk (max, sum of exp(z - max))
    float *za;                // [N]: the target's logit, written by the chunk holding it
    int *status;              // device status word
    float inv_temp;           // 1 / temperature (1 for raw logits)
    int32_t N, D, V;
    int32_t w_segments;       // 1: W bf16 [V, D]; 3: fp32 W split into three bf16 parts, [V][3][Dp]
    int32_t num_m_tiles, num_chunks;
    int32_t cluster;          // CTAs per cluster: K1_CLUSTER, or 1 for a batch of one m-tile
    int32_t num_m_groups;     // ceil(num_m_tiles / cluster): m-tiles of one cluster
    int32_t band, units;      // units = num_m_groups * num_chunks, one per cluster
    int32_t tail_mt;          // m-tile read through the padded tail map, or -1
    uint64_t wait_budget_ns;
    // backward (mode 1) only
    const float *grad;        // [N] upstream gradient of each l_t
    const float *lse_in;      // [N] the forward's lse
    uint16_t *dz;             // [N][dz_ld] bf16 gradient of the logits
    int64_t dz_ld;
};

// A batch of one m-tile (at most K1_BM rows) runs in clusters of one CTA that
// stream their own W tiles: a cluster peer would only multiply a tile of
// padding rows (measured: the W stream then left HBM at 0.74 of the copy rate).
// Larger batches run in clusters of K1_CLUSTER m-tiles that share each W tile.
// Sets cluster, num_m_groups, band (m-groups whose h rows stay in L2) and units.
inline void k1_set_units(K1Args &a, int64_t m_tiles, int64_t chunks, int64_t D)
{
    const int cl = m_tiles <= 1 ? 1 : K1_CLUSTER;
    const int64_t m_groups = (m_tiles + cl - 1) / cl;
    const int64_t band = k1_band_bytes() / (int64_t(cl) * K1_BM * D * 2);
    a.cluster = cl;
    a.num_m_groups = static_cast<int32_t>(m_groups);
    a.band = static_cast<int32_t>(band < 1 ? 1 : band < m_groups ? band : m_groups);
    a.units = static_cast<int32_t>(m_groups * chunks);
}

// Launches one cluster of a.cluster CTAs per unit, at most as many clusters
// as fit on the device at once (persistent).  mode 0: forward; 1: backward dz.
cudaError_t k1_launch_main(const CUtensorMap &tmap_h, const CUtensorMap &tmap_w, const CUtensorMap &tmap_h_tail,
                           const K1Args &a, cudaStream_t stream, int mode = 0);
cudaError_t k1_launch_combine(const float2 *part, const float *za, const int32_t *targets,
                              int32_t N, int32_t V, int32_t num_chunks, float inv_temp, float *out_logp,
                              float *out_lse, cudaStream_t stream);
cudaError_t k1_prepare_device();   // per-device function attributes
// Copies `rows` rows of h (D bf16 each, 16-byte aligned) into a K1_BM-row pad, zero past them.
cudaError_t k1_launch_pad_tail(const void *src, int64_t rows, int64_t D, void *dst, cudaStream_t stream);

// FP32 LM head: W fp32 [V, D] -> three bf16 parts [V][3][Dp], Dp = D rounded up
// to K1_BK, padding zero; w = part0 + part1 + part2 exactly.
inline int64_t k1_split_cols(int64_t D) { return (D + K1_BK - 1) / K1_BK * K1_BK; }
cudaError_t k1_launch_split(const float *W, int64_t V, int64_t D, void *W_split, int num_sms, cudaStream_t stream);

} // namespace tim
