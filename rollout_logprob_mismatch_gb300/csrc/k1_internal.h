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
constexpr int K1_BM = 128;        // rows (tokens) per tile = TMEM lanes of one CTA
constexpr int K1_BN = 256;        // vocabulary columns per tile = UMMA N
constexpr int K1_BK = 64;         // bf16 elements per 128-byte swizzled row
constexpr int K1_VCHUNK = 1024;   // vocabulary columns per split-V partial
constexpr int K1_THREADS = 192;   // warp 0 TMA, warp 1 UMMA + TMEM, warps 2-5 epilogue
constexpr int K1_CLUSTER = 2;     // CTAs per cluster: a CTA pair running one 2-SM UMMA (M = 256)
constexpr int K1_W_BOX_ROWS = K1_BN / 2;   // W rows of one TMA box: one pair CTA's half of a W tile
// Units walk the vocabulary in bands of m-tiles whose h rows (at most this many
// bytes) stay in L2 while the band's clusters stream each W chunk from HBM once.
// (TIM_K1_BAND_MB overrides it; the band changes the order of work, never a result.)
constexpr int64_t K1_BAND_BYTES = int64_t(32) << 20;   // measured best on the 8192 x 4096 x 151936 head
int64_t k1_band_bytes();

// Shared memory per CTA and pipeline stage: the CTA's h tile [128 x 64] and its
// W rows [rows x 64] -- in a CTA pair its own 128-row half of the 256-row W tile
// (the pair UMMA reads the other half from the peer), alone both halves.
constexpr uint32_t K1_A_BYTES = K1_BM * K1_BK * 2;
constexpr uint32_t k1_b_bytes(int cl) { return static_cast<uint32_t>(cl == 1 ? K1_BN : K1_BN / 2) * K1_BK * 2; }
constexpr int k1_stages(int cl) { return cl == 1 ? 4 : 7; }   // TMA -> UMMA pipeline depth
constexpr uint32_t K1_BAR_BYTES = 512;   // the unit ring, mbarriers, TMEM address, abort flag
constexpr uint32_t k1_ring_bytes(int cl) { return static_cast<uint32_t>(k1_stages(cl)) * (K1_A_BYTES + k1_b_bytes(cl)); }
constexpr uint32_t K1_SMEM_BYTES =
    (k1_ring_bytes(1) > k1_ring_bytes(K1_CLUSTER) ? k1_ring_bytes(1) : k1_ring_bytes(K1_CLUSTER)) + K1_BAR_BYTES + 1024;

inline int64_t k1_num_chunks(int64_t V) { return (V + K1_VCHUNK - 1) / K1_VCHUNK; }

// TMA loads of an h tile run markedly slower (measured: 1.4x the whole call at
// N = 1) when the tensor map's row count is not a multiple of 16, so the last
// m-tile of such a batch is read from a zero-padded copy of K1_BM rows.
constexpr int64_t K1_TAIL_ROWS_ALIGN = 16;
constexpr size_t K1_SCHED_BYTES = 256;   // the unit counter's slot in a workspace
inline bool k1_needs_tail_pad(int64_t N) { return N % K1_TAIL_ROWS_ALIGN != 0; }

struct K1Args {
    const int32_t *targets;   // [N]
    float2 *part;             // [N][num_chunks]: per-chunk (max, sum of exp(z - max))
    float *za;                // [N]: the target's logit, written by the chunk holding it
    int *status;              // device status word
    int *sched;               // unit counter, zero at launch: units are claimed in order from it
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
// stream their own W tiles: a pair would only multiply a tile of padding rows
// (measured: the W stream then left HBM at 0.74 of the copy rate).  Larger
// batches run in CTA pairs, each pair CTA holding one m-tile and half of each
// W tile.
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

// Launches at most as many clusters of a.cluster CTAs as fit on the device at
// once (persistent; they claim the units in order from a.sched, which this
// zeroes first on the stream).  mode 0: forward; 1: backward dz.
cudaError_t k1_launch_main(const CUtensorMap &tmap_h, const CUtensorMap &tmap_w, const CUtensorMap &tmap_h_tail,
                           const K1Args &a, cudaStream_t stream, int mode = 0);
cudaError_t k1_launch_combine(const float2 *part, const float *za, const int32_t *targets,
                              int32_t N, int32_t V, int32_t num_chunks, float inv_temp, float *out_logp,
                              float *out_lse, int *status, cudaStream_t stream);
cudaError_t k1_prepare_device();   // per-device function attributes
// Copies `rows` rows of h (D bf16 each, 16-byte aligned) into a K1_BM-row pad, zero past them.
cudaError_t k1_launch_pad_tail(const void *src, int64_t rows, int64_t D, void *dst, cudaStream_t stream);

// FP32 LM head: W fp32 [V, D] -> three bf16 parts [V][3][Dp], Dp = D rounded up
// to K1_BK, padding zero; w = part0 + part1 + part2 exactly.
inline int64_t k1_split_cols(int64_t D) { return (D + K1_BK - 1) / K1_BK * K1_BK; }
cudaError_t k1_launch_split(const float *W, int64_t V, int64_t D, void *W_split, int num_sms, cudaStream_t stream);

} // namespace tim
