// monitor_internal.h -- launch parameters of the mismatch monitor (exact quantiles by radix select).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tim {

constexpr int MON_THREADS = 256;
constexpr int MON_CTAS_PER_SM = 3;         // pass 2 holds 64 KB of histograms per CTA
constexpr int MON_UNROLL = 4;         // 4-token groups per thread per iteration, loaded before use
constexpr int MON_TARGETS = 8;        // order statistics: ranks k and k + 1 of four quantiles
constexpr int MON_BINS1 = 2048;       // pass 1: key bits 31..21
constexpr int MON_BINS2 = 2048;       // pass 2: key bits 20..10
constexpr int MON_BINS3 = 1024;       // pass 3: key bits 9..0

// Device state of one call, at the start of the workspace (zeroed before pass 1).
struct MonState {
    unsigned long long n_used;
    unsigned long long n_extreme;
    long long rank[MON_TARGETS];      // rank still to find inside the current prefix
    uint32_t prefix[MON_TARGETS];     // key bits fixed so far (high bits, rest zero)
    double frac[MON_TARGETS / 2];     // interpolation weight of each quantile
    int empty;                        // no used token: no selection
};

// Workspace: state, then the histograms of the three passes (32-bit counts).
constexpr size_t MON_STATE_BYTES = 512;
static_assert(sizeof(MonState) <= MON_STATE_BYTES, "state block");
constexpr size_t MON_HIST1_WORDS = MON_BINS1;                 // delta's key only
constexpr size_t MON_HIST2_WORDS = MON_TARGETS * MON_BINS2;   // one per target
constexpr size_t MON_HIST3_WORDS = MON_TARGETS * MON_BINS3;
constexpr size_t MON_WORKSPACE_BYTES = MON_STATE_BYTES + 4 * (MON_HIST1_WORDS + MON_HIST2_WORDS + MON_HIST3_WORDS);

struct MonArgs {
    const float *l_tr, *l_ro;
    const uint8_t *mask;
    int64_t N;
    float tau_tok;
    uint8_t *reject;     // optional [N]
    double *out;         // [TIM_MON_FIELDS]
    MonState *st;
    uint32_t *hist1, *hist2, *hist3;
    int *status;
};

cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream);
cudaError_t monitor_prepare_device();

} // namespace tim
