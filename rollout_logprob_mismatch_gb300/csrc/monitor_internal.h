// monitor_internal.h -- launch parameters of the mismatch monitor (exact quantiles by selection).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace tim {

constexpr int MON_THREADS = 256;
constexpr int MON_CTAS_PER_SM = 3;     // pass 2 holds 64 KB of histograms per CTA
constexpr int MON_UNROLL = 4;          // 4-token groups per thread per iteration, loaded before use
constexpr int MON_QUANTILES = 4;       // p95 |delta|; ratio 0.01, 0.5, 0.99
constexpr int MON_TARGETS = 8;         // order statistics: ranks k and k + 1 of each quantile
constexpr int MON_BINS1 = 2048;        // radix pass 1: 11 key bits
constexpr int MON_BINS2 = 2048;        // pass 2: 11 bits
constexpr int MON_BINS3 = 1024;        // pass 3: 10 bits
constexpr int MON_SAMPLE_RUNS = 1024;  // the sample: up to 1024 runs of MON_SAMPLE_RUN consecutive tokens
constexpr int MON_SAMPLE_RUN = 1024;
constexpr int MON_SBINS = 16384;       // sample histogram of delta's key >> 18 (|delta|'s follows from it)

// Device state of one call, at the start of the workspace (zeroed before the sample).
struct MonState {
    unsigned long long n_used, n_extreme, sample_used;
    unsigned long long below[MON_QUANTILES];   // used tokens with key < lo
    unsigned long long count[MON_QUANTILES];   // used tokens with lo <= key <= hi (kept up to cap)
    long long rank[MON_TARGETS];               // rank still to find inside the current prefix
    uint32_t lo[MON_QUANTILES], hi[MON_QUANTILES];
    uint32_t prefix[MON_TARGETS];              // bits fixed so far (of the key, or of key - lo)
    int span_bits[MON_QUANTILES];              // collected mode: bit length of hi - lo
    double frac[MON_QUANTILES];                // interpolation weight of each quantile
    int empty;                                 // no used token
    int fallback;                              // 1: select over all tokens (a bound missed)
    unsigned ticket[5];                        // CTAs finished: sample, full pass, passes 1..3
};

// Workspace: state, the radix histograms (pass 1: one per candidate list, then
// the one of the selection over all tokens), the sample histogram (all zeroed
// per call), then four candidate lists of `cap` keys.
constexpr size_t MON_STATE_BYTES = 512;
static_assert(sizeof(MonState) <= MON_STATE_BYTES, "state block");
constexpr size_t MON_HIST1_WORDS = (MON_QUANTILES + 1) * MON_BINS1;
constexpr size_t MON_HIST2_WORDS = MON_TARGETS * MON_BINS2;
constexpr size_t MON_HIST3_WORDS = MON_TARGETS * MON_BINS3;
constexpr size_t MON_SHIST_WORDS = MON_SBINS;
constexpr size_t MON_ZEROED_BYTES =
    MON_STATE_BYTES + 4 * (MON_HIST1_WORDS + MON_HIST2_WORDS + MON_HIST3_WORDS + MON_SHIST_WORDS);

inline unsigned long long monitor_cap(int64_t N) { return static_cast<unsigned long long>(N / 16 + 65536); }
inline size_t monitor_workspace_bytes(int64_t N)
{
    return MON_ZEROED_BYTES + 4ull * MON_QUANTILES * monitor_cap(N);
}

struct MonArgs {
    const float *l_tr, *l_ro;
    const uint8_t *mask;
    int64_t N;
    float tau_tok;
    uint8_t *reject;     // optional [N]
    double *out;         // [TIM_MON_FIELDS]
    MonState *st;
    uint32_t *hist1, *hist2, *hist3;
    uint32_t *shist;     // sample histogram of delta's key [MON_SBINS]
    uint32_t *cand;      // [MON_QUANTILES][cap] collected keys
    unsigned long long cap;
    int *status;
    uint64_t wait_budget_ns;   // bound of each pipeline wait in the kernels
};

cudaError_t monitor_launch(const MonArgs &a, int num_sms, cudaStream_t stream);
cudaError_t monitor_prepare_device();

} // namespace tim
