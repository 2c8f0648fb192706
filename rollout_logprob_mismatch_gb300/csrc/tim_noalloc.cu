// tim_noalloc.cu -- tim_token_logprob_noalloc: the fused token logprob for
// callers that cannot let a library allocate device memory.
//
// Who needs it: an engine that reserves its whole device-memory budget up front
// and hands out pieces itself (a trainer or serving process with its own
// caching allocator), or code running where the stream-ordered allocator is
// unavailable.  A hidden cudaMallocFromPoolAsync in such a process either fails
// for lack of free memory or escapes the owner's accounting, so this variant
// takes nothing at call time: the split-V scratch lives in one fixed device
// array of this library, and the caller still passes inputs and outputs.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds TIM_NOALLOC_SCRATCH_BYTES of it until the process exits.  All
// calls share it and it keeps the last call's contents: every partial a call
// reads is written by that call first, and the one word that must start at
// zero (the fused kernel's unit counter) is cleared on the stream before each
// launch (cudaMemsetAsync, which allocates nothing).
// Two calls whose kernels overlap on the GPU (other streams, other threads)
// race on the array: the caller must order them.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/tim.h"
#include "k1_internal.h"
#include "tim_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[TIM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct NoallocDevice {
    bool ready = false;
    int sms = 0;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    int *status = nullptr;              // device address of the library status word
};

std::mutex g_mu;
NoallocDevice g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int err(int code, const char *fmt, long long a = 0, long long b = 0)
{
    char msg[256];
    std::snprintf(msg, sizeof msg, fmt, a, b);
    return tim::record_error(code, msg);
}

int cuda_err(cudaError_t e, const char *what)
{
    char msg[256];
    std::snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return tim::record_error(TIM_ERR_CUDA, msg);
}

uint64_t wait_budget_ns()
{
    const char *s = std::getenv("TIM_WAIT_BUDGET_MS");
    const long long ms = s ? std::atoll(s) : 0;
    return ms > 0 ? static_cast<uint64_t>(ms) * 1000000ull : 4000000000ull;
}

// Set-up once per device, run by the first call on that device while it is the
// current device: sm_103 check, SM count, the scratch array's and the status
// word's device addresses (host code only has a stand-in symbol for them), the
// kernel's shared-memory attribute and the driver's tensor-map encoder.
int setup(NoallocDevice **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_err(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return err(TIM_ERR_UNSUPPORTED_DEVICE, "device ordinal %lld out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    NoallocDevice &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_err(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return err(TIM_ERR_UNSUPPORTED_DEVICE, "device is sm_%lld%lld; this library needs sm_103a", major,
                       minor);
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return cuda_err(e, "cudaGetSymbolAddress(scratch)");
        d.scratch = static_cast<unsigned char *>(p);
        if ((e = tim::status_word_address(&d.status)) != cudaSuccess)
            return cuda_err(e, "cudaGetSymbolAddress(status)");
        if ((e = tim::k1_prepare_device()) != cudaSuccess)
            return cuda_err(e, "cudaFuncSetAttribute");
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return err(TIM_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    *out = &d;
    return TIM_OK;
}

int encode(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(tim::K1_BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return err(TIM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%lld)", static_cast<long long>(r));
    return TIM_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

} // namespace

extern "C" int tim_token_logprob_noalloc(const void *h, const void *W, const int32_t *targets, int64_t N,
                                         int64_t D, int64_t V, float *out_logp, float *out_lse,
                                         tim_stream_t stream)
{
    if (N < 0 || N >= (int64_t(1) << 31))
        return err(TIM_ERR_INVALID_ARG, "N = %lld out of range [0, 2^31)", N);
    if (D <= 0 || D % 8 != 0 || D > 65536)
        return err(TIM_ERR_INVALID_ARG, "D = %lld must be positive, a multiple of 8 and <= 65536", D);
    if (V <= 0 || V >= (int64_t(1) << 31))
        return err(TIM_ERR_INVALID_ARG, "V = %lld out of range (0, 2^31)", V);
    if (N == 0)
        return tim::record_error(TIM_OK, "");
    if (!h || !W || !targets || !out_logp || !out_lse)
        return err(TIM_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned(h, 16) || !aligned(W, 16))
        return err(TIM_ERR_INVALID_ARG, "h and W must be 16-byte aligned");
    if (!aligned(targets, 4) || !aligned(out_logp, 4) || !aligned(out_lse, 4))
        return err(TIM_ERR_INVALID_ARG, "targets / outputs must be 4-byte aligned");
    const int64_t m_tiles = (N + tim::K1_BM - 1) / tim::K1_BM;
    const int64_t chunks = tim::k1_num_chunks(V);
    // scratch layout: per-chunk partials | target logits | padded last m-tile
    // (only when N % 16 != 0) | the unit counter
    const size_t part_bytes = round_up(static_cast<size_t>(chunks) * N * sizeof(float2), 256);
    const size_t za_bytes = round_up(static_cast<size_t>(N) * sizeof(float), 256);
    const size_t pad_bytes =
        tim::k1_needs_tail_pad(N) ? round_up(static_cast<size_t>(tim::K1_BM) * D * 2, 256) : 0;
    const size_t need = part_bytes + za_bytes + pad_bytes + tim::K1_SCHED_BYTES;
    if (need > static_cast<size_t>(TIM_NOALLOC_SCRATCH_BYTES))
        return err(TIM_ERR_INVALID_ARG,
                   "N x ceil(V / 1024) too large for the fixed scratch: needs %lld bytes, the limit is %lld "
                   "(TIM_NOALLOC_SCRATCH_BYTES); use tim_token_logprob or split the rows",
                   static_cast<long long>(need), static_cast<long long>(TIM_NOALLOC_SCRATCH_BYTES));

    NoallocDevice *dev = nullptr;
    int rc = setup(&dev);
    if (rc != TIM_OK)
        return rc;
    CUtensorMap th, tw;
    if ((rc = encode(&th, h, N, D, tim::K1_BM)) != TIM_OK)
        return rc;
    if ((rc = encode(&tw, W, V, D, tim::K1_W_BOX_ROWS)) != TIM_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *pad = dev->scratch + part_bytes + za_bytes;
    // TMA reads of h through a map whose row count is not a multiple of 16 are
    // slow, so such a batch's last m-tile is read from a zero-padded copy in
    // the scratch (same values, so the same result bits)
    CUtensorMap th_tail = th;
    int32_t tail_mt = -1;
    if (pad_bytes > 0) {
        const int64_t r0 = (m_tiles - 1) * tim::K1_BM;
        const cudaError_t ep = tim::k1_launch_pad_tail(static_cast<const char *>(h) + r0 * D * 2, N - r0, D, pad, s);
        if (ep != cudaSuccess)
            return cuda_err(ep, "tail pad copy");
        if ((rc = encode(&th_tail, pad, tim::K1_BM, D, tim::K1_BM)) != TIM_OK)
            return rc;
        tail_mt = static_cast<int32_t>(m_tiles - 1);
    }

    tim::K1Args a{};
    a.targets = targets;
    a.part = reinterpret_cast<float2 *>(dev->scratch);
    a.za = reinterpret_cast<float *>(dev->scratch + part_bytes);
    a.sched = reinterpret_cast<int *>(pad + pad_bytes);
    a.status = dev->status;
    a.inv_temp = 1.f;
    a.N = static_cast<int32_t>(N);
    a.D = static_cast<int32_t>(D);
    a.w_segments = 1;
    a.V = static_cast<int32_t>(V);
    a.num_m_tiles = static_cast<int32_t>(m_tiles);
    a.num_chunks = static_cast<int32_t>(chunks);
    tim::k1_set_units(a, m_tiles, chunks, D);
    a.wait_budget_ns = wait_budget_ns();
    a.tail_mt = tail_mt;
    cudaError_t e = tim::k1_launch_main(th, tw, th_tail, a, s);
    if (e == cudaSuccess)
        e = tim::k1_launch_combine(a.part, a.za, targets, a.N, a.V, a.num_chunks, a.inv_temp, out_logp, out_lse,
                                   a.status, s);
    if (e != cudaSuccess)
        return cuda_err(e, "token_logprob_noalloc launch");
    return tim::record_error(TIM_OK, "");
}
