// fp32_head.cu -- weights of the FP32 LM head as three bf16 parts, for sm_103a.
//
// LoongSage "Train-Inference Consistency" section 3 keeps the LM head's
// weights and arithmetic in fp32, so that rounding the logits to bf16 does not
// feed the log-probabilities.  The tensor cores take bf16 operands; an fp32
// weight w is the exact sum of three bf16 numbers: w1 = w with the low 16 bits
// of its encoding cleared, w2 the same of w - w1, w3 = w - w1 - w2 (both
// differences are exact in fp32; the 24-bit significand is cut into 8-bit
// pieces, so w3 has at most 8 significant bits; exact down to |w| ~ 2^-110,
// below which bf16 cannot hold the last piece).  A bf16 hidden value times a
// bf16 part is exact in fp32, so the fused kernel, run over the three parts
// with fp32 accumulation, forms h . w with fp32 weights and fp32 arithmetic
// at three times the tensor work.
//
// Layout: row v of the split is [w1 of the row | w2 | w3], each part Dp =
// D rounded up to 64 columns (the kernel's k-tile) with zero padding, so each
// k-tile of the split lies inside one part.  Non-finite weights go whole into
// w1 (w2 = w3 = 0).
#include <algorithm>
#include <cstdint>

#include "k1_internal.h"
#include "tim_internal.h"

namespace tim {
namespace {

__device__ __forceinline__ uint16_t hi16(float x) { return static_cast<uint16_t>(__float_as_uint(x) >> 16); }

__device__ __forceinline__ float trunc_bf16(float x) { return __uint_as_float(__float_as_uint(x) & 0xffff0000u); }

// One weight into its three parts (encodings of the bf16 parts).
__device__ __forceinline__ void split3(float w, uint16_t &p1, uint16_t &p2, uint16_t &p3)
{
    if (fabsf(w) <= 3.402823466e38f) {   // finite
        const float w1 = trunc_bf16(w);
        const float r1 = __fsub_rn(w, w1);
        const float w2 = trunc_bf16(r1);
        p1 = hi16(w1);
        p2 = hi16(w2);
        p3 = hi16(__fsub_rn(r1, w2));      // at most 8 significant bits: exact in bf16
    } else {
        p1 = hi16(w);
        p2 = p3 = 0;
    }
}

__device__ __forceinline__ uint2 pack4(const uint16_t (&p)[4])
{
    return make_uint2(static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 16),
                      static_cast<uint32_t>(p[2]) | (static_cast<uint32_t>(p[3]) << 16));
}

// Grid-stride over groups of 4 columns (D and Dp are multiples of 4, W is
// 16-byte aligned): one 16-byte load, three 8-byte stores per group.
__global__ void __launch_bounds__(256) k1_split_kernel(const float *__restrict__ W, int64_t V, int64_t D, int64_t Dp,
                                                      uint16_t *__restrict__ out)
{
    const int64_t gpr = Dp / 4;   // groups per row
    const int64_t total = V * gpr;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t v = i / gpr, k = (i - v * gpr) * 4;
        const float4 w = k < D ? __ldcs(reinterpret_cast<const float4 *>(W + v * D + k)) : make_float4(0, 0, 0, 0);
        uint16_t a[4], b[4], c[4];
        split3(w.x, a[0], b[0], c[0]);
        split3(w.y, a[1], b[1], c[1]);
        split3(w.z, a[2], b[2], c[2]);
        split3(w.w, a[3], b[3], c[3]);
        uint16_t *row = out + v * 3 * Dp + k;
        __stcs(reinterpret_cast<uint2 *>(row), pack4(a));
        __stcs(reinterpret_cast<uint2 *>(row + Dp), pack4(b));
        __stcs(reinterpret_cast<uint2 *>(row + 2 * Dp), pack4(c));
    }
}

} // namespace

cudaError_t k1_launch_split(const float *W, int64_t V, int64_t D, void *W_split, int num_sms, cudaStream_t stream)
{
    const int64_t Dp = k1_split_cols(D);
    const int64_t total = V * (Dp / 4);
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms) * 16);
    k1_split_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, stream>>>(
        W, V, D, Dp, static_cast<uint16_t *>(W_split));
    return cudaGetLastError();
}

} // namespace tim
