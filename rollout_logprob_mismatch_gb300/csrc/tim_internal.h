// tim_internal.h -- declarations shared by the library's own translation units
// (kernels and the C-ABI layer).  Not installed; not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace tim {

// Launch attribute list that makes a launch a programmatic dependent of the
// previous kernel in its stream (its kernel calls pdl_wait() before reading).
inline cudaLaunchAttribute pdl_attribute()
{
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

// ---------------------------------------------------------------- status block
// The device status block: word 0 the status (first error wins), word 1 the
// TIM_CHECK_* id of the first checked-build violation, words 2-3 its index,
// words 4-5 its value.  Kernels get its address as `int *status`.
constexpr int STATUS_WORDS = 8;

#ifdef TIM_DEBUG
// First violation wins the record; every violation sets the status.
__device__ __forceinline__ void debug_report(int *status, int check, int64_t index, uint64_t value)
{
    if (atomicCAS(status + 1, 0, check) == 0) {
        *reinterpret_cast<volatile long long *>(status + 2) = static_cast<long long>(index);
        *reinterpret_cast<volatile unsigned long long *>(status + 4) = static_cast<unsigned long long>(value);
    }
    atomicCAS(status, 0, -5);   // TIM_ERR_BAD_INPUT
}
#define TIM_DCHECK(cond, status, check, index, value)                                          \
    do {                                                                                        \
        if (!(cond))                                                                            \
            ::tim::debug_report((status), (check), static_cast<int64_t>(index), static_cast<uint64_t>(value)); \
    } while (0)
#else
#define TIM_DCHECK(cond, status, check, index, value) \
    do {                                              \
    } while (0)
#endif

// ---------------------------------------------------------------- shared by the C-ABI files
cudaError_t status_word_address(int **out);   // the library's device status block
int record_error(int code, const char *msg);  // message for tim_last_error()

} // namespace tim
