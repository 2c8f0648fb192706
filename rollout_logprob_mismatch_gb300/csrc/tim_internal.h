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

// ---------------------------------------------------------------- shared by the C-ABI files
cudaError_t status_word_address(int **out);   // the library's device status word
int record_error(int code, const char *msg);  // message for tim_last_error()

} // namespace tim
