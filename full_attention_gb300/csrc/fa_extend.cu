// Chunked-prefill / extend attention (placeholder until the tensor-core kernel lands).
#include "fa_internal.h"

namespace fa {

cudaError_t launch_extend(const ExtendArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
