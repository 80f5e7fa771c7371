// gdn_chunked.cu — tensor-core chunked prefill (placeholder until the kernel lands).
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {
int launch_chunked_prefill(const PrefillArgs&, void*) { return (int)cudaErrorNotSupported; }
int chunked_prefill_smem_bytes() { return 0; }
}  // namespace gdn
