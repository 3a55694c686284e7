// Tensor-core chunked forward kernel (tcgen05 / TMEM / TMA). Placeholder
// until the kernel lands: reports itself unsupported so AUTO uses the
// recurrent kernel.
#include "internal.h"

namespace dp {
bool chunk_tc_supported(const Problem &) { return false; }
size_t chunk_tc_scratch_bytes(const Problem &) { return 0; }
cudaError_t launch_chunk_tc(const Problem &) { return cudaErrorNotSupported; }
}  // namespace dp
