// Tensor-core (tcgen05 / TMEM / TMA) kernels of the chunked SSD core.
#include "ssd_internal.h"

namespace ssd {

bool tc_supported(const Problem&) { return false; }
cudaError_t tc_forward_scan(const Problem&) { return cudaErrorNotSupported; }
cudaError_t tc_backward(const Problem&) { return cudaErrorNotSupported; }

}  // namespace ssd
