// tcgen05 decode kernel: not built yet; the dispatcher uses the mma kernel.
#include "common.cuh"

namespace nvmla {

bool tc_supported(int) { return false; }

cudaError_t launch_decode_tc(int, const void*, const void*, const uint8_t*, const RowSelect&, const int32_t*, int,
                             int, int, float, void*, float*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace nvmla
