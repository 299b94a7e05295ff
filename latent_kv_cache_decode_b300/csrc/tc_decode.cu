// Tensor-core path of libslimkv (tcgen05 + TMA). Not built yet: every shape is
// routed to the SIMT path.
#include "tc_decode.cuh"

namespace slimkv {

bool tc_supported(int, int, int, int, int, int) { return false; }

cudaError_t tc_run(const TcCall&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace slimkv
