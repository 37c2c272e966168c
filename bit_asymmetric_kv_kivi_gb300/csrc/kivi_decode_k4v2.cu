// Decode attention kernels for 4-bit keys and 2-bit values: the instantiations of
// kivi_decode_impl.cuh for this pair of code widths.
#include "kivi_decode_impl.cuh"

namespace kivi {

cudaError_t launch_decode_k4v2(const DecodeArgs& a, cudaStream_t stream) { return launch_kv<4, 2>(a, stream); }

}  // namespace kivi
