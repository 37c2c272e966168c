// Multi-query attention kernels for 4-bit keys and 4-bit values: the instantiations of
// kivi_multi_impl.cuh for this pair of code widths.
#include "kivi_multi_impl.cuh"

namespace kivi {

cudaError_t launch_multi_k4v4(const DecodeArgs& a, cudaStream_t stream) { return launch_multi_kv<4, 4>(a, stream); }

}  // namespace kivi
