// Instantiation of the paged decode attention kernels for 4-bit K/V caches.
#include "decode_kernel.cuh"

namespace pkv {
namespace kern {
template int launch_d<PKV_I4>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
}  // namespace kern
}  // namespace pkv
