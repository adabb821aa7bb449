// Instantiation of the paged decode attention kernels for f32 K/V caches.
#include "decode_kernel.cuh"

namespace pkv {
namespace kern {
template int launch_d<PKV_F32>(const pkv_pool *, int, const Params &, int, int, cudaStream_t);
}  // namespace kern
}  // namespace pkv
