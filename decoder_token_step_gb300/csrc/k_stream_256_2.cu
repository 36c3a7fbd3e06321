// k_stream_256_2.cu -- the streaming decode-step kernel for head dimension 256 and 2 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_256_2() { return reinterpret_cast<const void *>(k_stream<256, 2>); }

}  // namespace syn
