// k_stream_256_1.cu -- the streaming decode-step kernel for head dimension 256 and 1 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_256_1() { return reinterpret_cast<const void *>(k_stream<256, 1>); }

}  // namespace syn
