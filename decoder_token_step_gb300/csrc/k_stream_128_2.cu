// k_stream_128_2.cu -- the streaming decode-step kernel for head dimension 128 and 2 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_128_2() { return reinterpret_cast<const void *>(k_stream<128, 2>); }

}  // namespace syn
