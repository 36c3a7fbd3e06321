// k_stream_128_1.cu -- the streaming decode-step kernel for head dimension 128 and 1 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_128_1() { return reinterpret_cast<const void *>(k_stream<128, 1>); }

}  // namespace syn
