// k_stream_128_4.cu -- the streaming decode-step kernel for head dimension 128 and 4 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_128_4() { return reinterpret_cast<const void *>(k_stream<128, 4>); }

}  // namespace syn
