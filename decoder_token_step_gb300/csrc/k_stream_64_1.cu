// k_stream_64_1.cu -- the streaming decode-step kernel for head dimension 64 and 1 (padded) query heads per
// KV head: one instantiation per translation unit, so that they compile in parallel.
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_64_1() { return reinterpret_cast<const void *>(k_stream<64, 1>); }

}  // namespace syn
