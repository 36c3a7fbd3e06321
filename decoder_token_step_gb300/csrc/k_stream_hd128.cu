// k_stream_hd128.cu -- the streaming decode-step kernel for head dimension 128, one instantiation per
// padded query-group size (a translation unit per head dimension, so they compile in parallel).
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_hd128(int gp) {
    switch (gp) {
    case 1: return reinterpret_cast<const void *>(k_stream<128, 1>);
    case 2: return reinterpret_cast<const void *>(k_stream<128, 2>);
    case 4: return reinterpret_cast<const void *>(k_stream<128, 4>);
    case 8: return reinterpret_cast<const void *>(k_stream<128, 8>);
    }
    return nullptr;
}

}  // namespace syn
