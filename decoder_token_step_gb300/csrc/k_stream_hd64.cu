// k_stream_hd64.cu -- the streaming decode-step kernel for head dimension 64, one instantiation per
// padded query-group size (a translation unit per head dimension, so they compile in parallel).
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_hd64(int gp) {
    switch (gp) {
    case 1: return reinterpret_cast<const void *>(k_stream<64, 1>);
    case 2: return reinterpret_cast<const void *>(k_stream<64, 2>);
    case 4: return reinterpret_cast<const void *>(k_stream<64, 4>);
    case 8: return reinterpret_cast<const void *>(k_stream<64, 8>);
    }
    return nullptr;
}

}  // namespace syn
