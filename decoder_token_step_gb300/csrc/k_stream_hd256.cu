// k_stream_hd256.cu -- the streaming decode-step kernel for head dimension 256, one instantiation per
// padded query-group size (a translation unit per head dimension, so they compile in parallel).
#include "k_stream.cuh"

namespace syn {

const void *stream_kernel_hd256(int gp) {
    switch (gp) {
    case 1: return reinterpret_cast<const void *>(k_stream<256, 1>);
    case 2: return reinterpret_cast<const void *>(k_stream<256, 2>);
    case 4: return reinterpret_cast<const void *>(k_stream<256, 4>);
    }
    return nullptr;
}

}  // namespace syn
