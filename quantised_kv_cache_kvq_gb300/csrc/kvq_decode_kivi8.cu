// kvq_decode_kivi8.cu -- decode kernels for 8-bit KIVI caches (one translation unit per bit
// width so the build compiles them in parallel).
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi8(DecodeArgs& a, cudaStream_t stream) {
    const bool wide = a.lo.gqa > 4;
    switch (a.lo.D) {
        case 64: return wide ? launch_decode_t<64, 8, 2>(a, stream) : launch_decode_t<64, 8, 1>(a, stream);
        case 128: return wide ? launch_decode_t<128, 8, 2>(a, stream) : launch_decode_t<128, 8, 1>(a, stream);
        case 256: return wide ? launch_decode_t<256, 8, 2>(a, stream) : launch_decode_t<256, 8, 1>(a, stream);
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

}  // namespace kvq
