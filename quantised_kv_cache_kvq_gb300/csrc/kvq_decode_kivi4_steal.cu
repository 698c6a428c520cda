// kvq_decode_kivi4_steal.cu -- 4-bit KIVI decode kernels for the on-demand split (blocks of a long unit take its chunks from a counter);
// a translation unit of their own so the build compiles them in parallel with the others.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi4_steal(DecodeArgs& a, cudaStream_t stream) {
    return launch_kivi_family<4, true, false>(a, stream);
}

}  // namespace kvq
