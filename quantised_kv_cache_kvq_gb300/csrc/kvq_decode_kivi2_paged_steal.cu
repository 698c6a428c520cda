// kvq_decode_kivi2_paged_steal.cu -- 2-bit KIVI decode kernels for the paged layout
// with the on-demand split; a translation unit of their own so the build compiles them in
// parallel with the others.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi2_paged_steal(DecodeArgs& a, cudaStream_t stream) {
    return launch_kivi_family<2, true, true>(a, stream);
}

}  // namespace kvq
