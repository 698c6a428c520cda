// kvq_decode_kivi2_sparse_paged.cu -- 2-bit KIVI decode kernels for dense-and-sparse
// records in the paged layout, fixed split.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi2_sparse_paged(DecodeArgs& a, cudaStream_t stream) {
    return launch_kivi_family<2, false, true, true>(a, stream);
}

}  // namespace kvq
