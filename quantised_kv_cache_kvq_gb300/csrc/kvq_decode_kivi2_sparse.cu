// kvq_decode_kivi2_sparse.cu -- 2-bit KIVI decode kernels for dense-and-sparse records
// (outliers kept aside in bf16), fixed split; the paged layout's are in
// kvq_decode_kivi2_sparse_paged.cu.  Translation units of their own so the build compiles
// them in parallel with the others.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi2_sparse(DecodeArgs& a, cudaStream_t stream) {
    if (a.lo.PG > 0) return launch_decode_kivi2_sparse_paged(a, stream);
    return launch_kivi_family<2, false, false, true>(a, stream);
}

}  // namespace kvq
