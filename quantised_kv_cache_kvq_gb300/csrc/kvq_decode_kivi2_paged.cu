// kvq_decode_kivi2_paged.cu -- 2-bit KIVI decode kernels for the paged layout (group
// records found through the block table), fixed split; a translation unit of their own so
// the build compiles them in parallel with the others.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi2_paged(DecodeArgs& a, cudaStream_t stream) {
    if (a.plan.steal) {   // the on-demand split, when its kernel has the same wave
        const int rc = launch_decode_kivi2_paged_steal(a, stream);
        if (rc != KVQ_ERR_UNSUPPORTED) return rc;
    }
    return launch_kivi_family<2, false, true>(a, stream);
}

}  // namespace kvq
