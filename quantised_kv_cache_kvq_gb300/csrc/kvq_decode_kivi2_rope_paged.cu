// kvq_decode_kivi2_rope_paged.cu -- 2-bit KIVI decode kernels for keys cached before the
// rotary embedding, paged layout, fixed split.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi2_rope_paged(DecodeArgs& a, cudaStream_t stream) {
    return launch_kivi_family<2, false, true, false, true>(a, stream);
}

}  // namespace kvq
