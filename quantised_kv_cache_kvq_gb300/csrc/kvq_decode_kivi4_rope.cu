// kvq_decode_kivi4_rope.cu -- 4-bit KIVI decode kernels for keys cached before the rotary
// embedding (keys turned in registers, scored on the tensor cores), fixed split; the paged
// layout's are in kvq_decode_kivi4_rope_paged.cu.
#include "kvq_decode.cuh"

namespace kvq {

int launch_decode_kivi4_rope(DecodeArgs& a, cudaStream_t stream) {
    if (a.lo.PG > 0) return launch_decode_kivi4_rope_paged(a, stream);
    return launch_kivi_family<4, false, false, false, true>(a, stream);
}

}  // namespace kvq
