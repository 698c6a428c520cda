// kvq_decode_rope.cu -- decode attention over KIVI caches whose keys were cached before the
// rotary position embedding ("KVQuant: Towards 10 Million Context Length ...", "Key points":
// keys are quantised before RoPE, which mixes channel pairs and would blur their outlier
// channels).  Every dequantised key is rotated at its position before its scores.
//   * Plain records: the KIVI kernels with ROPE set (kvq_decode_kivi*_rope*.cu) rotate the
//     keys of each tile in registers and score them on the tensor cores; the values and the
//     softmax are the packed path's, the bf16 window goes through rope_item.
//   * Dense-and-sparse records (outliers kept aside in bf16, "Summary" of the same page):
//     k_decode_rope below, rope_item for every part, where an outlier's side entry replaces
//     its dequantised value before the rotation.
// The split, the partial-result slots and the merge are the KIVI decode's.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

template <int D, int BITS>
__global__ void __launch_bounds__(kDecodeThreads, 4) k_decode_rope(const __grid_constant__ DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    grid_dependency_wait();
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    if (threadIdx.x == 0) {
        mbar_init(bars, 1);
        mbar_init(bars + 1, 1);
        mbar_init(bars + kSelfTestBar, 1);
    }
    __syncthreads();
    uint32_t phase = selftest_bits(a);
    for_each_segment<false>(
        a, reinterpret_cast<int64_t*>(smem + so.red), reinterpret_cast<int2*>(smem + so.sst),
        [&](int part, int b, int h, int64_t slot, int64_t t0, int64_t t1, const StealCtx&) -> bool {
            const int r = rope_item<D, BITS>(a, smem, b, h, slot, part, t0, t1, phase);
            if (r < 0) return false;
            phase = static_cast<uint32_t>(r);
            return true;
        },
        [&](int64_t slot) { empty_partial(a, slot); });
}

template <int D>
int launch_rope_bits(DecodeArgs& a, cudaStream_t stream) {
    switch (a.lo.bits) {
        case 2: return launch_wave(k_decode_rope<D, 2>, a, stream);
        case 4: return launch_wave(k_decode_rope<D, 4>, a, stream);
        default: return launch_wave(k_decode_rope<D, 8>, a, stream);
    }
}

}  // namespace

int launch_decode_rope(DecodeArgs& a, cudaStream_t stream) {
    if (a.lo.K == 0) {
        return a.lo.bits == 2 ? launch_decode_kivi2_rope(a, stream)
             : a.lo.bits == 4 ? launch_decode_kivi4_rope(a, stream)
                              : launch_decode_kivi8_rope(a, stream);
    }
    switch (a.lo.D) {
        case 64: return launch_rope_bits<64>(a, stream);
        case 128: return launch_rope_bits<128>(a, stream);
        case 256: return launch_rope_bits<256>(a, stream);
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

}  // namespace kvq
