// kvq_decode_rows.cu -- decode kernels for INT8 and FP8 caches, the log-sum-exp merge of
// the per-chunk partial results, and the decode dispatcher.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

// Combine the chunks of one (sequence, query head): with chunk i holding m_i (max score,
// base 2), l_i = sum 2^(s - m_i) and o_i = sum 2^(s - m_i) v, the output is
// sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i.  Warps take chunks in turn,
// lanes hold D/32 channels each, four chunks in flight per warp.
template <int D>
__global__ void __launch_bounds__(128) k_merge(DecodeArgs a) {
    constexpr int CPL = D / 32;
    __shared__ float red[4];
    __shared__ float part_o[4][D];
    __shared__ float part_l[4];
    const Layout& lo = a.lo;
    const int hq = blockIdx.x, b = blockIdx.y;
    const int h = hq / lo.gqa, head = hq % lo.gqa;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* st = state_ptr(lo, a.cache, a.layer, b);
    const int64_t n = st[0], qn = st[1];
    const int S = a.plan.S;
    const float* ml = reinterpret_cast<const float*>(a.ws + a.plan.ws_ml_off);
    const float* o = reinterpret_cast<const float*>(a.ws + a.plan.ws_o_off);
    const int64_t slot0 = (((int64_t)b * lo.H + h) * S) * lo.gqa + head;   // + item * gqa
    float mx = -INFINITY;
    for (int it = tid; it < S; it += blockDim.x) {
        const ItemRange r = item_range(lo, a.plan, it, n, qn);
        if (r.t0 < r.t1) mx = fmaxf(mx, ml[2 * (slot0 + (int64_t)it * lo.gqa)]);
    }
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    const float M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float acc[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) acc[e] = 0.0f;
    float l = 0.0f;
    for (int it0 = warp; it0 < S; it0 += 16) {
        float w4[4];
        float v4[4][CPL];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int it = it0 + 4 * k;
            w4[k] = 0.0f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) v4[k][e] = 0.0f;
            if (it < S) {
                const ItemRange r = item_range(lo, a.plan, it, n, qn);
                if (r.t0 < r.t1) {
                    const int64_t sl = slot0 + (int64_t)it * lo.gqa;
                    const float2 mlv = *reinterpret_cast<const float2*>(ml + 2 * sl);
                    w4[k] = fast_exp2(mlv.x - M);
                    if (lane == 0) l = fmaf(mlv.y, w4[k], l);
#pragma unroll
                    for (int e = 0; e < CPL; ++e) v4[k][e] = o[sl * D + lane + 32 * e];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int e = 0; e < CPL; ++e) acc[e] = fmaf(v4[k][e], w4[k], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < CPL; ++e) part_o[warp][lane + 32 * e] = acc[e];
    if (lane == 0) part_l[warp] = l;
    __syncthreads();
    const float L = part_l[0] + part_l[1] + part_l[2] + part_l[3];
    float* out = a.out + ((int64_t)b * lo.Hq + hq) * D;
    for (int d = tid; d < D; d += blockDim.x) {
        const float v = part_o[0][d] + part_o[1][d] + part_o[2][d] + part_o[3][d];
        out[d] = L > 0.0f ? v / L : 0.0f;
    }
}

}  // namespace

int launch_decode_rows(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.lo.D) {
        case 32: return launch_decode_t<32, 0, 1>(a, stream);
        case 64: return launch_decode_t<64, 0, 1>(a, stream);
        case 128: return launch_decode_t<128, 0, 1>(a, stream);
        case 256: return launch_decode_t<256, 0, 1>(a, stream);
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

int launch_decode(const Layout& lo, const DecodePlan& plan, const uint8_t* cache, int layer,
                  const void* q, float softmax_scale, float* out, uint8_t* ws, cudaStream_t stream) {
    DecodeArgs a;
    a.lo = lo;
    a.plan = plan;
    a.cache = cache;
    a.layer = layer;
    a.q = q;
    a.qscale = softmax_scale * 1.4426950408889634f;
    a.out = out;
    a.ws = ws;
    int rc;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        rc = lo.bits == 2 ? launch_decode_kivi2(a, stream)
           : lo.bits == 4 ? launch_decode_kivi4(a, stream)
                          : launch_decode_kivi8(a, stream);
    } else {
        rc = launch_decode_rows(a, stream);
    }
    if (rc != KVQ_OK) return rc;
    const dim3 mgrid(lo.Hq, lo.B);
    switch (lo.D) {
        case 32: k_merge<32><<<mgrid, 128, 0, stream>>>(a); break;
        case 64: k_merge<64><<<mgrid, 128, 0, stream>>>(a); break;
        case 128: k_merge<128><<<mgrid, 128, 0, stream>>>(a); break;
        default: k_merge<256><<<mgrid, 128, 0, stream>>>(a); break;
    }
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
