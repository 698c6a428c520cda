// kvq_decode_rows.cu -- decode kernels for INT8 and FP8 caches, the log-sum-exp merge of
// the per-chunk partial results, and the decode dispatcher.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

// Combine the chunks of one (sequence, query head): with chunk i holding m_i (max score,
// base 2), l_i = sum 2^(s - m_i) and o_i = sum 2^(s - m_i) v, the output is
// sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i.
__global__ void __launch_bounds__(128) k_merge(DecodeArgs a) {
    extern __shared__ float wts[];
    __shared__ float red[4];
    __shared__ float bc;
    const Layout& lo = a.lo;
    const int hq = blockIdx.x, b = blockIdx.y;
    const int h = hq / lo.gqa, head = hq % lo.gqa;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* st = state_ptr(lo, a.cache, a.layer, b);
    const int64_t n = st[0], qn = st[1];
    const int S = a.plan.S;
    const float* ml = reinterpret_cast<const float*>(a.ws + a.plan.ws_ml_off);
    const float* o = reinterpret_cast<const float*>(a.ws + a.plan.ws_o_off);
    auto slot = [&](int item) { return (((int64_t)b * lo.H + h) * S + item) * lo.gqa + head; };
    float mx = -INFINITY;
    for (int it = tid; it < S; it += blockDim.x) {
        const ItemRange r = item_range(lo, a.plan, it, n, qn);
        if (r.t0 < r.t1) mx = fmaxf(mx, ml[2 * slot(it)]);
    }
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (tid == 0) bc = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    const float M = bc;
    float l = 0.0f;
    for (int it = tid; it < S; it += blockDim.x) {
        const ItemRange r = item_range(lo, a.plan, it, n, qn);
        float w = 0.0f;
        if (r.t0 < r.t1) {
            w = exp2f(ml[2 * slot(it)] - M);
            l += ml[2 * slot(it) + 1] * w;
        }
        wts[it] = w;
    }
    l = warp_sum(l);
    __syncthreads();
    if (lane == 0) red[warp] = l;
    __syncthreads();
    const float L = red[0] + red[1] + red[2] + red[3];
    float* out = a.out + ((int64_t)b * lo.Hq + hq) * lo.D;
    for (int d = tid; d < lo.D; d += blockDim.x) {
        float acc = 0.0f;
        for (int it = 0; it < S; ++it) {
            const float w = wts[it];
            if (w != 0.0f) acc = fmaf(o[slot(it) * lo.D + d], w, acc);
        }
        out[d] = L > 0.0f ? acc / L : 0.0f;
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
    const size_t msmem = static_cast<size_t>(plan.S) * sizeof(float);
    if (msmem > 48 * 1024 &&
        cudaFuncSetAttribute(k_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(msmem)) !=
            cudaSuccess)
        return KVQ_ERR_CUDA;
    k_merge<<<dim3(lo.Hq, lo.B), 128, msmem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
