// kvq_decode_rows.cu -- the INT8 decode dispatch, the log-sum-exp merge of the per-chunk
// partial results, and the decode dispatcher.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

constexpr int kMergeThreads = 256;

// Combine the chunks of one (sequence, query head): with chunk i holding m_i (max score,
// base 2), l_i = sum 2^(s - m_i) and o_i = sum 2^(s - m_i) v, the output is
// sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i.  A block of 8 warps takes
// 32 * nwc channels of one (sequence, query head): warp w holds channels 32 (w % nwc) + lane
// and the chunks w / nwc + nwi * k, twelve per round, every load of a round issued before
// any is used.  The host picks nwi (and nwc = 8 / nwi) so that most merges take one round.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) k_merge(DecodeArgs a, int nwc) {
    constexpr int NW = kMergeThreads / 32, R = 12;
    __shared__ float red_m[2][NW];
    __shared__ float part_o[NW][32];
    __shared__ float part_l[NW];
    grid_dependency_wait();
    const Layout& lo = a.lo;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int h = hq / lo.gqa, head = hq % lo.gqa;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwi = NW / nwc, wc = warp % nwc, wi = warp / nwc;
    const int S = a.plan.S;
    const float* ml = reinterpret_cast<const float*>(a.ws + a.plan.ws_ml_off);
    const float* o = reinterpret_cast<const float*>(a.ws + a.plan.ws_o_off);
    const int64_t slot0 = (((int64_t)b * lo.H + h) * S) * lo.gqa + head;   // + item * gqa
    const int c = 32 * (blockIdx.x * nwc + wc) + lane;
    float M = -INFINITY, acc = 0.0f, l = 0.0f;
    const int rounds = (S + nwi * R - 1) / (nwi * R);     // the same in every warp (barriers inside)
    for (int round = 0; round < rounds; ++round) {
        const int it0 = wi + round * nwi * R;
        float mv[R], lv[R], ov[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int it = it0 + nwi * k;
            mv[k] = -INFINITY;
            lv[k] = 0.0f;
            ov[k] = 0.0f;
            if (it < S) {
                // every item leaves a partial (an empty one has l = 0: weight 0, and its o
                // is not used), so all loads go out at once without the cache state
                const int64_t sl = slot0 + (int64_t)it * lo.gqa;
                const float2 mlv = *reinterpret_cast<const float2*>(ml + 2 * sl);
                const float ovl = o[sl * D + c];
                mv[k] = mlv.y > 0.0f ? mlv.x : -INFINITY;
                lv[k] = mlv.y > 0.0f ? mlv.y : 0.0f;
                ov[k] = mlv.y > 0.0f ? ovl : 0.0f;
            }
        }
        // the round's maximum over the block (the same in every lane of a warp)
        float mr = mv[0];
#pragma unroll
        for (int k = 1; k < R; ++k) mr = fmaxf(mr, mv[k]);
        if (lane == 0) red_m[round & 1][warp] = mr;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < NW; ++w) mr = fmaxf(mr, red_m[round & 1][w]);
        const float mnew = fmaxf(M, mr);
        if (mnew > M && M > -INFINITY) {
            const float f = fast_exp2(M - mnew);
            acc *= f;
            l *= f;
        }
        M = mnew;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const float w = lv[k] > 0.0f ? fast_exp2(mv[k] - M) : 0.0f;
            acc = fmaf(ov[k], w, acc);
            l = fmaf(lv[k], w, l);
        }
    }
    part_o[warp][lane] = acc;
    if (lane == 0) part_l[warp] = l;
    __syncthreads();
    if (wi == 0) {
        float L = 0.0f, v = 0.0f;
        for (int j = 0; j < nwi; ++j) {
            L += part_l[j * nwc + wc];
            v += part_o[j * nwc + wc][lane];
        }
        a.out[((int64_t)b * lo.Hq + hq) * D + c] = L > 0.0f ? v / L : 0.0f;
    }
}

// The same merge for plans with at most kSmallS chunks per (sequence, query head): one
// thread per output element loads all of its chunks' partials at once, so the whole merge
// is one wave of small blocks with two rounds of loads.
constexpr int kSmallS = 4;
template <int D>
__global__ void __launch_bounds__(kMergeThreads) k_merge_small(DecodeArgs a) {
    grid_dependency_wait();
    const Layout& lo = a.lo;
    const int64_t idx = (int64_t)blockIdx.x * kMergeThreads + threadIdx.x;   // (b, hq, c)
    if (idx >= (int64_t)lo.B * lo.Hq * D) return;
    const int c = static_cast<int>(idx % D);
    const int64_t bh = idx / D;
    const int hq = static_cast<int>(bh % lo.Hq), b = static_cast<int>(bh / lo.Hq);
    const int h = hq / lo.gqa, head = hq % lo.gqa;
    const int S = a.plan.S;
    const float* ml = reinterpret_cast<const float*>(a.ws + a.plan.ws_ml_off);
    const float* o = reinterpret_cast<const float*>(a.ws + a.plan.ws_o_off);
    const int64_t slot0 = (((int64_t)b * lo.H + h) * S) * lo.gqa + head;
    float mv[kSmallS], lv[kSmallS], ov[kSmallS];
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < kSmallS; ++k) {
        mv[k] = -INFINITY;
        lv[k] = 0.0f;
        ov[k] = 0.0f;
        if (k < S) {
            const int64_t sl = slot0 + (int64_t)k * lo.gqa;
            const float2 mlv = *reinterpret_cast<const float2*>(ml + 2 * sl);
            const float ovl = o[sl * D + c];
            mv[k] = mlv.y > 0.0f ? mlv.x : -INFINITY;
            lv[k] = mlv.y > 0.0f ? mlv.y : 0.0f;
            ov[k] = mlv.y > 0.0f ? ovl : 0.0f;
        }
        M = fmaxf(M, mv[k]);
    }
    float L = 0.0f, v = 0.0f;
#pragma unroll
    for (int k = 0; k < kSmallS; ++k) {
        const float w = lv[k] > 0.0f ? fast_exp2(mv[k] - M) : 0.0f;
        v = fmaf(ov[k], w, v);
        L = fmaf(lv[k], w, L);
    }
    a.out[idx] = L > 0.0f ? v / L : 0.0f;
}

template <int D>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t stream) {
    const Layout& lo = a.lo;
    if (a.plan.S <= kSmallS) {
        const int64_t n = (int64_t)lo.B * lo.Hq * D;
        return launch_dependent(k_merge_small<D>, dim3(static_cast<unsigned>((n + kMergeThreads - 1) / kMergeThreads)),
                                kMergeThreads, 0, stream, a);
    }
    // warps over chunks: enough for one round of 12 chunks each (at most all 8), the rest
    // of the block's warps over channels (at most D / 32)
    int nwi = 1;
    while (nwi < kMergeThreads / 32 && nwi * 12 < a.plan.S) nwi *= 2;
    int nwc = kMergeThreads / 32 / nwi;
    if (nwc > D / 32) {
        nwc = D / 32;
        nwi = kMergeThreads / 32 / nwc;
    }
    return launch_dependent(k_merge<D>, dim3(D / (32 * nwc), lo.Hq, lo.B), kMergeThreads, 0, stream, a, nwc);
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
    } else if (lo.scheme == KVQ_SCHEME_FP8_E4M3) {
        rc = launch_decode_fp8(a, stream);
    } else {
        rc = launch_decode_rows(a, stream);
    }
    if (rc != KVQ_OK) return rc;
    cudaError_t e;
    switch (lo.D) {
        case 32: e = launch_merge<32>(a, stream); break;
        case 64: e = launch_merge<64>(a, stream); break;
        case 128: e = launch_merge<128>(a, stream); break;
        default: e = launch_merge<256>(a, stream); break;
    }
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
