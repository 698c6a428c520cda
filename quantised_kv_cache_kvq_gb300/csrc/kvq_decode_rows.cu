// kvq_decode_rows.cu -- the INT8 / INT4 decode dispatch, the log-sum-exp merge of the partial
// results, and the decode dispatcher.
#include <cmath>

#include "kvq_decode.cuh"

namespace kvq {
namespace {

constexpr int kMaxCand = KVQ_MAX_DECODE_BLOCKS;   // candidate blocks of one part of a unit

// Combine the partials of one (sequence, kv head) unit for one query head: with partial i
// holding m_i (max score, base 2), l_i = sum 2^(s - m_i) and o_i = sum 2^(s - m_i) v, the
// output is sum_i o_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M = max_i m_i (log-sum-exp).
//
// A block takes one query head of one unit, or 32 of its channels (SLICED: a lane per
// channel, for batches of few units with many partials each; otherwise a lane holds D / 32
// channels, read by vector loads), with W warps: warp w takes every W-th partial, with the
// loads of UNR partials in flight, so one round of loads covers up to W UNR partials.  Everything up to the slot list (the layer's
// totals, the unit's prefixes, the decode blocks that took chunks of the unit) depends
// only on the token counts that the kernels before the decode wrote: it runs while the
// decode is still finishing (this grid is its programmatic dependent), and only the
// partial loads wait for the decode.  The warps are combined in shared memory.
template <int NT>
__device__ __forceinline__ int64_t merge_sum64(int64_t v, int64_t* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int64_t t = 0;
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    __syncthreads();
    return t;
}

template <int D, int W, bool SLICED>
__global__ void __launch_bounds__(32 * W) k_merge(const __grid_constant__ DecodeArgs a) {
    constexpr int NT = 32 * W, Z = SLICED ? D / 32 : 1, CPL = SLICED ? 1 : D / 32;
    constexpr int UNR = CPL > 4 ? 6 : 12;
    __shared__ int cand[2 * kMaxCand];
    __shared__ int ncand;
    __shared__ int64_t red[W];
    __shared__ float gm[W], gl[W];
    __shared__ __align__(16) float go[W][32 * CPL];
    const Layout& lo = a.lo;
    const int z = blockIdx.x % Z, uh = blockIdx.x / Z;
    const int u = uh / lo.gqa, hh = uh % lo.gqa;
    const int b = u / lo.H, h = u % lo.H;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    SplitCtx x;
    {
        int64_t c0s = 0, c1s = 0, lv = 0, p0 = 0, p1 = 0;
        for (int bb = tid; bb < lo.B; bb += NT) {
            int64_t c0, c1;
            part_costs(a, seq_state(a, bb), c0, c1);
            c0s += c0;
            c1s += c1;
            lv += c0 + c1 > 0;
            if (bb < b) {
                p0 += c0;
                p1 += c1;
            }
        }
        x.C0 = lo.H * merge_sum64<NT>(c0s, red);
        x.C = x.C0 + lo.H * merge_sum64<NT>(c1s, red);
        x.live = lo.H * merge_sum64<NT>(lv, red);
        x.P0 = lo.H * merge_sum64<NT>(p0, red);
        x.P1 = lo.H * merge_sum64<NT>(p1, red);
        x.K = 0;
        if (a.plan.unit_aligned && x.C > 0) {
            int64_t kk = 0;
            for (int bb = tid; bb < b; bb += NT) {
                int64_t c0, c1;
                part_costs(a, seq_state(a, bb), c0, c1);
                kk += unit_blocks(c0 + c1, x.C, a.plan.NB - x.live);
            }
            x.K = lo.H * merge_sum64<NT>(kk, red);
        }
    }
    const int2 st = seq_state(a, b);
    const int total = unit_candidates(a, u, st, x, cand, NT);
    if (tid == 0) ncand = total;
    grid_dependency_wait();
    // the decode is complete: its chunk counter of this unit goes back to zero
    if (a.plan.steal && z == 0 && hh == 0 && tid == 0)
        reinterpret_cast<int*>(a.ws + a.plan.ws_ctr_off)[u] = 0;
    __syncthreads();
    const int n = ncand;
    const int c0 = 32 * z + lane * CPL;  // this lane's first channel
    float M = -INFINITY, L = 0.0f, O[CPL];
#pragma unroll
    for (int e = 0; e < CPL; ++e) O[e] = 0.0f;
    for (int i0 = warp; i0 < n; i0 += W * UNR) {
        float mv[UNR], lvv[UNR], ov[UNR][CPL];
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const int i = i0 + k * W;
            const int slot = i < n ? cand[i] : -1;
            mv[k] = -INFINITY;
            lvv[k] = 0.0f;
#pragma unroll
            for (int e = 0; e < CPL; ++e) ov[k][e] = 0.0f;
            if (slot >= 0) {
                const float2 ml = *reinterpret_cast<const float2*>(slot_ml(a, slot, hh));
                const float* op = slot_o(a, slot, hh) + c0;
                if constexpr (CPL % 4 == 0) {
#pragma unroll
                    for (int e = 0; e < CPL; e += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(op + e);
                        ov[k][e] = v.x;
                        ov[k][e + 1] = v.y;
                        ov[k][e + 2] = v.z;
                        ov[k][e + 3] = v.w;
                    }
                } else if constexpr (CPL == 2) {
                    const float2 v = *reinterpret_cast<const float2*>(op);
                    ov[k][0] = v.x;
                    ov[k][1] = v.y;
                } else {
                    ov[k][0] = op[0];
                }
                if (ml.y > 0.0f) {
                    mv[k] = ml.x;
                    lvv[k] = ml.y;
                }
            }
        }
        float mr = M;
#pragma unroll
        for (int k = 0; k < UNR; ++k) mr = fmaxf(mr, mv[k]);
        if (mr == -INFINITY) continue;
        const float f = M > -INFINITY ? fast_exp2(M - mr) : 0.0f;
        L *= f;
#pragma unroll
        for (int e = 0; e < CPL; ++e) O[e] *= f;
#pragma unroll
        for (int k = 0; k < UNR; ++k) {
            const float w = lvv[k] > 0.0f ? fast_exp2(mv[k] - mr) : 0.0f;
            L = fmaf(lvv[k], w, L);
#pragma unroll
            for (int e = 0; e < CPL; ++e) O[e] = fmaf(ov[k][e], w, O[e]);
        }
        M = mr;
    }
    float* outp = a.out + ((int64_t)b * lo.Hq + (int64_t)h * lo.gqa + hh) * D;
    if constexpr (W == 1) {
        const float inv = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
        for (int e = 0; e < CPL; ++e) outp[c0 + e] = O[e] * inv;
    } else {
        if (lane == 0) {
            gm[warp] = M;
            gl[warp] = L;
        }
#pragma unroll
        for (int e = 0; e < CPL; ++e) go[warp][lane * CPL + e] = O[e];
        __syncthreads();
        for (int c = tid; c < 32 * CPL; c += NT) {
            float Mx = -INFINITY;
            for (int w = 0; w < W; ++w) Mx = fmaxf(Mx, gm[w]);
            float Ls = 0.0f, Os = 0.0f;
            if (Mx > -INFINITY) {
                for (int w = 0; w < W; ++w) {
                    if (gm[w] == -INFINITY) continue;
                    const float f = fast_exp2(gm[w] - Mx);
                    Ls = fmaf(gl[w], f, Ls);
                    Os = fmaf(go[w][c], f, Os);
                }
            }
            outp[32 * z + c] = Ls > 0.0f ? Os / Ls : 0.0f;
        }
    }
}

// Warps per block from the slot list a unit has when its length is the mean: one wave of
// NB blocks over B H units gives each unit about NB / (B H) blocks.  Whole-block split
// (units <= NB / 2): 2 k entries, merged in 32-channel slices by one round of 12 loads per
// warp.  Cost ranges (more units): fewer than 2 blocks per unit, each part's range widened
// by two on each side, merged a whole head per block.
template <int D, int W>
cudaError_t launch_merge_sliced(const DecodeArgs& a, cudaStream_t stream) {
    const int64_t heads = (int64_t)a.lo.B * a.lo.Hq;
    return launch_dependent(k_merge<D, W, true>, dim3(static_cast<unsigned>(heads * (D / 32))), 32 * W, 0, stream, a);
}

template <int D>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t stream) {
    const int64_t units = (int64_t)a.lo.B * a.lo.H;
    if (!a.plan.unit_aligned) {
        const dim3 grid(static_cast<unsigned>((int64_t)a.lo.B * a.lo.Hq));
        if (2 * (a.plan.NB / units + 6) <= 12) return launch_dependent(k_merge<D, 1, false>, grid, 32, 0, stream, a);
        return launch_dependent(k_merge<D, 2, false>, grid, 64, 0, stream, a);
    }
    const int64_t per_unit = 2 * (a.plan.NB / units + 1);
    if (per_unit <= 12) return launch_merge_sliced<D, 1>(a, stream);
    if (per_unit <= 24) return launch_merge_sliced<D, 2>(a, stream);
    if (per_unit <= 48) return launch_merge_sliced<D, 4>(a, stream);
    if (per_unit <= 96) return launch_merge_sliced<D, 8>(a, stream);
    if (per_unit <= 192) return launch_merge_sliced<D, 16>(a, stream);
    return launch_merge_sliced<D, 32>(a, stream);
}

}  // namespace

int launch_decode_rows(DecodeArgs& a, cudaStream_t stream) {
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
    if (lo.scheme == KVQ_SCHEME_KIVI && lo.rope_base > 0.0f) {
        // keys cached before RoPE: w_i = base^(-2i/D), binary64 power rounded to binary32
        for (int i = 0; i < lo.D / 2; ++i)
            a.rope_w[i] = static_cast<float>(std::pow(static_cast<double>(lo.rope_base), -2.0 * i / lo.D));
        rc = launch_decode_rope(a, stream);
    } else if (lo.scheme == KVQ_SCHEME_KIVI && lo.K > 0) {
        // dense-and-sparse records: the kernels that add the outliers' corrections
        rc = lo.bits == 2 ? launch_decode_kivi2_sparse(a, stream)
           : lo.bits == 4 ? launch_decode_kivi4_sparse(a, stream)
                          : launch_decode_kivi8_sparse(a, stream);
    } else if (lo.scheme == KVQ_SCHEME_KIVI) {
        rc = lo.bits == 2 ? launch_decode_kivi2(a, stream)
           : lo.bits == 4 ? launch_decode_kivi4(a, stream)
                          : launch_decode_kivi8(a, stream);
    } else if (is_fp8(lo.scheme)) {
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
