// kvq_decode_fp8.cu -- single-query decode attention over FP8 (E4M3 or E5M2) caches on the
// tensor cores.
//
// An E4M3 value is exactly an fp16 value (3 mantissa bits, exponents inside fp16's
// range), and an E5M2 value is the upper byte of its fp16 value, so the codes go straight
// into mma.sync.m16n8k16 (f16 -> f32) after one conversion per code pair.  The key and value scales are per (layer, kv head)
// ("How the KV cache is quantized": one scale per tensor or head), so the query operand
// (query * key scale, split into fp16 major + minor parts) is built once per block and
// stays in registers, and the value scale is applied once to the block's output.
//
// Storage order (see the cache layout): a key row keeps, per 16-channel block, the
// channels 2i, 2i + 1, 2i + 8, 2i + 9 of lane quarter i side by side; values come in
// tiles of 16 tokens stored [channel][16 bytes] with tokens 2i, 2i + 8, 2i + 1, 2i + 9
// side by side.  One 32-bit shared load then gives a lane both halves of an A fragment
// row, and the value pairs (tt, tt + 8) match the score rows a lane holds.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

// The four FP8 codes of `w` as two fp16 pairs: lo <- bytes 0, 1 and hi <- bytes 2, 3 (the
// lower byte of each 16-bit half to the lower fp16).  One conversion per pair, straight
// from the register halves; both FP8 formats convert to fp16 exactly.
template <bool E5M2>
__device__ __forceinline__ void fp8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if constexpr (E5M2)
        asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e5m2x2 %0, l;\n cvt.rn.f16x2.e5m2x2 %1, h;\n}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    else
        asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n cvt.rn.f16x2.e4m3x2 %0, l;\n cvt.rn.f16x2.e4m3x2 %1, h;\n}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
}

// One FP8 work item: a run of chunks of CH = 4 * W tokens of one (sequence, kv head).
// Each warp takes W tokens (whole 16-token tiles but the sequence's last) of a chunk and
// keeps an online softmax across the item's chunks.
template <int D, int NT, bool E5M2>
__device__ __forceinline__ int fp8_item(const DecodeArgs& a, uint8_t* smem, int b, int h, int64_t slot, int64_t t0,
                                     int64_t t1, uint32_t phase) {
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    constexpr int NPAIR = D / 8;            // B words per lane and head block
    constexpr int KSTEPS = D / 16;
    constexpr int MTV = D / 16;             // 16-channel tiles of the value contraction
    constexpr int KQ = D / 16;              // words of a key row's lane quarter
    constexpr int QROW = NPAIR + 4;         // words per row of the query table (padded)
    constexpr int MAXT = 8;
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
    const int W = a.plan.W, CH = a.plan.CH, gqa = lo.gqa, nstage = a.plan.NSTAGE;
    const int ntok = static_cast<int>(t1 - t0);
    const int nch = (ntok + CH - 1) / CH;
    const uint32_t stage_bytes = static_cast<uint32_t>(CH) * 2 * D;     // key rows, then value tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    uint32_t* qt = reinterpret_cast<uint32_t*>(smem + so.qpa);
    float* comb = reinterpret_cast<float*>(smem + so.sc);          // [warp][head][D]
    float* cml = comb + 4 * gqa * D;                               // [warp][head][m, l]
    const int64_t u = unit_index(lo, a.layer, b, h);
    const uint8_t* unit = a.cache + lo.data_off + u * lo.unit;
    const uint8_t* kbase = unit + t0 * D;                          // t0 is a multiple of 16
    const uint8_t* vbase = unit + (int64_t)lo.T16 * D + t0 * D;

    auto issue = [&](int j) {       // stage chunk j (thread 0 only)
        const int cnt = min(CH, ntok - j * CH);
        const uint32_t kb = static_cast<uint32_t>(cnt) * D;
        const uint32_t vb = static_cast<uint32_t>((cnt + 15) / 16) * 16 * D;   // whole value tiles
        const int sj = nstage == 2 ? (j & 1) : 0;
        uint64_t* bar = bars + sj;
        uint8_t* st = smem + so.data + sj * stage_bytes;
        mbar_arrive_expect_tx(bar, kb + vb);
        bulk_copy_pieces(st, kbase + (int64_t)j * CH * D, kb, bar);
        bulk_copy_pieces(st + CH * D, vbase + (int64_t)j * CH * D, vb, bar);
    };
    if (tid == 0) {
        for (int j = 0; j < nstage && j < nch; ++j) issue(j);
    }
    // query prep while the copies are in flight: the fp32 scaled query and its largest
    // magnitude, then per lane (row 32 * nt + lane) the B column of the lane: (q * key
    // scale * 2^E) as fp16 major (part 0) or minor (part 1), E bringing the key scale to
    // [2^14, 2^15) so that no fp16 product overflows
    float qmax = 0.0f;
    {
        const int64_t base = ((int64_t)b * lo.Hq + (int64_t)h * gqa) * D;
        if (lo.dtype == KVQ_DTYPE_BF16) {
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.q) + base);
            for (int i = tid; i < gqa * D / 8; i += blockDim.x) {
                const uint4 v = src[i];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(w[e] << 16) * a.qscale;
                    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * a.qscale;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) qmax = fmaxf(qmax, fabsf(f[e]));
                reinterpret_cast<float4*>(qs)[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
                reinterpret_cast<float4*>(qs)[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
            }
        } else {
            const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.q) + base);
            for (int i = tid; i < gqa * D / 4; i += blockDim.x) {
                float4 v = src[i];
                v.x *= a.qscale;
                v.y *= a.qscale;
                v.z *= a.qscale;
                v.w *= a.qscale;
                qmax = fmaxf(fmaxf(qmax, fmaxf(fabsf(v.x), fabsf(v.y))), fmaxf(fabsf(v.z), fabsf(v.w)));
                reinterpret_cast<float4*>(qs)[i] = v;
            }
        }
    }
    qmax = warp_max(qmax);
    if (lane == 0) red[warp * 32] = qmax;
    __syncthreads();
    qmax = fmaxf(fmaxf(red[0], red[32]), fmaxf(red[64], red[96]));
    int qexp = 0;
    if (qmax > 0.0f) frexpf(qmax, &qexp);
    const float* tab = reinterpret_cast<const float*>(a.cache + lo.scales_off) + ((int64_t)a.layer * lo.H + h) * 2;
    const float kscale = tab[0], vscale = tab[1];
    int kexp = 0;
    if (kscale > 0.0f) frexpf(kscale, &kexp);
    const int E = max(-100, min(100, 15 - kexp));
    const float kse = ldexpf(kscale, E - qexp);             // key scale * 2^E * query prescale
    const float kf = ldexpf(1.0f, qexp - E);                // undoes both on the fp32 scores
    for (int i = tid; i < 16 * NT * NPAIR; i += blockDim.x) {
        const int m = i % NPAIR, r = i / NPAIR;
        const int hh = r >> 2, tg = r & 3;
        const int c = 16 * (m >> 1) + 8 * (m & 1) + 2 * tg;    // channels c, c + 1 of pair m
        float vlo = 0.0f, vhi = 0.0f;
        if (hh < gqa) {
            vlo = qs[hh * D + c] * kse;
            vhi = qs[hh * D + c + 1] * kse;
        }
        const __half2 major = __floats2half2_rn(vlo, vhi);
        const float2 mf = __half22float2(major);
        const int row0 = 32 * (hh >> 2) + 8 * (hh & 3) + tg;   // lane of part 0; part 1 is 4 lanes on
        qt[row0 * QROW + m] = h2_as_u32(major);
        qt[(row0 + 4) * QROW + m] = h2_as_u32(__floats2half2_rn(vlo - mf.x, vhi - mf.y));
    }
    __syncthreads();
    uint32_t bq[NT][NPAIR];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
        lds_words<NPAIR>(smem_addr(qt) + (32 * nt + lane) * QROW * 4, bq[nt]);

    const uint32_t sbase = smem_addr(smem);
    const int part = g & 1;                 // B column g = 2 * head + part
    const int src1 = (2 * tig) * 4 + (g >> 1), src2 = (2 * tig + 1) * 4 + (g >> 1);
    float mrun[NT], lrun[NT];
    float oacc[MTV][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrun[nt] = -INFINITY;
        lrun[nt] = 0.0f;
#pragma unroll
        for (int mt = 0; mt < MTV; ++mt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.0f;
    }
    const int wt0 = warp * W;               // the warp's first token of every chunk
    for (int j = 0; j < nch; ++j) {
        const int sj = nstage == 2 ? (j & 1) : 0;
        if (!wait_stage(bars, sj, phase, a.ws)) {
            // the next chunk's copy may already be armed on the other stage
            if (nstage == 2 && j + 1 < nch) drain_stage(bars, sj ^ 1, phase);
            empty_partial(a, slot);
            return -1;
        }
        const int cnt = min(CH, ntok - j * CH);
        const int wtok = cnt - wt0 < 0 ? 0 : (cnt - wt0 > W ? W : cnt - wt0);
        const uint32_t st = sbase + static_cast<uint32_t>(so.data) + sj * stage_bytes;
        if (wtok > 0) {
            const int ntl = (wtok + 15) >> 4;
            float2* wsc = reinterpret_cast<float2*>(smem + so.sc) + (int64_t)warp * MAXT * NT * 32 + lane;
            float cmax[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) cmax[nt] = -INFINITY;
            // ---- pass 1: scores (rows g and g + 8 of each tile are tokens g and g + 8)
#pragma unroll 1
            for (int i = 0; i < ntl; ++i) {
                const int tv = wtok - 16 * i;                 // valid tokens of this tile
                const uint32_t kr = st + (wt0 + 16 * i) * D + tig * (D / 4);
                uint32_t wa[KQ], wb[KQ];
                lds_words<KQ>(kr + g * D, wa);
                lds_words<KQ>(kr + (g + 8) * D, wb);
                float acc[2][NT][4];
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) acc[e][nt][0] = acc[e][nt][1] = acc[e][nt][2] = acc[e][nt][3] = 0.0f;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    uint32_t af[4];
                    fp8x4_to_f16x2x2<E5M2>(wa[ks], af[0], af[2]);
                    fp8x4_to_f16x2x2<E5M2>(wb[ks], af[1], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_16816(acc[ks & 1][nt], af, bq[nt][2 * ks], bq[nt][2 * ks + 1]);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float s0 = ((acc[0][nt][0] + acc[1][nt][0]) + (acc[0][nt][1] + acc[1][nt][1])) * kf;
                    float s1 = ((acc[0][nt][2] + acc[1][nt][2]) + (acc[0][nt][3] + acc[1][nt][3])) * kf;
                    if (g >= tv) s0 = -INFINITY;              // rows past the sequence's end
                    if (g + 8 >= tv) s1 = -INFINITY;
                    wsc[(i * NT + nt) * 32] = make_float2(s0, s1);
                    cmax[nt] = fmaxf(cmax[nt], fmaxf(s0, s1));
                }
            }
            // running maximum per head; rescale what the warp accumulated when it grows
            float mE[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float m = cmax[nt];
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                const float mnew = fmaxf(mrun[nt], m);
                if (mnew > mrun[nt] && mrun[nt] > -INFINITY) {
                    const float alpha = fast_exp2(mrun[nt] - mnew);
                    lrun[nt] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) oacc[mt][nt][e] *= alpha;
                }
                mrun[nt] = mnew;
                // p' = 2^(s - max + 15) <= 2^15: the value operand's power-of-two scale rides
                // in the exponent and cancels between the output and its sum
                mE[nt] = mnew - 15.0f;
            }
            // ---- pass 2: p' and the value contraction, tile by tile
#pragma unroll 1
            for (int i = 0; i < ntl; ++i) {
                uint32_t b0[NT], b1[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 sv = wsc[(i * NT + nt) * 32];
                    const float p0 = fast_exp2(sv.x - mE[nt]);
                    const float p1 = fast_exp2(sv.y - mE[nt]);
                    lrun[nt] += p0 + p1;
                    const __half2 pa = __floats2half2_rn(p0, p1);
                    const float2 pf = __half22float2(pa);
                    const __half2 pb = __floats2half2_rn(p0 - pf.x, p1 - pf.y);
                    const uint32_t ua = h2_as_u32(pa), ub = h2_as_u32(pb);
                    const uint32_t x1 = __shfl_sync(0xffffffffu, ua, src1);
                    const uint32_t y1 = __shfl_sync(0xffffffffu, ub, src1);
                    const uint32_t x2 = __shfl_sync(0xffffffffu, ua, src2);
                    const uint32_t y2 = __shfl_sync(0xffffffffu, ub, src2);
                    b0[nt] = part ? y1 : x1;
                    b1[nt] = part ? y2 : x2;
                }
                // this lane's bytes of a value tile row: tokens 2t, 2t + 8 (low half) and
                // 2t + 1, 2t + 9 (high half); tokens past the sequence's end are masked to
                // zero codes (their p' is 0, and stale bytes could read as NaN)
                const int tv = wtok - 16 * i;
                uint32_t vmask = 0xffffffffu;
                if (tv < 16)
                    vmask = (2 * tig < tv ? 0x000000ffu : 0u) | (2 * tig + 8 < tv ? 0x0000ff00u : 0u) |
                            (2 * tig + 1 < tv ? 0x00ff0000u : 0u) | (2 * tig + 9 < tv ? 0xff000000u : 0u);
                const uint32_t vt = st + CH * D + (wt0 + 16 * i) * D + 16 * g + 4 * tig;
#pragma unroll
                for (int q = 0; q < MTV; ++q) {
                    const uint32_t w0 = lds32(vt + 256 * q) & vmask;          // channel 16q + g
                    const uint32_t w1 = lds32(vt + 256 * q + 128) & vmask;    // channel 16q + g + 8
                    uint32_t af[4];
                    fp8x4_to_f16x2x2<E5M2>(w0, af[0], af[2]);
                    fp8x4_to_f16x2x2<E5M2>(w1, af[1], af[3]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[q][nt], af, b0[nt], b1[nt]);
                }
            }
        }
        __syncthreads();            // every warp is done with this stage
        if (tid == 0 && j + nstage < nch) issue(j + nstage);
    }
    // ---- warp partial (o carries the value scale; o and l share the factor 2^15), then
    // the 4 warps combined in shared memory
    float* cw = comb + warp * gqa * D;
    const bool wlive = mrun[0] > -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int head = 4 * nt + tig;
        float l = lrun[nt];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        if (head < gqa && wlive) {
#pragma unroll
            for (int mt = 0; mt < MTV; ++mt) {
                const int c0 = 16 * mt + g;
                cw[head * D + c0] = (oacc[mt][nt][0] + oacc[mt][nt][1]) * vscale;
                cw[head * D + c0 + 8] = (oacc[mt][nt][2] + oacc[mt][nt][3]) * vscale;
            }
        }
        if (g == 0 && head < gqa) {
            cml[2 * (warp * gqa + head)] = wlive ? mrun[nt] : -INFINITY;
            cml[2 * (warp * gqa + head) + 1] = wlive ? l : 0.0f;
        }
    }
    __syncthreads();
    combine_warps<D>(a, comb, cml, red, slot);
    return static_cast<int>(phase);
}

// One wave of blocks; block j takes its share of the layer's chunks (for_each_segment).
template <int D, int NT, bool E5M2>
__global__ void __launch_bounds__(kDecodeThreads, (NT == 1 && D <= 128) ? 4 : 2)
    k_decode_fp8(const __grid_constant__ DecodeArgs a) {
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
        [&](int, int b, int h, int64_t slot, int64_t t0, int64_t t1, const StealCtx&) -> bool {
            const int r = fp8_item<D, NT, E5M2>(a, smem, b, h, slot, t0, t1, phase);
            if (r < 0) return false;
            phase = static_cast<uint32_t>(r);
            return true;
        },
        [&](int64_t slot) { empty_partial(a, slot); });
}

template <int D, int NT>
int launch_fp8_t(DecodeArgs& a, cudaStream_t stream) {
    if (a.lo.scheme == KVQ_SCHEME_FP8_E5M2) return launch_wave(k_decode_fp8<D, NT, true>, a, stream);
    return launch_wave(k_decode_fp8<D, NT, false>, a, stream);
}

}  // namespace

int launch_decode_fp8(DecodeArgs& a, cudaStream_t stream) {
    const bool wide = a.lo.gqa > 4;
    switch (a.lo.D) {
        case 32: return wide ? launch_fp8_t<32, 2>(a, stream) : launch_fp8_t<32, 1>(a, stream);
        case 64: return wide ? launch_fp8_t<64, 2>(a, stream) : launch_fp8_t<64, 1>(a, stream);
        case 128: return wide ? launch_fp8_t<128, 2>(a, stream) : launch_fp8_t<128, 1>(a, stream);
        case 256: return wide ? launch_fp8_t<256, 2>(a, stream) : launch_fp8_t<256, 1>(a, stream);
        default: return KVQ_ERR_UNSUPPORTED;
    }
}

}  // namespace kvq
