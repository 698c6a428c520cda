// kvq_append.cu -- quantise-and-pack kernels: appending tokens to the cache and flushing
// full groups out of the KIVI window.
//
// Arithmetic (bit-exact contract): binary32 min/max, one IEEE subtraction and one IEEE
// division per step with round-to-nearest (the __f*_rn intrinsics), round-half-even to
// integer, binary16 parameters rounded with __float2half_rd / _ru.  This file is built
// with --fmad=false so no multiply-add is ever contracted.
//
// Quantisers:
//  * KIVI Q_b ("Quantizing the KV cache", "Per-channel and per-token grouping"):
//    s = (max - min) / (2^b - 1), code = round((x - min) / s); keys per channel over a
//    group of G tokens, values per token over Gv channels ("Keys and values are shaped
//    differently"; "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
//    "How It Works").  The window keeps the newest tokens in bf16 and quantises the
//    oldest G as a group whenever it would reach R + G tokens.
//  * INT8 per-token symmetric ("Quantising the Cache", "Workshop"): scale = max|x| / 127;
//    INT4 the same at 4 bits (the glossary "kv cache quantization"): scale = max|x| / 7.
//  * FP8 E4M3 or E5M2 with a per-(layer, KV head) scale ("Quantizing the KV cache", "How the
//    KV cache is quantized").
#include <cuda_fp8.h>

#include "kvq_internal.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float load_input(const void* p, int64_t idx, int dtype) {
    if (dtype == KVQ_DTYPE_BF16)
        return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p)[idx]);
    return reinterpret_cast<const float*>(p)[idx];
}

// Element offset of channel 0 of input row (sequence bi, new-token j, kv head h).
__device__ __forceinline__ int64_t input_row(const Layout& lo, int n_new, int bi, int64_t j, int h) {
    return (((int64_t)bi * n_new + j) * lo.H + h) * lo.D;
}

// Tokens a sequence takes in this append, or -1 when it is skipped (capacity or a full
// window); sets the matching status bit in *st.
// qn after taking m tokens (the window is flushed while it would hold >= R + G tokens).
__device__ __forceinline__ int qn_after(const Layout& lo, int n, int qn, int m, uint32_t flags) {
    if (lo.scheme != KVQ_SCHEME_KIVI) return n + m;
    if (flags & KVQ_NO_AUTOFLUSH) return qn;
    int over = n + m - qn - lo.R;
    return over >= lo.G ? qn + lo.G * (over / lo.G) : qn;
}

__device__ __forceinline__ int tokens_taken(const Layout& lo, int b, int n, int qn, int m, uint32_t flags,
                                            uint32_t* st) {
    if ((int64_t)n + m > lo.T) {
        *st |= KVQ_STATUS_CAPACITY;
        return -1;
    }
    if (lo.scheme == KVQ_SCHEME_KIVI && (flags & KVQ_NO_AUTOFLUSH) && n + m - qn > lo.C) {
        *st |= KVQ_STATUS_RING_FULL;
        return -1;
    }
    // paged layout: every group this append packs needs a page of the pool
    if (lo.PG > 0 && !pages_ok(lo, b, qn / lo.G, qn_after(lo, n, qn, m, flags) / lo.G)) {
        *st |= KVQ_STATUS_BAD_PAGE;
        return -1;
    }
    return m;
}

// Q_b parameters of one group: offset = min rounded down to binary16, scale = (max -
// offset) / levels rounded up to binary16.
struct QbParams {
    __half s, z;
    float sf, zf;
};
__device__ __forceinline__ QbParams qb_params(float mn, float mx, float levels) {
    QbParams p;
    p.z = __float2half_rd(mn);
    p.zf = __half2float(p.z);
    float s32 = __fdiv_rn(__fsub_rn(mx, p.zf), levels);
    p.s = __float2half_ru(s32);
    p.sf = __half2float(p.s);
    return p;
}
__device__ __forceinline__ uint32_t qb_code(float x, const QbParams& p, int levels) {
    if (p.sf == 0.0f) return 0u;
    int c = __float2int_rn(__fdiv_rn(__fsub_rn(x, p.zf), p.sf));
    c = c < 0 ? 0 : (c > levels ? levels : c);
    return static_cast<uint32_t>(c);
}

__device__ __forceinline__ bool nonfinite(float x) { return !isfinite(x); }

// Source of window/input token t of unit (l, b, h) for the group quantiser.
struct TokenSource {
    const uint8_t* ring_unit;  // first slot of the unit's window
    const void* k_new;
    const void* v_new;
    int64_t n;                 // tokens before this append
    int n_new, bi;
};
// Quantise the KIVI group of G tokens starting at absolute token t0 of unit (l, b, h)
// into its record.  Token t < s.n comes from window slot t % C, later tokens from the
// new input rows.  Cooperative over the whole block.  The group's bf16 keys and values
// are first staged into shared memory with 16-byte loads; `smem` holds 5*G*D bytes
// (keys G*D bf16, values G*D bf16, codes G*D bytes).  Returns the non-finite flag
// seen by this thread.
__device__ uint32_t quantise_group(const Layout& lo, uint8_t* cache, int l, int b, int h,
                                   int64_t t0, const TokenSource& s, uint8_t* smem) {
    const int D = lo.D, G = lo.G, Gv = lo.Gv, bits = lo.bits;
    const int levels = (1 << bits) - 1;
    const float flevels = static_cast<float>(levels);
    // (a paged record's page was checked by the caller's admission rule)
    uint8_t* rec = cache + group_offset(lo, l, b, h, t0 / G);
    __half* kpar = reinterpret_cast<__half*>(rec + lo.kc + lo.vc);
    __half* vpar = reinterpret_cast<__half*>(rec + lo.kc + lo.vc + lo.kp);
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem);
    uint16_t* vs = ks + G * D;
    uint8_t* codes = reinterpret_cast<uint8_t*>(vs + G * D);
    uint32_t bad = 0;

    // stage the G key and value rows (16-byte pieces; rows are 2*D bytes)
    {
        const int cpr = D / 8;
        for (int idx = threadIdx.x; idx < G * cpr; idx += blockDim.x) {
            const int i = idx / cpr, piece = idx % cpr;
            const int64_t t = t0 + i;
            const uint16_t* kr;
            const uint16_t* vr;
            if (t < s.n) {
                kr = reinterpret_cast<const uint16_t*>(s.ring_unit + (t % lo.C) * (int64_t)(4 * D));
                vr = kr + D;
            } else {
                const int64_t row = input_row(lo, s.n_new, s.bi, t - s.n, h);
                kr = reinterpret_cast<const uint16_t*>(s.k_new) + row;
                vr = reinterpret_cast<const uint16_t*>(s.v_new) + row;
            }
            reinterpret_cast<uint4*>(ks + i * D)[piece] = reinterpret_cast<const uint4*>(kr)[piece];
            reinterpret_cast<uint4*>(vs + i * D)[piece] = reinterpret_cast<const uint4*>(vr)[piece];
        }
    }
    __syncthreads();
    // keys: one thread per channel, statistics over the G tokens of the group
    if (lo.K == 0) {
        for (int c = threadIdx.x; c < D; c += blockDim.x) {
            float mn = bf16_bits_to_float(ks[c]), mx = mn;
            bad |= nonfinite(mn);
            for (int i = 1; i < G; ++i) {
                const float x = bf16_bits_to_float(ks[i * D + c]);
                bad |= nonfinite(x);
                mn = fminf(mn, x);
                mx = fmaxf(mx, x);
            }
            QbParams p = qb_params(mn, mx, flevels);
            kpar[c] = p.s;
            kpar[D + c] = p.z;
            for (int i = 0; i < G; ++i)
                codes[i * D + c] = static_cast<uint8_t>(qb_code(bf16_bits_to_float(ks[i * D + c]), p, levels));
        }
    } else {
        // dense-and-sparse ("KVQuant ...", "Summary"): the channel's K elements of largest
        // magnitude (bf16 pattern without its sign, as an integer; the lower token first on
        // equal magnitudes) go to the side list, entry e the e-th largest; the Q_b
        // parameters are fitted to the other G - K tokens and the outliers' codes are 0.
        // The channel's column of `codes` marks the chosen tokens (1) while selecting.
        uint32_t* kside = reinterpret_cast<uint32_t*>(rec + lo.kc + lo.vc + lo.kp + lo.vp);
        for (int c = threadIdx.x; c < D; c += blockDim.x) {
            for (int i = 0; i < G; ++i) codes[i * D + c] = 0;
            for (int e = 0; e < lo.K; ++e) {
                int best = -1;
                uint32_t bm = 0;
                for (int i = 0; i < G; ++i) {
                    if (codes[i * D + c]) continue;
                    const uint32_t m = ks[i * D + c] & 0x7fffu;
                    if (best < 0 || m > bm) {
                        best = i;
                        bm = m;
                    }
                }
                codes[best * D + c] = 1;
                kside[e * D + c] = (static_cast<uint32_t>(ks[best * D + c]) << 16) | static_cast<uint32_t>(best);
            }
            float mn = 0.0f, mx = 0.0f;
            bool first = true;      // min and max start at the first element kept
            for (int i = 0; i < G; ++i) {
                const float x = bf16_bits_to_float(ks[i * D + c]);
                bad |= nonfinite(x);
                if (codes[i * D + c]) continue;
                mn = first ? x : fminf(mn, x);
                mx = first ? x : fmaxf(mx, x);
                first = false;
            }
            QbParams p = qb_params(mn, mx, flevels);
            kpar[c] = p.s;
            kpar[D + c] = p.z;
            for (int i = 0; i < G; ++i)
                codes[i * D + c] = codes[i * D + c]
                                       ? 0
                                       : static_cast<uint8_t>(qb_code(bf16_bits_to_float(ks[i * D + c]), p, levels));
        }
    }
    __syncthreads();
    // pack token-major: code index i*D + c at bit (i*D + c)*bits, 16-byte stores
    {
        const int per16 = 128 / bits;  // codes per 16-byte chunk
        const int chunks = G * D / per16;
        for (int k = threadIdx.x; k < chunks; k += blockDim.x) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            const uint8_t* src = codes + k * per16;
            for (int e = 0; e < per16; ++e) w[(e * bits) >> 5] |= static_cast<uint32_t>(src[e]) << ((e * bits) & 31);
            reinterpret_cast<uint4*>(rec)[k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    __syncthreads();
    // values: one warp per token, each lane holds D/32 consecutive channels; a channel
    // group of Gv spans Gv / (D/32) lanes and its min/max is a shuffle reduction
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int cpl = D / 32;               // channels per lane
        const int lpg = Gv / cpl;             // lanes per value group
        for (int i = warp; i < G; i += blockDim.x / 32) {
            float x[8];
            const int gv = (lane * cpl) / Gv;
            // scale[gv][G] then zero[gv][G], tokens of a 16-token tile in the order 0, 8, 1, 9, ...
            const int tt = i % 16, pos = gv * G + (i - tt) + 2 * (tt % 8) + tt / 8;
            // dense-and-sparse: the group's K elements of largest magnitude leave the dense
            // part (bit e of `skip`: the lane's element e), chosen by K rounds of a shuffle
            // maximum over the group's lanes of (magnitude, lower channel first)
            uint32_t skip = 0;
            for (int r = 0; r < lo.K; ++r) {
                uint32_t key = 0;
                for (int e = 0; e < cpl; ++e) {
                    if (skip & (1u << e)) continue;
                    const uint32_t ch = (lane * cpl + e) % Gv;
                    const uint32_t k = ((static_cast<uint32_t>(vs[i * D + lane * cpl + e]) & 0x7fffu) << 16) |
                                       (0xffffu - ch);
                    key = k > key ? k : key;
                }
                uint32_t best = key;
                for (int off = 1; off < lpg; off <<= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, off));
                const int ch = static_cast<int>(0xffffu - (best & 0xffffu));
                const int owner = ch / cpl, e = ch % cpl;      // lane (within the group) and element
                if (lane % lpg == owner) {
                    skip |= 1u << e;
                    uint32_t* vside = reinterpret_cast<uint32_t*>(rec + lo.kc + lo.vc + lo.kp + lo.vp + lo.ko);
                    vside[r * lo.NGv * G + pos] =
                        (static_cast<uint32_t>(vs[i * D + lane * cpl + e]) << 16) | static_cast<uint32_t>(ch);
                }
            }
            float mn = INFINITY, mx = -INFINITY;
            for (int e = 0; e < cpl; ++e) {
                x[e] = bf16_bits_to_float(vs[i * D + lane * cpl + e]);
                bad |= nonfinite(x[e]);
                if (skip & (1u << e)) continue;
                mn = fminf(mn, x[e]);
                mx = fmaxf(mx, x[e]);
            }
            for (int off = 1; off < lpg; off <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            }
            QbParams p = qb_params(mn, mx, flevels);
            if ((lane % lpg) == 0) {
                vpar[pos] = p.s;
                vpar[G * lo.NGv + pos] = p.z;
            }
            // channel-major staging: code of (channel c, token i) at c*G + i
            for (int e = 0; e < cpl; ++e)
                codes[(lane * cpl + e) * G + i] =
                    (skip & (1u << e)) ? 0 : static_cast<uint8_t>(qb_code(x[e], p, levels));
        }
    }
    __syncthreads();
    // value codes: per 16-token tile, 32 lanes of wpl = D * bits / 64 words in the order
    // of the decode's value fragments.  Lane 4g + i, word w = 2 (j / hw) + s: its halves
    // hold tokens 2i + s and 2i + s + 8, and index j = 2q + r (channel 16q + g + 8r) sits at
    // bit bits * (j mod hw) of each half (hw = 16 / bits).  A lane's words go in slabs of
    // sw = min(wpl, 4) so that a warp reads one slab of a tile with one contiguous
    // 16-byte (or 8-byte) load per lane.
    {
        uint32_t* vrec = reinterpret_cast<uint32_t*>(rec + lo.kc);
        const int hw = 16 / bits, wpl = D * bits / 64, sw = wpl < 4 ? wpl : 4;
        const int words = (G / 16) * 32 * wpl;
        for (int k = threadIdx.x; k < words; k += blockDim.x) {
            const int tile = k / (32 * wpl), kk = k % (32 * wpl);
            const int slab = kk / (32 * sw), lane = (kk / sw) % 32;
            const int w = slab * sw + kk % sw;
            const int g = lane >> 2, i = lane & 3, sbit = w & 1;
            const int tlo = tile * 16 + 2 * i + sbit;          // token of the low half
            uint32_t word = 0u;
            for (int m = 0; m < hw; ++m) {
                const int j = (w >> 1) * hw + m;
                const int ch = 16 * (j >> 1) + g + 8 * (j & 1);
                const uint8_t* src = codes + ch * G;
                word |= static_cast<uint32_t>(src[tlo]) << (bits * m);
                word |= static_cast<uint32_t>(src[tlo + 8]) << (16 + bits * m);
            }
            vrec[k] = word;
        }
    }
    __syncthreads();
    return bad;
}

// Copy input row j (new token t = n + j) of (bi, h) into window slot t % C; one warp.
__device__ __forceinline__ uint32_t ring_write_row(const Layout& lo, uint8_t* cache, int l, int b,
                                                   int h, int64_t t, int64_t n, const void* k_new,
                                                   const void* v_new, int n_new, int bi, int lane) {
    const int D = lo.D;
    uint16_t* slot = reinterpret_cast<uint16_t*>(cache + lo.ring_off +
                                                 (unit_index(lo, l, b, h) * lo.C + t % lo.C) *
                                                     (int64_t)(4 * D));
    const int64_t src = input_row(lo, n_new, bi, t - n, h);
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(k_new) + src;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(v_new) + src;
    uint32_t bad = 0;
    // D/32 consecutive channels per lane (2 to 8 bf16 values): one vector load and store
    // each for keys and values; input rows are 16-byte aligned (16-byte aligned base, D a
    // multiple of 64)
    const int cpl = D / 32;
    for (int c = lane * cpl; c < D; c += 32 * cpl) {
        uint32_t kw[4] = {0u, 0u, 0u, 0u}, vw[4] = {0u, 0u, 0u, 0u};
        if (cpl == 8) {
            const uint4 k4 = *reinterpret_cast<const uint4*>(ks + c), v4 = *reinterpret_cast<const uint4*>(vs + c);
            kw[0] = k4.x; kw[1] = k4.y; kw[2] = k4.z; kw[3] = k4.w;
            vw[0] = v4.x; vw[1] = v4.y; vw[2] = v4.z; vw[3] = v4.w;
            *reinterpret_cast<uint4*>(slot + c) = k4;
            *reinterpret_cast<uint4*>(slot + D + c) = v4;
        } else if (cpl == 4) {
            const uint2 k2 = *reinterpret_cast<const uint2*>(ks + c), v2 = *reinterpret_cast<const uint2*>(vs + c);
            kw[0] = k2.x; kw[1] = k2.y; vw[0] = v2.x; vw[1] = v2.y;
            *reinterpret_cast<uint2*>(slot + c) = k2;
            *reinterpret_cast<uint2*>(slot + D + c) = v2;
        } else {
            kw[0] = *reinterpret_cast<const uint32_t*>(ks + c);
            vw[0] = *reinterpret_cast<const uint32_t*>(vs + c);
            *reinterpret_cast<uint32_t*>(slot + c) = kw[0];
            *reinterpret_cast<uint32_t*>(slot + D + c) = vw[0];
        }
        for (int e = 0; e < (cpl + 1) / 2; ++e) {
            bad |= nonfinite(__uint_as_float(kw[e] << 16)) | nonfinite(__uint_as_float(kw[e] & 0xffff0000u));
            bad |= nonfinite(__uint_as_float(vw[e] << 16)) | nonfinite(__uint_as_float(vw[e] & 0xffff0000u));
        }
    }
    return bad;
}

// INT8 / INT4 / FP8: quantise one token row of (l, b, h) at absolute position t; one warp.
__device__ __forceinline__ uint32_t quantise_row(const Layout& lo, uint8_t* cache, int l, int b,
                                                 int h, int64_t t, const void* src_k,
                                                 const void* src_v, int64_t row,
                                                 const float* fp8_scales, int lane) {
    const int D = lo.D;
    uint8_t* base = cache + lo.data_off + unit_index(lo, l, b, h) * lo.unit;
    uint32_t bad = 0;
    for (int kv = 0; kv < 2; ++kv) {
        const void* src = kv ? src_v : src_k;
        uint8_t* codes = base + (int64_t)kv * lo.T16 * D + t * D;
        if (lo.scheme == KVQ_SCHEME_INT8) {
            float x[8];
            const int cpl = (D + 31) / 32;
            float a = 0.0f;
            for (int e = 0; e < cpl; ++e) {
                int c = lane + 32 * e;
                x[e] = c < D ? load_input(src, row + c, lo.dtype) : 0.0f;
                bad |= nonfinite(x[e]);
                a = fmaxf(a, fabsf(x[e]));
            }
            for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
            float s = __fdiv_rn(a, 127.0f);
            for (int e = 0; e < cpl; ++e) {
                int c = lane + 32 * e;
                if (c >= D) continue;
                int code = 0;
                if (s != 0.0f) {
                    code = __float2int_rn(__fdiv_rn(x[e], s));
                    code = code < -127 ? -127 : (code > 127 ? 127 : code);
                }
                codes[c] = static_cast<uint8_t>(static_cast<int8_t>(code));
            }
            if (lane == 0)
                reinterpret_cast<float*>(base + 2 * (int64_t)lo.T16 * D)[(int64_t)kv * lo.T16 + t] = s;
        } else if (lo.scheme == KVQ_SCHEME_INT4) {
            // two channels per byte: lane takes channel pairs (2p, 2p + 1), p = lane + 32 e
            const int ppl = (D / 2 + 31) / 32;   // pairs per lane (1..4)
            float x[8];
            float a = 0.0f;
            for (int e = 0; e < ppl; ++e) {
                const int pr = lane + 32 * e;
                x[2 * e] = pr < D / 2 ? load_input(src, row + 2 * pr, lo.dtype) : 0.0f;
                x[2 * e + 1] = pr < D / 2 ? load_input(src, row + 2 * pr + 1, lo.dtype) : 0.0f;
                bad |= nonfinite(x[2 * e]) | nonfinite(x[2 * e + 1]);
                a = fmaxf(a, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
            }
            for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
            const float s = __fdiv_rn(a, 7.0f);
            uint8_t* codes4 = base + (int64_t)kv * lo.T16 * (D / 2) + t * (D / 2);
            for (int e = 0; e < ppl; ++e) {
                const int pr = lane + 32 * e;
                if (pr >= D / 2) continue;
                int c2[2] = {0, 0};
                if (s != 0.0f) {
                    for (int u = 0; u < 2; ++u) {
                        int code = __float2int_rn(__fdiv_rn(x[2 * e + u], s));
                        c2[u] = code < -7 ? -7 : (code > 7 ? 7 : code);
                    }
                }
                codes4[pr] = static_cast<uint8_t>((c2[0] & 15) | ((c2[1] & 15) << 4));
            }
            if (lane == 0)
                reinterpret_cast<float*>(base + (int64_t)lo.T16 * D)[(int64_t)kv * lo.T16 + t] = s;
        } else {
            // keys: channel r of 16-channel block kb at quarter (r mod 8) / 2 of the row,
            // byte 4 kb + 2 (r / 8) + (r mod 2) of it; values: tiles of 16 tokens stored
            // [channel][16], token tt at byte 4 ((tt mod 8) / 2) + 2 (tt mod 2) + tt / 8
            const float s = fp8_scales[2 * h + kv];
            const __nv_fp8_interpretation_t fmt = lo.scheme == KVQ_SCHEME_FP8_E4M3 ? __NV_E4M3 : __NV_E5M2;
            const int tt = static_cast<int>(t % 16);
            uint8_t* vtile = base + (int64_t)lo.T16 * D + (t - tt) * D + 4 * ((tt % 8) / 2) + 2 * (tt % 2) + tt / 8;
            uint8_t* krow = base + t * D;
            for (int c = lane; c < D; c += 32) {
                float x = load_input(src, row + c, lo.dtype);
                bad |= nonfinite(x);
                const uint8_t code = static_cast<uint8_t>(
                    __nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, fmt));
                const int r = c % 16;
                if (kv == 0)
                    krow[((r % 8) / 2) * (D / 4) + 4 * (c / 16) + 2 * (r / 8) + (r % 2)] = code;
                else
                    vtile[c * 16] = code;
            }
        }
    }
    return bad;
}

struct AppendArgs {
    Layout lo;
    uint8_t* cache;
    int layer, seq_begin, seq_count, n_new;
    const void* k_new;
    const void* v_new;
    const int32_t* n_valid;
    const float* fp8_scales;
    uint32_t flags;
};

__device__ __forceinline__ int new_tokens(const AppendArgs& a, int bi) {
    return a.n_valid ? a.n_valid[bi] : a.n_new;
}

// Small appends: one block per (kv head, sequence).  Each block flushes its head's full
// groups (reading the window) before writing its head's new window rows, so the reads
// and writes of the same slots are ordered by a block barrier.  Every block of a
// sequence reads the old token counts first; the last block of the sequence to finish
// (an arrival counter in the sequence's state entry, zero at rest) writes the new ones.
__global__ void __launch_bounds__(kThreads) k_append_small(AppendArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const Layout& lo = a.lo;
    const int h = blockIdx.x, bi = blockIdx.y, b = a.seq_begin + bi;
    if (lo.scheme == KVQ_SCHEME_KIVI && (threadIdx.x >> 5) < a.n_new) {
        // the new rows' addresses do not depend on the cache state: start bringing them
        // into L2 (a hint only; nothing is read before the wait below)
        const int64_t row = input_row(lo, a.n_new, bi, threadIdx.x >> 5, h) + (threadIdx.x & 31) * (lo.D / 32);
        prefetch_l2(reinterpret_cast<const uint16_t*>(a.k_new) + row);
        prefetch_l2(reinterpret_cast<const uint16_t*>(a.v_new) + row);
    }
    // launched as a dependent of the stream's previous kernel: everything it wrote (the
    // inputs, the cache) is visible after this wait, and nothing is read before it
    grid_dependency_wait();
    grid_launch_dependents();   // a decode launched next may start launching (it waits for us)
    int32_t* st = state_ptr(lo, a.cache, a.layer, b);
    const int n = st[0], qn = st[1];
    uint32_t status = 0;
    int m = new_tokens(a, bi);
    m = m < 0 ? 0 : (m > a.n_new ? a.n_new : m);
    if (tokens_taken(lo, b, n, qn, m, a.flags, &status) < 0) {
        if (threadIdx.x == 0 && h == 0) atomicOr(reinterpret_cast<uint32_t*>(a.cache), status);
        return;
    }
    uint32_t bad = 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    int qn2 = n + m;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        qn2 = qn_after(lo, n, qn, m, a.flags);
        TokenSource s;
        s.ring_unit = a.cache + lo.ring_off + unit_index(lo, a.layer, b, h) * lo.C * (int64_t)(4 * lo.D);
        s.k_new = a.k_new;
        s.v_new = a.v_new;
        s.n = n;
        s.n_new = a.n_new;
        s.bi = bi;
        for (int64_t t0 = qn; t0 < qn2; t0 += lo.G)
            bad |= quantise_group(lo, a.cache, a.layer, b, h, t0, s, smem);
        __syncthreads();
        const int64_t first = n > qn2 ? n : qn2;
        for (int64_t t = first + warp; t < (int64_t)n + m; t += nwarps)
            bad |= ring_write_row(lo, a.cache, a.layer, b, h, t, n, a.k_new, a.v_new, a.n_new, bi, lane);
    } else {
        if (is_fp8(lo.scheme) && bi == 0 && h == 0)
            for (int i = threadIdx.x; i < 2 * lo.H; i += blockDim.x)
                reinterpret_cast<float*>(a.cache + lo.scales_off)[(int64_t)a.layer * lo.H * 2 + i] = a.fp8_scales[i];
        for (int j = warp; j < m; j += nwarps)
            bad |= quantise_row(lo, a.cache, a.layer, b, h, (int64_t)n + j, a.k_new, a.v_new,
                                input_row(lo, a.n_new, bi, j, h), a.fp8_scales, lane);
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (bad) atomicOr(reinterpret_cast<uint32_t*>(a.cache), KVQ_STATUS_NONFINITE);
        // every block has used its reads of the old counts before it arrives here (its
        // control flow depends on them); the rows it wrote are for later kernels, which see
        // them at this kernel's end, so no fence is needed before the arrival
        if (atomicAdd(&st[2], 1) == lo.H - 1) {
            st[0] = n + m;
            st[1] = qn2;
            st[2] = 0;
        }
    }
}

// Bulk appends, step 1 (KIVI): one block per (group to quantise, kv head, sequence).
__global__ void __launch_bounds__(kThreads) k_append_groups(AppendArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const Layout& lo = a.lo;
    const int bi = blockIdx.z, b = a.seq_begin + bi, h = blockIdx.y;
    const int32_t* st = state_ptr(lo, a.cache, a.layer, b);
    const int n = st[0], qn = st[1];
    uint32_t dummy = 0;
    int m = new_tokens(a, bi);
    m = m < 0 ? 0 : (m > a.n_new ? a.n_new : m);
    if (tokens_taken(lo, b, n, qn, m, a.flags, &dummy) < 0) return;
    const int qn2 = qn_after(lo, n, qn, m, a.flags);
    const int64_t t0 = qn + (int64_t)blockIdx.x * lo.G;
    if (t0 >= qn2) return;
    TokenSource s;
    s.ring_unit = a.cache + lo.ring_off + unit_index(lo, a.layer, b, h) * lo.C * (int64_t)(4 * lo.D);
    s.k_new = a.k_new;
    s.v_new = a.v_new;
    s.n = n;
    s.n_new = a.n_new;
    s.bi = bi;
    uint32_t bad = quantise_group(lo, a.cache, a.layer, b, h, t0, s, smem);
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0 && bad) atomicOr(reinterpret_cast<uint32_t*>(a.cache), KVQ_STATUS_NONFINITE);
}

// Bulk appends, step 2: rows that do not become part of a group -- window rows (KIVI)
// or quantised rows (INT8, FP8).  One warp per (row, kv head); grid (row blocks, seq).
__global__ void __launch_bounds__(kThreads) k_append_rows(AppendArgs a) {
    const Layout& lo = a.lo;
    const int bi = blockIdx.y, b = a.seq_begin + bi;
    const int32_t* st = state_ptr(lo, a.cache, a.layer, b);
    const int n = st[0], qn = st[1];
    uint32_t dummy = 0;
    int m = new_tokens(a, bi);
    m = m < 0 ? 0 : (m > a.n_new ? a.n_new : m);
    if (tokens_taken(lo, b, n, qn, m, a.flags, &dummy) < 0) return;
    const int lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    uint32_t bad = 0;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        const int qn2 = qn_after(lo, n, qn, m, a.flags);
        const int64_t first = n > qn2 ? n : qn2;
        const int64_t rows = (int64_t)n + m - first;
        if (r < rows * lo.H) {
            const int h = static_cast<int>(r % lo.H);
            bad = ring_write_row(lo, a.cache, a.layer, b, h, first + r / lo.H, n, a.k_new, a.v_new,
                                 a.n_new, bi, lane);
        }
    } else if (r < (int64_t)m * lo.H) {
        const int h = static_cast<int>(r % lo.H);
        const int64_t j = r / lo.H;
        bad = quantise_row(lo, a.cache, a.layer, b, h, n + j, a.k_new, a.v_new,
                           input_row(lo, a.n_new, bi, j, h), a.fp8_scales, lane);
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0 && bad) atomicOr(reinterpret_cast<uint32_t*>(a.cache), KVQ_STATUS_NONFINITE);
}

// Bulk appends, step 3: new per-sequence counts and status bits (and the FP8 scale table).
__global__ void k_append_commit(AppendArgs a) {
    const Layout& lo = a.lo;
    if (is_fp8(lo.scheme) && blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * lo.H; i += blockDim.x)
            reinterpret_cast<float*>(a.cache + lo.scales_off)[(int64_t)a.layer * lo.H * 2 + i] = a.fp8_scales[i];
    const int bi = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t status = 0;
    if (bi < a.seq_count) {
        const int b = a.seq_begin + bi;
        int32_t* st = state_ptr(lo, a.cache, a.layer, b);
        const int n = st[0], qn = st[1];
        int m = new_tokens(a, bi);
        m = m < 0 ? 0 : (m > a.n_new ? a.n_new : m);
        if (tokens_taken(lo, b, n, qn, m, a.flags, &status) >= 0) {
            st[1] = qn_after(lo, n, qn, m, a.flags);
            st[0] = n + m;
        }
    }
    if (status) atomicOr(reinterpret_cast<uint32_t*>(a.cache), status);
}

// Explicit flush (KIVI): one block per (group index, kv head, sequence) quantises window
// groups [qn + g*G, ...) while n - qn >= R + G; a second kernel commits qn.
__global__ void __launch_bounds__(kThreads) k_flush_groups(Layout lo, uint8_t* cache, int layer) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int b = blockIdx.z, h = blockIdx.y;
    const int32_t* st = state_ptr(lo, cache, layer, b);
    const int n = st[0], qn = st[1];
    const int ready = (n - qn - lo.R) >= lo.G ? (n - qn - lo.R) / lo.G : 0;
    if (static_cast<int>(blockIdx.x) >= ready) return;
    if (!pages_ok(lo, b, qn / lo.G, qn / lo.G + ready)) return;   // k_flush_commit reports it
    TokenSource s;
    s.ring_unit = cache + lo.ring_off + unit_index(lo, layer, b, h) * lo.C * (int64_t)(4 * lo.D);
    s.k_new = nullptr;
    s.v_new = nullptr;
    s.n = n;
    s.n_new = 0;
    s.bi = 0;
    uint32_t bad = quantise_group(lo, cache, layer, b, h, qn + (int64_t)blockIdx.x * lo.G, s, smem);
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0 && bad) atomicOr(reinterpret_cast<uint32_t*>(cache), KVQ_STATUS_NONFINITE);
}

__global__ void k_flush_commit(Layout lo, uint8_t* cache, int layer) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= lo.B) return;
    int32_t* st = state_ptr(lo, cache, layer, b);
    const int n = st[0], qn = st[1];
    const int ready = (n - qn - lo.R) >= lo.G ? (n - qn - lo.R) / lo.G : 0;
    if (!pages_ok(lo, b, qn / lo.G, qn / lo.G + ready)) {   // the window stays as it is
        atomicOr(reinterpret_cast<uint32_t*>(cache), KVQ_STATUS_BAD_PAGE);
        return;
    }
    st[1] = qn + ready * lo.G;
}

}  // namespace

static size_t group_smem(const Layout& lo) {
    return lo.scheme == KVQ_SCHEME_KIVI ? static_cast<size_t>(5) * lo.G * lo.D : 0;
}

static int set_smem(const void* fn, size_t bytes) {
    if (bytes > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
            cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int launch_append(const Layout& lo, uint8_t* cache, int layer, int seq_begin, int seq_count,
                  const void* k_new, const void* v_new, int n_new, const int32_t* n_valid,
                  const float* fp8_scales, uint32_t flags, cudaStream_t stream) {
    if (seq_count == 0) return KVQ_OK;
    AppendArgs a;
    a.lo = lo;
    a.cache = cache;
    a.layer = layer;
    a.seq_begin = seq_begin;
    a.seq_count = seq_count;
    a.n_new = n_new;
    a.k_new = k_new;
    a.v_new = v_new;
    a.n_valid = n_valid;
    a.fp8_scales = fp8_scales;
    a.flags = flags;
    const size_t smem = group_smem(lo);
    if (n_new <= kSmallAppend) {
        if (set_smem(reinterpret_cast<const void*>(k_append_small), smem)) return KVQ_ERR_CUDA;
        return launch_dependent(k_append_small, dim3(lo.H, seq_count), kThreads, smem, stream, a) == cudaSuccess
                   ? KVQ_OK
                   : KVQ_ERR_CUDA;
    }
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        // at most (window - 1 + n_new) / G groups leave the window in one append
        const int64_t max_groups = ((int64_t)lo.C - 1 + n_new) / lo.G;
        if (max_groups > 0) {
            if (set_smem(reinterpret_cast<const void*>(k_append_groups), smem)) return KVQ_ERR_CUDA;
            dim3 grid(static_cast<unsigned>(max_groups), lo.H, seq_count);
            k_append_groups<<<grid, kThreads, smem, stream>>>(a);
        }
        const int64_t rows = (int64_t)(n_new < lo.C ? n_new : lo.C) * lo.H;
        dim3 grid2(static_cast<unsigned>((rows + 3) / 4), seq_count);
        k_append_rows<<<grid2, kThreads, 0, stream>>>(a);
    } else {
        const int64_t rows = (int64_t)n_new * lo.H;
        dim3 grid2(static_cast<unsigned>((rows + 3) / 4), seq_count);
        k_append_rows<<<grid2, kThreads, 0, stream>>>(a);
    }
    k_append_commit<<<(seq_count + 127) / 128, 128, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int launch_flush(const Layout& lo, uint8_t* cache, int layer, cudaStream_t stream) {
    if (lo.scheme != KVQ_SCHEME_KIVI) return KVQ_OK;
    // the window never holds more than R + G tokens, so at most one group per sequence
    // and kv head is ready
    const int max_groups = 1;
    const size_t smem = group_smem(lo);
    if (set_smem(reinterpret_cast<const void*>(k_flush_groups), smem)) return KVQ_ERR_CUDA;
    dim3 grid(max_groups, lo.H, lo.B);
    k_flush_groups<<<grid, kThreads, smem, stream>>>(lo, cache, layer);
    k_flush_commit<<<(lo.B + 127) / 128, 128, 0, stream>>>(lo, cache, layer);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq
