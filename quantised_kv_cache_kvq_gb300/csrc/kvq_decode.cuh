// kvq_decode.cuh -- single-query decode attention over the packed cache (kernel templates,
// instantiated by the kvq_decode_*.cu translation units).
//
// What is computed ("Quantizing the KV cache", "Why values per token"): for every query
// head, o = sum_t p_t * Vhat_t with p = softmax_t(softmax_scale * q . Khat_t) over all
// cached tokens of the sequence; query head hq reads KV head hq / gqa.
//
// Work split: a block handles one (sequence, kv head, chunk of tokens) item and leaves
// the chunk's partial softmax (m, l, o[D]) for all gqa query heads of the kv head, so
// every cache byte is read once per step.  k_merge combines the chunks by log-sum-exp.
//
// Packed KIVI chunks (runs of group records) are staged into shared memory by one bulk
// asynchronous copy, then both contractions run on the tensor cores with operands built
// in registers:
//   scores  S[token][col] = sum_c code[token][c] * Bq[c][col], A = 2/4/8-bit key codes
//           turned into exact fp16 integers, Bq = (query * per-channel key scale) split
//           into an fp16 major part and an fp16 minor part (cols 2h, 2h+1), so the fp32
//           accumulator sees the product to ~22 bits; the per-group offset term
//           sum_c q_c * zero_c is added in fp32.  (Q_b equation: xhat = code*s + min.)
//   values  O[c][col] = sum_t code[t][c] * Bp[t][col], A = value codes (stored
//           channel-major so one 32-bit word holds a channel's consecutive tokens),
//           Bp = p_t * value scale split into major/minor parts; the offset term
//           sum_t p_t * zero_t is added in fp32.
// The bf16 window (KIVI), INT8 rows and FP8 rows go through a CUDA-core row path.
#pragma once

#include <cuda_fp8.h>

#include "kvq_internal.cuh"
#include "kvq_launch.h"

namespace kvq {

constexpr int kDecodeThreads = 128;

struct DecodeArgs {
    Layout lo;
    DecodePlan plan;
    const uint8_t* cache;
    int layer;
    const void* q;
    float qscale;  // softmax_scale * log2(e): scores live in the base-2 domain
    float* out;
    uint8_t* ws;
};

struct ItemRange {
    int64_t t0, t1;
};

// Token range of work item `item` of a unit with n cached tokens, qn of them packed.
__host__ __device__ inline ItemRange item_range(const Layout& lo, const DecodePlan& p, int item,
                                                int64_t n, int64_t qn) {
    ItemRange r;
    if (item < p.NRC) {
        const int64_t base = lo.scheme == KVQ_SCHEME_KIVI ? qn : 0;
        r.t0 = base + (int64_t)item * p.CHR;
        r.t1 = r.t0 + p.CHR < n ? r.t0 + p.CHR : n;
    } else {
        r.t0 = (int64_t)(item - p.NRC) * p.CH;
        r.t1 = r.t0 + p.CH < qn ? r.t0 + p.CH : qn;
    }
    return r;
}

__device__ __forceinline__ float load_q(const void* q, int64_t idx, int dtype) {
    if (dtype == KVQ_DTYPE_BF16) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(q)[idx]);
    return reinterpret_cast<const float*>(q)[idx];
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Issue bulk copies of `bytes` bytes (a multiple of 16) in pieces of at most 32 KiB.
__device__ __forceinline__ void bulk_copy_pieces(uint8_t* dst, const uint8_t* src, uint32_t bytes,
                                                 uint64_t* bar) {
    for (uint32_t off = 0; off < bytes; off += 32768u) {
        const uint32_t len = bytes - off < 32768u ? bytes - off : 32768u;
        bulk_copy_g2s(dst + off, src + off, len, bar);
    }
}

// All threads wait for the staged bytes; on a timeout the decode status gets
// KVQ_STATUS_TIMEOUT, the block waits once more (bounded) for its copies and returns false.
__device__ __forceinline__ bool wait_staged(uint64_t* bar, uint8_t* ws) {
    bool ok = mbar_wait_bounded(bar, 0, kWaitLimit);
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(reinterpret_cast<uint32_t*>(ws), KVQ_STATUS_TIMEOUT);
        mbar_wait_bounded(bar, 0, kWaitLimit);
        __syncthreads();
    }
    return ok;
}

// Partial-result slots of the workspace.
__device__ __forceinline__ int64_t slot_index(const DecodeArgs& a, int b, int h, int item, int head) {
    return (((int64_t)b * a.lo.H + h) * a.plan.S + item) * a.lo.gqa + head;
}

// Scaled query of the block's kv head into shared fp32 qs[gqa][D].
__device__ __forceinline__ void load_query(const DecodeArgs& a, int b, int h, float* qs) {
    const Layout& lo = a.lo;
    const int64_t base = ((int64_t)b * lo.Hq + (int64_t)h * lo.gqa) * lo.D;
    for (int i = threadIdx.x; i < lo.gqa * lo.D; i += blockDim.x)
        qs[i] = load_q(a.q, base + i, lo.dtype) * a.qscale;
}

// Softmax over the chunk: per-head max (from per-warp maxima in red[warp][head]), then
// p = 2^(s - max) in place and l = sum p.  Leaves max and l in hstat[0..31], [32..63].
__device__ __forceinline__ void chunk_softmax(const Layout& lo, float* sc, int ntok, int sc_stride,
                                              float* red, float* hstat) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < lo.gqa) {
        float m = -INFINITY;
        for (int w = 0; w < 4; ++w) m = fmaxf(m, red[w * 32 + tid]);
        hstat[tid] = m;
    }
    __syncthreads();
    for (int hh = 0; hh < lo.gqa; ++hh) {
        const float m = hstat[hh];
        float part = 0.0f;
        for (int t = tid; t < ntok; t += blockDim.x) {
            const float p = exp2f(sc[hh * sc_stride + t] - m);
            sc[hh * sc_stride + t] = p;
            part += p;
        }
        part = warp_sum(part);
        if (lane == 0) red[warp * 32 + hh] = part;
    }
    __syncthreads();
    if (tid < lo.gqa) {
        float l = 0.0f;
        for (int w = 0; w < 4; ++w) l += red[w * 32 + tid];
        hstat[32 + tid] = l;
    }
    __syncthreads();
}

// ------------------------------------------------------------------------ row path
// Tokens held as whole rows: the bf16 window of a KIVI cache, or INT8 / FP8 rows.
template <int D>
__device__ void rows_item(const DecodeArgs& a, uint8_t* smem, const SmemOffsets& so, int b, int h,
                          int item, int64_t t0, int64_t t1) {
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cnt = static_cast<int>(t1 - t0);
    const int CHR = a.plan.CHR;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* hstat = reinterpret_cast<float*>(smem + so.hstat);
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    float* sc = reinterpret_cast<float*>(smem + so.sc);
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);

    if (tid == 0) mbar_init(bar, 1);
    __syncthreads();
    if (tid == 0) {
        if (lo.scheme == KVQ_SCHEME_KIVI) {
            const uint8_t* ring = a.cache + lo.ring_off + u * lo.C * (int64_t)(4 * D);
            const int s0 = static_cast<int>(t0 % lo.C);
            const int first = cnt < lo.C - s0 ? cnt : lo.C - s0;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt) * 4 * D);
            bulk_copy_pieces(data, ring + (int64_t)s0 * 4 * D, static_cast<uint32_t>(first) * 4 * D, bar);
            if (cnt > first)
                bulk_copy_pieces(data + (int64_t)first * 4 * D, ring, static_cast<uint32_t>(cnt - first) * 4 * D, bar);
        } else {
            const uint8_t* unit = a.cache + lo.data_off + u * lo.unit;
            const uint32_t cb = static_cast<uint32_t>(cnt) * D;
            if (lo.scheme == KVQ_SCHEME_INT8) {
                const uint32_t sb = static_cast<uint32_t>((cnt + 3) / 4 * 4) * 4;
                mbar_arrive_expect_tx(bar, 2 * cb + 2 * sb);
                bulk_copy_pieces(data, unit + t0 * D, cb, bar);
                bulk_copy_pieces(data + (int64_t)CHR * D, unit + (int64_t)lo.T16 * D + t0 * D, cb, bar);
                const uint8_t* scales = unit + 2 * (int64_t)lo.T16 * D;
                bulk_copy_pieces(data + 2 * (int64_t)CHR * D, scales + 4 * t0, sb, bar);
                bulk_copy_pieces(data + 2 * (int64_t)CHR * D + 4 * CHR, scales + 4 * (int64_t)lo.T16 + 4 * t0, sb, bar);
            } else {
                mbar_arrive_expect_tx(bar, 2 * cb);
                bulk_copy_pieces(data, unit + t0 * D, cb, bar);
                bulk_copy_pieces(data + (int64_t)CHR * D, unit + (int64_t)lo.T16 * D + t0 * D, cb, bar);
            }
        }
    }
    load_query(a, b, h, qs);
    float kscale = 1.0f, vscale = 1.0f;
    if (lo.scheme == KVQ_SCHEME_FP8_E4M3) {
        const float* tab = reinterpret_cast<const float*>(a.cache + lo.scales_off) + ((int64_t)a.layer * lo.H + h) * 2;
        kscale = tab[0];
        vscale = tab[1];
    }
    if (!wait_staged(bar, a.ws)) return;

    auto kval = [&](int i, int c) -> float {
        if (lo.scheme == KVQ_SCHEME_KIVI)
            return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D)[c]);
        if (lo.scheme == KVQ_SCHEME_INT8)
            return static_cast<float>(reinterpret_cast<const int8_t*>(data)[i * D + c]) *
                   reinterpret_cast<const float*>(data + 2 * (int64_t)CHR * D)[i];
        const __half_raw hr = __nv_cvt_fp8_to_halfraw(data[i * D + c], __NV_E4M3);
        return __half2float(__half(hr)) * kscale;
    };
    auto vval = [&](int i, int c) -> float {
        if (lo.scheme == KVQ_SCHEME_KIVI)
            return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D + 2 * D)[c]);
        if (lo.scheme == KVQ_SCHEME_INT8)
            return static_cast<float>(reinterpret_cast<const int8_t*>(data + (int64_t)CHR * D)[i * D + c]) *
                   reinterpret_cast<const float*>(data + 2 * (int64_t)CHR * D + 4 * CHR)[i];
        const __half_raw hr = __nv_cvt_fp8_to_halfraw(data[(int64_t)CHR * D + i * D + c], __NV_E4M3);
        return __half2float(__half(hr)) * vscale;
    };

    // scores: a warp per token, lanes over channels, one reduction per head
    constexpr int CPL = (D + 31) / 32;
    float hmax[8];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) hmax[hh] = -INFINITY;
    for (int i = warp; i < cnt; i += 4) {
        float kv[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) kv[j] = kval(i, lane + 32 * j);
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            if (hh >= lo.gqa) break;
            float acc = 0.0f;
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc = fmaf(qs[hh * D + lane + 32 * j], kv[j], acc);
            acc = warp_sum(acc);
            if (lane == 0) sc[hh * CHR + i] = acc;
            hmax[hh] = fmaxf(hmax[hh], acc);
        }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh)
        if (lane == 0 && hh < lo.gqa) red[warp * 32 + hh] = hmax[hh];
    __syncthreads();
    chunk_softmax(lo, sc, cnt, CHR, red, hstat);

    // values: a thread per channel
    for (int c = tid; c < D; c += blockDim.x) {
        float o[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) o[hh] = 0.0f;
        for (int i = 0; i < cnt; ++i) {
            const float v = vval(i, c);
#pragma unroll
            for (int hh = 0; hh < 8; ++hh)
                if (hh < lo.gqa) o[hh] = fmaf(sc[hh * CHR + i], v, o[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
            if (hh < lo.gqa)
                reinterpret_cast<float*>(a.ws + a.plan.ws_o_off)[slot_index(a, b, h, item, hh) * D + c] = o[hh];
    }
    if (tid < lo.gqa) {
        float* ml = reinterpret_cast<float*>(a.ws + a.plan.ws_ml_off) + 2 * slot_index(a, b, h, item, tid);
        ml[0] = hstat[tid];
        ml[1] = hstat[32 + tid];
    }
}

// ------------------------------------------------------------------------ packed path
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&w)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(p + 4 * i);
            w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
        }
    } else if constexpr (N == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = reinterpret_cast<const uint32_t*>(p)[i];
    }
}

// Two codes of a 32-bit word (the one at bit `shift` and the one 16 bits above it) as an
// exact fp16 pair: OR the code into the mantissa of 1024.0 and subtract 1024.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int shift) {
    constexpr uint32_t mask = ((1u << BITS) - 1u) * 0x00010001u;
    const uint32_t x = ((w >> shift) & mask) | 0x64006400u;
    return h2_as_u32(__hsub2(u32_as_h2(x), __half2(__half(1024.0f), __half(1024.0f))));
}

template <int D, int BITS, int NT>
__device__ void packed_item(const DecodeArgs& a, uint8_t* smem, const SmemOffsets& so, int b, int h,
                            int item, int64_t t0, int64_t t1) {
    constexpr int CPW = 32 / BITS;         // key channels per 32-bit word
    constexpr int HPW = CPW / 2;           // code pairs per word
    constexpr int NPAIR = D / 8;           // code pairs per thread per token row
    constexpr int KSTEPS = D / 16;
    constexpr int ROWW = D * BITS / 128;   // words per thread per token row
    constexpr int MT = D / 64;             // 16-channel tiles per warp in the value pass
    constexpr int TPW = 32 / BITS;         // value tokens per word
    constexpr int HW = TPW / 2;
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
    const int G = lo.G, CH = a.plan.CH;
    const int ntok = static_cast<int>(t1 - t0);
    const int gqa = lo.gqa;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* hstat = reinterpret_cast<float*>(smem + so.hstat);
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    uint32_t* qpa = reinterpret_cast<uint32_t*>(smem + so.qpa);
    uint32_t* qpb = reinterpret_cast<uint32_t*>(smem + so.qpb);
    float* sc = reinterpret_cast<float*>(smem + so.sc);
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);

    if (tid == 0) mbar_init(bar, 1);
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = static_cast<uint32_t>(ntok / G) * lo.rec;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_copy_pieces(data, a.cache + lo.data_off + u * lo.unit + (t0 / G) * (int64_t)lo.rec, bytes, bar);
    }
    // query prep while the copy is in flight: scaled query, a power-of-two prescale that
    // brings max|q| into [0.5, 1) (so fp16 products cannot overflow), and the query in
    // the thread-pair order of the key fragments as fp16 major + minor parts
    load_query(a, b, h, qs);
    __syncthreads();
    float qmax = 0.0f;
    for (int i = tid; i < gqa * D; i += blockDim.x) qmax = fmaxf(qmax, fabsf(qs[i]));
    qmax = warp_max(qmax);
    if (lane == 0) red[warp * 32] = qmax;
    __syncthreads();
    qmax = fmaxf(fmaxf(red[0], red[32]), fmaxf(red[64], red[96]));
    int qexp = 0;
    if (qmax > 0.0f) frexpf(qmax, &qexp);
    const float qdown = ldexpf(1.0f, -qexp), qup = ldexpf(1.0f, qexp);
    for (int i = tid; i < 4 * NT * 4 * NPAIR; i += blockDim.x) {
        const int m = i % NPAIR, tg = (i / NPAIR) % 4, hh = i / (NPAIR * 4);
        const int wi = m / HPW, j = m % HPW;
        const int clo = tg * (D / 4) + wi * CPW + j, chi = clo + HPW;
        float vlo = 0.0f, vhi = 0.0f;
        if (hh < gqa) {
            vlo = qs[hh * D + clo] * qdown;
            vhi = qs[hh * D + chi] * qdown;
        }
        const __half2 major = __floats2half2_rn(vlo, vhi);
        const float2 mf = __half22float2(major);
        const __half2 minor = __floats2half2_rn(vlo - mf.x, vhi - mf.y);
        qpa[i] = h2_as_u32(major);
        qpb[i] = h2_as_u32(minor);
    }
    __syncthreads();
    if (!wait_staged(bar, a.ws)) return;

    // ---------------- scores
    const int kc_bytes = lo.kc, vc_bytes = lo.vc;
    const int rowbytes = D * BITS / 8;
    const int tiles_per_warp = CH / 64;
    const int tile_lo = warp * tiles_per_warp;
    int tile_hi = tile_lo + tiles_per_warp;
    if (tile_hi > ntok / 16) tile_hi = ntok / 16;
    uint32_t bq[NT][NPAIR];
    float cst[NT];
    float hmax[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) hmax[nt] = -INFINITY;
    int cur = -1;
    for (int mt = tile_lo; mt < tile_hi; ++mt) {
        const int tok0 = mt * 16, grp = tok0 / G;
        const uint8_t* rec = data + (int64_t)grp * lo.rec;
        if (grp != cur) {
            cur = grp;
            const __half* sK = reinterpret_cast<const __half*>(rec + kc_bytes + vc_bytes);
            const __half* zK = sK + D;
            uint32_t sreg[D / 8];
            load_words<D / 8>(reinterpret_cast<const uint8_t*>(sK + tig * (D / 4)), sreg);
            const int part = g & 1;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hh = 4 * nt + (g >> 1);
                const uint32_t* pa = qpa + (hh * 4 + tig) * NPAIR;
                const uint32_t* pb = qpb + (hh * 4 + tig) * NPAIR;
#pragma unroll
                for (int m = 0; m < NPAIR; ++m) {
                    const int wi = m / HPW, j = m % HPW;
                    const int lo_l = wi * CPW + j, hi_l = lo_l + HPW;
                    const __half2 s2 = u32_as_h2(prmt(sreg[lo_l / 2], sreg[hi_l / 2], (j & 1) ? 0x7632u : 0x5410u));
                    const __half2 qa = u32_as_h2(pa[m]), qb = u32_as_h2(pb[m]);
                    const __half2 major = __hmul2(s2, qa);
                    __half2 minor = __hfma2(s2, qa, __hneg2(major));
                    minor = __hfma2(s2, qb, minor);
                    bq[nt][m] = part ? h2_as_u32(minor) : h2_as_u32(major);
                }
                // offset term sum_c qs[hh][c] * zero[c]; the two threads of a (major, minor)
                // pair split the thread's channel block in halves
                float zsum = 0.0f;
                if (hh < gqa) {
                    const int c0 = tig * (D / 4) + part * (D / 8);
#pragma unroll 8
                    for (int c = 0; c < D / 8; ++c) zsum = fmaf(qs[hh * D + c0 + c], __half2float(zK[c0 + c]), zsum);
                }
                zsum += __shfl_xor_sync(0xffffffffu, zsum, 4);
                zsum += __shfl_xor_sync(0xffffffffu, zsum, 1);
                zsum += __shfl_xor_sync(0xffffffffu, zsum, 2);
                cst[nt] = __shfl_sync(0xffffffffu, zsum, 8 * tig);
            }
        }
        uint32_t wa[ROWW], wb[ROWW];
        const int ti = tok0 % G + g;
        load_words<ROWW>(rec + ti * rowbytes + tig * (ROWW * 4), wa);
        load_words<ROWW>(rec + (ti + 8) * rowbytes + tig * (ROWW * 4), wb);
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const int m0 = 2 * ks, m1 = 2 * ks + 1;
            uint32_t af[4];
            af[0] = code_pair<BITS>(wa[m0 / HPW], BITS * (m0 % HPW));
            af[1] = code_pair<BITS>(wb[m0 / HPW], BITS * (m0 % HPW));
            af[2] = code_pair<BITS>(wa[m1 / HPW], BITS * (m1 % HPW));
            af[3] = code_pair<BITS>(wb[m1 / HPW], BITS * (m1 % HPW));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(acc[nt], af, bq[nt][m0], bq[nt][m1]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = 4 * nt + tig;
            if (head < gqa) {
                const float s0 = fmaf(acc[nt][0] + acc[nt][1], qup, cst[nt]);
                const float s1 = fmaf(acc[nt][2] + acc[nt][3], qup, cst[nt]);
                sc[head * CH + tok0 + g] = s0;
                sc[head * CH + tok0 + g + 8] = s1;
                hmax[nt] = fmaxf(hmax[nt], fmaxf(s0, s1));
            }
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float m = hmax[nt];
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (g == 0) red[warp * 32 + 4 * nt + tig] = m;
    }
    __syncthreads();
    chunk_softmax(lo, sc, ntok, CH, red, hstat);

    // ---------------- values
    const int wi = (2 * tig) / HW, j0 = (2 * tig) % HW;
    const int tA = wi * TPW + j0, tB = tA + HW, tC = tA + 1, tD = tB + 1;
    const int cw0 = warp * (D / 4);
    float oacc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.0f;
    const int part = g & 1;
    for (int ks = 0; ks < ntok / 16; ++ks) {
        const int tokbase = ks * 16, grp = tokbase / G, tb = tokbase % G;
        const uint8_t* rec = data + (int64_t)grp * lo.rec;
        const uint32_t* vcw = reinterpret_cast<const uint32_t*>(rec + kc_bytes);
        const __half* sV = reinterpret_cast<const __half*>(rec + kc_bytes + vc_bytes + lo.kp);
        // p of this thread's four tokens, split into fp16 major + minor parts
        __half2 pa01[NT], pb01[NT], pa23[NT], pb23[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hp = 4 * nt + (g >> 1);
            float p0 = 0.0f, p1 = 0.0f, p2 = 0.0f, p3 = 0.0f;
            if (hp < gqa) {
                const float* ps = sc + hp * CH + tokbase;
                p0 = ps[tA]; p1 = ps[tB]; p2 = ps[tC]; p3 = ps[tD];
            }
            pa01[nt] = __floats2half2_rn(p0, p1);
            pa23[nt] = __floats2half2_rn(p2, p3);
            const float2 f01 = __half22float2(pa01[nt]), f23 = __half22float2(pa23[nt]);
            pb01[nt] = __floats2half2_rn(p0 - f01.x, p1 - f01.y);
            pb23[nt] = __floats2half2_rn(p2 - f23.x, p3 - f23.y);
        }
        uint32_t bp[NT][2];
        int gv_cur = -1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int c0 = cw0 + mt * 16 + g;
            const int gv = (cw0 + mt * 16) / lo.Gv;
            if (gv != gv_cur) {
                gv_cur = gv;
                const __half2 s01 = __halves2half2(sV[(tb + tA) * lo.NGv + gv], sV[(tb + tB) * lo.NGv + gv]);
                const __half2 s23 = __halves2half2(sV[(tb + tC) * lo.NGv + gv], sV[(tb + tD) * lo.NGv + gv]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const __half2 M01 = __hmul2(s01, pa01[nt]);
                    __half2 m01 = __hfma2(s01, pa01[nt], __hneg2(M01));
                    m01 = __hfma2(s01, pb01[nt], m01);
                    const __half2 M23 = __hmul2(s23, pa23[nt]);
                    __half2 m23 = __hfma2(s23, pa23[nt], __hneg2(M23));
                    m23 = __hfma2(s23, pb23[nt], m23);
                    bp[nt][0] = part ? h2_as_u32(m01) : h2_as_u32(M01);
                    bp[nt][1] = part ? h2_as_u32(m23) : h2_as_u32(M23);
                }
            }
            const uint32_t w0 = vcw[(c0 * G + tb) * BITS / 32 + wi];
            const uint32_t w1 = vcw[((c0 + 8) * G + tb) * BITS / 32 + wi];
            uint32_t af[4];
            af[0] = code_pair<BITS>(w0, BITS * j0);
            af[1] = code_pair<BITS>(w1, BITS * j0);
            af[2] = code_pair<BITS>(w0, BITS * (j0 + 1));
            af[3] = code_pair<BITS>(w1, BITS * (j0 + 1));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[mt][nt], af, bp[nt][0], bp[nt][1]);
        }
    }
    // offset term of the values: oz[head][gv] = sum_t p[head][t] * zero[t][gv]
    float oz[MT][NT];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const int gv = (cw0 + mt * 16) / lo.Gv;
        float zs[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) zs[hh] = 0.0f;
        for (int t = lane; t < ntok; t += 32) {
            const uint8_t* rec = data + (int64_t)(t / G) * lo.rec;
            const __half* zV = reinterpret_cast<const __half*>(rec + kc_bytes + vc_bytes + lo.kp) + G * lo.NGv;
            const float z = __half2float(zV[(t % G) * lo.NGv + gv]);
#pragma unroll
            for (int hh = 0; hh < 8; ++hh)
                if (hh < gqa) zs[hh] = fmaf(sc[hh * CH + t], z, zs[hh]);
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
            if (hh < gqa) zs[hh] = warp_sum(zs[hh]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float v = 0.0f;
#pragma unroll
            for (int hh = 0; hh < 8; ++hh)
                if (hh == 4 * nt + tig) v = zs[hh];
            oz[mt][nt] = v;
        }
    }
    float* wso = reinterpret_cast<float*>(a.ws + a.plan.ws_o_off);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = 4 * nt + tig;
            if (head < gqa) {
                const int c0 = cw0 + mt * 16 + g;
                float* o = wso + slot_index(a, b, h, item, head) * D;
                o[c0] = (oacc[mt][nt][0] + oacc[mt][nt][1]) + oz[mt][nt];
                o[c0 + 8] = (oacc[mt][nt][2] + oacc[mt][nt][3]) + oz[mt][nt];
            }
        }
    if (tid < gqa) {
        float* ml = reinterpret_cast<float*>(a.ws + a.plan.ws_ml_off) + 2 * slot_index(a, b, h, item, tid);
        ml[0] = hstat[tid];
        ml[1] = hstat[32 + tid];
    }
}

// One block per (item, kv head, sequence).  BITS == 0: no packed path (INT8 / FP8).
template <int D, int BITS, int NT>
__global__ void __launch_bounds__(kDecodeThreads) k_decode(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int item = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int32_t* st = state_ptr(a.lo, a.cache, a.layer, b);
    const int64_t n = st[0], qn = st[1];
    const ItemRange r = item_range(a.lo, a.plan, item, n, qn);
    if (r.t0 >= r.t1) return;
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    if constexpr (BITS != 0) {
        if (item >= a.plan.NRC) {
            packed_item<D, BITS, NT>(a, smem, so, b, h, item, r.t0, r.t1);
            return;
        }
    }
    rows_item<D>(a, smem, so, b, h, item, r.t0, r.t1);
}

template <int D, int BITS, int NT>
int launch_decode_t(const DecodeArgs& a, cudaStream_t stream) {
    auto fn = k_decode<D, BITS, NT>;
    if (a.plan.smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(a.plan.smem)) !=
            cudaSuccess)
        return KVQ_ERR_CUDA;
    dim3 grid(a.plan.S, a.lo.H, a.lo.B);
    fn<<<grid, kDecodeThreads, a.plan.smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// Dispatchers, one per translation unit.
int launch_decode_kivi2(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_rows(const DecodeArgs& a, cudaStream_t stream);

}  // namespace kvq
