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
//           turned into exact fp16 subnormals (code * 2^(p - 24), powers of two undone
//           exactly on the other operand and the result), Bq = (query * per-channel key scale) split
//           into an fp16 major part and an fp16 minor part (cols 2h, 2h+1), so the fp32
//           accumulator sees the product to ~22 bits; the per-group offset term
//           sum_c q_c * zero_c is added in fp32.  (Q_b equation: xhat = code*s + min.)
//   values  O[c][col] = sum_t code[t][c] * Bp[t][col], A = value codes (stored per tile
//           in the order of the A fragments, so a lane reads its codes of a tile with
//           one or two wide loads), Bp = p_t * value scale split into major/minor parts;
//           the offset term sum_t p_t * zero_t is one more small product.
// The bf16 window of a KIVI cache runs on the tensor cores too (window_item); INT8 rows
// go through a CUDA-core row path; FP8 caches run on the tensor cores in
// kvq_decode_fp8.cu.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

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
        const int64_t span = (int64_t)p.CPI * p.CH;
        r.t0 = (int64_t)(item - p.NRC) * span;
        r.t1 = r.t0 + span < qn ? r.t0 + span : qn;
    }
    return r;
}

// The work of one decode block.  Blocks are numbered item-major over the units (sequence,
// kv head): first every unit's packed items (the long ones; a unit's last, possibly
// partial, item last), then the window or row items.  The blocks left over for a second
// wave of resident blocks are then the short ones.
struct BlockWork {
    int item, h, b;
};
__device__ __forceinline__ BlockWork block_work(const Layout& lo, const DecodePlan& p) {
    const uint32_t units = static_cast<uint32_t>(lo.B) * static_cast<uint32_t>(lo.H);
    const uint32_t k = blockIdx.x / units, u = blockIdx.x - k * units;
    BlockWork w;
    w.item = static_cast<int>(k) < p.NQ ? p.NRC + static_cast<int>(k) : static_cast<int>(k) - p.NQ;
    w.b = static_cast<int>(u / static_cast<uint32_t>(lo.H));
    w.h = static_cast<int>(u) - w.b * lo.H;
    return w;
}
// Grid of the decode kernels: one block per (item, unit).
inline dim3 decode_grid(const DecodeArgs& a) {
    return dim3(static_cast<unsigned>((int64_t)a.plan.S * a.lo.B * a.lo.H));
}

__device__ __forceinline__ float load_q(const void* q, int64_t idx, int dtype) {
    if (dtype == KVQ_DTYPE_BF16) return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(q)[idx]);
    return reinterpret_cast<const float*>(q)[idx];
}

// 2^x by the hardware approximation (relative error about 2^-22; flushes subnormals)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

// An item without tokens (or whose chunks never arrived) leaves an empty partial: m = -inf,
// l = 0, so the merge gives it weight 0 without reading the cache state.
__device__ __forceinline__ void empty_partial(const DecodeArgs& a, int b, int h, int item) {
    if (threadIdx.x < a.lo.gqa) {
        float* ml = reinterpret_cast<float*>(a.ws + a.plan.ws_ml_off) + 2 * slot_index(a, b, h, item, threadIdx.x);
        ml[0] = -INFINITY;
        ml[1] = 0.0f;
    }
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
// Tokens held as whole rows: the bf16 window of a KIVI cache, or INT8 rows.
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
            // INT8 rows (FP8 has its own tensor-core path)
            const uint8_t* unit = a.cache + lo.data_off + u * lo.unit;
            const uint32_t cb = static_cast<uint32_t>(cnt) * D;
            const uint32_t sb = static_cast<uint32_t>((cnt + 3) / 4 * 4) * 4;
            mbar_arrive_expect_tx(bar, 2 * cb + 2 * sb);
            bulk_copy_pieces(data, unit + t0 * D, cb, bar);
            bulk_copy_pieces(data + (int64_t)CHR * D, unit + (int64_t)lo.T16 * D + t0 * D, cb, bar);
            const uint8_t* scales = unit + 2 * (int64_t)lo.T16 * D;
            bulk_copy_pieces(data + 2 * (int64_t)CHR * D, scales + 4 * t0, sb, bar);
            bulk_copy_pieces(data + 2 * (int64_t)CHR * D + 4 * CHR, scales + 4 * (int64_t)lo.T16 + 4 * t0, sb, bar);
        }
    }
    load_query(a, b, h, qs);
    if (!wait_staged(bar, a.ws)) {
        empty_partial(a, b, h, item);
        return;
    }

    auto kval = [&](int i, int c) -> float {
        if (lo.scheme == KVQ_SCHEME_KIVI)
            return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D)[c]);
        return static_cast<float>(reinterpret_cast<const int8_t*>(data)[i * D + c]) *
               reinterpret_cast<const float*>(data + 2 * (int64_t)CHR * D)[i];
    };
    auto vval = [&](int i, int c) -> float {
        if (lo.scheme == KVQ_SCHEME_KIVI)
            return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D + 2 * D)[c]);
        return static_cast<float>(reinterpret_cast<const int8_t*>(data + (int64_t)CHR * D)[i * D + c]) *
               reinterpret_cast<const float*>(data + 2 * (int64_t)CHR * D + 4 * CHR)[i];
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

// Combine the 4 warps' partials of one work item (comb[warp][head][D] = o, cml[warp][head]
// = (m, l)) into the item's workspace slots.  Called by the whole block after a barrier.
// A warp without tokens leaves m = -inf, l = 0 and its o unwritten; it gets weight 0 and
// its o is never read.
template <int D>
__device__ __forceinline__ void combine_warps(const DecodeArgs& a, const float* comb, const float* cml,
                                              float* red, int b, int h, int item) {
    const int tid = threadIdx.x;
    const int gqa = a.lo.gqa;
    float* wgt = red;   // [head][4 warps]
    if (tid < gqa) {
        float M = -INFINITY, l = 0.0f;
        for (int w = 0; w < 4; ++w) M = fmaxf(M, cml[2 * (w * gqa + tid)]);
        for (int w = 0; w < 4; ++w) {
            const float* mlw = cml + 2 * (w * gqa + tid);
            const float wt = mlw[1] > 0.0f ? fast_exp2(mlw[0] - M) : 0.0f;
            wgt[tid * 4 + w] = wt;
            l = fmaf(mlw[1], wt, l);
        }
        float* ml = reinterpret_cast<float*>(a.ws + a.plan.ws_ml_off) + 2 * slot_index(a, b, h, item, tid);
        ml[0] = M;
        ml[1] = l;
    }
    __syncthreads();
    // the item's gqa slots are consecutive: gqa * D floats, four per thread and step
    float4* wso = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.ws + a.plan.ws_o_off) +
                                            slot_index(a, b, h, item, 0) * D);
    for (int i = tid; i < gqa * D / 4; i += blockDim.x) {
        const int head = (4 * i) / D;
        float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float wt = wgt[head * 4 + w];
            if (wt != 0.0f) {
                const float4 v = reinterpret_cast<const float4*>(comb + w * gqa * D)[i];
                o.x = fmaf(v.x, wt, o.x);
                o.y = fmaf(v.y, wt, o.y);
                o.z = fmaf(v.z, wt, o.z);
                o.w = fmaf(v.w, wt, o.w);
            }
        }
        wso[i] = o;
    }
}

// ------------------------------------------------------------------------ window path
// The bf16 window of a KIVI cache.  Keys and queries are exact bf16 values, so the scores
// go straight to the tensor cores (no conversion, no operand split): rows = 16 tokens,
// columns = up to 8 query heads.  Each warp takes one 16-token tile and keeps its own
// softmax partial; P.V runs on the tensor cores too, with V^T fragments read from the
// token-major rows by ldmatrix.trans and p split into bf16 major and minor parts.  The
// block then combines its 4 warps.
template <int D, int NT>
__device__ void window_item(const DecodeArgs& a, uint8_t* smem, const SmemOffsets& so, int b, int h,
                            int item, int64_t t0, int64_t t1) {
    constexpr int KSTEPS = D / 16;
    constexpr int MTV = D / 16;
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
    const int cnt = static_cast<int>(t1 - t0);
    const int gqa = lo.gqa;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* comb = reinterpret_cast<float*>(smem + so.sc);       // [warp][head][D]
    float* cml = comb + 4 * gqa * D;                            // [warp][head][m, l]
    float* pw = reinterpret_cast<float*>(smem + so.pw);         // [warp][16 tokens][8 heads]
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);

    if (tid == 0) mbar_init(bar, 1);
    __syncthreads();
    if (tid == 0) {
        const uint8_t* ring = a.cache + lo.ring_off + u * lo.C * (int64_t)(4 * D);
        const int s0 = static_cast<int>(t0 % lo.C);
        const int first = cnt < lo.C - s0 ? cnt : lo.C - s0;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt) * 4 * D);
        bulk_copy_pieces(data, ring + (int64_t)s0 * 4 * D, static_cast<uint32_t>(first) * 4 * D, bar);
        if (cnt > first)
            bulk_copy_pieces(data + (int64_t)first * 4 * D, ring, static_cast<uint32_t>(cnt - first) * 4 * D, bar);
    }
    // query operand: column g = head g (zero beyond gqa), k = channel pairs (2t, 2t+1) and
    // (2t+8, 2t+9) of each 16-channel step, straight from the caller's bf16 query
    uint32_t bq[KSTEPS][2];
    {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const uint16_t*>(a.q) + ((int64_t)b * lo.Hq + (int64_t)h * gqa + g) * D);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            bq[ks][0] = g < gqa ? qrow[(16 * ks + 2 * tig) / 2] : 0u;
            bq[ks][1] = g < gqa ? qrow[(16 * ks + 8 + 2 * tig) / 2] : 0u;
        }
    }
    const bool ok = wait_staged(bar, a.ws);
    const int tok0 = 16 * warp;
    const int ntok = cnt - tok0 < 0 ? 0 : (cnt - tok0 > 16 ? 16 : cnt - tok0);
    float oacc[MTV][NT][4];
#pragma unroll
    for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.0f;
    float mh = -INFINITY, lh = 0.0f;      // this lane's head (lane < gqa): max and sum
    if (ok && ntok > 0) {
        // scores: rows g, g + 8 of the tile (tokens beyond the window read as zero rows)
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint8_t* r0 = data + (int64_t)(tok0 + g) * 4 * D;
        const uint8_t* r1 = data + (int64_t)(tok0 + g + 8) * 4 * D;
        const bool v0 = g < ntok, v1 = g + 8 < ntok;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t af[4];
            af[0] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + 2 * (16 * ks + 2 * tig)) : 0u;
            af[1] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + 2 * (16 * ks + 2 * tig)) : 0u;
            af[2] = v0 ? *reinterpret_cast<const uint32_t*>(r0 + 2 * (16 * ks + 8 + 2 * tig)) : 0u;
            af[3] = v1 ? *reinterpret_cast<const uint32_t*>(r1 + 2 * (16 * ks + 8 + 2 * tig)) : 0u;
            mma_16816_bf16(acc, af, bq[ks][0], bq[ks][1]);
        }
        // lane (g, t) holds heads 2t, 2t+1 for tokens g and g + 8
        float sc[2][2];
        sc[0][0] = v0 ? acc[0] * a.qscale : -INFINITY;
        sc[0][1] = v0 ? acc[1] * a.qscale : -INFINITY;
        sc[1][0] = v1 ? acc[2] * a.qscale : -INFINITY;
        sc[1][1] = v1 ? acc[3] * a.qscale : -INFINITY;
        float m0 = fmaxf(sc[0][0], sc[1][0]), m1 = fmaxf(sc[0][1], sc[1][1]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
            m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
        }
        float* pt = pw + warp * 16 * 8;
        const float p00 = v0 ? fast_exp2(sc[0][0] - m0) : 0.0f, p01 = v0 ? fast_exp2(sc[0][1] - m1) : 0.0f;
        const float p10 = v1 ? fast_exp2(sc[1][0] - m0) : 0.0f, p11 = v1 ? fast_exp2(sc[1][1] - m1) : 0.0f;
        pt[g * 8 + 2 * tig] = p00;
        pt[g * 8 + 2 * tig + 1] = p01;
        pt[(g + 8) * 8 + 2 * tig] = p10;
        pt[(g + 8) * 8 + 2 * tig + 1] = p11;
        float l0 = p00 + p10, l1 = p01 + p11;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        // lane hh (< gqa) keeps head hh's max and sum: heads 2t, 2t+1 live in lanes t
        const int src = (lane < 8 ? lane : 0) >> 1;
        const float mm0 = __shfl_sync(0xffffffffu, m0, src), mm1 = __shfl_sync(0xffffffffu, m1, src);
        const float ll0 = __shfl_sync(0xffffffffu, l0, src), ll1 = __shfl_sync(0xffffffffu, l1, src);
        mh = (lane & 1) ? mm1 : mm0;
        lh = (lane & 1) ? ll1 : ll0;
        // value rows past the window's end hold stale bytes: zero them (their p is 0,
        // and a stale pattern could read as NaN)
        if (ntok < 16) {
            for (int i = ntok + (lane >> 4); i < 16; i += 2) {
                uint4* vr = reinterpret_cast<uint4*>(data + (int64_t)(tok0 + i) * 4 * D + 2 * D);
                for (int e = lane & 15; e < D / 8; e += 16) vr[e] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncwarp();
        // values on the tensor cores: A = the 16 x 16 (channels x tokens) tile of V^T, read
        // from the token-major bf16 rows by ldmatrix.trans; B = p (k = tokens, column
        // 2h + part) split into bf16 major and minor parts, from the warp's p table
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head = 4 * nt + (g >> 1);
            const float p0 = pt[(2 * tig) * 8 + head], p1 = pt[(2 * tig + 1) * 8 + head];
            const float p2 = pt[(2 * tig + 8) * 8 + head], p3 = pt[(2 * tig + 9) * 8 + head];
            const __nv_bfloat162 m01 = __floats2bfloat162_rn(p0, p1), m23 = __floats2bfloat162_rn(p2, p3);
            const float2 f01 = __bfloat1622float2(m01), f23 = __bfloat1622float2(m23);
            const __nv_bfloat162 r01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
            const __nv_bfloat162 r23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
            const uint32_t um01 = *reinterpret_cast<const uint32_t*>(&m01), um23 = *reinterpret_cast<const uint32_t*>(&m23);
            const uint32_t ur01 = *reinterpret_cast<const uint32_t*>(&r01), ur23 = *reinterpret_cast<const uint32_t*>(&r23);
            b0[nt] = (g & 1) ? ur01 : um01;
            b1[nt] = (g & 1) ? ur23 : um23;
        }
        // ldmatrix rows: lane l addresses token (l mod 8) + 8 (l / 16), channels from
        // 16 q + 8 ((l / 8) mod 2): the four 8 x 8 blocks land as a0..a3
        const uint32_t vrow = smem_addr(data) + (tok0 + (lane & 7) + 8 * (lane >> 4)) * 4 * D + 2 * D +
                              2 * 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int q = 0; q < MTV; ++q) {
            uint32_t af[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                         : "=r"(af[0]), "=r"(af[1]), "=r"(af[2]), "=r"(af[3])
                         : "r"(vrow + 32 * q)
                         : "memory");
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816_bf16(oacc[q][nt], af, b0[nt], b1[nt]);
        }
    }
    // warp partial into shared memory, then the 4 warps combined
    float* cw = comb + warp * gqa * D;
    const bool wlive = ok && ntok > 0;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int head = 4 * nt + tig;
        if (head < gqa && wlive) {
#pragma unroll
            for (int mt = 0; mt < MTV; ++mt) {
                const int c0 = 16 * mt + g;
                cw[head * D + c0] = oacc[mt][nt][0] + oacc[mt][nt][1];
                cw[head * D + c0 + 8] = oacc[mt][nt][2] + oacc[mt][nt][3];
            }
        }
    }
    if (lane < gqa) {
        cml[2 * (warp * gqa + lane)] = wlive ? mh : -INFINITY;
        cml[2 * (warp * gqa + lane) + 1] = wlive ? lh : 0.0f;
    }
    __syncthreads();
    combine_warps<D>(a, comb, cml, red, b, h, item);
}

// ------------------------------------------------------------------------ packed path
// Loads from the staged chunk by 32-bit shared-window address.  They are volatile so the
// compiler keeps them after the barrier waits (volatile asm with a memory clobber) that
// make the bulk copies visible, and before the barrier that frees the stage.
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
template <int N>
__device__ __forceinline__ void lds_words(uint32_t a, uint32_t (&w)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const uint4 v = lds128(a + 4 * i);
            w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
        }
    } else if constexpr (N == 2) {
        const uint2 v = lds64(a);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = lds32(a + 4 * i);
    }
}

// 2^k as a float for -126 <= k <= 127 (exact).
__device__ __forceinline__ float exp2i(int k) { return __int_as_float((127 + k) << 23); }
// 2^k as an fp16 pair for -14 <= k <= 15 (exact).
__device__ __forceinline__ uint32_t exp2i_h2(int k) { return static_cast<uint32_t>((15 + k) << 10) * 0x00010001u; }

// Code extraction.  A b-bit code c at bit p of a 16-bit half, with every other bit of the
// half cleared, is the fp16 subnormal c * 2^(p - 24) -- exact, and made for the code pair
// of both halves of a 32-bit word by one AND, as long as p + b <= 10 (the code stays in
// the mantissa).  The factor 2^(p - 24) is undone exactly: 2^-p goes into the other MMA
// operand as a power-of-two scale, 2^24 onto the fp32 result.
template <int BITS>
__device__ __forceinline__ uint32_t code_bits(uint32_t w, int p) {
    return w & ((((1u << BITS) - 1u) << p) * 0x00010001u);
}
// Code pair jj of a word (codes at bits BITS*jj and 16 + BITS*jj): codes reaching past
// bit 10 are first shifted down by 6 (one shift per word), everything else stays in place;
// the pair then sits at bit code_pos of each half.
template <int BITS> constexpr int code_shift(int jj) { return BITS * jj + BITS > 10 ? 6 : 0; }
template <int BITS> constexpr int code_pos(int jj) { return BITS * jj - code_shift<BITS>(jj); }

// (s * x) of fp16 pairs split in two fp16 parts by an error-free product: with x = (0,
// major) -> the rounded product of s and `major`; with x = (major, minor) -> the rounding
// error of s * major plus s * minor.  The lanes holding B column 2h take the first form,
// the lanes of column 2h + 1 the second, so no lane selects between results.
__device__ __forceinline__ uint32_t split_mul(__half2 s, uint32_t x, uint32_t y) {
    const __half2 t = __hmul2(s, u32_as_h2(x));
    const __half2 e = __hfma2(s, u32_as_h2(x), __hneg2(t));
    return h2_as_u32(__hfma2(s, u32_as_h2(y), e));
}

// One packed work item: a run of chunks of CH = 4 * W tokens of one (sequence, kv head).
// Chunks are staged by bulk copies into NSTAGE shared-memory buffers (double-buffered
// when they fit), each warp takes W tokens of a chunk, and every warp keeps an online
// softmax (running max, sum and output) across the chunks of the item.
//
// Scales.  Scores: A = key codes c * 2^(p - 24), B = q * s_c * 2^(E - p) with E per group
// such that the largest key scale of the group times 2^E is below 2^15, so the product
// is c * q * s_c * 2^(E - 24) and the score is the fp32 sum times 2^(24 - E).  Values:
// A = value codes c * 2^(p - 24), B = P * s_t * 2^Ev with Ev per warp such that the
// largest value scale seen so far times 2^Ev is below 2^15 (lowered, and what was
// accumulated rescaled by the exact power of two, when a larger scale arrives); the code
// position p is fixed per accumulator element, so 2^(24 - p) is applied at the end.
template <int D, int BITS, int NT>
__device__ void packed_item(const DecodeArgs& a, uint8_t* smem, const SmemOffsets& so, int b, int h,
                            int item, int64_t t0, int64_t t1) {
    constexpr int CPW = 32 / BITS;          // key channels per 32-bit word
    constexpr int HPW = CPW / 2;            // code pairs per word (keys and values)
    constexpr int NPAIR = D / 8;            // code pairs per thread per token row
    constexpr int KSTEPS = D / 16;
    constexpr int ROWW = D * BITS / 128;    // words per thread per key row
    constexpr int ROWB = D * BITS / 8;      // bytes per key row
    constexpr int MTV = D / 16;             // 16-channel tiles of the value contraction
    constexpr int WPL = D * BITS / 64;      // value-code words per lane per tile
    constexpr int SW = WPL < 4 ? WPL : 4;   // words per lane per slab (one wide load)
    constexpr int MAXT = 8;                 // a warp holds at most 8 tiles (W <= 128 tokens)
    constexpr int QROW = NPAIR + 4;         // words per row of the query tables (padded)
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
    const int G = lo.G, W = a.plan.W, CH = a.plan.CH, gqa = lo.gqa, NGv = lo.NGv;
    const int nstage = a.plan.NSTAGE;
    const uint32_t rec = static_cast<uint32_t>(lo.rec);
    const uint32_t stage_bytes = static_cast<uint32_t>(CH / G) * rec;
    const int ntok = static_cast<int>(t1 - t0);
    const int nch = (ntok + CH - 1) / CH;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    uint32_t* qx = reinterpret_cast<uint32_t*>(smem + so.qpa);
    uint32_t* qy = reinterpret_cast<uint32_t*>(smem + so.qpb);
    float* comb = reinterpret_cast<float*>(smem + so.sc);          // [warp][head][D]
    float* cml = comb + 4 * gqa * D;                               // [warp][head][m, l]
    const int64_t u = unit_index(lo, a.layer, b, h);
    const uint8_t* src_unit = a.cache + lo.data_off + u * lo.unit;

    // the item's groups (t0 and t1 are group boundaries): chunk j holds gpc of them
    const int gpc = CH / G;
    const uint8_t* src_groups = src_unit + (t0 / G) * (int64_t)rec;
    const int ngroups = ntok / G;
    auto issue = [&](int j) {       // stage chunk j (thread 0 only)
        const int gj = min(gpc, ngroups - j * gpc);
        const uint32_t bytes = static_cast<uint32_t>(gj) * rec;
        const int sj = nstage == 2 ? (j & 1) : 0;   // stage of chunk j
        uint64_t* bar = bars + sj;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_copy_pieces(smem + so.data + sj * stage_bytes, src_groups + (int64_t)j * gpc * rec, bytes, bar);
    };
    if (tid == 0) {
        for (int s2 = 0; s2 < nstage; ++s2) mbar_init(bars + s2, 1);
    }
    __syncthreads();
    if (tid == 0) {
        for (int j = 0; j < nstage && j < nch; ++j) issue(j);
    }
    // query prep (whole block) while the copies are in flight: fp32 scaled query, a
    // power-of-two prescale bringing max|q| into [0.5, 1) so fp16 products cannot
    // overflow, and per-lane tables of the query in the lanes' key-pair order split into
    // fp16 major + minor parts: row 32 * nt + lane holds x = (0 | major) and y = (major |
    // minor) for B column g = 2 * head + part of that lane (split_mul)
    float qmax = 0.0f;
    {
        // scaled query of the kv head's gqa query heads into shared fp32, vector loads
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
    const float qdown = ldexpf(1.0f, -qexp), qup = ldexpf(1.0f, qexp);
    // one entry per (head hh, lane quarter tg, key pair m), written to the rows of the two
    // lanes (parts) of B columns 2 (hh mod 4) and 2 (hh mod 4) + 1
    for (int i = tid; i < 16 * NT * NPAIR; i += blockDim.x) {
        const int m = i % NPAIR, r = i / NPAIR;
        const int hh = r >> 2, tg = r & 3;
        const int wi = m / HPW, jj = m % HPW;
        const int clo = tg * (D / 4) + wi * CPW + jj, chi = clo + HPW;
        float vlo = 0.0f, vhi = 0.0f;
        if (hh < gqa) {
            vlo = qs[hh * D + clo] * qdown;
            vhi = qs[hh * D + chi] * qdown;
        }
        const __half2 major = __floats2half2_rn(vlo, vhi);
        const float2 mf = __half22float2(major);
        const uint32_t mj = h2_as_u32(major), mn = h2_as_u32(__floats2half2_rn(vlo - mf.x, vhi - mf.y));
        const int row0 = 32 * (hh >> 2) + 8 * (hh & 3) + tg;   // lane of part 0; part 1 is 4 lanes on
        qx[row0 * QROW + m] = 0u;
        qy[row0 * QROW + m] = mj;
        qx[(row0 + 4) * QROW + m] = mj;
        qy[(row0 + 4) * QROW + m] = mn;
    }
    __syncthreads();

    const uint32_t sbase = smem_addr(smem);
    const uint32_t qx_lane = sbase + static_cast<uint32_t>(so.qpa) + lane * QROW * 4;
    const uint32_t qy_lane = sbase + static_cast<uint32_t>(so.qpb) + lane * QROW * 4;
    const int part = g & 1;                 // B column g = 2 * head + part
    const uint32_t kpar = lo.kc + lo.vc;                    // key params in a record
    const uint32_t vpar = kpar + lo.kp;                     // value params in a record
    const uint32_t kscale_lane = kpar + tig * (D / 2);      // the lane's quarter of the key scales
    const uint32_t kzero_lane = kscale_lane + 2 * D;
    // score tile rows: lane (g, tig) scores tokens g and g + 8 of each 16-token tile, so the
    // lane pair (2t', h') and (2t' + 1, h') holds the tokens of the value fragment of lane
    // (g', t') (h' = g' / 2): 2t' and 2t' + 8 (k slots 2t', 2t' + 1), 2t' + 1 and 2t' + 9
    // (k slots 2t' + 8, 2t' + 9)
    const uint32_t krow0 = g * ROWB + tig * (ROWW * 4), krow1 = (g + 8) * ROWB + tig * (ROWW * 4);
    // value codes of a tile: 32 lanes of WPL words in slabs of SW; lane (g, t) holds, for
    // every 16-channel tile q, its A fragment: the codes of channels 16q + g (r = 0) and
    // 16q + g + 8 (r = 1) for tokens 2t, 2t + 8 (even words, k slots 2t, 2t + 1) and
    // 2t + 1, 2t + 9 (odd words, k slots 2t + 8, 2t + 9), index j = 2q + r at bits
    // BITS * (j mod HPW) of word pair j / HPW
    const uint32_t vlane = lo.kc + lane * SW * 4;
    // value scales and zeros: [group][G] fp16 with tile token tt at position 2 (tt mod 8) +
    // tt / 8, so this lane's four tokens are the 8 bytes at tile position 4t
    const uint32_t vscale_lane = vpar + 8 * tig;
    const uint32_t vzero_lane = vpar + 2 * G * NGv + 8 * tig;
    const int src1 = (2 * tig) * 4 + (g >> 1), src2 = (2 * tig + 1) * 4 + (g >> 1);
    const uint32_t pmask = part ? 0xffffffffu : 0u;
    const uint32_t zg = g < NGv ? 2 * G * g : 0u, zmask = g < NGv ? 0xffffffffu : 0u;
    const uint32_t zg8 = g + 8 < NGv ? 2 * G * (g + 8) : 0u, zmask8 = g + 8 < NGv ? 0xffffffffu : 0u;
    const int gvs = __ffs(lo.Gv) - 5;       // value groups are powers of two >= 16

    float mrun[NT], lrun[NT];
    float oacc[MTV][NT][4];
    float ozacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        mrun[nt] = -INFINITY;
        lrun[nt] = 0.0f;
        ozacc[nt][0] = ozacc[nt][1] = ozacc[nt][2] = ozacc[nt][3] = 0.0f;
#pragma unroll
        for (int mt = 0; mt < MTV; ++mt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.0f;
    }
    int Ev = 15;
    bool live = true;
    // the warp's tokens start W * warp tokens into every chunk: group g0 of the chunk's
    // records, offset ti0 in it (a group may be shared by two warps)
    const int g0 = (warp * W) / G, ti0 = (warp * W) % G;
    for (int j = 0; j < nch; ++j) {
        const int sj = nstage == 2 ? (j & 1) : 0;                       // stage of chunk j
        const uint32_t par = nstage == 2 ? ((j >> 1) & 1) : (j & 1);    // its barrier phase
        bool ok = mbar_wait_bounded(bars + sj, par, kWaitLimit);
        ok = __syncthreads_and(ok);
        if (!ok) {
            if (tid == 0) atomicOr(reinterpret_cast<uint32_t*>(a.ws), KVQ_STATUS_TIMEOUT);
            mbar_wait_bounded(bars + sj, par, kWaitLimit);
            live = false;
            break;
        }
        const int ctok = min(ntok - j * CH, CH);
        const int wtok = ctok - warp * W < 0 ? 0 : (ctok - warp * W > W ? W : ctok - warp * W);   // multiple of 16
        const uint32_t st0 = sbase + static_cast<uint32_t>(so.data) + sj * stage_bytes + g0 * rec;
        int ngrp = 0;                                  // groups the warp's tokens touch (<= 8)
        for (int x = ti0 + wtok; x > 0; x -= G) ++ngrp;
        if (wtok > 0) {
            const int ntl = wtok >> 4;
            // offset term of every group of the warp: cst[group][head] = sum_c q_c zero_c,
            // as one small tensor-core product (rows = groups, k = channels in pair order)
            float cstf[NT][4];
            {
                uint32_t zreg[D / 8];
                if (g < ngrp) {
                    lds_words<D / 8>(st0 + g * rec + kzero_lane, zreg);
                } else {
#pragma unroll
                    for (int i = 0; i < D / 8; ++i) zreg[i] = 0u;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    cstf[nt][0] = cstf[nt][1] = cstf[nt][2] = cstf[nt][3] = 0.0f;
                    uint32_t qt[NPAIR];
                    lds_words<NPAIR>(qy_lane + nt * 32 * QROW * 4, qt);
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        uint32_t af[4];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int m = 2 * ks + e, wi = m / HPW, jj = m % HPW;
                            const int lo_l = wi * CPW + jj, hi_l = lo_l + HPW;
                            af[2 * e] = prmt(zreg[lo_l / 2], zreg[hi_l / 2], (jj & 1) ? 0x7632u : 0x5410u);
                            af[2 * e + 1] = 0u;
                        }
                        mma_16816(cstf[nt], af, qt[2 * ks], qt[2 * ks + 1]);
                    }
                }
            }
            // ---- pass 1: scores of the warp's tiles, parked in the warp's shared scratch
            // (rolled loops keep the kernel within the instruction cache)
            float2* wsc = reinterpret_cast<float2*>(smem + so.sc) + (int64_t)warp * MAXT * NT * 32 + lane;
            float cmax[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) cmax[nt] = -INFINITY;
            {
                int i = 0, grp = 0, ti = ti0;
                uint32_t ro = st0;
#pragma unroll 1
                while (i < ntl) {
                    // key-score operand of the group: (q * key scale * 2^(E - p)) as fp16
                    // major + minor, E from the group's largest key scale
                    uint32_t bq[NT][NPAIR];
                    float kf, cst[NT];
                    {
                        uint32_t sreg[D / 8];
                        lds_words<D / 8>(ro + kscale_lane, sreg);
                        // the group's largest key scale (scales are >= 0, so fp16 bit patterns
                        // order as integers): each lane takes D / 32 of the D scales
                        uint32_t mb;
                        {
                            uint32_t part_w[D / 64];
                            lds_words<D / 64>(ro + kpar + lane * (D / 16), part_w);
                            __half2 mx = u32_as_h2(part_w[0]);
#pragma unroll
                            for (int k = 1; k < D / 64; ++k) mx = __hmax2(mx, u32_as_h2(part_w[k]));
                            mb = h2_as_u32(mx);
                            mb = max(mb & 0xffffu, mb >> 16);
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
                        }
                        const int E = min(15, 29 - static_cast<int>((mb >> 10) & 31u));
                        kf = exp2i(24 - E) * qup;
                        __half2 sp[NPAIR];
#pragma unroll
                        for (int m = 0; m < NPAIR; ++m) {
                            const int wi = m / HPW, jj = m % HPW;
                            const int lo_l = wi * CPW + jj, hi_l = lo_l + HPW;
                            sp[m] = __hmul2(u32_as_h2(prmt(sreg[lo_l / 2], sreg[hi_l / 2], (jj & 1) ? 0x7632u : 0x5410u)),
                                            u32_as_h2(exp2i_h2(E - code_pos<BITS>(jj))));
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint32_t xq[NPAIR], yq[NPAIR];
                            lds_words<NPAIR>(qx_lane + nt * 32 * QROW * 4, xq);
                            lds_words<NPAIR>(qy_lane + nt * 32 * QROW * 4, yq);
#pragma unroll
                            for (int m = 0; m < NPAIR; ++m) bq[nt][m] = split_mul(sp[m], xq[m], yq[m]);
                            const float c = __shfl_sync(0xffffffffu, cstf[nt][0] + cstf[nt][1], grp * 4 + tig);
                            cst[nt] = c * qup;
                        }
                    }
                    const int nseg = min(ntl - i, (G - ti) >> 4);
                    uint32_t kro = ro + ti * ROWB;
#pragma unroll 1
                    for (int k = 0; k < nseg; ++k, ++i, kro += 16 * ROWB) {
                        uint32_t wa[ROWW], wb[ROWW];
                        lds_words<ROWW>(kro + krow0, wa);
                        lds_words<ROWW>(kro + krow1, wb);
                        // two accumulator chains (even and odd k steps) for instruction-level
                        // parallelism between the dependent tensor-core operations
                        float acc[2][NT][4];
#pragma unroll
                        for (int e = 0; e < 2; ++e)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) acc[e][nt][0] = acc[e][nt][1] = acc[e][nt][2] = acc[e][nt][3] = 0.0f;
#pragma unroll
                        for (int ks = 0; ks < KSTEPS; ++ks) {
                            const int m0 = 2 * ks, m1 = 2 * ks + 1;
                            const int j0 = m0 % HPW, j1 = m1 % HPW;
                            uint32_t af[4];
                            af[0] = code_bits<BITS>(wa[m0 / HPW] >> code_shift<BITS>(j0), code_pos<BITS>(j0));
                            af[1] = code_bits<BITS>(wb[m0 / HPW] >> code_shift<BITS>(j0), code_pos<BITS>(j0));
                            af[2] = code_bits<BITS>(wa[m1 / HPW] >> code_shift<BITS>(j1), code_pos<BITS>(j1));
                            af[3] = code_bits<BITS>(wb[m1 / HPW] >> code_shift<BITS>(j1), code_pos<BITS>(j1));
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) mma_16816(acc[ks & 1][nt], af, bq[nt][m0], bq[nt][m1]);
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const float s0 = fmaf((acc[0][nt][0] + acc[1][nt][0]) + (acc[0][nt][1] + acc[1][nt][1]), kf, cst[nt]);
                            const float s1 = fmaf((acc[0][nt][2] + acc[1][nt][2]) + (acc[0][nt][3] + acc[1][nt][3]), kf, cst[nt]);
                            wsc[(i * NT + nt) * 32] = make_float2(s0, s1);
                            cmax[nt] = fmaxf(cmax[nt], fmaxf(s0, s1));
                        }
                    }
                    ro += rec;
                    ti = 0;
                    ++grp;
                }
            }
            // value-scale exponent: the largest value scale of the records the warp's tokens
            // lie in must stay below 2^(15 - Ev); lower Ev (and rescale) when it does not
            {
                uint32_t smx = 0;
                const int nv = NGv * G / 8;      // 16-byte runs of value scales per record
#pragma unroll 1
                for (int r = 0; r < ngrp; ++r) {
#pragma unroll 1
                    for (int o = lane; o < nv; o += 32) {
                        const uint4 v = lds128(st0 + r * rec + vpar + 16 * o);
                        const __half2 m2 = __hmax2(__hmax2(u32_as_h2(v.x), u32_as_h2(v.y)),
                                                   __hmax2(u32_as_h2(v.z), u32_as_h2(v.w)));
                        const uint32_t mb = h2_as_u32(m2);
                        smx = max(smx, max(mb & 0xffffu, mb >> 16));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) smx = max(smx, __shfl_xor_sync(0xffffffffu, smx, o));
                const int en = min(15, 29 - static_cast<int>((smx >> 10) & 31u));
                if (en < Ev) {
                    const float f = exp2i(en - Ev);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        lrun[nt] *= f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) ozacc[nt][e] *= f;
#pragma unroll
                        for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) oacc[mt][nt][e] *= f;
                    }
                    Ev = en;
                }
            }
            // running maximum per head (lanes of a head share tig); rescale what the warp
            // accumulated over earlier chunks when it grows
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
                    for (int e = 0; e < 4; ++e) ozacc[nt][e] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) oacc[mt][nt][e] *= alpha;
                }
                mrun[nt] = mnew;
                // p' = 2^(s - max + Ev): the value operand's power-of-two scale, applied
                // in the exponent
                mE[nt] = mnew - static_cast<float>(Ev);
            }
            // ---- pass 2: p' and the value contraction, tile by tile; the value-group
            // size is a template parameter so the per-group operand rebuilds unroll
            auto pass2 = [&](auto gvs_c) {
                constexpr int GVS = decltype(gvs_c)::value;
                constexpr int QM = (1 << GVS) - 1;
                int i = 0, ti = ti0;
                uint32_t ro = st0;
#pragma unroll 1
                while (i < ntl) {
                    const int nseg = min(ntl - i, (G - ti) >> 4);
#pragma unroll 1
                    for (int k = 0; k < nseg; ++k, ++i, ti += 16) {
                        uint32_t px1[NT], py1[NT], px2[NT], py2[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const float2 sv = wsc[(i * NT + nt) * 32];
                            const float p0 = fast_exp2(sv.x - mE[nt]);
                            const float p1 = fast_exp2(sv.y - mE[nt]);
                            lrun[nt] += p0 + p1;
                            // p' as fp16 major + minor, moved to the lanes of the value fragment
                            const __half2 pa = __floats2half2_rn(p0, p1);
                            const float2 pf = __half22float2(pa);
                            const __half2 pb = __floats2half2_rn(p0 - pf.x, p1 - pf.y);
                            const uint32_t ua = h2_as_u32(pa), ub = h2_as_u32(pb);
                            const uint32_t x1 = __shfl_sync(0xffffffffu, ua, src1);
                            const uint32_t y1 = __shfl_sync(0xffffffffu, ub, src1);
                            const uint32_t x2 = __shfl_sync(0xffffffffu, ua, src2);
                            const uint32_t y2 = __shfl_sync(0xffffffffu, ub, src2);
                            px1[nt] = x1 & pmask;
                            py1[nt] = part ? y1 : x1;
                            px2[nt] = x2 & pmask;
                            py2[nt] = part ? y2 : x2;
                        }
                        // values: O[c][col] += sum_t code[t][c] * (p'_t * scale[t][gv(c)]); the
                        // offset term OZ[gv][col] += sum_t zero[t][gv] * p_t.  Zero pairs of value
                        // groups g and g + 8 (rows of the offset product); lanes past the last
                        // group read group 0 and mask it out.
                        const uint2 z2 = lds64(ro + vzero_lane + 2 * ti + zg);
                        const uint32_t zA = z2.x & zmask, zC = z2.y & zmask;
                        uint32_t zA8 = 0u, zC8 = 0u;
                        if constexpr (D > 128) {
                            const uint2 z8 = lds64(ro + vzero_lane + 2 * ti + zg8);
                            zA8 = z8.x & zmask8;
                            zC8 = z8.y & zmask8;
                        }
                        const uint32_t vsc = ro + vscale_lane + 2 * ti;
                        const uint32_t vtile = ro + vlane + (ti / 16) * (2 * D * BITS);
                        uint32_t vw[WPL <= 8 ? WPL : SW];
                        if constexpr (WPL <= 8) {
                            // the whole tile: slab sl of the lane's words is 128 * SW bytes on
#pragma unroll
                            for (int sl = 0; sl < WPL / SW; ++sl) {
                                uint32_t part[SW];
                                lds_words<SW>(vtile + sl * 128 * SW, part);
#pragma unroll
                                for (int x = 0; x < SW; ++x) vw[sl * SW + x] = part[x];
                            }
                        }
                        uint32_t bv[NT][2];
#pragma unroll
                        for (int q = 0; q < MTV; ++q) {
                            if ((q & QM) == 0) {
                                const int gv = q >> GVS;
                                const uint2 sc = lds64(vsc + 2 * G * gv);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    bv[nt][0] = split_mul(u32_as_h2(sc.x), px1[nt], py1[nt]);
                                    bv[nt][1] = split_mul(u32_as_h2(sc.y), px2[nt], py2[nt]);
                                }
                            }
                            // word pair of q: even word (k slots 2t, 2t + 1), odd word (2t + 8,
                            // 2t + 9); rows g at pair j = 2q, rows g + 8 at pair 2q + 1
                            const int w0 = 2 * ((2 * q) / HPW), m0 = (2 * q) % HPW, m1 = m0 + 1;
                            if constexpr (WPL > 8) {
                                // wide codes: one slab at a time, loaded by its first q
                                if (w0 % SW == 0 && m0 == 0) lds_words<SW>(vtile + (w0 / SW) * 128 * SW, vw);
                            }
                            const uint32_t e = vw[(WPL <= 8 ? w0 : w0 % SW)];
                            const uint32_t o = vw[(WPL <= 8 ? w0 : w0 % SW) + 1];
                            uint32_t af[4];
                            af[0] = code_bits<BITS>(e >> code_shift<BITS>(m0), code_pos<BITS>(m0));
                            af[1] = code_bits<BITS>(e >> code_shift<BITS>(m1), code_pos<BITS>(m1));
                            af[2] = code_bits<BITS>(o >> code_shift<BITS>(m0), code_pos<BITS>(m0));
                            af[3] = code_bits<BITS>(o >> code_shift<BITS>(m1), code_pos<BITS>(m1));
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[q][nt], af, bv[nt][0], bv[nt][1]);
                        }
                        {
                            uint32_t af[4] = {zA, zA8, zC, zC8};
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) mma_16816(ozacc[nt], af, py1[nt], py2[nt]);
                        }
                    }
                    ro += rec;
                    ti = 0;
                }
            };
            switch (gvs) {
                case 0: pass2(std::integral_constant<int, 0>{}); break;
                case 1: if constexpr (MTV > 1) pass2(std::integral_constant<int, 1>{}); break;
                case 2: if constexpr (MTV > 2) pass2(std::integral_constant<int, 2>{}); break;
                case 3: if constexpr (MTV > 4) pass2(std::integral_constant<int, 3>{}); break;
                default: if constexpr (MTV > 8) pass2(std::integral_constant<int, 4>{}); break;
            }
        }
        __syncthreads();            // every warp is done with this stage
        if (tid == 0 && j + nstage < nch) issue(j + nstage);
    }
    // ---- warp partial: undo the power-of-two scales, reduce l over the lanes of a head,
    // add the value offset term, combine the 4 warps in shared memory
    float* cw = comb + warp * gqa * D;
    const bool wlive = live && mrun[0] > -INFINITY;
    const float zfac = exp2i(-Ev), lfac = exp2i(-Ev);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int head = 4 * nt + tig;
        float l = lrun[nt] * lfac;
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        const float oz01 = ozacc[nt][0] + ozacc[nt][1], oz23 = ozacc[nt][2] + ozacc[nt][3];
#pragma unroll
        for (int mt = 0; mt < MTV; ++mt) {
            const int gv = mt >> gvs;
            const float zsrc = gv < 8 ? oz01 : oz23;
            const float oz = __shfl_sync(0xffffffffu, zsrc, (gv & 7) * 4 + tig) * zfac;
            // codes of rows g sat at bit code_pos of pair 2 mt, rows g + 8 of pair 2 mt + 1
            const int m0 = (2 * mt) % HPW;
            const float f0 = exp2i(24 - code_pos<BITS>(m0) - Ev), f1 = exp2i(24 - code_pos<BITS>(m0 + 1) - Ev);
            if (head < gqa && wlive) {
                const int c0 = 16 * mt + g;
                cw[head * D + c0] = fmaf(oacc[mt][nt][0] + oacc[mt][nt][1], f0, oz);
                cw[head * D + c0 + 8] = fmaf(oacc[mt][nt][2] + oacc[mt][nt][3], f1, oz);
            }
        }
        if (g == 0 && head < gqa) {
            cml[2 * (warp * gqa + head)] = wlive ? mrun[nt] : -INFINITY;
            cml[2 * (warp * gqa + head) + 1] = wlive ? l : 0.0f;
        }
    }
    __syncthreads();
    grid_launch_dependents();   // the merge may start launching; it waits for this grid
    combine_warps<D>(a, comb, cml, red, b, h, item);
}

// One block per (item, kv head, sequence), in the order of block_work.  BITS == 0: no
// packed path (INT8 rows).
template <int D, int BITS, int NT>
__global__ void __launch_bounds__(kDecodeThreads, (NT == 1 && D <= 128) ? 4 : 2) k_decode(DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    grid_dependency_wait();
    const BlockWork bw = block_work(a.lo, a.plan);
    const int item = bw.item, h = bw.h, b = bw.b;
    const int32_t* st = state_ptr(a.lo, a.cache, a.layer, b);
    const int64_t n = st[0], qn = st[1];
    const ItemRange r = item_range(a.lo, a.plan, item, n, qn);
    if (r.t0 >= r.t1) {
        empty_partial(a, b, h, item);
        return;
    }
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    if constexpr (BITS != 0) {
        if (item >= a.plan.NRC)
            packed_item<D, BITS, NT>(a, smem, so, b, h, item, r.t0, r.t1);
        else
            window_item<D, NT>(a, smem, so, b, h, item, r.t0, r.t1);
        return;
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
    return launch_dependent(fn, decode_grid(a), kDecodeThreads, static_cast<size_t>(a.plan.smem), stream, a) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
}

// Dispatchers, one per translation unit.
int launch_decode_kivi2(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_rows(const DecodeArgs& a, cudaStream_t stream);
int launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream);

}  // namespace kvq
