// kvq_rope.cuh -- pieces of the decode over KIVI caches whose keys were cached before the
// rotary position embedding ("KVQuant: Towards 10 Million Context Length ...", "Key points":
// keys are quantised before RoPE, which mixes channel pairs).  The angle of channel pair i
// at position t is the binary32 product t * w_i; rope_sincos gives its cosine and sine.
// rope_item is the CUDA-core pass over a run of one unit's tokens (a warp per token for
// the scores, a thread per channel for the values), used for the bf16 window of every
// pre-RoPE decode and, for dense-and-sparse records, for the packed groups too.
// Included by kvq_decode.cuh after the helpers it uses.
#pragma once

namespace kvq {

// Bit, within a group record's value codes, of the code of (token t of the group, channel
// ch), and byte, within its value parameters, of the (token t, value group j) scale: the
// record layout described in kvq_internal.cuh (16-token tiles of 32 lane slabs).
template <int D, int BITS>
__device__ __forceinline__ int value_code_bit(int t, int ch) {
    constexpr int HW = 16 / BITS, WPL = D * BITS / 64, SW = WPL < 4 ? WPL : 4;
    const int tile = t >> 4, tt = t & 15, half = tt >> 3, i = (tt & 7) >> 1, s = tt & 1;
    const int q = ch >> 4, g = ch & 7, r = (ch & 15) >> 3;
    const int lane = 4 * g + i, j = 2 * q + r;
    const int w = 2 * (j / HW) + s;
    const int word = tile * 32 * WPL + (w / SW) * 32 * SW + lane * SW + (w % SW);
    return word * 32 + 16 * half + BITS * (j % HW);
}
__device__ __forceinline__ int value_param_byte(int G, int j, int t) {
    const int tt = t & 15;
    return 2 * (j * G + (t - tt) + 2 * (tt & 7) + (tt >> 3));
}
// The BITS-bit code at bit `bit` of `p` (codes never straddle a byte).
template <int BITS>
__device__ __forceinline__ int code_at(const uint8_t* p, int bit) {
    return (p[bit >> 3] >> (bit & 7)) & ((1 << BITS) - 1);
}
__device__ __forceinline__ float half_at(const uint8_t* p, int byte) {
    return __half2float(*reinterpret_cast<const __half*>(p + byte));
}
// cos and sin of a binary32 angle a.  For |a| < 2^17, Cody and Waite's reduction by 2 pi
// in three binary32 parts (the first, 6.28125, has 8 significant bits, so k * C1 is exact
// for the |k| < 2^15 that occur; C2 and C3 carry the rest of 2 pi), then the hardware sine
// and cosine on the reduced |r| <= pi (absolute error about 1e-6).  Larger angles take the
// library's sincosf with its full argument reduction.
__device__ __forceinline__ void rope_sincos(float a, float* sn, float* cs) {
    if (fabsf(a) < 131072.0f) {
        constexpr float kInv2Pi = 0.159154943091895336f;
        constexpr float C1 = 6.28125f, C2 = 1.9353072e-3f, C3 = 1.0253132e-11f;
        const float k = rintf(a * kInv2Pi);
        float r = fmaf(-k, C1, a);
        r = fmaf(-k, C2, r);
        r = fmaf(-k, C3, r);
        __sincosf(r, sn, cs);
    } else {
        sincosf(a, sn, cs);
    }
}

// Dequantised value of a code: code * scale + zero, a binary32 product, then a sum.
__device__ __forceinline__ float dequant(int code, float s, float z) {
    return __fadd_rn(__fmul_rn(static_cast<float>(code), s), z);
}

// One run of a unit's tokens: part 0, whole groups [t0, t1) of the packed records (chunks
// of up to 128 tokens); part 1, window tokens [t0, t1) (chunks of CHR).
template <int D, int BITS>
__device__ int rope_item(const DecodeArgs& a, uint8_t* smem, int b, int h, int64_t slot, int part, int64_t t0,
                         int64_t t1, uint32_t phase) {
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    constexpr int CPL = D / 32;                                       // channels per lane (scores)
    constexpr int HP = CPL / 2;                                       // rotation pairs per lane
    constexpr int CPT = (D + kDecodeThreads - 1) / kDecodeThreads;    // channels per thread (values)
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gqa = lo.gqa, G = lo.G, rec = lo.rec;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* hstat = reinterpret_cast<float*>(smem + so.hstat);       // M[32], L[32], alpha[32]
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    float* sc = reinterpret_cast<float*>(smem + so.sc);              // [head][CH] scores, then p
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);
    const uint8_t* ring = a.cache + lo.ring_off + u * lo.C * (int64_t)(4 * D);
    const int64_t qn = seq_state(a, b).y;                             // window token i is token qn + i
    const int CH = part == 0 ? (G < 128 ? 128 / G : 1) * G : a.plan.CHR;

    load_query(a, b, h, qs);
    if (tid < 32) {
        hstat[tid] = -INFINITY;
        hstat[32 + tid] = 0.0f;
    }
    float o[CPT][8];
#pragma unroll
    for (int x = 0; x < CPT; ++x)
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) o[x][hh] = 0.0f;

    for (int64_t c0 = t0; c0 < t1; c0 += CH) {
        const int cnt = static_cast<int>(t1 - c0 < CH ? t1 - c0 : CH);
        __syncthreads();    // the previous chunk is done with the stage
        if (tid == 0) {
            if (part == 0) {            // whole group records, one copy each (either layout)
                const int ng = cnt / G;
                mbar_arrive_expect_tx(bars, static_cast<uint32_t>(ng * rec));
                for (int r = 0; r < ng; ++r) {
                    const int64_t g = c0 / G + r;
                    int64_t off = group_offset(lo, a.layer, b, h, g);
                    if (off < 0) {      // a table entry outside the pool: read page 0, report it
                        atomicOr(reinterpret_cast<uint32_t*>(a.ws), KVQ_STATUS_BAD_PAGE);
                        off = lo.data_off + (((int64_t)a.layer * lo.H + h) * lo.PG + g % lo.PG) * rec;
                    }
                    bulk_copy_pieces(data + (int64_t)r * rec, a.cache + off, static_cast<uint32_t>(rec), bars);
                }
            } else {                    // window rows, slot (qn + t) mod C
                const int C = lo.C;
                const int s0 = static_cast<int>((qn + c0) % C);
                const int first = cnt < C - s0 ? cnt : C - s0;
                mbar_arrive_expect_tx(bars, static_cast<uint32_t>(cnt) * 4 * D);
                bulk_copy_pieces(data, ring + (int64_t)s0 * 4 * D, static_cast<uint32_t>(first) * 4 * D, bars);
                if (cnt > first)
                    bulk_copy_pieces(data + (int64_t)first * 4 * D, ring, static_cast<uint32_t>(cnt - first) * 4 * D,
                                     bars);
            }
        }
        if (!wait_stage(bars, 0, phase, a.ws)) {
            empty_partial(a, slot);
            return -1;
        }
        // scores: a warp per token; the key is dequantised, turned by its position, dotted
        float hmax[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) hmax[hh] = -INFINITY;
        for (int i = warp; i < cnt; i += 4) {
            float k[CPL];
            if (part == 0) {
                const uint8_t* rp = data + (int64_t)(i / G) * rec;
                const int ig = i % G;
                const uint8_t* kpar = rp + lo.kc + lo.vc;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int c = lane + 32 * j;
                    k[j] = dequant(code_at<BITS>(rp, (ig * D + c) * BITS), half_at(kpar, 2 * c),
                                   half_at(kpar, 2 * D + 2 * c));
                }
                // dense-and-sparse records: a key outlier of this token holds its bf16 value
                // (side entry [e][c]: bf16 bits << 16 | token in the group)
                if (lo.K > 0) {
                    const uint32_t* side = reinterpret_cast<const uint32_t*>(kpar + lo.kp + lo.vp);
                    for (int e = 0; e < lo.K; ++e) {
#pragma unroll
                        for (int j = 0; j < CPL; ++j) {
                            const uint32_t w = side[e * D + lane + 32 * j];
                            if (static_cast<int>(w & 0xffffu) == ig) k[j] = bf16_bits_to_float(static_cast<uint16_t>(w >> 16));
                        }
                    }
                }
            } else {
                const uint16_t* row = reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D);
#pragma unroll
                for (int j = 0; j < CPL; ++j) k[j] = bf16_bits_to_float(row[lane + 32 * j]);
            }
            const float pos = static_cast<float>((part == 0 ? c0 : qn + c0) + i);
#pragma unroll
            for (int j = 0; j < HP; ++j) {
                float sn, cs;
                rope_sincos(__fmul_rn(pos, a.rope_w[lane + 32 * j]), &sn, &cs);
                const float x = k[j], y = k[j + HP];
                k[j] = x * cs - y * sn;
                k[j + HP] = y * cs + x * sn;
            }
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                if (hh >= gqa) break;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < CPL; ++j) acc = fmaf(qs[hh * D + lane + 32 * j], k[j], acc);
                acc = warp_sum(acc);
                if (lane == 0) sc[hh * CH + i] = acc;
                hmax[hh] = fmaxf(hmax[hh], acc);
            }
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
            if (lane == 0 && hh < gqa) red[warp * 32 + hh] = hmax[hh];
        __syncthreads();
        // running max per head, the rescale factor of what came before, p in place
        if (tid < gqa) {
            float m = hstat[tid];
            for (int w = 0; w < 4; ++w) m = fmaxf(m, red[w * 32 + tid]);
            hstat[64 + tid] = hstat[tid] > -INFINITY ? fast_exp2(hstat[tid] - m) : 0.0f;
            hstat[tid] = m;
        }
        __syncthreads();
        for (int hh = 0; hh < gqa; ++hh) {
            const float m = hstat[hh];
            float psum = 0.0f;
            for (int t = tid; t < cnt; t += blockDim.x) {
                const float p = fast_exp2(sc[hh * CH + t] - m);
                sc[hh * CH + t] = p;
                psum += p;
            }
            psum = warp_sum(psum);
            if (lane == 0) red[warp * 32 + hh] = psum;
        }
        __syncthreads();
        if (tid < gqa) {
            float l = 0.0f;
            for (int w = 0; w < 4; ++w) l += red[w * 32 + tid];
            hstat[32 + tid] = fmaf(hstat[32 + tid], hstat[64 + tid], l);
        }
        // values: a thread per channel
#pragma unroll
        for (int x = 0; x < CPT; ++x) {
            const int c = tid + kDecodeThreads * x;
            if (c < D) {
#pragma unroll
                for (int hh = 0; hh < 8; ++hh)
                    if (hh < gqa) o[x][hh] *= hstat[64 + hh];
                const int jv = c / lo.Gv;
                if (part == 0) {
                    // a 16-token tile at a time: the channel's codes of tokens tt and tt + 8
                    // share a word (value_code_bit), the tile's 16 scales (and zeros) are 32
                    // contiguous bytes in the order 2 (tt mod 8) + tt / 8
                    for (int i0 = 0; i0 < cnt; i0 += 16) {
                        const uint8_t* rp = data + (int64_t)(i0 / G) * rec;
                        const int ig0 = i0 % G;
                        const uint8_t* vpar = rp + lo.kc + lo.vc + lo.kp + value_param_byte(G, jv, ig0);
                        const uint4* sp = reinterpret_cast<const uint4*>(vpar);
                        const uint4* zp = reinterpret_cast<const uint4*>(vpar + 2 * G * lo.NGv);
                        const uint4 s0 = sp[0], s1 = sp[1], z0 = zp[0], z1 = zp[1];
                        const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        const uint32_t zw[8] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) {       // tokens tt = e and e + 8
                            const int bit = value_code_bit<D, BITS>(ig0 + e, c);   // low half: token e
                            const uint32_t word = *reinterpret_cast<const uint32_t*>(rp + lo.kc + 4 * (bit >> 5));
                            const int sh = bit & 31;
                            const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&sw[e]));
                            const float2 zf = __half22float2(*reinterpret_cast<const __half2*>(&zw[e]));
                            float v0 = dequant((word >> sh) & ((1u << BITS) - 1u), sf.x, zf.x);
                            float v1 = dequant((word >> (sh + 16)) & ((1u << BITS) - 1u), sf.y, zf.y);
                            if (lo.K > 0) {
                                // value outliers of tokens e and e + 8 (side positions 2e and
                                // 2e + 1 of the tile): index = channel within the value group
                                const uint32_t* side = reinterpret_cast<const uint32_t*>(
                                    rp + lo.kc + lo.vc + lo.kp + lo.vp + lo.ko);
                                const int base = jv * G + ig0 + 2 * e, cg = c - jv * lo.Gv;
                                for (int ee = 0; ee < lo.K; ++ee) {
                                    const uint32_t w0 = side[ee * lo.NGv * G + base];
                                    const uint32_t w1 = side[ee * lo.NGv * G + base + 1];
                                    if (static_cast<int>(w0 & 0xffffu) == cg) v0 = bf16_bits_to_float(static_cast<uint16_t>(w0 >> 16));
                                    if (static_cast<int>(w1 & 0xffffu) == cg) v1 = bf16_bits_to_float(static_cast<uint16_t>(w1 >> 16));
                                }
                            }
#pragma unroll
                            for (int hh = 0; hh < 8; ++hh)
                                if (hh < gqa)
                                    o[x][hh] = fmaf(sc[hh * CH + i0 + e + 8], v1, fmaf(sc[hh * CH + i0 + e], v0, o[x][hh]));
                        }
                    }
                } else {
                    for (int i = 0; i < cnt; ++i) {
                        const float v = bf16_bits_to_float(
                            reinterpret_cast<const uint16_t*>(data + (int64_t)i * 4 * D)[D + c]);
#pragma unroll
                        for (int hh = 0; hh < 8; ++hh)
                            if (hh < gqa) o[x][hh] = fmaf(sc[hh * CH + i], v, o[x][hh]);
                    }
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int x = 0; x < CPT; ++x) {
        const int c = tid + kDecodeThreads * x;
        if (c < D) {
#pragma unroll
            for (int hh = 0; hh < 8; ++hh)
                if (hh < gqa) slot_o(a, slot, hh)[c] = o[x][hh];
        }
    }
    if (tid < gqa) {
        float* ml = slot_ml(a, slot, tid);
        ml[0] = hstat[tid];
        ml[1] = hstat[32 + tid];
    }
    return static_cast<int>(phase);
}

}  // namespace kvq
