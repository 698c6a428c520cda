// kvq_decode.cuh -- single-query decode attention over the packed cache (kernel templates,
// instantiated by the kvq_decode_*.cu translation units).
//
// What is computed ("Quantizing the KV cache", "Why values per token"): for every query
// head, o = sum_t p_t * Vhat_t with p = softmax_t(softmax_scale * q . Khat_t) over all
// cached tokens of the sequence; query head hq reads KV head hq / gqa.
//
// Work split: the grid is one wave of resident blocks.  The layer's work is measured by
// the real token counts in the cache state (the bytes each token reads), and block j takes
// a contiguous 1/NB of it: runs of chunks of one or more (sequence, kv head) units.  For
// every part of a unit it touches (the packed tokens, the rows) a block leaves one partial
// softmax (m, l, o[D]) for all gqa query heads of the kv head, so every cache byte is read
// once per step.  k_merge combines a unit's partials by log-sum-exp.
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
    float rope_w[128];   // keys cached before RoPE: w_i = base^(-2i/D) in binary32, i < D/2
};

// ------------------------------------------------------------------------ scheduling
// Tokens of the two parts of a unit holding n tokens, qn of them packed: part 0 (KIVI
// groups, FP8 tiles) and part 1 (KIVI window, INT8 or INT4 rows).
__host__ __device__ __forceinline__ void unit_parts(const Layout& lo, int64_t n, int64_t qn, int64_t& n0,
                                                    int64_t& n1) {
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        n0 = qn;
        n1 = n - qn;
    } else if (is_fp8(lo.scheme)) {
        n0 = n;
        n1 = 0;
    } else {
        n0 = 0;
        n1 = n;
    }
}

// The scheduling arithmetic below divides by multiplying with binary32 reciprocals made
// on the host (integer division and binary64 arithmetic are long or slow on the GPU).  A
// block boundary or a chunk index may then differ a little from the exact quotient, which
// only moves work between neighbouring blocks: the decode and the merge call these same
// functions with the same arguments, block ranges are nondecreasing in j with
// range_lo(C, 0) = 0 and range_lo(C, nb) = C, and block j's chunks end where block j + 1's
// begin, so every chunk is taken by exactly one block.

// First cost position of block j of nb over a total cost C: about ceil(C j / nb).
__host__ __device__ __forceinline__ int64_t range_lo(int64_t C, int64_t j, int64_t nb, float inv_nb) {
    if (j >= nb) return C;
    const int64_t r = static_cast<int64_t>(ceilf(static_cast<float>(C) * (static_cast<float>(j) * inv_nb)));
    return r < C ? r : C;
}

// Chunks [k_lo, k_hi) of a part whose chunk k starts at cost position base + k * cc (nch
// chunks, inv_cc = 1 / cc) that start inside the block range [lo, hi), up to the rounding
// described above.
__host__ __device__ __forceinline__ void chunks_in(int64_t base, int64_t nch, float inv_cc, int64_t lo, int64_t hi,
                                                   int64_t& k_lo, int64_t& k_hi) {
    k_lo = lo > base ? static_cast<int64_t>(ceilf(static_cast<float>(lo - base) * inv_cc)) : 0;
    k_hi = hi > base ? static_cast<int64_t>(ceilf(static_cast<float>(hi - base) * inv_cc)) : 0;
    if (k_lo > nch) k_lo = nch;
    if (k_hi > nch) k_hi = nch;
}

// floor(N r / k) for chunk counts N < 2^31 and 0 <= r <= k <= 2048 in 32-bit integer
// arithmetic, as (N / k) r + floor((N mod k) r / k) (a 64-bit division is a long
// instruction sequence on the GPU).
__host__ __device__ __forceinline__ int64_t share_lo(int N, int r, int k) {
    const int q = N / k, m = N - q * k;
    return (int64_t)q * r + (m * r) / k;
}

// Tokens n, qn of sequence b in this layer's state.
__device__ __forceinline__ int2 seq_state(const DecodeArgs& a, int b) {
    return *reinterpret_cast<const int2*>(state_ptr(a.lo, a.cache, a.layer, b));
}

// Scheduling costs of one unit's packed part and row part for a sequence with state st.
__device__ __forceinline__ void part_costs(const DecodeArgs& a, int2 st, int64_t& c0, int64_t& c1) {
    int64_t n0, n1;
    unit_parts(a.lo, st.x, st.y, n0, n1);
    c0 = n0 * a.plan.cpt0;
    c1 = n1 * a.plan.cpt1;
}

__device__ __forceinline__ int64_t warp_scan64(int64_t v) {   // inclusive
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Block-wide inclusive scan of one int64 per thread over a tile of kDecodeThreads values;
// returns the thread's inclusive prefix within the tile and sets *tile_total.  Two block
// barriers; `scratch` holds NW int64.
__device__ __forceinline__ int64_t block_scan64(int64_t v, int64_t* scratch, int64_t* tile_total) {
    constexpr int NW = kDecodeThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int64_t inc = warp_scan64(v);
    if (lane == 31) scratch[warp] = inc;
    __syncthreads();
    int64_t woff = 0, tot = 0;
    for (int w = 0; w < NW; ++w) {
        if (w < warp) woff += scratch[w];
        tot += scratch[w];
    }
    __syncthreads();
    *tile_total = tot;
    return inc + woff;
}

// The layer's work in cost order: first the packed parts of every unit (sequence-major,
// then kv head), then the row parts of every unit.  Keeping the two apart means a block
// never interleaves a unit's bf16 window with packed groups.  C0 is the packed total, C
// the whole.  block_range finds this block's range [lo, hi) and the (part, sequence) at
// position lo with the cost P before that sequence in its part; part = 2 when the range
// is empty.  Whole block; `scratch` holds at least 16 int64 of shared memory and `sst` B
// int2 when B <= kDecodeThreads (the sequences' states, kept for the walk).
struct BlockRange {
    int64_t C0, C, lo, hi, P;
    int part, b;
};
__device__ inline BlockRange block_range(const DecodeArgs& a, int64_t* scratch, int2* sst, int blk) {
    const int tid = threadIdx.x;
    const int B = a.lo.B, H = a.lo.H;
    BlockRange r;
    int64_t f0 = 0, f1 = 0, C0 = 0, C1 = 0;
    for (int base = 0; base < B; base += kDecodeThreads) {
        const int b = base + tid;
        int2 st = make_int2(0, 0);
        if (b < B) st = seq_state(a, b);
        if (B <= kDecodeThreads && b < B) sst[b] = st;
        int64_t c0, c1;
        part_costs(a, st, c0, c1);
        c0 *= H;
        c1 *= H;
        if (base == 0) {
            f0 = c0;
            f1 = c1;
        }
        int64_t t0, t1;
        block_scan64(c0, scratch, &t0);
        block_scan64(c1, scratch, &t1);
        C0 += t0;
        C1 += t1;
    }
    r.C0 = C0;
    r.C = C0 + C1;
    r.lo = range_lo(r.C, blk, a.plan.NB, a.plan.inv_nb);
    r.hi = range_lo(r.C, blk + 1, a.plan.NB, a.plan.inv_nb);
    r.part = 2;
    r.b = B;
    r.P = 0;
    if (r.lo >= r.hi) return r;
    // the part holding lo, then the sequence within it
    const int part = r.lo < C0 ? 0 : 1;
    const int64_t pos = part ? r.lo - C0 : r.lo;
    if (tid == 0) scratch[8] = -1;
    int64_t run = 0;
    for (int base = 0; base < B; base += kDecodeThreads) {
        const int b = base + tid;
        int64_t c;
        if (base == 0) {
            c = part ? f1 : f0;
        } else {
            int64_t c0 = 0, c1 = 0;
            if (b < B) part_costs(a, seq_state(a, b), c0, c1);
            c = H * (part ? c1 : c0);
        }
        int64_t tile;
        const int64_t inc = block_scan64(c, scratch, &tile) + run;
        const int64_t exc = inc - c;
        if (c > 0 && exc <= pos && pos < inc) {
            scratch[8] = b;
            scratch[9] = exc;
        }
        __syncthreads();
        const int64_t found = scratch[8];
        __syncthreads();
        if (found >= 0) {
            r.part = part;
            r.b = static_cast<int>(found);
            r.P = scratch[9];
            break;
        }
        run += tile;
    }
    __syncthreads();
    return r;
}

// The unit-aligned split, used when the batch has at most half as many units as the grid
// has blocks.  A unit of cost U > 0 gets k = 1 + floor(U NB' / C) whole blocks (NB' = NB
// minus the number of non-empty units, so that sum k <= NB), units in order (sequence-
// major, then kv head) on consecutive blocks.  The unit's N chunks (packed part, then rows)
// are shared by count: block r of k takes chunks [N r / k, N (r + 1) / k), so that no
// block holds a chunk more than another (a cost split can give one block three chunk
// starts where the next gets two).  No
// block then spans two units, and block j's partial results go to slots 2 j + part.  (The
// cost-range slots j + part B H + unit would collide here: a unit's rows can end on a
// block a few blocks before the next unit's packed part begins.)  unit_plan finds this
// block's unit (b = B when it has none) and r, k.
struct UnitPlan {
    int b, h, r, k;
    int64_t n0, n1;
};
// 1 + floor(U nbp / C) in binary32, scaled down by 1e-6 so that the rounding never makes it
// exceed the exact value (the error of the few binary32 operations is below 3e-7): the
// sum over the units then stays within NB.
__device__ __forceinline__ int unit_blocks(int64_t U, int64_t C, int64_t nbp) {
    if (U <= 0) return 0;
    const float x = static_cast<float>(U) * (static_cast<float>(nbp) / static_cast<float>(C)) * 0.999999f;
    return 1 + static_cast<int>(x);
}
__device__ inline UnitPlan unit_plan(const DecodeArgs& a, int64_t* scratch, int2* sst, int blk) {
    const int tid = threadIdx.x;
    const int B = a.lo.B, H = a.lo.H;
    UnitPlan up;
    up.b = B;
    if (B <= 32) {
        // one warp, a sequence per lane, one block barrier
        if (tid < 32) {
            const int b = tid;
            int2 st = make_int2(0, 0);
            if (b < B) st = seq_state(a, b);
            sst[b] = st;
            int64_t c0, c1;
            part_costs(a, st, c0, c1);
            const int64_t U = b < B ? c0 + c1 : 0;
            int64_t C = H * U, live = U > 0 ? H : 0;
            for (int o = 16; o > 0; o >>= 1) {
                C += __shfl_xor_sync(0xffffffffu, C, o);
                live += __shfl_xor_sync(0xffffffffu, live, o);
            }
            const int64_t nbp = a.plan.NB - live;
            const int k = C > 0 ? unit_blocks(U, C, nbp) : 0;
            const int64_t inc = warp_scan64((int64_t)H * k), exc = inc - (int64_t)H * k;
            const bool mine = k > 0 && exc <= blk && blk < inc;
            const unsigned m = __ballot_sync(0xffffffffu, mine);
            if (tid == 0) scratch[8] = m ? static_cast<int64_t>(__ffs(m) - 1) : -1;
            if (mine) {
                scratch[9] = exc;
                scratch[10] = k;
            }
        }
        __syncthreads();
        const int64_t found = scratch[8];
        if (found >= 0) {
            up.b = static_cast<int>(found);
            up.k = static_cast<int>(scratch[10]);
            const int off = blk - static_cast<int>(scratch[9]);
            up.h = off / up.k;
            up.r = off - up.h * up.k;
            const int2 st = sst[up.b];
            unit_parts(a.lo, st.x, st.y, up.n0, up.n1);
        }
        return up;
    }
    int64_t C = 0, live = 0, fU = 0;
    for (int base = 0; base < B; base += kDecodeThreads) {
        const int b = base + tid;
        int2 st = make_int2(0, 0);
        if (b < B) st = seq_state(a, b);
        if (B <= kDecodeThreads && b < B) sst[b] = st;
        int64_t c0, c1;
        part_costs(a, st, c0, c1);
        if (base == 0) fU = c0 + c1;
        int64_t t0, t1;
        block_scan64(H * (c0 + c1), scratch, &t0);
        block_scan64(c0 + c1 > 0 ? H : 0, scratch, &t1);
        C += t0;
        live += t1;
    }
    if (C == 0) return up;
    const int64_t nbp = a.plan.NB - live;
    int64_t run = 0;
    if (tid == 0) scratch[8] = -1;
    for (int base = 0; base < B; base += kDecodeThreads) {
        const int b = base + tid;
        int64_t U = fU;
        if (base != 0 || B > kDecodeThreads) {
            int64_t c0 = 0, c1 = 0;
            if (b < B) part_costs(a, B <= kDecodeThreads ? sst[b] : seq_state(a, b), c0, c1);
            U = c0 + c1;
        }
        if (b >= B) U = 0;
        const int k = unit_blocks(U, C, nbp);
        int64_t tile;
        const int64_t inc = block_scan64((int64_t)H * k, scratch, &tile) + run;
        const int64_t exc = inc - (int64_t)H * k;
        if (k > 0 && exc <= blk && blk < inc) {
            scratch[8] = b;
            scratch[9] = exc;
            scratch[10] = k;
        }
        __syncthreads();
        const int64_t found = scratch[8];
        if (found >= 0) break;
        run += tile;
        __syncthreads();
    }
    __syncthreads();
    const int64_t found = scratch[8];
    if (found >= 0) {
        up.b = static_cast<int>(found);
        up.k = static_cast<int>(scratch[10]);
        const int off = blk - static_cast<int>(scratch[9]);
        up.h = off / up.k;
        up.r = off - up.h * up.k;
        const int2 st = B <= kDecodeThreads ? sst[up.b] : seq_state(a, up.b);
        unit_parts(a.lo, st.x, st.y, up.n0, up.n1);
    }
    __syncthreads();
    return up;
}

// Chunks taken on demand (the unit-aligned split of the KIVI kernels, plan.steal, for a
// unit with at least 4 packed chunks per block): the k blocks of the unit share its packed
// chunks through a counter in the workspace instead of a fixed split, so blocks that run
// faster (or hold no window rows) take more chunks and the unit's blocks finish together.
// The window's row chunks go, by count, to the last kw = min(nc1, max(k - 1, 1)) blocks,
// which take them first; each of the other nw = k - kw blocks r starts with the fixed
// chunks r + s nw (s < NSTAGE), so no block waits on the counter before its first copy;
// every further chunk is NSTAGE nw + an atomic increment of the unit's counter (the merge
// sets it back to zero).  on == 0: the chunks of [t0, t1) in order.
struct StealCtx {
    int on, r, nw;
    int* ctr;
};
__device__ __forceinline__ bool unit_steals(const DecodePlan& p, int64_t n0, int k) {
    return p.steal && n0 > (4 * (int64_t)k - 1) * p.CH;   // ceil(n0 / CH) >= 4 k
}
__device__ __forceinline__ int window_blocks(const DecodePlan& p, int64_t n1, int k) {
    const int nc1 = (static_cast<int>(n1) + p.CHR - 1) / p.CHR;
    return nc1 == 0 ? 0 : min(nc1, max(k - 1, 1));
}

// Calls fn(part, b, h, slot, t0, t1, steal) for every run of chunks of one part of one
// unit that this block takes, in cost order (whole block, uniform).  The run's partial
// result goes to slot j + part * B H + unit: unique, because block ranges are contiguous in
// cost order (slot 2 j + part in the unit-aligned split).  fn returns false once the block
// cannot go on (a bounded wait gave up); the remaining runs then get empty partials via
// dead(slot).  STEAL: the kernel variant that may share a unit's chunks on demand.
template <bool STEAL, typename F, typename E>
__device__ void for_each_segment(const DecodeArgs& a, int64_t* scratch, int2* sst, F&& fn, E&& dead) {
    const Layout& lo = a.lo;
    const int64_t units = (int64_t)lo.B * lo.H;
    StealCtx none;
    none.on = 0;
    none.r = none.nw = 0;
    none.ctr = nullptr;
    if (a.plan.unit_aligned) {
        const UnitPlan up = unit_plan(a, scratch, sst, blockIdx.x);
        grid_launch_dependents();   // the merge may start its own planning; it waits for this grid
        if (up.b >= lo.B) return;
        if (STEAL && unit_steals(a.plan, up.n0, up.k)) {
            // slot 2 j + 1 only on the kw window blocks, slot 2 j on every block
            const int nc1 = (static_cast<int>(up.n1) + a.plan.CHR - 1) / a.plan.CHR;
            const int kw = window_blocks(a.plan, up.n1, up.k);
            const int w = up.r - (up.k - kw);
            const int64_t slot0 = 2 * (int64_t)blockIdx.x, slot1 = slot0 + 1;
            bool go = true;
            if (w >= 0) {
                const int64_t t0 = (int64_t)a.plan.CHR * (nc1 * w / kw);
                const int64_t t1e = (int64_t)a.plan.CHR * (nc1 * (w + 1) / kw);
                __syncthreads();
                go = fn(1, up.b, up.h, slot1, t0, t1e < up.n1 ? t1e : up.n1, none);
            }
            StealCtx sc;
            sc.on = 1;
            sc.r = up.r;
            sc.nw = up.k - kw;
            sc.ctr = reinterpret_cast<int*>(a.ws + a.plan.ws_ctr_off) + (up.b * lo.H + up.h);
            __syncthreads();   // the window run is done with shared memory
            if (go && up.n0 > 0)
                fn(0, up.b, up.h, slot0, 0, up.n0, sc);
            else
                dead(slot0);
            return;
        }
        const int64_t nc0 = (static_cast<int>(up.n0) + a.plan.CH - 1) / a.plan.CH;
        const int64_t nc1 = (static_cast<int>(up.n1) + a.plan.CHR - 1) / a.plan.CHR;
        const int N = static_cast<int>(nc0 + nc1);
        const int64_t clo = share_lo(N, up.r, up.k), chi = share_lo(N, up.r + 1, up.k);
        bool go = true;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int64_t nt = part ? up.n1 : up.n0, gs = part ? a.plan.CHR : a.plan.CH;
            if (nt > 0) {
                const int64_t off = part ? nc0 : 0, nch = part ? nc1 : nc0;
                int64_t k_lo = clo - off, k_hi = chi - off;
                k_lo = k_lo < 0 ? 0 : (k_lo > nch ? nch : k_lo);
                k_hi = k_hi < 0 ? 0 : (k_hi > nch ? nch : k_hi);
                if (k_lo < k_hi) {
                    const int64_t slot = 2 * (int64_t)blockIdx.x + part;   // one unit per block
                    const int64_t t1 = k_hi * gs < nt ? k_hi * gs : nt;
                    __syncthreads();   // the previous run is done with shared memory
                    if (go)
                        go = fn(part, up.b, up.h, slot, k_lo * gs, t1, none);
                    else
                        dead(slot);
                }
            }
        }
        return;
    }
    const BlockRange r = block_range(a, scratch, sst, blockIdx.x);
    grid_launch_dependents();   // the merge may start its own planning; it waits for this grid
    bool live = true;
    for (int part = r.part; part < 2; ++part) {
        const int64_t gs = part ? a.plan.CHR : a.plan.CH, cpt = part ? a.plan.cpt1 : a.plan.cpt0;
        const float inv_cc = part ? a.plan.inv_cc1 : a.plan.inv_cc0;
        // cost position of the part's first sequence considered, in the whole order
        int64_t P = (part ? r.C0 : 0) + (part == r.part ? r.P : 0);
        if (P >= r.hi) break;
        for (int b = part == r.part ? r.b : 0; b < lo.B && P < r.hi; ++b) {
            const int2 st = lo.B <= kDecodeThreads ? sst[b] : seq_state(a, b);
            int64_t n0, n1;
            unit_parts(lo, st.x, st.y, n0, n1);
            const int64_t nt = part ? n1 : n0;
            const int64_t U = nt * cpt;
            if (U == 0) continue;
            // the first head whose cost range reaches lo (a reciprocal estimate, made exact)
            int h0 = 0;
            if (r.lo > P) {
                h0 = static_cast<int>(static_cast<float>(r.lo - P) / static_cast<float>(U));
                h0 = h0 < 0 ? 0 : (h0 > lo.H - 1 ? lo.H - 1 : h0);
                while (h0 > 0 && P + h0 * U > r.lo) --h0;
                while (h0 + 1 < lo.H && P + (h0 + 1) * U <= r.lo) ++h0;
            }
            for (int h = h0; h < lo.H && P + h * U < r.hi; ++h) {
                int64_t k_lo, k_hi;
                chunks_in(P + h * U, (nt + gs - 1) / gs, inv_cc, r.lo, r.hi, k_lo, k_hi);
                if (k_lo < k_hi) {
                    const int64_t slot = blockIdx.x + part * units + (int64_t)b * lo.H + h;
                    const int64_t t1 = k_hi * gs < nt ? k_hi * gs : nt;
                    __syncthreads();   // the previous run is done with shared memory
                    if (live)
                        live = fn(part, b, h, slot, k_lo * gs, t1, none);
                    else
                        dead(slot);
                }
            }
            P += (int64_t)lo.H * U;
        }
    }
}

// The layer's totals and one sequence's prefixes, as the decode's split uses them: C0 the
// packed total, C the whole, P0 and P1 the packed and row costs of the sequences before
// b (cost-range split); live the non-empty units and K the first block of sequence b
// (unit-aligned split).
struct SplitCtx {
    int64_t C0, C, P0, P1, live, K;
};

// The partial-result slots of unit u (sequence b = u / H, kv head h = u % H, state st):
// the decode blocks that may have taken chunks of the unit, by the same arithmetic as the
// decode's split; cand[i] is the block's slot, or -1 when the block took no chunk of the
// unit (in the cost-range split the range is widened by two blocks on each side for the
// rounding of that arithmetic).  Written by the block's `nthreads` threads (no barrier);
// returns the list's length (at most 2 KVQ_MAX_DECODE_BLOCKS).
__device__ inline int unit_candidates(const DecodeArgs& a, int u, int2 st, const SplitCtx& x, int* cand,
                                      int nthreads) {
    const Layout& lo = a.lo;
    const int h = u % lo.H;
    const int tid = threadIdx.x;
    const int64_t units = (int64_t)lo.B * lo.H;
    const int NB = a.plan.NB;
    int64_t n0, n1;
    unit_parts(lo, st.x, st.y, n0, n1);
    int total = 0;
    if (a.plan.unit_aligned) {
        // the unit's k blocks from K + h k; block r takes chunks starting in its share
        const int64_t U = n0 * a.plan.cpt0 + n1 * a.plan.cpt1;
        const int k = x.C > 0 ? unit_blocks(U, x.C, NB - x.live) : 0;
        const int64_t K = x.K + (int64_t)h * k;
        if (unit_steals(a.plan, n0, k)) {   // slot 2 j of every block, 2 j + 1 of the window blocks
            const int kw = window_blocks(a.plan, n1, k);
            for (int i = tid; i < k + kw; i += nthreads)
                cand[i] = i < k ? static_cast<int>(2 * (K + i)) : static_cast<int>(2 * (K + k - kw + (i - k)) + 1);
            return k + kw;
        }
        const int64_t nc0 = (static_cast<int>(n0) + a.plan.CH - 1) / a.plan.CH;
        const int64_t nc1 = (static_cast<int>(n1) + a.plan.CHR - 1) / a.plan.CHR;
        const int N = static_cast<int>(nc0 + nc1);
        for (int i = tid; i < 2 * k; i += nthreads) {
            const int part = i / k, r = i - part * k;
            const int64_t clo = share_lo(N, r, k), chi = share_lo(N, r + 1, k);
            const int64_t lo_c = part ? nc0 : 0, hi_c = part ? N : nc0;
            const bool any = (clo > lo_c ? clo : lo_c) < (chi < hi_c ? chi : hi_c);
            cand[i] = any ? static_cast<int>(2 * (K + r) + part) : -1;
        }
        return 2 * k;
    }
    const int64_t C0 = x.C0, C = x.C;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        const int64_t nt = part ? n1 : n0, gs = part ? a.plan.CHR : a.plan.CH;
        const int64_t cpt = part ? a.plan.cpt1 : a.plan.cpt0;
        if (nt > 0 && C > 0) {
            const int64_t base = (part ? C0 + x.P1 : x.P0) + (int64_t)h * nt * cpt;
            const int64_t nch = (nt + gs - 1) / gs;
            const float inv_cc = part ? a.plan.inv_cc1 : a.plan.inv_cc0;
            const float per = static_cast<float>(NB) / static_cast<float>(C);
            int j0 = static_cast<int>(static_cast<float>(base) * per) - 2;
            int j1 = static_cast<int>(static_cast<float>(base + (nch - 1) * gs * cpt) * per) + 2;
            j0 = j0 < 0 ? 0 : j0;
            j1 = j1 > NB - 1 ? NB - 1 : j1;
            const int count = j1 - j0 + 1;
            for (int i = tid; i < count; i += nthreads) {
                const int j = j0 + i;
                int64_t k_lo, k_hi;
                chunks_in(base, nch, inv_cc, range_lo(C, j, NB, a.plan.inv_nb), range_lo(C, j + 1, NB, a.plan.inv_nb),
                          k_lo, k_hi);
                cand[total + i] = k_lo < k_hi ? static_cast<int>(j + part * units + u) : -1;
            }
            total += count;
        }
    }
    return total;
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

// Staging barriers: bit s of `phase` is the parity the next completion of barrier s
// carries (items take the bits and return them updated, or -1 once a wait gave up).  All
// threads wait; on a timeout the decode status gets KVQ_STATUS_TIMEOUT, the block waits
// once more (bounded) for the copy and false is returned.  With kSelfTestBit set in
// `phase` (the workspace self-test, see kvq_decode_attention) the wait is made on a
// barrier that nothing completes, so it gives up, and the real copy is then waited for.
__device__ __forceinline__ bool wait_stage(uint64_t* bars, int s, uint32_t& phase, uint8_t* ws) {
    const uint32_t par = (phase >> s) & 1u;
    bool ok = mbar_wait_bounded(bars + ((phase & kSelfTestBit) ? kSelfTestBar : s), par, kWaitLimitNs);
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (threadIdx.x == 0) atomicOr(reinterpret_cast<uint32_t*>(ws), KVQ_STATUS_TIMEOUT);
        mbar_wait_bounded(bars + s, par, kWaitLimitNs);
        return false;
    }
    phase ^= 1u << s;
    return true;
}
// After a timeout: a bounded wait for a copy still armed on barrier s.
__device__ __forceinline__ void drain_stage(uint64_t* bars, int s, uint32_t phase) {
    mbar_wait_bounded(bars + s, (phase >> s) & 1u, kWaitLimitNs);
}

// The workspace self-test word (bytes 8..15 of the workspace header).
__device__ __forceinline__ uint32_t selftest_bits(const DecodeArgs& a) {
    return *reinterpret_cast<const unsigned long long*>(a.ws + 8) == KVQ_SELFTEST_WAIT_MAGIC ? kSelfTestBit : 0u;
}

// Partial-result slots of the workspace: slot * gqa + head.
__device__ __forceinline__ float* slot_o(const DecodeArgs& a, int64_t slot, int head) {
    return reinterpret_cast<float*>(a.ws + a.plan.ws_o_off) + (slot * a.lo.gqa + head) * a.lo.D;
}
__device__ __forceinline__ float* slot_ml(const DecodeArgs& a, int64_t slot, int head) {
    return reinterpret_cast<float*>(a.ws + a.plan.ws_ml_off) + 2 * (slot * a.lo.gqa + head);
}

// An empty partial: m = -inf, l = 0, so the merge gives it weight 0.
__device__ __forceinline__ void empty_partial(const DecodeArgs& a, int64_t slot) {
    if (threadIdx.x < a.lo.gqa) {
        float* ml = slot_ml(a, slot, threadIdx.x);
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

}  // namespace kvq

#include "kvq_rope.cuh"

namespace kvq {

// ------------------------------------------------------------------------ row path (INT8, INT4)
// Per-token rows, CHR tokens per chunk: a warp per token for the scores, a thread per
// channel for the values, and a running softmax (per-head max M and sum L in shared memory,
// per-thread outputs in registers) across the chunks of the run.  INT4 rows hold two
// channels per byte (even channel in the low four bits, two's complement).
template <int D>
__device__ __forceinline__ int rows_item(const DecodeArgs& a, uint8_t* smem, int b, int h, int64_t slot, int64_t t0,
                                      int64_t t1, uint32_t phase) {
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    constexpr int CPL = (D + 31) / 32;              // channels per lane (scores)
    constexpr int CPT = (D + kDecodeThreads - 1) / kDecodeThreads;   // channels per thread (values)
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int CHR = a.plan.CHR, gqa = lo.gqa;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* hstat = reinterpret_cast<float*>(smem + so.hstat);    // M[32], L[32], alpha[32]
    float* qs = reinterpret_cast<float*>(smem + so.qs);
    float* sc = reinterpret_cast<float*>(smem + so.sc);
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);
    const uint8_t* unit = a.cache + lo.data_off + u * lo.unit;
    const bool int4 = lo.scheme == KVQ_SCHEME_INT4;
    const int RB = int4 ? D / 2 : D;                 // code bytes per row

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

    for (int64_t c0 = t0; c0 < t1; c0 += CHR) {
        const int cnt = static_cast<int>(t1 - c0 < CHR ? t1 - c0 : CHR);
        __syncthreads();    // the previous chunk is done with the stage
        if (tid == 0) {
            const uint32_t cb = static_cast<uint32_t>(cnt) * RB;
            const uint32_t sb = static_cast<uint32_t>((cnt + 3) / 4 * 4) * 4;
            mbar_arrive_expect_tx(bars, 2 * cb + 2 * sb);
            bulk_copy_pieces(data, unit + c0 * RB, cb, bars);
            bulk_copy_pieces(data + (int64_t)CHR * D, unit + (int64_t)lo.T16 * RB + c0 * RB, cb, bars);
            const uint8_t* scales = unit + 2 * (int64_t)lo.T16 * RB;
            bulk_copy_pieces(data + 2 * (int64_t)CHR * D, scales + 4 * c0, sb, bars);
            bulk_copy_pieces(data + 2 * (int64_t)CHR * D + 4 * CHR, scales + 4 * (int64_t)lo.T16 + 4 * c0, sb, bars);
        }
        if (!wait_stage(bars, 0, phase, a.ws)) {
            empty_partial(a, slot);
            return -1;
        }
        const int8_t* kc = reinterpret_cast<const int8_t*>(data);
        const int8_t* vc = reinterpret_cast<const int8_t*>(data + (int64_t)CHR * D);
        const float* ks = reinterpret_cast<const float*>(data + 2 * (int64_t)CHR * D);
        const float* vs = ks + CHR;
        // the integer code of channel c of row i (a sign-extended nibble for INT4)
        auto code = [&](const int8_t* rows, int i, int c) -> int {
            if (!int4) return rows[i * D + c];
            const uint32_t byte = static_cast<uint8_t>(rows[i * (D / 2) + c / 2]);
            return static_cast<int>(byte << ((c & 1) ? 24 : 28)) >> 28;
        };
        // scores: a warp per token, lanes over channels, one reduction per head
        float hmax[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) hmax[hh] = -INFINITY;
        for (int i = warp; i < cnt; i += 4) {
            float kv[CPL];
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int c = lane + 32 * j;
                kv[j] = c < D ? static_cast<float>(code(kc, i, c)) * ks[i] : 0.0f;
            }
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                if (hh >= gqa) break;
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < CPL; ++j) {
                    const int c = lane + 32 * j;
                    if (c < D) acc = fmaf(qs[hh * D + c], kv[j], acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) sc[hh * CHR + i] = acc;
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
            float part = 0.0f;
            for (int t = tid; t < cnt; t += blockDim.x) {
                const float p = fast_exp2(sc[hh * CHR + t] - m);
                sc[hh * CHR + t] = p;
                part += p;
            }
            part = warp_sum(part);
            if (lane == 0) red[warp * 32 + hh] = part;
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
                for (int i = 0; i < cnt; ++i) {
                    const float v = static_cast<float>(code(vc, i, c)) * vs[i];
#pragma unroll
                    for (int hh = 0; hh < 8; ++hh)
                        if (hh < gqa) o[x][hh] = fmaf(sc[hh * CHR + i], v, o[x][hh]);
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

// Combine the 4 warps' partials of one run (comb[warp][head][D] = o, cml[warp][head] =
// (m, l)) into the workspace slot.  Called by the whole block after a barrier.  A warp
// without tokens leaves m = -inf, l = 0 and its o unwritten; it gets weight 0 and its o is
// never read.
template <int D>
__device__ __forceinline__ void combine_warps(const DecodeArgs& a, const float* comb, const float* cml,
                                              float* red, int64_t slot) {
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
        float* ml = slot_ml(a, slot, tid);
        ml[0] = M;
        ml[1] = l;
    }
    __syncthreads();
    // the slot's gqa heads are consecutive: gqa * D floats, four per thread and step
    float4* wso = reinterpret_cast<float4*>(slot_o(a, slot, 0));
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
// The bf16 window of a KIVI cache, CHR = 64 tokens per chunk.  Keys and queries are exact
// bf16 values, so the scores go straight to the tensor cores (no conversion, no operand
// split): rows = 16 tokens, columns = up to 8 query heads.  Each warp takes one 16-token
// tile of every chunk and keeps its own running softmax (max and sum per head, rescaled
// output); P.V runs on the tensor cores too, with V^T fragments read from the
// token-major rows by ldmatrix.trans and p split into bf16 major and minor parts.  The
// block then combines its 4 warps.
template <int D, int NT>
__device__ __forceinline__ int window_item(const DecodeArgs& a, uint8_t* smem, int b, int h, int64_t slot,
                                        int64_t t0, int64_t t1, uint32_t phase) {
    const SmemOffsets so = decode_smem(a.lo, a.plan);
    constexpr int KSTEPS = D / 16;
    constexpr int MTV = D / 16;
    const Layout& lo = a.lo;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
    const int gqa = lo.gqa, CHR = a.plan.CHR;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + so.bar);
    float* red = reinterpret_cast<float*>(smem + so.red);
    float* comb = reinterpret_cast<float*>(smem + so.sc);       // [warp][head][D]
    float* cml = comb + 4 * gqa * D;                            // [warp][head][m, l]
    float* pw = reinterpret_cast<float*>(smem + so.pw);         // [warp][16 tokens][8 heads]
    uint8_t* data = smem + so.data;
    const int64_t u = unit_index(lo, a.layer, b, h);
    const uint8_t* ring = a.cache + lo.ring_off + u * lo.C * (int64_t)(4 * D);
    // the window's tokens follow the packed ones: part-1 token i is absolute token qn + i
    const int64_t qn = seq_state(a, b).y;

    // query operand: column g = head g (zero beyond gqa), k = channel pairs (2t, 2t+1) and
    // (2t+8, 2t+9) of each 16-channel step: the caller's bf16 query rows, staged once in
    // shared memory (rows gqa..7 zero) and read per tile
    uint32_t* qw = reinterpret_cast<uint32_t*>(smem + so.qs);   // [8 heads][D / 2] words
    {
        const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(
            reinterpret_cast<const uint16_t*>(a.q) + ((int64_t)b * lo.Hq + (int64_t)h * gqa) * D);
        for (int i = tid; i < 8 * D / 2; i += blockDim.x) qw[i] = i < gqa * D / 2 ? qsrc[i] : 0u;
    }
    const uint32_t qlane = smem_addr(qw) + (g * (D / 2) + tig) * 4;
    float oacc[MTV][NT][4];
#pragma unroll
    for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.0f;
    // running max of heads 2 tig, 2 tig + 1 (the lane's score columns) and the lane's
    // partial sums of their p
    float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
    for (int64_t c0 = t0; c0 < t1; c0 += CHR) {
        const int cnt = static_cast<int>(t1 - c0 < CHR ? t1 - c0 : CHR);
        __syncthreads();    // the previous chunk is done with the stage
        if (tid == 0) {
            const int C = lo.C;
            const int s0 = static_cast<int>((qn + c0) % C);
            const int first = cnt < C - s0 ? cnt : C - s0;
            mbar_arrive_expect_tx(bars, static_cast<uint32_t>(cnt) * 4 * D);
            bulk_copy_pieces(data, ring + (int64_t)s0 * 4 * D, static_cast<uint32_t>(first) * 4 * D, bars);
            if (cnt > first)
                bulk_copy_pieces(data + (int64_t)first * 4 * D, ring, static_cast<uint32_t>(cnt - first) * 4 * D, bars);
        }
        if (!wait_stage(bars, 0, phase, a.ws)) {
            empty_partial(a, slot);
            return -1;
        }
        const int tok0 = 16 * warp;
        const int ntok = cnt - tok0 < 0 ? 0 : (cnt - tok0 > 16 ? 16 : cnt - tok0);
        if (ntok > 0) {
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
                mma_16816_bf16(acc, af, lds32(qlane + 32 * ks), lds32(qlane + 32 * ks + 16));
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
            // new running maxima (finite: the tile has a token) and the factors that
            // rescale what the warp accumulated before
            const float MA = fmaxf(mA, m0), MB = fmaxf(mB, m1);
            const float aA = mA > -INFINITY ? fast_exp2(mA - MA) : 0.0f;
            const float aB = mB > -INFINITY ? fast_exp2(mB - MB) : 0.0f;
            mA = MA;
            mB = MB;
            float* pt = pw + warp * 16 * 8;
            const float p00 = v0 ? fast_exp2(sc[0][0] - MA) : 0.0f, p01 = v0 ? fast_exp2(sc[0][1] - MB) : 0.0f;
            const float p10 = v1 ? fast_exp2(sc[1][0] - MA) : 0.0f, p11 = v1 ? fast_exp2(sc[1][1] - MB) : 0.0f;
            pt[g * 8 + 2 * tig] = p00;
            pt[g * 8 + 2 * tig + 1] = p01;
            pt[(g + 8) * 8 + 2 * tig] = p10;
            pt[(g + 8) * 8 + 2 * tig + 1] = p11;
            lA = fmaf(lA, aA, p00 + p10);
            lB = fmaf(lB, aB, p01 + p11);
            // the value accumulators of lane (g, t) hold head 4 nt + t: its factor comes
            // from lane (4 nt + t) / 2 of the score layout
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hv = 4 * nt + tig;
                const float xa = __shfl_sync(0xffffffffu, aA, hv >> 1);
                const float xb = __shfl_sync(0xffffffffu, aB, hv >> 1);
                const float f = (hv & 1) ? xb : xa;
#pragma unroll
                for (int mt = 0; mt < MTV; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) oacc[mt][nt][e] *= f;
            }
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
    }
    // warp partial into shared memory, then the 4 warps combined
    float* cw = comb + warp * gqa * D;
    const bool wlive = mA > -INFINITY;
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
    // lane hh (< gqa) keeps head hh's max and sum: heads 2t, 2t+1 live in lanes t
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        lA += __shfl_xor_sync(0xffffffffu, lA, off);
        lB += __shfl_xor_sync(0xffffffffu, lB, off);
    }
    const int src = (lane < 8 ? lane : 0) >> 1;
    const float mm0 = __shfl_sync(0xffffffffu, mA, src), mm1 = __shfl_sync(0xffffffffu, mB, src);
    const float ll0 = __shfl_sync(0xffffffffu, lA, src), ll1 = __shfl_sync(0xffffffffu, lB, src);
    if (lane < gqa) {
        cml[2 * (warp * gqa + lane)] = wlive ? ((lane & 1) ? mm1 : mm0) : -INFINITY;
        cml[2 * (warp * gqa + lane) + 1] = wlive ? ((lane & 1) ? ll1 : ll0) : 0.0f;
    }
    __syncthreads();
    combine_warps<D>(a, comb, cml, red, slot);
    return static_cast<int>(phase);
}

// ------------------------------------------------------------------------ packed path
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

// Keys cached before RoPE: the BITS-bit codes of channels c0, c0 + 1, c0 + 8, c0 + 9 (c0 =
// 16 p + 2 t, t < 4) of one token-major key row: one 32-bit word (2-bit), two (4-bit) or
// two 16-bit loads (8-bit).
template <int BITS>
__device__ __forceinline__ void row_codes4(const uint8_t* row, int c0, int (&q)[4]) {
    constexpr int M = (1 << BITS) - 1;
    if constexpr (BITS == 2) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(row + 4 * (c0 >> 4));
        const int sh = 2 * (c0 & 15);
        q[0] = (w >> sh) & M;
        q[1] = (w >> (sh + 2)) & M;
        q[2] = (w >> (sh + 16)) & M;
        q[3] = (w >> (sh + 18)) & M;
    } else if constexpr (BITS == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(row + 8 * (c0 >> 4));
        const int sh = 4 * (c0 & 7);
        q[0] = (w.x >> sh) & M;
        q[1] = (w.x >> (sh + 4)) & M;
        q[2] = (w.y >> sh) & M;
        q[3] = (w.y >> (sh + 4)) & M;
    } else {
        const uint32_t lo = *reinterpret_cast<const uint16_t*>(row + c0);
        const uint32_t hi = *reinterpret_cast<const uint16_t*>(row + c0 + 8);
        q[0] = lo & M;
        q[1] = lo >> 8;
        q[2] = hi & M;
        q[3] = hi >> 8;
    }
}
// Two binary32 values as fp16 pairs: the rounded values, and the rounded remainders.
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& major, uint32_t& minor) {
    const __half2 m = __floats2half2_rn(x, y);
    const float2 f = __half22float2(m);
    major = h2_as_u32(m);
    minor = h2_as_u32(__floats2half2_rn(x - f.x, y - f.y));
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
//
// ROPE (keys cached before the rotary embedding): the key pass dequantises each tile's keys
// in binary32 (code * s + z), turns every channel pair (c, c + D/2) by its token's angle,
// and scores the turned keys on the tensor cores: A = the keys times 2^(14 - e) (e from the
// group's largest possible |key|, so that no fp16 part overflows) as fp16 major + minor
// parts, B = the query in natural channel order (major and minor in the columns of each
// head).  Lane (g, t) holds, for k-steps p and p + D/32, the channels 16 p + 2 t + {0, 1, 8,
// 9} and their partners, so each rotation pair stays in one lane.  The values and the
// softmax are those of the other keys.
template <int D, int BITS, int NT, bool STEAL, bool PAGED, bool SPARSE, bool ROPE = false>
__device__ __forceinline__ int packed_item(const DecodeArgs& a, uint8_t* smem, int b, int h, int64_t slot,
                                        int64_t t0, int64_t t1, uint32_t phase, const StealCtx& sc) {
    const SmemOffsets so = decode_smem(a.lo, a.plan);
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

    // the item's groups (t0 and t1 are group boundaries): chunk c holds gpc of them
    const int gpc = CH / G;
    const uint8_t* src_groups = src_unit + (int64_t)(static_cast<int>(t0) / G) * rec;
    const int ngroups = ntok / G;
    auto issue = [&](int c, int sj) {       // stage chunk c into stage sj (thread 0 only)
        const int gj = min(gpc, ngroups - c * gpc);
        const uint32_t bytes = static_cast<uint32_t>(gj) * rec;
        uint64_t* bar = bars + sj;
        uint8_t* dst = smem + so.data + sj * stage_bytes;
        mbar_arrive_expect_tx(bar, bytes);
        if constexpr (!PAGED) {
            bulk_copy_pieces(dst, src_groups + (int64_t)c * gpc * rec, bytes, bar);
        } else {
            // paged layout: one copy per run of the chunk's groups that shares a page.  The
            // item's sequence, kv head and first group come back from shared memory (kept
            // there so that they hold no registers through the chunk loop).
            const int* pi = reinterpret_cast<const int*>(smem + so.hstat) + 16;
            const int pb = pi[0], ph = pi[1];
            int g = pi[2] + c * gpc;
            for (int x = 0; x < gj;) {
                const int pg = g / lo.PG, slot = g - pg * lo.PG;
                const int run = min(lo.PG - slot, gj - x);
                int p = lo.table[(int64_t)pb * lo.MP + pg];
                if (p < 0 || p >= lo.NP) {   // a table entry outside the pool: read page 0, report it
                    atomicOr(reinterpret_cast<uint32_t*>(a.ws), KVQ_STATUS_BAD_PAGE);
                    p = 0;
                }
                const int64_t off = lo.data_off + (int64_t)p * lo.page + (((int64_t)a.layer * lo.H + ph) * lo.PG + slot) * rec;
                bulk_copy_pieces(dst + (int64_t)x * rec, a.cache + off, static_cast<uint32_t>(run) * rec, bar);
                x += run;
                g += run;
            }
        }
    };
    if constexpr (PAGED) {
        if (tid == 0) {
            int* pi = reinterpret_cast<int*>(smem + so.hstat) + 16;
            pi[0] = b;
            pi[1] = h;
            pi[2] = static_cast<int>(t0 / G);
        }
    }

    // the chunk each stage holds (-1: none; the chunks come in increasing order, so the
    // first stage without one ends the item): chunks 0, 1, ... of the run, or (sc.on) the
    // block's fixed chunks and then counter grabs.  Thread 0 writes an entry before a
    // block barrier that precedes every read of it.
    int* chunk_of = reinterpret_cast<int*>(smem + so.hstat);
    const int dyn0 = nstage * sc.nw;    // chunk of counter value 0
    int pending = 0;                    // thread 0: the counter value fetched for the next chunk
    if constexpr (STEAL) {
        if (tid == 0) {
            for (int s2 = 0; s2 < nstage; ++s2) {
                int c;
                if (!sc.on) {
                    c = s2;
                } else if (sc.r < sc.nw) {
                    c = sc.r + s2 * sc.nw;
                } else {
                    c = dyn0 + atomicAdd(sc.ctr, 1);
                }
                c = c < nch ? c : -1;
                chunk_of[s2] = c;
                if (c >= 0) issue(c, s2);
            }
            if (sc.on) pending = atomicAdd(sc.ctr, 1);   // lands while the first chunks run
        }
    } else if (tid == 0) {
        for (int j = 0; j < nstage && j < nch; ++j) issue(j, j);   // chunk j into stage j
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
    if constexpr (ROPE) {
        // row 32 nt + lane (lane = 4 g + t): for k-step ks, words 2 ks and 2 ks + 1 hold the
        // query part (g & 1: 0 major, 1 minor) of head 4 nt + g / 2 at channels 16 ks + 2 t
        // + {0, 1} and {8, 9}; and the rotation frequencies w_i
        float* rw = reinterpret_cast<float*>(smem + so.rw);
        for (int i = tid; i < D / 2; i += blockDim.x) rw[i] = a.rope_w[i];
        for (int i = tid; i < 32 * NT * KSTEPS; i += blockDim.x) {
            const int ks = i % KSTEPS, row = i / KSTEPS;
            const int ln = row & 31, gg = ln >> 2, tt = ln & 3;
            const int hh = 4 * (row >> 5) + (gg >> 1);
            uint32_t w2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int c = 16 * ks + 2 * tt + 8 * e;
                float v0 = 0.0f, v1 = 0.0f;
                if (hh < gqa) {
                    v0 = qs[hh * D + c] * qdown;
                    v1 = qs[hh * D + c + 1] * qdown;
                }
                uint32_t mj, mn;
                split_pair(v0, v1, mj, mn);
                w2[e] = (gg & 1) ? mn : mj;
            }
            qx[row * QROW + 2 * ks] = w2[0];
            qx[row * QROW + 2 * ks + 1] = w2[1];
        }
    }
    // one entry per (head hh, lane quarter tg, key pair m), written to the rows of the two
    // lanes (parts) of B columns 2 (hh mod 4) and 2 (hh mod 4) + 1
    for (int i = tid; i < (ROPE ? 0 : 16 * NT * NPAIR); i += blockDim.x) {
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
    // dense-and-sparse records: the value outliers' corrections p' (x - zero) are summed per
    // warp in shared memory [head][D], in the units (and under the rescales) of oacc
    float* ocw = reinterpret_cast<float*>(smem + so.oc) + warp * gqa * D;
    if constexpr (SPARSE) {
        for (int x = lane; x < gqa * D; x += 32) ocw[x] = 0.0f;
    }
    // the warp's tokens start W * warp tokens into every chunk: group g0 of the chunk's
    // records, offset ti0 in it (a group may be shared by two warps)
    const int g0 = (warp * W) / G, ti0 = (warp * W) % G;
    for (int j = 0; STEAL || j < nch; ++j) {
        const int sj = nstage == 2 ? (j & 1) : 0;                       // stage of step j
        int c = j;
        if constexpr (STEAL) {
            c = chunk_of[sj];
            if (c < 0) break;
        }
        if (!wait_stage(bars, sj, phase, a.ws)) {
            // the next chunk's copy may already be armed on the other stage
            if (nstage == 2 && (STEAL ? chunk_of[sj ^ 1] >= 0 : j + 1 < nch)) drain_stage(bars, sj ^ 1, phase);
            empty_partial(a, slot);
            return -1;
        }
        const int ctok = min(ntok - c * CH, CH);
        const int wtok = ctok - warp * W < 0 ? 0 : (ctok - warp * W > W ? W : ctok - warp * W);   // multiple of 16
        const uint32_t st0 = sbase + static_cast<uint32_t>(so.data) + sj * stage_bytes + g0 * rec;
        int ngrp = 0;                                  // groups the warp's tokens touch (<= 8)
        for (int x = ti0 + wtok; x > 0; x -= G) ++ngrp;
        if (wtok > 0) {
            const int ntl = wtok >> 4;
            // offset term of every group of the warp: cst[group][head] = sum_c q_c zero_c,
            // as one small tensor-core product (rows = groups, k = channels in pair order)
            float cstf[NT][4];
            if constexpr (!ROPE) {
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
            if constexpr (ROPE) {
                const float* rw = reinterpret_cast<const float*>(smem + so.rw);
                const uint32_t qt_lane = qx_lane;      // the natural-order query table
                const float lv = static_cast<float>((1 << BITS) - 1);
                // position of the warp's first token (the item starts at token t0)
                const int64_t wpos = t0 + (int64_t)c * CH + warp * W;
                int i = 0, ti = ti0;
                const uint8_t* rp = smem + so.data + sj * stage_bytes + (int64_t)g0 * rec;
#pragma unroll 1
                while (i < ntl) {
                    const uint8_t* kp = rp + kpar;     // fp16 scale[D], then zero[D]
                    // the group's largest possible |key| (before and after rotation, up to
                    // sqrt 2): scale 2^(14 - e) keeps every fp16 part finite
                    float ksc, kf;
                    {
                        float m = 0.0f;
                        for (int cc = lane; cc < D; cc += 32) {
                            const float sv = half_at(kp, 2 * cc), zv = half_at(kp, 2 * D + 2 * cc);
                            m = fmaxf(m, fmaxf(fabsf(zv), fabsf(fmaf(sv, lv, zv))));
                        }
                        m = warp_max(m);
                        int e = 0;
                        if (m > 0.0f) frexpf(m * 1.41421366f, &e);
                        e = e < -100 ? -100 : (e > 120 ? 120 : e);
                        ksc = exp2i(14 - e);
                        kf = exp2i(e - 14) * qup;
                    }
                    const int nseg = min(ntl - i, (G - ti) >> 4);
#pragma unroll 1
                    for (int k = 0; k < nseg; ++k, ++i, ti += 16) {
                        const uint8_t* rowg = rp + (int64_t)(ti + g) * ROWB;
                        const uint8_t* rowg8 = rowg + 8 * ROWB;
                        const float posg = static_cast<float>(wpos + 16 * i + g);
                        const float posg8 = static_cast<float>(wpos + 16 * i + g + 8);
                        float acc[NT][4];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
#pragma unroll
                        for (int pp = 0; pp < KSTEPS / 2; ++pp) {
                            const int c0 = 16 * pp + 2 * tig, c2 = c0 + D / 2;
                            int xg[4], xg8[4], yg[4], yg8[4];
                            row_codes4<BITS>(rowg, c0, xg);
                            row_codes4<BITS>(rowg8, c0, xg8);
                            row_codes4<BITS>(rowg, c2, yg);
                            row_codes4<BITS>(rowg8, c2, yg8);
                            float xr[2][4], yr[2][4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int cl = c0 + (e & 1) + 8 * (e >> 1), ch = cl + D / 2;
                                const float s1 = half_at(kp, 2 * cl), z1 = half_at(kp, 2 * D + 2 * cl);
                                const float s2 = half_at(kp, 2 * ch), z2 = half_at(kp, 2 * D + 2 * ch);
                                const float w = rw[cl];
                                float sn, cs;
                                {
                                    const float x = dequant(xg[e], s1, z1), y = dequant(yg[e], s2, z2);
                                    rope_sincos(__fmul_rn(posg, w), &sn, &cs);
                                    xr[0][e] = (x * cs - y * sn) * ksc;
                                    yr[0][e] = (y * cs + x * sn) * ksc;
                                }
                                {
                                    const float x = dequant(xg8[e], s1, z1), y = dequant(yg8[e], s2, z2);
                                    rope_sincos(__fmul_rn(posg8, w), &sn, &cs);
                                    xr[1][e] = (x * cs - y * sn) * ksc;
                                    yr[1][e] = (y * cs + x * sn) * ksc;
                                }
                            }
                            // A fragments of k-steps pp (x) and pp + D/32 (y): rows g, g + 8,
                            // columns 2t, 2t + 1 (registers 0, 1) and 2t + 8, 2t + 9 (2, 3)
                            uint32_t xm[4], xn[4], ym[4], yn[4];
                            split_pair(xr[0][0], xr[0][1], xm[0], xn[0]);
                            split_pair(xr[1][0], xr[1][1], xm[1], xn[1]);
                            split_pair(xr[0][2], xr[0][3], xm[2], xn[2]);
                            split_pair(xr[1][2], xr[1][3], xm[3], xn[3]);
                            split_pair(yr[0][0], yr[0][1], ym[0], yn[0]);
                            split_pair(yr[1][0], yr[1][1], ym[1], yn[1]);
                            split_pair(yr[0][2], yr[0][3], ym[2], yn[2]);
                            split_pair(yr[1][2], yr[1][3], ym[3], yn[3]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint2 qa = lds64(qt_lane + nt * 32 * QROW * 4 + 8 * pp);
                                const uint2 qb = lds64(qt_lane + nt * 32 * QROW * 4 + 8 * (pp + KSTEPS / 2));
                                mma_16816(acc[nt], xm, qa.x, qa.y);
                                mma_16816(acc[nt], xn, qa.x, qa.y);
                                mma_16816(acc[nt], ym, qb.x, qb.y);
                                mma_16816(acc[nt], yn, qb.x, qb.y);
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const float s0 = (acc[nt][0] + acc[nt][1]) * kf;
                            const float s1 = (acc[nt][2] + acc[nt][3]) * kf;
                            wsc[(i * NT + nt) * 32] = make_float2(s0, s1);
                            cmax[nt] = fmaxf(cmax[nt], fmaxf(s0, s1));
                        }
                    }
                    rp += rec;
                    ti = 0;
                }
            } else {
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
            if constexpr (SPARSE) {
                // key outliers of the warp's tokens: their dense code 0 scored q_c zero_c, the
                // element is x, so s[t][head] += qs[head][c] (x - zero_c); several outliers of
                // one token meet in one score, hence the shared-memory atomics
                __syncwarp();
                float* wsc0 = reinterpret_cast<float*>(smem + so.sc) + (int64_t)warp * MAXT * NT * 32 * 2;
                const uint8_t* rp = smem + so.data + sj * stage_bytes + (int64_t)g0 * rec;
                for (int r = 0; r < ngrp; ++r, rp += rec) {
                    const uint32_t* side = reinterpret_cast<const uint32_t*>(rp + lo.kc + lo.vc + lo.kp + lo.vp);
                    const __half* kz = reinterpret_cast<const __half*>(rp + kpar + 2 * D);
                    for (int x = lane; x < lo.K * D; x += 32) {
                        const uint32_t w = side[x];
                        const int c = x & (D - 1);
                        const int wt = r * G + static_cast<int>(w & 0xffffu) - ti0;   // warp token
                        if (wt < 0 || wt >= wtok) continue;
                        const float d = __fsub_rn(bf16_bits_to_float(static_cast<uint16_t>(w >> 16)), __half2float(kz[c]));
                        const int it = wt >> 4, tt = wt & 15;
                        float* dst = wsc0 + 2 * ((it * NT) * 32 + (tt & 7) * 4) + (tt >> 3);
#pragma unroll
                        for (int hh = 0; hh < NT * 4; ++hh)
                            if (hh < gqa) atomicAdd(dst + 2 * ((hh >> 2) * 32 + (hh & 3)), qs[hh * D + c] * d);
                    }
                }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    cmax[nt] = -INFINITY;
                    for (int it = 0; it < ntl; ++it) {
                        const float2 v = wsc[(it * NT + nt) * 32];
                        cmax[nt] = fmaxf(cmax[nt], fmaxf(v.x, v.y));
                    }
                }
            }
            float ocf[NT];          // rescale factor of this chunk for the value corrections
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) ocf[nt] = 1.0f;
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
                        ocf[nt] = f;
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
                    ocf[nt] *= alpha;
                }
                mrun[nt] = mnew;
                // p' = 2^(s - max + Ev): the value operand's power-of-two scale, applied
                // in the exponent
                mE[nt] = mnew - static_cast<float>(Ev);
            }
            if constexpr (SPARSE) {
                // the value corrections follow oacc's rescales (lanes g of a head: channels
                // g + 8 x)
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int head = 4 * nt + tig;
                    if (ocf[nt] != 1.0f && head < gqa)
                        for (int x = g; x < D; x += 8) ocw[head * D + x] *= ocf[nt];
                }
                __syncwarp();
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
                            if constexpr (SPARSE) {
                                // value outliers of this lane's tokens g and g + 8 (side-list
                                // positions 2g and 2g + 1 of the tile, like their zeros): the
                                // dense code 0 gave zero, the element is x
                                const int head = 4 * nt + tig;
                                if (head < gqa) {
                                    for (int jv = 0; jv < NGv; ++jv) {
                                        const uint32_t zw = lds32(ro + vpar + 2 * G * NGv + 2 * (jv * G + ti) + 4 * g);
                                        const float2 zf = __half22float2(u32_as_h2(zw));
                                        for (int e = 0; e < lo.K; ++e) {
                                            const uint2 w2 = lds64(ro + vpar + lo.vp + lo.ko +
                                                                   4 * (e * NGv * G + jv * G + ti) + 8 * g);
                                            const float d0 = __fsub_rn(bf16_bits_to_float(static_cast<uint16_t>(w2.x >> 16)), zf.x);
                                            const float d1 = __fsub_rn(bf16_bits_to_float(static_cast<uint16_t>(w2.y >> 16)), zf.y);
                                            // (the index is masked into the group: a record read
                                            // through a bad page cannot write past the buffer)
                                            const int gm = lo.Gv - 1;
                                            atomicAdd(ocw + head * D + jv * lo.Gv + (static_cast<int>(w2.x) & gm), p0 * d0);
                                            atomicAdd(ocw + head * D + jv * lo.Gv + (static_cast<int>(w2.y) & gm), p1 * d1);
                                        }
                                    }
                                }
                            }
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
        if constexpr (STEAL) {
            if (tid == 0) {         // this stage's next chunk
                const int nx = sc.on ? dyn0 + pending : j + nstage;
                chunk_of[sj] = nx < nch ? nx : -1;
            }
            __syncthreads();        // every warp is done with this stage
            if (tid == 0 && chunk_of[sj] >= 0) {
                issue(chunk_of[sj], sj);
                if (sc.on) pending = atomicAdd(sc.ctr, 1);
            }
        } else {
            __syncthreads();        // every warp is done with this stage
            if (tid == 0 && j + nstage < nch) issue(j + nstage, sj);
        }
    }
    // ---- warp partial: undo the power-of-two scales, reduce l over the lanes of a head,
    // add the value offset term, combine the 4 warps in shared memory
    float* cw = comb + warp * gqa * D;
    const bool wlive = mrun[0] > -INFINITY;
    const float zfac = exp2i(-Ev), lfac = exp2i(-Ev);
    if constexpr (SPARSE) __syncwarp();     // every lane's value corrections have landed
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
                float o0 = fmaf(oacc[mt][nt][0] + oacc[mt][nt][1], f0, oz);
                float o1 = fmaf(oacc[mt][nt][2] + oacc[mt][nt][3], f1, oz);
                if constexpr (SPARSE) {
                    o0 = fmaf(ocw[head * D + c0], zfac, o0);
                    o1 = fmaf(ocw[head * D + c0 + 8], zfac, o1);
                }
                cw[head * D + c0] = o0;
                cw[head * D + c0 + 8] = o1;
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
// BITS == 0: no packed part (INT8 rows).  STEAL: units may share their packed chunks on
// demand (a separate instantiation: the extra code slows the kernels that never use it).
// PAGED: the group records are found through the block table (paged layout).
// ROPE: keys cached before the rotary embedding (packed tokens on the tensor cores,
// window rows through rope_item).
template <int D, int BITS, int NT, bool STEAL, bool PAGED, bool SPARSE = false, bool ROPE = false>
__global__ void __launch_bounds__(kDecodeThreads, (NT == 1 && D <= 128) ? 4 : 2)
    k_decode(const __grid_constant__ DecodeArgs a) {
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
    for_each_segment<STEAL>(
        a, reinterpret_cast<int64_t*>(smem + so.red), reinterpret_cast<int2*>(smem + so.sst),
        [&](int part, int b, int h, int64_t slot, int64_t t0, int64_t t1, const StealCtx& sc) -> bool {
            int r;
            if constexpr (BITS != 0) {
                if (part == 0)
                    r = packed_item<D, BITS, NT, STEAL, PAGED, SPARSE, ROPE>(a, smem, b, h, slot, t0, t1, phase, sc);
                else if constexpr (ROPE)
                    r = rope_item<D, BITS>(a, smem, b, h, slot, 1, t0, t1, phase);
                else
                    r = window_item<D, NT>(a, smem, b, h, slot, t0, t1, phase);
            } else {
                r = rows_item<D>(a, smem, b, h, slot, t0, t1, phase);
            }
            if (r < 0) return false;
            phase = static_cast<uint32_t>(r);
            return true;
        },
        [&](int64_t slot) { empty_partial(a, slot); });
}

// The decode's wave: NB = one wave of resident blocks of kernel fn (SM count times the
// occupancy calculator's blocks per SM), the split (unit_aligned) and whether the blocks of
// a unit should take its chunks on demand: when some unit could get 4 packed chunks per
// block, i.e. when the layer's packed capacity holds 4 NB chunks (a unit of cost U gets
// about U NB / C blocks and holds U / (CH cpt0) packed chunks, so the ratio is
// C / (NB CH cpt0) for every unit).
template <typename K>
int plan_wave(K fn, DecodeArgs& a) {
    int nb = 0;
    const int rc = decode_blocks(reinterpret_cast<const void*>(fn), kDecodeThreads, a.plan.smem, &nb);
    if (rc != KVQ_OK) return rc;
    a.plan.NB = nb;
    a.plan.inv_nb = 1.0f / nb;
    a.plan.unit_aligned = 2 * (int64_t)a.lo.B * a.lo.H <= nb ? 1 : 0;
    const int64_t packed_chunks = (int64_t)a.lo.B * a.lo.H * (((int64_t)a.lo.NG * a.lo.G) / a.plan.CH);
    a.plan.steal = a.plan.unit_aligned && a.lo.scheme == KVQ_SCHEME_KIVI && packed_chunks >= 4 * (int64_t)nb;
    return KVQ_OK;
}

// Launches fn over the wave plan_wave sized (a.plan.NB blocks); KVQ_ERR_UNSUPPORTED, with
// nothing launched, when fn has another number of resident blocks.
template <typename K>
int launch_on_wave(K fn, DecodeArgs& a, cudaStream_t stream) {
    int nb = 0;
    const int rc = decode_blocks(reinterpret_cast<const void*>(fn), kDecodeThreads, a.plan.smem, &nb);
    if (rc != KVQ_OK) return rc;
    if (nb != a.plan.NB) return KVQ_ERR_UNSUPPORTED;
    return launch_dependent(fn, dim3(static_cast<unsigned>(nb)), kDecodeThreads, static_cast<size_t>(a.plan.smem),
                            stream, a) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
}

// One kernel on its own wave, the fixed split (FP8, rows).
template <typename K>
int launch_wave(K fn, DecodeArgs& a, cudaStream_t stream) {
    const int rc = plan_wave(fn, a);
    if (rc != KVQ_OK) return rc;
    a.plan.steal = 0;
    return launch_on_wave(fn, a, stream);
}

// KIVI variants beyond the base kernel, each family in translation units of its own (so
// the builds run in parallel): on demand (STEAL), paged layout (PAGED) and both.  The
// paged fixed-split kernel plans its own wave (it is the paged fallback).
// SPARSE: dense-and-sparse records (side lists of outliers); ROPE: keys cached before the
// rotary embedding.  These kernels use the fixed split and plan their own wave.
template <int D, int BITS, int NT, bool STEAL, bool PAGED, bool SPARSE, bool ROPE>
int launch_kivi_variant(DecodeArgs& a, cudaStream_t stream) {
    if constexpr ((PAGED || SPARSE || ROPE) && !STEAL) {   // the fixed split, on the kernel's own wave
        const int rc = plan_wave(k_decode<D, BITS, NT, false, PAGED, SPARSE, ROPE>, a);
        if (rc != KVQ_OK) return rc;
        a.plan.steal = 0;
    }
    return launch_on_wave(k_decode<D, BITS, NT, STEAL, PAGED, SPARSE, ROPE>, a, stream);
}
template <int BITS, bool STEAL, bool PAGED, bool SPARSE = false, bool ROPE = false>
int launch_kivi_family(DecodeArgs& a, cudaStream_t stream) {
    const bool wide = a.lo.gqa > 4;
    switch (a.lo.D) {
        case 64:
            return wide ? launch_kivi_variant<64, BITS, 2, STEAL, PAGED, SPARSE, ROPE>(a, stream)
                        : launch_kivi_variant<64, BITS, 1, STEAL, PAGED, SPARSE, ROPE>(a, stream);
        case 128:
            return wide ? launch_kivi_variant<128, BITS, 2, STEAL, PAGED, SPARSE, ROPE>(a, stream)
                        : launch_kivi_variant<128, BITS, 1, STEAL, PAGED, SPARSE, ROPE>(a, stream);
        case 256:
            return wide ? launch_kivi_variant<256, BITS, 2, STEAL, PAGED, SPARSE, ROPE>(a, stream)
                        : launch_kivi_variant<256, BITS, 1, STEAL, PAGED, SPARSE, ROPE>(a, stream);
        default: return KVQ_ERR_UNSUPPORTED;
    }
}
int launch_decode_kivi2_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_paged_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_paged_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_paged_steal(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_sparse(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_sparse(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_sparse(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_rope(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_rope(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_rope(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_rope_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_rope_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_rope_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi2_sparse_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4_sparse_paged(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8_sparse_paged(DecodeArgs& a, cudaStream_t stream);

// The base kernel sizes the wave; paged caches and on-demand splits go to their variants.
template <int D, int BITS, int NT>
int launch_decode_t(DecodeArgs& a, cudaStream_t stream) {
    int rc = plan_wave(k_decode<D, BITS, NT, false, false>, a);
    if (rc != KVQ_OK) return rc;
    if constexpr (BITS != 0) {
        if (a.lo.PG > 0) {
            if constexpr (BITS == 2) return launch_decode_kivi2_paged(a, stream);
            else if constexpr (BITS == 4) return launch_decode_kivi4_paged(a, stream);
            else return launch_decode_kivi8_paged(a, stream);
        }
        if (a.plan.steal) {
            if constexpr (BITS == 2) rc = launch_decode_kivi2_steal(a, stream);
            else if constexpr (BITS == 4) rc = launch_decode_kivi4_steal(a, stream);
            else rc = launch_decode_kivi8_steal(a, stream);
            if (rc != KVQ_ERR_UNSUPPORTED) return rc;
        }
    }
    a.plan.steal = 0;   // the fixed split
    return launch_on_wave(k_decode<D, BITS, NT, false, false>, a, stream);
}

// Dispatchers, one per translation unit.
int launch_decode_kivi2(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi4(DecodeArgs& a, cudaStream_t stream);
int launch_decode_kivi8(DecodeArgs& a, cudaStream_t stream);
int launch_decode_rows(DecodeArgs& a, cudaStream_t stream);
int launch_decode_fp8(DecodeArgs& a, cudaStream_t stream);
int launch_decode_rope(DecodeArgs& a, cudaStream_t stream);

}  // namespace kvq
