// kvq_internal.cuh -- cache layout and device helpers shared by the CUDA translation units
// of libkvq.so (not part of the public ABI).
//
// Cache image (little-endian, every region starts on a 256-byte boundary):
//   header   256 B; u32 status word at byte 0.
//   state    16 B per (layer, sequence): int32 n tokens cached, int32 qn of them in packed
//            groups (KIVI; qn == n for INT8 and FP8), an int32 arrival counter of the
//            one-kernel append (zero whenever no call runs) and a reserved zero word.
//   KIVI     "group records", one per (layer, sequence, kv head, group slot), NG =
//            (max_tokens - R) / G slots per (layer, sequence, kv head).  A record holds
//            everything a decode block needs for G tokens, so a run of groups is one
//            contiguous span (one bulk copy):
//              K codes  G*D*b/8 B, token-major: (token t, channel c) at bit (t*D + c)*b
//              V codes  D*G*b/8 B of 32-bit words, 2*D*b B per 16-token tile, in the
//                       order of the decode's value fragments: 32 lanes of wpl = D*b/64
//                       words, lane 4g + i holding tokens 2i + s (low half) and 2i + s + 8
//                       (high half) in its words 2m + s, with channel 16q + g + 8r
//                       (j = 2q + r) at bit b * (j mod 16/b) of word pair j / (16/b); a
//                       lane's words sit in slabs of min(wpl, 4), lanes contiguous
//              K params 4*D B: fp16 scale[D] then fp16 zero[D] (per channel, "min")
//              V params 4*G*(D/Gv) B: fp16 scale[D/Gv][G] then fp16 zero[D/Gv][G], tile
//                       token tt of a group's row at position 2 (tt mod 8) + tt / 8
//            then the bf16 window ("ring"): per (layer, sequence, kv head) C = R + G slots
//            of [K row bf16[D], V row bf16[D]]; token t (qn <= t < n) lives in slot t % C.
//   INT8     per (layer, sequence, kv head), T16 = max_tokens rounded up to 16:
//            K codes int8[T16][D], V codes int8[T16][D], K scale f32[T16], V scale f32[T16]
//   FP8      scale table f32[layers][kv heads][2] (K, V), then per (layer, sequence, kv
//            head): K codes e4m3[T16][D], each row's channels in fragment order (channel
//            r of 16-channel block kb in quarter (r mod 8)/2 at byte 4 kb + 2 (r/8) +
//            r mod 2); V codes e4m3 in 16-token tiles [channel][16], token tt at byte
//            4 ((tt mod 8)/2) + 2 (tt mod 2) + tt/8
// Bits are numbered LSB-first within a byte.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "kvq.h"

namespace kvq {

struct Layout {
    int32_t scheme, L, B, Hq, H, D, bits, G, Gv, R, T, dtype;
    int32_t gqa, C, NG, NGv, T16;
    int64_t state_off, scales_off, data_off, ring_off, total;
    int64_t unit;                    // bytes of one (layer, sequence, kv head) data block
    int32_t rec, kc, vc, kp, vp;     // KIVI record: total, K codes, V codes, K params, V params
};

inline int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// Streaming multiprocessors of the GB300 the decode work is sized for.
constexpr int kNumSMs = 152;

// How one decode step is split: every (sequence, kv head) "unit" gets NRC row chunks of
// CHR tokens (the bf16 window for KIVI, all tokens for INT8/FP8) and NQ packed chunks of
// CH tokens (KIVI groups), S = NRC + NQ work items in all.  A packed chunk is split among
// the block's 4 warps, W = CH / 4 tokens (whole groups) each; a packed item covers CPI
// consecutive chunks, staged through NSTAGE shared-memory buffers.  Each item leaves a
// partial softmax result (m, l, o[D]) per query head in the workspace.
struct DecodePlan {
    int CH, W, CPI, NSTAGE, NQ, CHR, NRC, S, NT;
    int64_t ws_o_off, ws_ml_off, ws_total;
    int64_t smem;
};

// Shared-memory carve of the decode block, identical on host and device.
struct SmemOffsets {
    int64_t bar, red, hstat, qs, qpa, qpb, pw, sc, data, total;
};
__host__ __device__ inline SmemOffsets decode_smem(const Layout& lo, const DecodePlan& p) {
    SmemOffsets o;
    int64_t off = 0;
    o.bar = off;   off += 64;                         // mbarriers, one per stage
    o.red = off;   off += 4 * 32 * 4;                 // [warp][32] floats
    o.hstat = off; off += 2 * 32 * 4;                 // per-head max and sum
    o.qs = off;    off += (int64_t)lo.gqa * lo.D * 4; // scaled query, fp32
    o.qpa = off;   off += (int64_t)32 * p.NT * (lo.D / 8 + 4) * 4;   // query tables: [32 NT][D/8 + 4]
    o.qpb = off;   off += (int64_t)32 * p.NT * (lo.D / 8 + 4) * 4;
    o.pw = off;    off += 4 * 16 * 8 * 4;                // window path: [warp][token][head] p
    o.sc = off;
    {
        const int64_t rows_sc = (int64_t)lo.gqa * p.CHR;                // row path scores
        const int64_t comb = (int64_t)4 * lo.gqa * (lo.D + 2);           // per-warp o and (m, l)
        const int64_t wsc = (int64_t)4 * 8 * p.NT * 32 * 2;              // per-warp tile scores
        int64_t big = rows_sc > comb ? rows_sc : comb;
        big = big > wsc ? big : wsc;
        off += 4 * big;
    }
    off = (off + 127) / 128 * 128;
    o.data = off;
    int64_t rows = 0, packed = 0;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        rows = (int64_t)p.CHR * 4 * lo.D;
        packed = (int64_t)p.NSTAGE * (p.CH / lo.G) * lo.rec;
    } else if (lo.scheme == KVQ_SCHEME_INT8) {
        rows = (int64_t)p.CHR * (2 * lo.D + 8);
    } else {
        rows = (int64_t)p.NSTAGE * p.CH * 2 * lo.D;      // FP8: key rows + value tiles per stage
    }
    off += rows > packed ? rows : packed;
    o.total = off;
    return o;
}

// Validates cfg (with `max_tokens` as the capacity) and fills the layout; returns KVQ_OK,
// KVQ_ERR_ARG or KVQ_ERR_UNSUPPORTED.
int make_layout(const kvq_config* cfg, int64_t max_tokens, Layout* out);

// ---------------------------------------------------------------------------- device helpers
__device__ __forceinline__ int32_t* state_ptr(const Layout& lo, uint8_t* cache, int l, int b) {
    return reinterpret_cast<int32_t*>(cache + lo.state_off) + 4 * ((int64_t)l * lo.B + b);
}
__device__ __forceinline__ const int32_t* state_ptr(const Layout& lo, const uint8_t* cache, int l,
                                                    int b) {
    return reinterpret_cast<const int32_t*>(cache + lo.state_off) + 4 * ((int64_t)l * lo.B + b);
}
__device__ __forceinline__ int64_t unit_index(const Layout& lo, int l, int b, int h) {
    return ((int64_t)l * lo.B + b) * lo.H + h;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t v) {
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// mbarrier + bulk asynchronous copy (the non-tensor TMA path): one thread arms the
// barrier with the byte count and issues the copies, every thread waits on phase 0.
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` polls (each poll may suspend the thread for a
// while), so a copy that never lands cannot hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
constexpr uint32_t kWaitLimit = 1u << 22;

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch.  A kernel launched by launch_dependent may begin while the
// kernel before it in the stream is still running; grid_dependency_wait, called before the
// kernel's first global read or write, returns once that kernel has completed and its
// writes are visible (at once when there is no such kernel).  grid_launch_dependents lets
// the next dependent kernel start launching early; it still waits in its own
// grid_dependency_wait for this grid to complete.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... P, typename... A>
inline cudaError_t launch_dependent(void (*fn)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    A&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, std::forward<A>(args)...);
}

// Bring the 128-byte line holding `p` into L2 (no register result, no fault semantics
// beyond those of a load of `p`).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

}  // namespace kvq
