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
//              with K = outliers > 0 (dense-and-sparse), two side lists of 32-bit entries
//              (bf16 bits of the element << 16 | its index in the vector), the e-th
//              largest magnitude first:
//              K side   4*K*D B: entry [e][c] of key channel c (index: token in the group)
//              V side   4*K*(D/Gv)*G B: entry [e][j][position] of value group j of a token
//                       (index: channel in the group), positions as the V params
//            Paged layout (page_groups PG > 0): the records live in a pool of NP pages of
//            L * H * PG records; record (l, b, h, g) is record (l * H + h) * PG + g mod PG
//            of page block_table[b * MP + g / PG], MP = ceil(NG / PG).
//            then the bf16 window ("ring"): per (layer, sequence, kv head) C = R + G slots
//            of [K row bf16[D], V row bf16[D]]; token t (qn <= t < n) lives in slot t % C.
//   INT8     per (layer, sequence, kv head), T16 = max_tokens rounded up to 16:
//            K codes int8[T16][D], V codes int8[T16][D], K scale f32[T16], V scale f32[T16]
//   INT4     the same with K and V codes of D / 2 bytes per row: channel c in byte c / 2,
//            low four bits for even c, high four for odd c (two's complement)
//   FP8      (E4M3 or E5M2) scale table f32[layers][kv heads][2] (K, V), then per (layer, sequence, kv
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
    int32_t K, ko, vo;               // KIVI dense-and-sparse: outliers per vector, K and V side lists
    int32_t PG, NP, MP;              // paged layout: records per page and sequence, pages, table row
    int64_t page;                    // paged layout: bytes of a page
    const int32_t* table;            // paged layout: the block table (device)
    float rope_base;                 // > 0: keys cached before the rotary embedding
};

inline int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

// FP8 caches (E4M3 or E5M2 codes, per-(layer, kv head) scales) and per-token row caches
// (INT8 or INT4 codes, per-(head, token) scales).
__host__ __device__ inline bool is_fp8(int scheme) {
    return scheme == KVQ_SCHEME_FP8_E4M3 || scheme == KVQ_SCHEME_FP8_E5M2;
}
__host__ __device__ inline bool is_rows(int scheme) {
    return scheme == KVQ_SCHEME_INT8 || scheme == KVQ_SCHEME_INT4;
}

// How one decode step is split.  Every (sequence, kv head) "unit" has two parts: part 0,
// the packed tokens (KIVI groups, FP8 tiles), cut into chunks of CH tokens; part 1, the row
// tokens (the KIVI bf16 window, INT8 rows), cut into chunks of CHR tokens.  A chunk costs
// its tokens times cpt0 or cpt1 (16-byte units of the bytes a token reads), so the layer's
// total cost C follows the real token counts in the cache state.  The decode runs NB
// blocks, one wave of resident blocks; block j takes the chunks whose cost position starts
// in [ceil(C j / NB), ceil(C (j + 1) / NB)) and leaves, for every part of a unit it
// touches, one partial softmax result (m, l, o[D]) per query head in workspace slot
// j + part B H + unit.  With at most half as many units as blocks, units instead get whole
// blocks (unit_aligned).  A packed chunk is split among the block's 4 warps,
// W = CH / 4 tokens (whole groups) each, staged through NSTAGE shared-memory buffers.
struct DecodePlan {
    int CH, W, NSTAGE, CHR, NT;
    int NB;                          // decode blocks of the launch (set by the launcher)
    int unit_aligned;                // 1: every unit gets whole blocks (set by the launcher)
    int steal;                       // 1: those blocks share the unit's packed chunks on demand
    int64_t cpt0, cpt1;              // scheduling cost of a packed token and of a row token
    float inv_nb, inv_cc0, inv_cc1;  // 1 / NB and 1 / (chunk cost) of each part
    int64_t nslot;                   // partial-result slots the workspace holds
    int64_t ws_ctr_off;              // per-unit chunk counters (zero between decodes)
    int64_t ws_o_off, ws_ml_off, ws_total;   // partial o, partial (m, l)
    int64_t smem;
};

// Shared-memory carve of the decode block, identical on host and device.
struct SmemOffsets {
    int64_t bar, red, hstat, sst, qs, qpa, qpb, pw, sc, oc, rw, data, total;
};
__host__ __device__ inline SmemOffsets decode_smem(const Layout& lo, const DecodePlan& p) {
    SmemOffsets o;
    int64_t off = 0;
    o.bar = off;   off += 64;                         // mbarriers, one per stage
    o.red = off;   off += 4 * 32 * 4;                 // [warp][32] floats
    o.hstat = off; off += 4 * 32 * 4;                 // per-head running max, sum, rescale
    o.sst = off;   off += 128 * 8;                    // sequence states (n, qn), batch <= 128
    o.qs = off;                                       // scaled query fp32 [gqa][D], or the
    off += (lo.gqa > 4 ? lo.gqa : 4) * (int64_t)lo.D * 4;   // window's bf16 query words [8][D / 2]
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
    o.oc = off;                                          // dense-and-sparse: per-warp value
    if (lo.K > 0) off += (int64_t)4 * lo.gqa * lo.D * 4;    // corrections [warp][head][D]
    o.rw = off;                                          // keys before RoPE: w_i, i < D/2
    if (lo.rope_base > 0.0f) off += (int64_t)2 * lo.D;
    off = (off + 127) / 128 * 128;
    o.data = off;
    int64_t rows = 0, packed = 0;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        rows = (int64_t)p.CHR * 4 * lo.D;
        packed = (int64_t)p.NSTAGE * (p.CH / lo.G) * lo.rec;
    } else if (is_rows(lo.scheme)) {
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

// Byte offset, from the cache base, of KIVI group record g of unit (l, b, h).  Paged
// layout: through the sequence's block table; -1 when its entry is outside the pool.
__device__ __forceinline__ int64_t group_offset(const Layout& lo, int l, int b, int h, int64_t g) {
    if (lo.PG == 0) return lo.data_off + unit_index(lo, l, b, h) * lo.unit + g * lo.rec;
    const int pg = static_cast<int>(g) / lo.PG;
    const int32_t p = lo.table[(int64_t)b * lo.MP + pg];
    if (p < 0 || p >= lo.NP) return -1;
    return lo.data_off + (int64_t)p * lo.page + (((int64_t)l * lo.H + h) * lo.PG + (g - (int64_t)pg * lo.PG)) * lo.rec;
}
// True when every group slot in [g0, g1) of sequence b has a page in the pool.
__device__ __forceinline__ bool pages_ok(const Layout& lo, int b, int64_t g0, int64_t g1) {
    if (lo.PG == 0 || g0 >= g1) return true;
    for (int64_t pg = g0 / lo.PG; pg <= (g1 - 1) / lo.PG; ++pg) {
        const int32_t p = lo.table[(int64_t)b * lo.MP + pg];
        if (p < 0 || p >= lo.NP) return false;
    }
    return true;
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
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: gives up once `limit_ns` nanoseconds of the GPU's global timer have passed,
// so a copy that never lands cannot hang the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}
// A staged copy of at most a few tens of KiB lands in microseconds; one second means it
// never will.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// Barrier slot (in the decode block's barrier area) that nothing ever completes: the
// workspace self-test of the bounded waits waits on it.
constexpr int kSelfTestBar = 2;
constexpr uint32_t kSelfTestBit = 1u << 30;   // phase bits stay non-negative as an int

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
