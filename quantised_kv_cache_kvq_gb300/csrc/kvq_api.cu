// kvq_api.cu -- the extern "C" entry points of libkvq.so: argument validation, the cache
// layout, the decode plan, and kernel launches on the caller's stream.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kvq_decode.cuh"
#include "kvq_internal.cuh"
#include "kvq_launch.h"

namespace kvq {

static bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

int make_layout(const kvq_config* c, int64_t max_tokens, Layout* out) {
    if (!c || !out) return KVQ_ERR_ARG;
    Layout lo;
    std::memset(&lo, 0, sizeof lo);
    if (c->scheme < 0 || c->scheme > 4) return KVQ_ERR_ARG;
    if (c->layers < 1 || c->batch < 1 || c->kv_heads < 1 || c->q_heads < c->kv_heads) return KVQ_ERR_ARG;
    if (c->q_heads % c->kv_heads != 0) return KVQ_ERR_ARG;
    if (max_tokens < 1 || max_tokens > (int64_t)1 << 30) return KVQ_ERR_ARG;
    if (c->in_dtype != KVQ_DTYPE_BF16 && c->in_dtype != KVQ_DTYPE_F32) return KVQ_ERR_ARG;
    if (c->page_groups < 0 || c->num_pages < 0) return KVQ_ERR_ARG;
    if (!(c->rope_base >= 0.0f) || c->rope_base > 3.0e38f) return KVQ_ERR_ARG;   // NaN, negative, inf
    const int gqa = c->q_heads / c->kv_heads;
    if (gqa != 1 && gqa != 2 && gqa != 4 && gqa != 8) return KVQ_ERR_UNSUPPORTED;
    const int D = c->head_dim;
    lo.scheme = c->scheme;
    lo.L = c->layers;
    lo.B = c->batch;
    lo.Hq = c->q_heads;
    lo.H = c->kv_heads;
    lo.D = D;
    lo.bits = c->bits;
    lo.G = c->group_k;
    lo.Gv = c->group_v;
    lo.R = c->residual;
    lo.T = static_cast<int32_t>(max_tokens);
    lo.dtype = c->in_dtype;
    lo.gqa = gqa;
    lo.T16 = static_cast<int32_t>((max_tokens + 15) / 16 * 16);
    const int64_t units = (int64_t)lo.L * lo.B * lo.H;
    lo.state_off = 256;
    int64_t pos = lo.state_off + align256((int64_t)lo.L * lo.B * 16);
    if (c->scheme == KVQ_SCHEME_KIVI) {
        if (!pow2_in(D, 64, 256)) return KVQ_ERR_UNSUPPORTED;
        if (c->bits != 2 && c->bits != 4 && c->bits != 8) return KVQ_ERR_ARG;
        if (c->group_k < 16 || c->group_k > 128 || c->group_k % 16 != 0) return KVQ_ERR_ARG;
        if (c->group_v < 16 || c->group_v % 16 != 0 || D % c->group_v != 0) return KVQ_ERR_ARG;
        if (c->residual < 0 || c->residual > (1 << 20)) return KVQ_ERR_ARG;
        if (c->in_dtype != KVQ_DTYPE_BF16) return KVQ_ERR_ARG;
        lo.C = lo.R + lo.G;
        lo.NG = max_tokens > lo.R ? static_cast<int32_t>((max_tokens - lo.R) / lo.G) : 0;
        lo.NGv = D / lo.Gv;
        lo.kc = lo.G * D * lo.bits / 8;
        lo.vc = D * lo.G * lo.bits / 8;
        lo.kp = 4 * D;
        lo.vp = 4 * lo.G * lo.NGv;
        if (c->outliers < 0 || c->outliers > 4) return KVQ_ERR_ARG;
        lo.K = c->outliers;
        lo.ko = 4 * lo.K * D;
        lo.vo = 4 * lo.K * lo.NGv * lo.G;
        lo.rec = lo.kc + lo.vc + lo.kp + lo.vp + lo.ko + lo.vo;
        lo.unit = (int64_t)lo.NG * lo.rec;
        lo.data_off = pos;
        if (c->page_groups > 0) {
            if (c->num_pages < 1) return KVQ_ERR_ARG;
            lo.PG = c->page_groups;
            lo.NP = c->num_pages;
            lo.MP = (lo.NG + lo.PG - 1) / lo.PG;
            lo.page = (int64_t)lo.L * lo.H * lo.PG * lo.rec;
            lo.table = c->block_table;
            pos += align256((int64_t)lo.NP * lo.page);
        } else {
            pos += align256(units * lo.unit);
        }
        lo.ring_off = pos;
        pos += align256(units * lo.C * 4 * (int64_t)D);
        lo.rope_base = c->rope_base;
    } else {
        if (c->page_groups > 0) return KVQ_ERR_UNSUPPORTED;   // pages hold KIVI group records
        if (c->rope_base > 0.0f) return KVQ_ERR_UNSUPPORTED;  // pre-RoPE keys: KIVI caches
        if (c->outliers != 0) return KVQ_ERR_UNSUPPORTED;     // dense-and-sparse: KIVI caches
        if (!pow2_in(D, 32, 256)) return KVQ_ERR_UNSUPPORTED;
        if (is_rows(c->scheme)) {
            lo.unit = (int64_t)lo.T16 * ((c->scheme == KVQ_SCHEME_INT8 ? 2 * D : D) + 8);
            lo.data_off = pos;
            pos += align256(units * lo.unit);
        } else {
            lo.scales_off = pos;
            pos += align256((int64_t)lo.L * lo.H * 8);
            lo.unit = (int64_t)lo.T16 * 2 * D;
            lo.data_off = pos;
            pos += align256(units * lo.unit);
        }
    }
    lo.total = pos;
    *out = lo;
    return KVQ_OK;
}

// Decode blocks resident per SM for `smem` bytes of dynamic shared memory, as used to
// choose between one and two staging buffers: 4 by the kernels' register bound, fewer
// when 228 KiB of shared memory per SM (1 KiB of it reserved per block) does not hold 4.
// The grid itself is sized on the device by the occupancy calculator (decode_blocks).
static int resident_blocks(int64_t smem) {
    const int64_t r = (228 * 1024) / (smem + 1024);
    return r < 4 ? static_cast<int>(r) : 4;
}

static int64_t ceil16(int64_t bytes) { return (bytes + 15) / 16; }

int make_plan(const Layout& lo, DecodePlan* p) {
    std::memset(p, 0, sizeof *p);
    p->NT = lo.gqa > 4 ? 2 : 1;
    p->NSTAGE = 1;
    if (lo.scheme == KVQ_SCHEME_KIVI) {
        p->CHR = 64;
        // a warp takes W tokens (a multiple of 16, at least 64) and a block 4 warps, with 4 * W
        // a whole number of groups: W = 16 * (G / gcd(G, 64)) scaled up to 64 or more
        int gg = lo.G, hh = 64;
        while (hh) { const int t = gg % hh; gg = hh; hh = t; }
        const int wstep = 16 * (lo.G / gg);
        p->W = wstep * ((64 + wstep - 1) / wstep);
        p->CH = 4 * p->W;
        p->cpt0 = ceil16((lo.rec + lo.G - 1) / lo.G);      // group record bytes per token
        p->cpt1 = ceil16(4 * (int64_t)lo.D);                // bf16 key and value row
    } else if (is_fp8(lo.scheme)) {
        p->CHR = 16;
        p->W = 32;
        p->CH = 4 * p->W;
        p->cpt0 = ceil16(2 * (int64_t)lo.D);
        p->cpt1 = 1;
    } else {
        p->CHR = 128;
        p->CH = 16;
        p->W = 4;
        p->cpt0 = 1;
        p->cpt1 = ceil16((lo.scheme == KVQ_SCHEME_INT8 ? 2 * (int64_t)lo.D : lo.D) + 8);
    }
    // double-buffer the packed chunks when that costs no resident block
    if (!is_rows(lo.scheme)) {
        const int res1 = resident_blocks(decode_smem(lo, *p).total);
        p->NSTAGE = 2;
        if (resident_blocks(decode_smem(lo, *p).total) < res1) p->NSTAGE = 1;
    }
    // slots: block j writes slot j + part * units + unit (cost ranges) or 2 j + part (whole
    // blocks per unit, used only when 2 units <= NB), j < NB <= KVQ_MAX_DECODE_BLOCKS
    const int64_t units = (int64_t)lo.B * lo.H;
    p->nslot = KVQ_MAX_DECODE_BLOCKS + (2 * units > KVQ_MAX_DECODE_BLOCKS ? 2 * units : KVQ_MAX_DECODE_BLOCKS);
    const int64_t slots = p->nslot * lo.gqa;
    p->ws_ctr_off = 256;                                    // KVQ_MAX_DECODE_BLOCKS / 2 int32
    p->ws_o_off = p->ws_ctr_off + 2 * KVQ_MAX_DECODE_BLOCKS;
    p->ws_ml_off = align256(p->ws_o_off + slots * lo.D * 4);
    p->ws_total = align256(p->ws_ml_off + slots * 8);
    p->smem = decode_smem(lo, *p).total;
    if (p->smem > 227 * 1024) return KVQ_ERR_UNSUPPORTED;
    p->NB = KVQ_MAX_DECODE_BLOCKS;   // the launcher lowers it to one wave on the device
    p->inv_nb = 1.0f / p->NB;
    p->inv_cc0 = 1.0f / static_cast<float>(p->CH * p->cpt0);
    p->inv_cc1 = 1.0f / static_cast<float>(p->CHR * p->cpt1);
    return KVQ_OK;
}

// Streaming multiprocessors of `device`, read once per device.
int device_sm_count(int device) {
    static std::mutex mu;
    static int sms[64] = {};
    if (device < 0 || device >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[device] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
        sms[device] = v;
    }
    return sms[device];
}

// One wave of resident blocks of kernel `fn` with `smem` bytes of dynamic shared memory on
// the current device (SM count times the occupancy calculator's blocks per SM), at most
// KVQ_MAX_DECODE_BLOCKS; remembered per (device, kernel, shared memory).  Also raises the
// kernel's dynamic shared-memory limit the first time it needs more than 48 KiB.
int decode_blocks(const void* fn, int threads, int64_t smem, int* nb) {
    struct Entry { int dev; const void* fn; int64_t smem; int nb; };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem) {
                *nb = cache[i].nb;
                return KVQ_OK;
            }
    }
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
        return KVQ_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, static_cast<size_t>(smem)) !=
            cudaSuccess ||
        per_sm < 1)
        return KVQ_ERR_CUDA;
    const int sms = device_sm_count(dev);
    if (sms < 1) return KVQ_ERR_CUDA;
    int64_t n = (int64_t)sms * per_sm;
    if (n > KVQ_MAX_DECODE_BLOCKS) n = KVQ_MAX_DECODE_BLOCKS;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = used < 64 ? cache[used++] : cache[next++ % 64];
    e.dev = dev;
    e.fn = fn;
    e.smem = smem;
    e.nb = static_cast<int>(n);
    *nb = e.nb;
    return KVQ_OK;
}

namespace {
__global__ void k_lengths(Layout lo, const uint8_t* cache, int layer, int32_t* n_out, int32_t* qn_out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= lo.B) return;
    const int32_t* st = state_ptr(lo, cache, layer, b);
    if (n_out) n_out[b] = st[0];
    if (qn_out) qn_out[b] = st[1];
}
}  // namespace

int launch_lengths(const Layout& lo, const uint8_t* cache, int layer, int32_t* n_out, int32_t* qn_out,
                   cudaStream_t stream) {
    k_lengths<<<(lo.B + 127) / 128, 128, 0, stream>>>(lo, cache, layer, n_out, qn_out);
    return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

using kvq::Layout;

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

extern "C" {

int kvq_cache_bytes(const kvq_config* cfg, int64_t tokens, int32_t mode, uint64_t* out_bytes) {
    if (!cfg || !out_bytes || tokens < 0) return KVQ_ERR_ARG;
    if (mode == KVQ_BYTES_FORMULA) {
        if (cfg->layers < 1 || cfg->kv_heads < 1 || cfg->head_dim < 1 || cfg->batch < 1 || cfg->bits < 1 ||
            cfg->bits > 32)
            return KVQ_ERR_ARG;
        // 2 (keys and values) x layers x KV heads x head size x tokens x bytes per value
        const uint64_t bits = 2ull * cfg->layers * cfg->kv_heads * cfg->head_dim * (uint64_t)tokens *
                              cfg->batch * cfg->bits;
        *out_bytes = bits / 8;
        return KVQ_OK;
    }
    if (mode != KVQ_BYTES_LAYOUT) return KVQ_ERR_ARG;
    Layout lo;
    const int rc = kvq::make_layout(cfg, tokens, &lo);
    if (rc != KVQ_OK) return rc;
    *out_bytes = static_cast<uint64_t>(lo.total);
    return KVQ_OK;
}

int kvq_cache_init(const kvq_config* cfg, void* cache, kvq_stream_t stream) {
    if (!cfg || !cache) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (!aligned(cache, 256)) return KVQ_ERR_ALIGN;
    // header, status and the per-sequence counts; the FP8 scale table too (unset scales
    // read as zero until the first append of a layer)
    const int64_t clear = kvq::is_fp8(lo.scheme) ? lo.data_off : lo.state_off + kvq::align256((int64_t)lo.L * lo.B * 16);
    if (cudaMemsetAsync(cache, 0, static_cast<size_t>(clear), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KVQ_ERR_CUDA;
    return KVQ_OK;
}

int kvq_quantize_append(const kvq_config* cfg, void* cache, int32_t layer, int32_t seq_begin,
                        int32_t seq_count, const void* k_new, const void* v_new, int32_t n_new,
                        const int32_t* n_valid, const float* fp8_scales, uint32_t flags,
                        kvq_stream_t stream) {
    if (!cfg || !cache) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (layer < 0 || layer >= lo.L || seq_begin < 0 || seq_count < 0 || seq_begin + (int64_t)seq_count > lo.B)
        return KVQ_ERR_ARG;
    if (n_new < 0) return KVQ_ERR_ARG;
    if (n_new > lo.T) return KVQ_ERR_CAPACITY;
    if (flags & ~static_cast<uint32_t>(KVQ_NO_AUTOFLUSH)) return KVQ_ERR_ARG;
    if (seq_count == 0 || n_new == 0) return KVQ_OK;
    if (!k_new || !v_new) return KVQ_ERR_ARG;
    if (kvq::is_fp8(lo.scheme) && !fp8_scales) return KVQ_ERR_ARG;
    if (lo.PG > 0 && !lo.table) return KVQ_ERR_ARG;
    if (!aligned(cache, 256) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        (n_valid && !aligned(n_valid, 4)) || (fp8_scales && !aligned(fp8_scales, 4)) ||
        (lo.table && !aligned(lo.table, 4)))
        return KVQ_ERR_ALIGN;
    return kvq::launch_append(lo, static_cast<uint8_t*>(cache), layer, seq_begin, seq_count, k_new, v_new,
                              n_new, n_valid, fp8_scales, flags, reinterpret_cast<cudaStream_t>(stream));
}

int kvq_flush_group(const kvq_config* cfg, void* cache, int32_t layer, kvq_stream_t stream) {
    if (!cfg || !cache) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (layer < 0 || layer >= lo.L) return KVQ_ERR_ARG;
    if (lo.PG > 0 && !lo.table) return KVQ_ERR_ARG;
    if (!aligned(cache, 256) || (lo.table && !aligned(lo.table, 4))) return KVQ_ERR_ALIGN;
    return kvq::launch_flush(lo, static_cast<uint8_t*>(cache), layer, reinterpret_cast<cudaStream_t>(stream));
}

int kvq_workspace_bytes(const kvq_config* cfg, uint64_t* out_bytes) {
    if (!cfg || !out_bytes) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    kvq::DecodePlan plan;
    rc = kvq::make_plan(lo, &plan);
    if (rc != KVQ_OK) return rc;
    *out_bytes = static_cast<uint64_t>(plan.ws_total);
    return KVQ_OK;
}

int kvq_decode_attention(const kvq_config* cfg, const void* cache, int32_t layer, const void* q,
                         float softmax_scale, float* out, void* workspace, uint64_t workspace_bytes,
                         kvq_stream_t stream) {
    if (!cfg || !cache || !q || !out || !workspace) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (layer < 0 || layer >= lo.L) return KVQ_ERR_ARG;
    kvq::DecodePlan plan;
    rc = kvq::make_plan(lo, &plan);
    if (rc != KVQ_OK) return rc;
    if (workspace_bytes < static_cast<uint64_t>(plan.ws_total)) return KVQ_ERR_WORKSPACE;
    if (lo.PG > 0 && !lo.table) return KVQ_ERR_ARG;
    if (!aligned(cache, 256) || !aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 256) ||
        (lo.table && !aligned(lo.table, 4)))
        return KVQ_ERR_ALIGN;
    return kvq::launch_decode(lo, plan, static_cast<const uint8_t*>(cache), layer, q, softmax_scale, out,
                              static_cast<uint8_t*>(workspace), reinterpret_cast<cudaStream_t>(stream));
}

int kvq_read_status(const void* cache, const void* workspace, uint32_t* out, kvq_stream_t stream) {
    if (!out) return KVQ_ERR_ARG;
    uint32_t words[2] = {0u, 0u};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cache && cudaMemcpyAsync(&words[0], cache, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVQ_ERR_CUDA;
    if (workspace && cudaMemcpyAsync(&words[1], workspace, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KVQ_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
    *out = words[0] | words[1];
    return KVQ_OK;
}

int kvq_sequence_lengths(const kvq_config* cfg, const void* cache, int32_t layer, int32_t* n_out,
                         int32_t* qn_out, kvq_stream_t stream) {
    if (!cfg || !cache) return KVQ_ERR_ARG;
    Layout lo;
    int rc = kvq::make_layout(cfg, cfg->max_tokens, &lo);
    if (rc != KVQ_OK) return rc;
    if (layer < 0 || layer >= lo.L) return KVQ_ERR_ARG;
    if (!aligned(cache, 256)) return KVQ_ERR_ALIGN;
    if (!n_out && !qn_out) return KVQ_OK;
    return kvq::launch_lengths(lo, static_cast<const uint8_t*>(cache), layer, n_out, qn_out,
                               reinterpret_cast<cudaStream_t>(stream));
}

const char* kvq_status_string(int code) {
    switch (code) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_ARG: return "invalid argument";
        case KVQ_ERR_ALIGN: return "misaligned pointer";
        case KVQ_ERR_CAPACITY: return "more new tokens than the cache capacity";
        case KVQ_ERR_WORKSPACE: return "decode workspace too small";
        case KVQ_ERR_CUDA: return "CUDA launch or copy failed";
        case KVQ_ERR_UNSUPPORTED: return "configuration not supported by this build";
        default: return "unknown status";
    }
}

}  // extern "C"
