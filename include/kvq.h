/*
 * kvq.h -- C ABI of the GB300 quantised KV cache library (libkvq.so).
 *
 * The library stores attention keys and values in a packed low-bit cache and runs
 * single-query decode attention over it on one GPU (sm_103a).  Five cache schemes:
 *
 *   KVQ_SCHEME_KIVI      asymmetric b-bit (b = 2, 4, 8): keys quantised per channel over
 *                        groups of G tokens, values per token over groups of Gv channels,
 *                        the newest R tokens kept unquantised in a bf16 window.
 *                        ("Quantizing the KV cache", "Keys and values are shaped
 *                        differently" and "Per-channel and per-token grouping", Q_b
 *                        equation; "KIVI: A Tuning-Free Asymmetric 2bit Quantization for
 *                        KV Cache", "How It Works".)
 *   KVQ_SCHEME_INT8      symmetric round-to-nearest, one fp32 scale per (head, token)
 *                        ("Quantising the Cache", "Workshop" and "Terms / Per-token").
 *   KVQ_SCHEME_FP8_E4M3  E4M3 codes with one fp32 scale per (layer, KV head) for keys and
 *                        one for values ("Quantizing the KV cache", "How the KV cache is
 *                        quantized", FP8 KV cache).
 *   KVQ_SCHEME_FP8_E5M2  the same with E5M2 codes (same section: FP8 as E4M3 or E5M2).
 *   KVQ_SCHEME_INT4      symmetric round-to-nearest at 4 bits, one fp32 scale per (head,
 *                        token), codes in [-7, 7] (the glossary "kv cache quantization":
 *                        INT4 and per-token quantization).
 *
 * Memory ownership: the caller allocates every buffer (the cache, the decode workspace,
 * inputs and outputs) in device memory, and every entry point that takes a workspace
 * allocates nothing.  The one exception is kvq_decode_attention_noalloc, which keeps its
 * scratch in a fixed array of KVQ_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 * library (with a small host-side record of that array's address per device); see its
 * declaration below.  The library also remembers, per device, the SM count and the
 * resident decode blocks per SM it sizes its decode grid by.  All device work is enqueued asynchronously on the caller's stream; no
 * call synchronises except kvq_read_status.  Pointers marked "device" must be device
 * (or managed) memory; the cache must be 256-byte aligned, every other device pointer
 * 16-byte aligned.  Pointers marked "device or mapped host" may also point into
 * page-locked host memory that is mapped into the device's address space under the same
 * address (cudaHostAlloc, or cudaHostRegister with mapping, on a system with unified
 * addressing), with the same alignment: the kernels then read the inputs, or write the
 * outputs, across the host link themselves, with no copy enqueued by the library.  The
 * caller keeps such memory unchanged (inputs) or unread (outputs) until the work on
 * `stream` has completed.
 *
 * Errors: each call returns KVQ_OK (0) or a negative KVQ_ERR_* code for problems found
 * on the host before any work is enqueued (nothing is enqueued then).  Problems that only
 * the GPU can see set sticky KVQ_STATUS_* bits in a status word (the first 4 bytes of the
 * cache for appends and flushes, of the workspace for decodes); read them with
 * kvq_read_status.  No kernel traps or asserts: a failed device check is a status bit.
 *
 * Token layout conventions (row-major, element = in_dtype unless stated):
 *   new keys / values   [seq_count][n_new][kv_heads][head_dim]
 *   queries             [batch][q_heads][head_dim]
 *   decode output       [batch][q_heads][head_dim] fp32
 * Query head hq attends with KV head hq / (q_heads / kv_heads) (grouped-query
 * attention, "Quantizing the KV cache", "The other big memory user").
 *
 * The byte layout of the cache is internal to the library (it is restated, for checking,
 * by the test oracle); callers need not depend on it: kvq_cache_bytes gives the size.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (cudaStream_t); NULL means the legacy default stream. */
typedef struct CUstream_st* kvq_stream_t;

enum kvq_scheme {
    KVQ_SCHEME_KIVI = 0,
    KVQ_SCHEME_INT8 = 1,
    KVQ_SCHEME_FP8_E4M3 = 2,
    KVQ_SCHEME_FP8_E5M2 = 3,
    KVQ_SCHEME_INT4 = 4
};

enum kvq_dtype {
    KVQ_DTYPE_BF16 = 0, /* bfloat16 inputs (required for KIVI: the window stores them as is) */
    KVQ_DTYPE_F32 = 1   /* fp32 inputs (INT8, INT4 and FP8 schemes) */
};

enum kvq_bytes_mode {
    KVQ_BYTES_FORMULA = 0, /* 2 x layers x kv_heads x head_dim x tokens x batch x bits / 8 */
    KVQ_BYTES_LAYOUT = 1   /* the real allocation: codes, scales, window, header */
};

enum kvq_append_flags {
    KVQ_NO_AUTOFLUSH = 1u  /* KIVI: leave full groups in the window until kvq_flush_group */
};

enum kvq_error {
    KVQ_OK = 0,
    KVQ_ERR_ARG = -1,        /* bad configuration, null pointer, out-of-range index */
    KVQ_ERR_ALIGN = -2,      /* a pointer is not aligned as required */
    KVQ_ERR_CAPACITY = -3,   /* n_new exceeds the per-sequence capacity */
    KVQ_ERR_WORKSPACE = -4,  /* workspace smaller than kvq_workspace_bytes */
    KVQ_ERR_CUDA = -5,       /* a CUDA launch or copy failed */
    KVQ_ERR_UNSUPPORTED = -6 /* a valid combination this build has no kernel for */
};

enum kvq_status_bits {
    KVQ_STATUS_CAPACITY = 1u,  /* an append would exceed max_tokens: that sequence was skipped */
    KVQ_STATUS_RING_FULL = 2u, /* KIVI no-autoflush append would overflow the window: skipped */
    KVQ_STATUS_NONFINITE = 4u, /* a NaN or infinity reached a quantiser (values still stored) */
    KVQ_STATUS_TIMEOUT = 8u,   /* a bounded wait for an asynchronous copy gave up: output invalid */
    KVQ_STATUS_BAD_PAGE = 16u  /* a block-table entry outside the page pool: appends and flushes
                                  left that sequence unchanged, a decode's output is invalid */
};

/*
 * Cache configuration.  The arguments follow the pages' formulation of the cache size
 * ("Quantizing the KV cache", "The other big memory user": layers, KV heads, head size,
 * tokens, bytes per value) and of KIVI (bit width, group size, residual length).
 *   scheme      kvq_scheme
 *   layers      number of layers held by this cache (>= 1)
 *   batch       number of sequences (>= 1)
 *   q_heads     query heads; q_heads / kv_heads must be 1, 2, 4 or 8
 *   kv_heads    key/value heads
 *   head_dim    channels per head: 64, 128 or 256 (KIVI); 32, 64, 128 or 256 (INT8, INT4, FP8)
 *   bits        KIVI: 2, 4 or 8; the other schemes fix their code width and ignore it (the
 *               formula mode uses it as the bits per value, and accepts 16 for an
 *               unquantised reference size)
 *   group_k     KIVI G: tokens per key group, a multiple of 16 in [16, 128]
 *   group_v     KIVI Gv: channels per value group, a multiple of 16 dividing head_dim
 *   residual    KIVI R: newest tokens kept in the bf16 window (>= 0)
 *   max_tokens  per-sequence capacity in tokens (>= 1)
 *   in_dtype    kvq_dtype of keys, values and queries (KIVI: bf16 only)
 *   page_groups KIVI paged layout: group records per page; 0 for the contiguous layout
 *               (the other schemes: 0 only)
 *   num_pages   paged layout: pages in the cache's pool (>= 1)
 *   rope_base   KIVI: keys are cached before the rotary position embedding and the decode
 *               rotates every dequantised key at its position ("KVQuant: Towards 10 Million
 *               Context Length ...", "Key points": keys quantised before RoPE, which mixes
 *               channel pairs); the embedding's base (e.g. 10000), or 0 for keys cached as
 *               given.  Channel i is paired with i + head_dim/2; the angle of pair i at
 *               position t is the binary32 product t * w_i, w_i = base^(-2i/head_dim)
 *               rounded to binary32; the query is passed already rotated.  The other
 *               schemes: 0 only.
 *   block_table paged layout, device int32 [batch][max_pages], max_pages = ceil(NG /
 *               page_groups) with NG = floor((max_tokens - residual) / group_k) group slots
 *               per sequence: the pool page holding each run of page_groups group slots of
 *               each sequence.  Read by every call that reads or writes group records
 *               (appends, flushes, decodes), so the caller may hand a sequence new pages
 *               between calls; unused for the contiguous layout.
 *   outliers    KIVI dense-and-sparse quantisation: in every quantisation vector (a key
 *               channel over the G tokens of a group, a token's values over one group of Gv
 *               channels) the `outliers` elements of largest magnitude are kept aside in
 *               bf16 and the Q_b parameters are fitted to the other elements ("KVQuant:
 *               Towards 10 Million Context Length ...", "Summary": a small fraction of
 *               outlier values is moved, per vector, into a separate sparse representation;
 *               "Key points": 1% outliers).  0 (plain KIVI) to 4, KIVI only.  Magnitude is
 *               the bf16 pattern with its sign cleared, compared as an integer (a NaN ranks
 *               above an infinity); equal magnitudes go to the lower index first.  The
 *               outliers' dense codes are 0 and the decode uses their bf16 values.
 * Paged layout ("KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache", "Key
 * Takeaways for Interviews": KIVI pairs with PagedAttention, whose fixed-size pages are
 * found through a per-sequence block table): the packed group records live in a pool of
 * num_pages pages instead of one fixed region per (layer, sequence, KV head).  A page holds
 * page_groups consecutive group slots of one sequence for every layer and KV head; group
 * slot g of sequence b is in page block_table[b][g / page_groups].  The bf16 window, the
 * token counts and the header stay where they are.  A table entry outside [0, num_pages)
 * sets KVQ_STATUS_BAD_PAGE: an append or flush that would write through it leaves that
 * sequence unchanged; a decode reads page 0 instead (its output is then invalid).
 */
typedef struct kvq_config {
    int32_t scheme;
    int32_t layers;
    int32_t batch;
    int32_t q_heads;
    int32_t kv_heads;
    int32_t head_dim;
    int32_t bits;
    int32_t group_k;
    int32_t group_v;
    int32_t residual;
    int32_t max_tokens;
    int32_t in_dtype;
    int32_t page_groups;
    int32_t num_pages;
    const int32_t* block_table;
    float rope_base;
    int32_t outliers;
} kvq_config;

/*
 * kvq_cache_bytes -- size of a cache, host arithmetic only (no GPU needed).
 *   mode KVQ_BYTES_FORMULA: the pages' formula ("The other big memory user") for `tokens`
 *        tokens per sequence over all layers and sequences, cfg->bits bits per value,
 *        scales ignored.  Validates only the dimensions it uses.
 *   mode KVQ_BYTES_LAYOUT: bytes to allocate for a cache whose per-sequence capacity is
 *        `tokens` (cfg->max_tokens is ignored); includes codes, scales, the KIVI window
 *        and the header.  Validates the whole configuration.
 *   out_bytes (host) receives the size.  Returns KVQ_OK or KVQ_ERR_ARG.
 */
int kvq_cache_bytes(const kvq_config* cfg, int64_t tokens, int32_t mode, uint64_t* out_bytes);

/*
 * kvq_cache_init -- make `cache` (device, kvq_cache_bytes(LAYOUT, max_tokens) bytes) an
 * empty cache: clears the header, status and per-sequence token counts.  Codes, scales
 * and window contents need no clearing.  Enqueued on `stream`.
 */
int kvq_cache_init(const kvq_config* cfg, void* cache, kvq_stream_t stream);

/*
 * kvq_quantize_append -- append new tokens' keys and values of one layer to sequences
 * [seq_begin, seq_begin + seq_count), quantising and packing them.
 *   k_new, v_new  device or mapped host, [seq_count][n_new][kv_heads][head_dim] in
 *                 cfg->in_dtype
 *   n_new         tokens per sequence in the input rows (0 <= n_new <= max_tokens)
 *   n_valid       device int32 [seq_count] or NULL: sequence i appends its first
 *                 n_valid[i] rows (0..n_new), the rest of its rows are ignored
 *   fp8_scales    FP8 only, device fp32 [kv_heads][2] = (key scale, value scale) of this
 *                 layer: codes are e4m3(x / scale) (saturating at +-448) or e5m2(x /
 *                 scale) (saturating at +-57344), round-to-nearest-even, NaN to 0x7f.  The
 *                 scales are also stored in the cache for decoding, so they must stay the
 *                 same for every append to a layer.  Ignored otherwise.
 *   flags         KVQ_NO_AUTOFLUSH or 0
 * KIVI: tokens enter the bf16 window; whenever the window would hold R + G tokens its
 * oldest G are quantised as one group ("Quantizing the KV cache", "Keys and values are
 * shaped differently" and "Per-channel and per-token grouping": recent tokens wait
 * unquantised in a window that is packed group by group, and the newest R always stay
 * unquantised).  Keys: per channel over the group's
 * G tokens; values: per token over each Gv channels; parameters s = (max - min) /
 * (2^b - 1) and min are stored as fp16 (min rounded down, s rounded up), codes are
 * round-half-even((x - min) / s) in fp32.  With KVQ_NO_AUTOFLUSH the groups wait in the
 * window (which holds R + G tokens) until kvq_flush_group; an append that would overflow
 * it sets KVQ_STATUS_RING_FULL and leaves that sequence unchanged.
 * INT8: each token's key and value per head get scale = max|x| / 127 and codes
 * round-half-even(x / scale) in [-127, 127]; INT4 the same with max|x| / 7 and codes in
 * [-7, 7], two per byte (even channel in the low four bits).  An append past max_tokens sets KVQ_STATUS_CAPACITY and
 * leaves that sequence unchanged.  Appends of at most 16 tokens run as one kernel.
 */
int kvq_quantize_append(const kvq_config* cfg, void* cache, int32_t layer, int32_t seq_begin,
                        int32_t seq_count, const void* k_new, const void* v_new, int32_t n_new,
                        const int32_t* n_valid, const float* fp8_scales, uint32_t flags,
                        kvq_stream_t stream);

/*
 * kvq_flush_group -- KIVI: quantise every full group waiting in the window of every
 * sequence of `layer`: while a window holds at least R + G tokens, its oldest G tokens
 * become one packed group.  This is the window rule of "Quantizing the KV cache": a full
 * window of recent keys is quantised together as one group ("Keys and values are shaped
 * differently"), and the newest R tokens stay in full precision ("Per-channel and
 * per-token grouping", residual length R; "KIVI: A Tuning-Free Asymmetric 2bit
 * Quantization for KV Cache", "How It Works").  The group's codes and parameters are
 * those of kvq_quantize_append.  A no-op for the other schemes and for caches appended
 * with automatic flushing.  Enqueued on `stream`; host argument errors as for
 * kvq_quantize_append.
 */
int kvq_flush_group(const kvq_config* cfg, void* cache, int32_t layer, kvq_stream_t stream);

/*
 * kvq_workspace_bytes -- device scratch needed by kvq_decode_attention for this
 * configuration: the per-chunk partial softmax results of the split context, plus a
 * 256-byte header holding the decode status word and a 4096-byte table of chunk counters
 * (bytes 256..4351) that the decode uses and leaves at zero.  The pages define no split of the
 * context: splitting a sequence's tokens into chunks that run in parallel and merging
 * their partial softmax results by log-sum-exp is this library's design for long
 * contexts (the merge is exact: the chunks' partials give the unsplit softmax).  Host
 * arithmetic only, no GPU needed: the size is an upper bound that holds for decode grids
 * of up to KVQ_MAX_DECODE_BLOCKS blocks (the decode uses fewer on smaller GPUs).
 * out_bytes (host) receives the size.  Returns KVQ_OK, KVQ_ERR_ARG or
 * KVQ_ERR_UNSUPPORTED.
 */
#define KVQ_MAX_DECODE_BLOCKS 2048
int kvq_workspace_bytes(const kvq_config* cfg, uint64_t* out_bytes);

/*
 * kvq_decode_attention -- one decode step of single-query attention for every sequence of
 * one layer ("Quantizing the KV cache", "Why values per token": o = sum_t p_t V_t with
 * p = softmax over the cached tokens of softmax_scale * q . K_t).
 *   cache       device, the cache (read only)
 *   q           device or mapped host, [batch][q_heads][head_dim] in cfg->in_dtype
 *   out         device or mapped host, fp32 [batch][q_heads][head_dim]; a sequence with
 *               no tokens gets 0
 *   workspace   device, at least kvq_workspace_bytes bytes, whose first 4352 bytes are
 *               zero before its first decode (every decode leaves bytes 4..4351 as it
 *               found them); its first 4 bytes are the decode status word (sticky; clear
 *               it with a memset to restart)
 * Every cache byte is read once per step for all the query heads that share it.  The
 * context is split into chunks processed in parallel; their partial results are merged
 * by log-sum-exp.  The split follows the token counts held in the cache: one wave of
 * blocks, each taking an equal share of the bytes the step reads (or, for few long
 * sequences, taking chunks of its sequence on demand until none is left).  Calls that
 * overlap on the GPU must not share a workspace.
 * Self-test of the bounded waits: when bytes 8..15 of the workspace hold
 * KVQ_SELFTEST_WAIT_MAGIC (little-endian uint64), every decode block makes its first
 * staging wait on a barrier that nothing completes.  The wait gives up after its limit
 * (about one second), the block sets KVQ_STATUS_TIMEOUT, waits for its copy in flight and
 * leaves empty partial results (the outputs are then 0); the GPU stays usable.  A zeroed
 * workspace header decodes normally.
 */
#define KVQ_SELFTEST_WAIT_MAGIC 0x4b56515449434b31ull
int kvq_decode_attention(const kvq_config* cfg, const void* cache, int32_t layer, const void* q,
                         float softmax_scale, float* out, void* workspace,
                         uint64_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_decode_attention_noalloc -- the same decode as kvq_decode_attention for callers that
 * cannot allocate device memory for a workspace: code running where cudaMalloc is not
 * allowed or not wanted (an allocator or memory-pool callback, a plugin whose host owns all
 * device memory, a path that must not synchronise the device the way an allocation can).
 * The pages have no counterpart: this is an interface convenience of this library.
 *   The split-context scratch lives in a fixed array of KVQ_NOALLOC_SCRATCH_BYTES that the
 *   library holds in device memory on every GPU that loads it, until the process exits.
 *   Configurations whose kvq_workspace_bytes exceeds it are rejected with
 *   KVQ_ERR_WORKSPACE before anything is enqueued.  The call allocates nothing.
 *   The first call on a device looks the array's device address up (with that device
 *   current) and remembers it for the device's current CUDA context; a later call in a
 *   new context (after cudaDeviceReset, for example) looks it up again.  Make the first
 *   call in each context before any stream capture.
 *   Every call on a device shares the one array and it keeps the previous call's
 *   contents: calls that overlap on the GPU (different streams, or threads) race and
 *   corrupt each other's results; serialise them.  Each call clears the array's status
 *   word; a device-side status (a bounded wait that gave up) is not reported by this
 *   variant.  Arguments, layouts and the output are those of kvq_decode_attention.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)
int kvq_decode_attention_noalloc(const kvq_config* cfg, const void* cache, int32_t layer, const void* q,
                                 float softmax_scale, float* out, kvq_stream_t stream);

/*
 * kvq_read_status -- OR of the status words of `cache` and `workspace` (either may be
 * NULL) into *out (host).  Synchronises `stream` to read them.  The pages define no error
 * reporting; the status bits name the conditions the pages' method leaves open on a
 * device: a sequence past its capacity, a window that must not be flushed yet
 * ("Quantizing the KV cache", "Keys and values are shaped differently": recent tokens
 * wait in a window of fixed size) and a non-finite value reaching the Q_b quantiser
 * ("Per-channel and per-token grouping", whose min, max and scale are then undefined).
 * Returns KVQ_OK, KVQ_ERR_ARG (out is NULL) or KVQ_ERR_CUDA.
 */
int kvq_read_status(const void* cache, const void* workspace, uint32_t* out, kvq_stream_t stream);

/* kvq_sequence_lengths -- copies the per-sequence token counts of `layer` (n, tokens cached,
 * and qn, tokens held in packed groups) into device int32 n_out[batch], qn_out[batch]
 * (either may be NULL).  Enqueued on `stream`. */
int kvq_sequence_lengths(const kvq_config* cfg, const void* cache, int32_t layer, int32_t* n_out,
                         int32_t* qn_out, kvq_stream_t stream);

/* kvq_status_string -- a static, NUL-terminated description of a KVQ_ERR_* code (never
 * NULL; unknown codes get "unknown status").  No counterpart on the pages: it only names
 * this library's host-side error codes. */
const char* kvq_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
