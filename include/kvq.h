/*
 * kvq.h -- C ABI of the sub-byte quantized KV cache for GB300 (sm_103a).
 *
 * What it computes (problem statement from four pages):
 *   [P1] "Hierarchical Token Routing and Sub-2-Bit Non-Linear KV Compression":
 *        outliers beyond a sigma threshold kept in FP8 E4M3 ("1. Dynamic Outlier
 *        Isolation"), the rest as a 4-centroid (2-bit) codebook ("2. Centroid
 *        Vector Quantization for Residuals"), read by one kernel that expands
 *        codes in registers and runs attention on the fly ("Hardware-Kernel
 *        Fusion: Eliminating DRAM Round-Trips").
 *   [P2] "Hierarchical Token Gating and Tiered KV-Cache Paging": a paged cache
 *        whose pages are either FP8 (tier 1) or 2-bit (tier 2)
 *        ("2. Entropy-Guided Tiered KV-Cache Quantization").
 *   [P3] "Sub-5ms MoE Inference: Sub-Byte KV Quantization and Expert Pipelining
 *        at Scale": FP16 outlier tensor beside sub-byte codes ("Sub-Byte
 *        KV-Cache Quantization"); the attention projection fused with the
 *        KV-cache write ("Engineering Real-Time Autonomous Workflows", item 1).
 *   [P4] "The Sub-10ms Barrier: Fusing Sparse MoE Routing with FP4 KV-Cache
 *        Quantization": block-wise asymmetric INT4 and FP4 E2M1 with per-group
 *        scales, dequantized during the flash-decoding reduction
 *        ("2. FP4/INT4 KV-Cache Quantization"), 128-byte aligned pages
 *        ("Key Production Engineering Takeaways").
 *
 * Conventions for every call:
 *   - The caller owns all memory (allocate it with any allocator: torch,
 *     cudaMalloc, a pool).  The library never allocates, never synchronises the
 *     host, and keeps no pointer after a call returns.
 *   - "device" pointers must be CUDA device memory of the current device;
 *     "host" pointers are ordinary host memory read before the call returns.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and runs asynchronously.
 *   - Argument errors return a status before anything is enqueued.  A failed
 *     launch returns KVQ_ERR_CUDA.  Problems only the device can see (a page
 *     table entry out of range, an append past the page table) set bits in the
 *     device word `cache->status` (KVQ_STATUS_*); the affected sequence is
 *     skipped, nothing outside the caller's buffers is touched, and the host
 *     reads the word whenever it chooses.  No call ever traps or spins forever:
 *     every wait in device code (for the asynchronous copies of a page, for a
 *     tensor-memory copy or MMA to complete) gives up after 100 ms and sets
 *     KVQ_STATUS_TIMEOUT.
 *   - No C++ exception crosses this interface.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size, a bad enum */
    KVQ_ERR_UNSUPPORTED = 2,   /* a valid but unimplemented shape (head_dim, group size) */
    KVQ_ERR_WORKSPACE = 3,     /* workspace smaller than kvq_decode_workspace_bytes() */
    KVQ_ERR_CAPACITY = 4,      /* sizes exceed what the layout can index */
    KVQ_ERR_CUDA = 5,          /* the CUDA runtime reported an error at launch */
    KVQ_ERR_TIMEOUT = 6        /* reserved for host-side waits (none today) */
} kvq_status;

/* Cache formats.  Pages hold KVQ_PAGE_TOKENS tokens of one sequence. */
typedef enum {
    /* [P4] asymmetric INT4, groups of 32 along head_dim, fp16 scale S and fp16
     * zero m (x ~ q*S + m); values beyond sigma standard deviations of their
     * group go to a per-token FP16 (channel, value) side-list ([P3]).
     * Quantized per token on arrival. */
    KVQ_FMT_INT4_G32 = 0,
    /* [P4] FP4 E2M1 codes with one FP8 E4M3 scale per 16 values (s =
     * e4m3(amax/6)); no outliers.  Quantized per token on arrival. */
    KVQ_FMT_FP4_E2M1_S16 = 1,
    /* [P1] per (page, channel) 4-centroid fp16 codebook fitted by Lloyd-Max
     * (k-means in one dimension, linspace start) over the page's non-outliers;
     * per-token outliers (sigma rule over the head vector) kept as FP8 E4M3 in
     * a per-page side-list: one (channel, token mask, 16 values) record per
     * channel holding outliers.  Quantized when a page fills; the partial last
     * page waits in fp32 staging. */
    KVQ_FMT_CB2_OUTLIER = 2,
    /* [P2] KVQ_FMT_CB2_OUTLIER pages plus FP8 E4M3 pages with one fp32 scale per
     * (page, head, K|V) (s = amax/448).  A page-table entry with bit 31 set
     * lives in the FP8 tier pool. */
    KVQ_FMT_TIERED = 3,
    /* [P4] "Key Production Engineering Takeaways" item 2: a static
     * high-precision channel mask -- the cfg->static_channels channels of each
     * (kv head, K|V) named by cache->static_mask keep fp16 values for every
     * token; every other channel gets the KVQ_FMT_CB2_OUTLIER codebook fitted
     * over all 16 of its page values (no per-token outlier detection, no
     * side-list).  kvq_select_static_channels picks the mask (top channels by
     * absolute magnitude) from calibration values.  Quantized when a page
     * fills; the partial last page waits in fp32 staging. */
    KVQ_FMT_CB2_STATIC = 4,
    /* [P3] "Sub-Byte KV-Cache Quantization": asymmetric 3-bit codes with
     * dynamic outlier preservation.  Per (page, channel) over its
     * non-outliers: S = fp16((max - min)/7), m = fp16(min), q =
     * clamp(rint((x - m)/S), 0, 7) (fp64); a code stands for
     * fp16(q*S + m).  Outliers as KVQ_FMT_CB2_OUTLIER (sigma rule per token,
     * e4m3 side-list).  Quantized when a page fills; the partial last page
     * waits in fp32 staging. */
    KVQ_FMT_ASYM3_OUTLIER = 5,
    /* [P1] "2. Centroid Vector Quantization for Residuals" (k-means "per
     * head-group block"): as KVQ_FMT_CB2_OUTLIER, but each channel's
     * 4-centroid codebook is fitted over a group of 4 consecutive pages (64
     * tokens) of one (sequence, kv head, K|V) and stored once, in the group's
     * first page; outliers and side-lists stay per page.  Quantized when a
     * group fills; the partial last group (up to 63 tokens) waits in fp32
     * staging [num_seqs][Hkv][2][64][D]. */
    KVQ_FMT_CB2_GROUP4 = 6
} kvq_format;

typedef enum { KVQ_BF16 = 0, KVQ_F16 = 1, KVQ_F32 = 2 } kvq_dtype;

/* Where decode runs the dense QK^T and PV products of the codebook pages.
 * KVQ_DECODE_TENSOR_CORES: mma.sync tiles (the query heads of a kv head are
 * the tile's N = 8 columns; G <= 4 leaves half of them empty).
 * KVQ_DECODE_CUDA_CORES: fp32 FMAs on the dequantized values, only for
 * KVQ_FMT_CB2_OUTLIER at G <= 4 (other formats and larger groups take the
 * tensor cores whatever is asked).  KVQ_DECODE_AUTO picks the one measured
 * faster for the format and group size.  Both give the same quantity within
 * the decode tolerance (different rounding, not the same bits). */
typedef enum { KVQ_DECODE_AUTO = 0, KVQ_DECODE_TENSOR_CORES = 1, KVQ_DECODE_CUDA_CORES = 2 } kvq_decode_math;

#define KVQ_PAGE_TOKENS 16
#define KVQ_TIER_BIT 0x80000000u

/* Bits of the device status word. */
#define KVQ_STATUS_BAD_PAGE     0x1u  /* page-table entry outside its pool: sequence skipped */
#define KVQ_STATUS_CAPACITY     0x2u  /* append past pages_per_seq_max pages: sequence skipped */
#define KVQ_STATUS_SEQ_TOO_LONG 0x4u  /* decode: seq_lens[b] > max_seq_len: tokens beyond ignored */
#define KVQ_STATUS_TIMEOUT      0x8u  /* a bounded device wait gave up */

typedef struct {
    int32_t num_seqs;           /* B: sequences (rows of the page table) */
    int32_t num_kv_heads;       /* Hkv */
    int32_t head_dim;           /* D: 64 or 128 */
    int32_t pages_per_seq_max;  /* columns of the page table */
    int32_t num_pages;          /* physical pages in the main pool */
    int32_t num_tier_pages;     /* physical pages in the FP8 tier pool (TIERED), else 0 */
    int32_t format;             /* kvq_format */
    int32_t lloyd_iters;        /* CB2: maximum Lloyd-Max assignment passes (16) */
    double sigma;               /* outlier threshold in standard deviations, >= 3 (3.0) */
    int32_t static_channels;    /* CB2_STATIC: fp16 channels per (kv head, K|V), 1..8
                                   (ceil(D / 100) for the pages' 1%); ignored otherwise */
    int32_t decode_math;        /* kvq_decode_math (KVQ_DECODE_AUTO = 0) */
} kvq_config;

/* The cache.  All pointers are device memory owned by the caller.
 *   pool        main pool: block (phys, head, role) at
 *               ((phys * Hkv + head) * 2 + role) * kvq_block_bytes(cfg, 0); role 0 = K, 1 = V.
 *               Zero-fill it once before first use.
 *   tier_pool   FP8 pool (TIERED only, else NULL), blocks of kvq_block_bytes(cfg, 1).
 *   page_table  int32 [num_seqs][pages_per_seq_max]: physical page of each
 *               logical page; bit 31 selects the tier pool (TIERED only).
 *               Entries are read only for pages a call touches.
 *   seq_lens    int32 [num_seqs]: tokens cached per sequence; appends advance it.
 *   staging     fp32 [num_seqs][Hkv][2][16][D]: partial last page of the page
 *               formats (CB2, TIERED, CB2_STATIC, ASYM3); [num_seqs][Hkv][2][64][D]
 *               (partial last group) for CB2_GROUP4; NULL for INT4 / E2M1.
 *   status      one uint32 word, OR-ed with KVQ_STATUS_* bits; the caller clears it.
 *   static_mask uint8 [Hkv][2][static_channels] (CB2_STATIC only, else NULL):
 *               the static channels of each (kv head, K|V), ascending, distinct,
 *               below D.  Fixed for the cache's lifetime (set before the first
 *               append, e.g. by kvq_select_static_channels).
 * The byte layout of a block (a definition of this library, chosen so the decode
 * kernel loads tensor-core fragments directly) is given at the end of this
 * header. */
typedef struct {
    void* pool;
    void* tier_pool;
    int32_t* page_table;
    int32_t* seq_lens;
    float* staging;
    uint32_t* status;
    const uint8_t* static_mask;
} kvq_cache;

/* Bytes of one block: tier = 0 for the pool's own format, 1 for an FP8 tier
 * block.  A multiple of 128 ([P4] cache-line aligned pages). */
kvq_status kvq_block_bytes(const kvq_config* cfg, int32_t tier, size_t* bytes);

/* Bytes the caller must allocate for the pool, the tier pool and the staging. */
kvq_status kvq_cache_bytes(const kvq_config* cfg, size_t* pool_bytes, size_t* tier_pool_bytes,
                           size_t* staging_bytes);

/* Quantize-on-append ([P4] "2. FP4/INT4 KV-Cache Quantization": group scales
 * are computed when a token is inserted; [P1] outlier isolation, then the
 * codebook fit).
 *   k_new, v_new  device, [num_seqs][t_new][Hkv][D] in in_dtype (bf16, f16, f32).
 *   t_per_seq     device int32 [num_seqs] or NULL: sequence b appends its first
 *                 t_per_seq[b] <= t_new tokens (ragged batches); NULL = t_new each.
 * Tokens land at positions seq_lens[b] .. ; per-token formats quantize each
 * token in place; page formats write fp32 staging and quantize each page that
 * fills (FP8 when its page-table entry carries the tier bit).  seq_lens is
 * advanced on the device.  The quantizer is defined in fp64 (outlier
 * statistics, the Lloyd-Max fit, scales and codes; ascending-index sums; each
 * result rounded once to its stored format) and the cache is bit-identical to
 * that definition: decisions are taken in binary32 with a certified error
 * bound, and a unit whose decision the bound does not settle (a value within
 * rounding of a threshold or a midpoint) is recomputed in fp64.  Sequences
 * that would overflow their page table or name a bad page are skipped and
 * flagged in the status word. */
kvq_status kvq_quantize_append(const kvq_config* cfg, const kvq_cache* cache, const void* k_new,
                               const void* v_new, kvq_dtype in_dtype, int32_t t_new,
                               const int32_t* t_per_seq, void* stream);

/* K/V projection fused with quantize-on-append ([P3] "Engineering Real-Time
 * Autonomous Workflows", item 1: the attention projection and the KV-cache
 * write in one kernel).  For appended token i of sequence b and kv head h,
 *   k = x[b][i] . W_k[h*D + j][:],  v = x[b][i] . W_v[h*D + j][:]   (j < D)
 * with bf16 operands and fp32 accumulation on the tensor cores; k and v are
 * then quantized into the cache exactly as kvq_quantize_append quantizes fp32
 * inputs (same blocks, staging, seq_lens and status behaviour), without being
 * written to global memory.  Every format.  A one-token append (t_new == 1,
 * the decode-time case) splits hidden across the CTAs of a thread-block
 * cluster and adds their fp32 partial sums in cluster order.
 *   x         device bf16 [num_seqs][t_new][hidden], 16-byte aligned.
 *   hidden    a positive multiple of 32.
 *   w_k, w_v  device bf16 [num_kv_heads * head_dim][hidden] (a linear layer's
 *             weight, output-major), 16-byte aligned.
 *   t_per_seq as for kvq_quantize_append.
 *   kv_out    NULL, or device fp32 [2][num_seqs][t_new][num_kv_heads][head_dim],
 *             16-byte aligned: receives the projected K (index 0) and V of the
 *             tokens appended; other rows are not written.
 * Errors: KVQ_ERR_INVALID_ARG for a null or misaligned pointer or a bad size,
 * KVQ_ERR_UNSUPPORTED for head_dim other than 64 / 128, num_seqs * t_new >= 2^31 or
 * t_new > 8,387,456 (65535 tiles of 128 positions),
 * KVQ_ERR_CAPACITY as for kvq_quantize_append, KVQ_ERR_CUDA when the driver
 * offers no tensor-map encoder or a launch fails.  A tensor-core wait that gives up sets
 * KVQ_STATUS_TIMEOUT and leaves that tile's blocks unwritten. */
kvq_status kvq_project_append(const kvq_config* cfg, const kvq_cache* cache, const void* x, int32_t hidden,
                              const void* w_k, const void* w_v, int32_t t_new, const int32_t* t_per_seq,
                              float* kv_out, void* stream);

/* Workspace bytes kvq_decode_attention needs for (num_q_heads, max_seq_len,
 * num_splits); num_splits = 0 asks for the library's choice. */
kvq_status kvq_decode_workspace_bytes(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len,
                                      int32_t num_splits, size_t* bytes);

/* The split count kvq_decode_attention uses when num_splits == 0. */
kvq_status kvq_decode_num_splits(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len,
                                 int32_t* num_splits);

/* Decode attention over the quantized cache with dequantization fused in
 * ([P1] "Hardware-Kernel Fusion"; [P4] flash-decoding over the compressed
 * cache; [P3] "Sub-Byte Dequantization on the Fly" in tensor-core fragment
 * registers).  One query token per sequence, grouped-query attention:
 *   q       device bf16 [num_seqs][num_q_heads][D]; query head h reads kv head
 *           h / (num_q_heads / Hkv).  Any finite bf16 value: each head is
 *           scaled by a power of two into fp16 range for the tensor cores and
 *           the scale is undone in its scores.
 *   out     device [num_seqs][num_q_heads][D] in out_dtype (bf16 or f32):
 *           softmax(softmax_scale * q K^T) V over the seq_lens[b] cached tokens
 *           (0 for an empty sequence).
 *   max_seq_len  host bound on seq_lens (sizes the split grid); tokens beyond it
 *           are ignored and flagged KVQ_STATUS_SEQ_TOO_LONG.
 *   num_splits   context splits per (sequence, kv head), at most 256
 *           (KVQ_ERR_CAPACITY beyond); 0 = library choice.
 *   workspace    device, >= kvq_decode_workspace_bytes(), 16-byte aligned:
 *           4 * num_seqs * Hkv bytes of arrival counters (padded to 256
 *           bytes), then the fp32 split partials.  The counters must be zero
 *           before a workspace's first use (zero the whole workspace once);
 *           every call leaves them zero again, so one workspace serves calls
 *           of any shape (splits, query heads, length) on the same cache.  Zero
 *           it again after a call that set KVQ_STATUS_TIMEOUT, and before using
 *           it for a cache with more (sequence, kv head) pairs.  The partials
 *           need no initialisation.
 * One kernel launch: split CTAs stream each page's packed blocks into shared
 * memory with bulk asynchronous copies, expand codes straight into
 * tensor-core fragments, correct outliers, run an online softmax and write
 * (m, l, o) partials; the last CTA of each (sequence, kv head) to finish
 * (counted on its arrival counter) merges the splits into `out`. */
kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                int32_t num_q_heads, float softmax_scale, int32_t max_seq_len,
                                int32_t num_splits, void* out, kvq_dtype out_dtype, void* workspace,
                                size_t workspace_bytes, void* stream);

/* The two stages of kvq_decode_attention as separate launches (same
 * arguments, same resolution of num_splits = 0): kvq_decode_split writes the
 * fp32 split partials (m, l, o) of every (sequence, query head, split) into
 * `workspace` and leaves its arrival counters alone; kvq_decode_combine
 * merges them into `out` with the same arithmetic as the fused merge, so
 * split then combine on one stream gives kvq_decode_attention's result. */
kvq_status kvq_decode_split(const kvq_config* cfg, const kvq_cache* cache, const void* q, int32_t num_q_heads,
                            float softmax_scale, int32_t max_seq_len, int32_t num_splits, void* workspace,
                            size_t workspace_bytes, void* stream);
kvq_status kvq_decode_combine(const kvq_config* cfg, int32_t num_q_heads, int32_t max_seq_len, int32_t num_splits,
                              const void* workspace, size_t workspace_bytes, void* out, kvq_dtype out_dtype,
                              void* stream);

/* Decode attention that allocates nothing and takes no workspace.  The pages
 * have no counterpart to this call; it exists for callers that may not
 * allocate device memory when they run decode -- a serving loop that reserves
 * all of its memory at start-up and treats any later allocation as an error,
 * code running inside an allocator or memory-pool callback (allocating there
 * would recurse or deadlock), a plugin whose host hands it only inputs and
 * outputs.  Same arguments and result as kvq_decode_attention without the
 * workspace: the split partials go to one scratch array compiled into the
 * library (KVQ_NOALLOC_SCRATCH_BYTES, a copy on every GPU that loads the
 * library, kept until the process exits).
 *   - Returns KVQ_ERR_WORKSPACE, before anything is enqueued, when the
 *     partials (kvq_decode_workspace_bytes) would exceed the scratch.
 *   - Calls no allocator.  Its first call on a device looks up the scratch's
 *     device address once (cudaGetSymbolAddress, with that device current);
 *     make that first call before any stream capture.
 *   - Every call on a device shares the one scratch, which keeps the last
 *     call's contents; calls that may overlap on the GPU (different streams)
 *     race on it -- serialise them.  Each call first clears its own arrival
 *     counters with a memset on `stream` (their place in the scratch depends
 *     on the call's shape), then launches the decode; the partials need no
 *     initialisation.
 *   - The looked-up address is kept per device ordinal for the life of the
 *     process: do not use this call on a device after cudaDeviceReset. */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_cache* cache, const void* q,
                                        int32_t num_q_heads, float softmax_scale, int32_t max_seq_len,
                                        int32_t num_splits, void* out, kvq_dtype out_dtype, void* stream);

/* The static channel mask of KVQ_FMT_CB2_STATIC ([P4] "Key Production
 * Engineering Takeaways" item 2: the top 1% channels by absolute magnitude stay
 * in FP16): for each (kv head, K|V), the cfg->static_channels channels with the
 * largest max |x| over `t` calibration tokens, ties to the lower channel,
 * written ascending to mask (device uint8 [Hkv][2][static_channels]).
 * k, v: device [t][Hkv][D] in in_dtype (bf16, f16 or f32), t >= 1. */
kvq_status kvq_select_static_channels(const kvq_config* cfg, const void* k, const void* v, kvq_dtype in_dtype,
                                      int32_t t, uint8_t* mask, void* stream);

/* Debug: the values tokens [tok_begin, tok_end) of (seq, kv_head, which = 0 K /
 * 1 V) stand for, as fp32 [tok_end - tok_begin][D] in device memory `out`.
 * Bit-identical to the CPU reference's dequantization. */
kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_cache* cache, int32_t seq, int32_t kv_head,
                          int32_t which, int32_t tok_begin, int32_t tok_end, float* out, void* stream);

/* Static, NUL-terminated description of a status code. */
const char* kvq_status_string(kvq_status status);

/* The CUDA runtime error code (a cudaError_t value) behind the most recent
 * KVQ_ERR_CUDA returned on the calling thread, or 0 if this thread has seen
 * none.  A later successful call does not clear it.  Host only, no GPU needed. */
int32_t kvq_last_cuda_error(void);

/* Static, NUL-terminated name of a CUDA runtime error code (as returned by
 * kvq_last_cuda_error), e.g. "cudaErrorInvalidValue"; the runtime's
 * "unrecognized error code" for values it does not know. */
const char* kvq_cuda_error_name(int32_t error);

/* Library version, "MAJOR.MINOR.PATCH". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

/*
 * Block layout.  A block is one (page, kv head, K|V) slice: 16 tokens x D
 * channels.  Element (t, c), j = c % 16, has a fragment position
 * (lane 0..31, step s = c / 16, slot k 0..7) -- the lane and register half of
 * an m16n8k16 A operand that holds it:
 *   K blocks: lane = 4*(t%8) + (j%8)/2,  k = 2*((t/8) + 2*(j/8)) + j%2
 *             (A = K rows are tokens, columns channels)
 *   V blocks: lane = 4*(j%8) + (t%8)/2,  k = 2*((j/8) + 2*(t/8)) + t%2
 *             (A = V^T rows are channels, columns tokens)
 * NS = D/16.  Offsets in bytes; every unlisted byte is zero.
 *   INT4_G32  [0, 8D)   codes: lane l at 4*NS*l, step s = u32 at +4s, slot k =
 *                       bits 4k..4k+3 (unsigned code 0..15)
 *             8D        {fp16 S, fp16 m} per (token t, group g): 8D + 4*(t*D/32 + g)
 *             10D       u8 outlier count per token [16]
 *             10D+16    u8 channel [16][cap], cap = 3*D/32
 *             10D+16+16*cap  fp16 value [16][cap]
 *             stride 1024 (D=64), 1920 (D=128)
 *   E2M1_S16  [0, 8D)   codes as INT4 (slot k = e2m1 nibble: sign, 2 exponent, 1 mantissa)
 *             8D        e4m3 scale [NS][16]: byte 8D + 16*s + t
 *             stride 640 (D=64), 1152 (D=128)
 *   CB2       [0, 4D)   codes: lane l at 2*NS*l, step s = u16 at +2s, slot k =
 *                       bits 4*(k%4) + 2*(k/4)
 *             4D        codebook: 8 bytes per slot sigma(c) = {u32 L, u32 H}, L byte
 *                       i = low byte of fp16 centroid i, H byte i = its high byte;
 *                       K: sigma(c) = c;  V: sigma(c) = 16*(c/16) + 2*(c%8) + (c%16)/8
 *             12D       outlier side-list, grouped by channel: u8 n_ch (channels
 *                       holding an outlier), u8 total (outliers), 2 zero bytes;
 *                       then n_ch 20-byte records at 12D + 4 + 20*i, channels
 *                       ascending: {u8 channel, 0, u16 token mask, u8 value[16]},
 *                       value[t] = e4m3 of the outlier at token t, 0 where t is
 *                       not an outlier of the channel (K and V alike).  The first
 *                       six records travel with the block's codes; decode reads
 *                       further ones six at a time.
 *             stride 2176 (D=64), 4224 (D=128)
 *   CB2_STATIC [0, 12D) codes and codebook as CB2; the static channels have code 0
 *                       and an all-zero codebook
 *             12D       u8 n_s, u8 channel[n_s] (ascending), zeros to 12D + 16
 *             12D + 16  fp16 value of static channel i, token t at 12D + 16 + 32*i + 2*t
 *             stride 1152 (D=64), 1920 (D=128)
 *   ASYM3     [0, 4D)   low 2 code bits: u32 word j of lane l (steps 2j, 2j+1) at
 *                       4*(l*NS/2 + j), slot k of step s at bit 8*(s%2) + 16*(k%2) + 2*(k/2)
 *             4D        high code bit: u32 word at 4D + 4*(l*NS/4 + s/4), bit
 *                       4*(s%4) + 16*(k%2) + k/2
 *             6D, 8D    fp16 S and m of channel c at +2*rho(c); K: rho(c) = 16*(c/16) +
 *                       4*((c%8)/2) + 2*((c%16)/8) + c%2, V: rho(c) = 16*(c/16) +
 *                       2*(c%8) + (c%16)/8
 *             10D       outlier side-list as CB2's (records at 10D + 4 + 20*i)
 *             stride 2048 (D=64), 3968 (D=128)
 *   CB2_GROUP4 [0, 8D)  the group's codebook, as CB2's (first page of a group; zeros
 *                       in the other three)
 *             8D        codes as CB2's
 *             12D       outlier side-list as CB2's (per page)
 *             stride 2176 (D=64), 4224 (D=128)
 *   FP8 tier  [0, 16D)  codes: lane l at 8*NS*l, step s at +8s, slot k = byte k (e4m3)
 *             16D       fp32 scale
 *             stride 1152 (D=64), 2176 (D=128)
 * A code slot that holds an outlier stores 0; the decoder adds the outlier's
 * difference from code 0's value.
 */

#endif /* KVQ_H_ */
