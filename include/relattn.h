/*
 * relattn.h -- C ABI of the paged relative-bias attention library (GB300,
 * sm_103a).
 *
 * The operation.  Inkling-family attention is grouped-query attention with no
 * RoPE.  The pre-softmax logit of query i (position P_i, head h) for key j is
 *
 *     q_i . k_j / sqrt(d_qk) + rel[i, h, P_i - j]
 *
 * ("Inkling-Small on Gaudi 2", section "Why it needed a port": rel[i, h, i-j]
 * is a per-query, per-distance term; "vLLM TML Inkling Support", section "TML
 * Inkling Model Architecture": a learned relative-position term added to the
 * pre-softmax logits instead of RoPE).  rel = r @ rel_logits_proj is computed
 * by the model per query and head over distances 0..rel_extent-1 ("Inkling-
 * Small on Gaudi 2", section "Attention with a relative bias"); this library
 * takes it as an input.  A distance at or beyond rel_extent adds 0.
 *
 * Window.  A sliding-window layer (window W > 0) lets the query at position P
 * see keys P-W+1 .. P: W keys counting its own ("Inkling-Small on Gaudi 2",
 * section "Decode window": the mask cuts a 512-key window at exactly 512).
 * W <= 0 is a global layer (every key 0..P).  Only blocks that hold a visible
 * key are read: ceil(W/128)+1 blocks at most on a local layer.
 *
 * Paged KV cache.  Keys and values live in a pool of 128-token blocks
 * ("Inkling-Small on Gaudi 2", section "At a glance": a pool of 2,560 blocks
 * holds 327,680 tokens).  Position pos of sequence b is slot pos % 128 of
 * physical block block_table[b * max_blocks_per_seq + pos / 128].  Layout
 * (row-major, bf16):  k: [num_blocks][128][num_kv_heads][d_qk],
 *                     v: [num_blocks][128][num_kv_heads][d_v].
 * GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 * Softmax scale: 1/sqrt(d_qk), also when d_v != d_qk ("Inkling on Two DGX
 * Sparks", section "Wall 1": head_dim 128, v_head_dim 64).
 *
 * Conventions shared by every entry point.
 *  - All tensor pointers are DEVICE pointers owned by the caller and must be
 *    16-byte aligned.  The library never allocates, frees or synchronises
 *    (except relattn_read_status, which reads a word back).  Work is enqueued
 *    on `stream` (a cudaStream_t; NULL = legacy default stream) and is safe to
 *    capture in a CUDA graph: no call reads device memory from the host.
 *  - Return value: RELATTN_OK or one of the RELATTN_ERR_* codes below.
 *    Argument errors are found on the host before anything is enqueued.
 *  - Errors that only the device can see (a block id outside the pool, a
 *    length beyond the block table) never fault: the kernel skips the
 *    affected tile or sequence, ORs a RELATTN_DEV_* bit into the workspace's
 *    status word and carries on.  A skipped sequence's output rows are zero.
 *  - The workspace (size from relattn_workspace_size) must be zero-filled
 *    once before first use (relattn_workspace_init).  Calls leave it ready for
 *    the next call, also a call whose waits gave up (its split counters still
 *    complete and return to zero); the status word keeps its bits until the
 *    workspace is zero-filled again.  Calls that share one workspace must be
 *    ordered on one stream: concurrent calls on the same workspace race.
 */
#ifndef RELATTN_H_
#define RELATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define RELATTN_OK               0
#define RELATTN_ERR_INVALID_ARG  1 /* null/misaligned pointer, bad size */
#define RELATTN_ERR_UNSUPPORTED  2 /* valid but not built: see relattn_decode */
#define RELATTN_ERR_WORKSPACE    3 /* workspace too small */
#define RELATTN_ERR_CUDA         4 /* a CUDA runtime/driver call failed */

/* Device status bits, ORed into the workspace status word. */
#define RELATTN_DEV_BAD_BLOCK_ID 0x1u /* a needed table entry was outside
                                         [0, num_blocks): its tile was skipped */
#define RELATTN_DEV_BAD_LENGTH   0x2u /* a length outside the block table's
                                         capacity: the sequence was skipped */
#define RELATTN_DEV_WAIT_TIMEOUT 0x4u /* an internal pipeline wait ran past its
                                         limit (about 2 s): the CTA gave up */
#define RELATTN_DEV_Q_RANGE      0x8u /* a call over an e4m3 cache, which computes
                                         in f16, met a query element outside f16's
                                         range (|q| > 65504 after rounding) or not
                                         finite: that row's output is inf or NaN */

/* The paged KV cache (device memory, caller-owned). */
typedef struct relattn_kv_cache {
  void*   k;            /* bf16 [num_blocks][block_size][num_kv_heads][d_qk],
                           or e4m3 [num_blocks][num_kv_heads][block_size][d_qk]
                           (relattn_options.kv)                              */
  void*   v;            /* the same with d_v                                 */
  int32_t num_blocks;   /* physical blocks in the pool                       */
  int32_t block_size;   /* tokens per block: must be 128                     */
  int32_t num_kv_heads; /* Hkv                                               */
  int32_t d_qk;         /* key/query head size: must be 128                  */
  int32_t d_v;          /* value head size: 64 or 128                        */
} relattn_kv_cache;

/* Host-side sizes of one call.  No field is read from device memory. */
typedef struct relattn_dims {
  int32_t batch;              /* B: sequences in the call                   */
  int32_t num_q_heads;        /* Hq: a multiple of Hkv, Hq/Hkv <= 16        */
  int32_t max_blocks_per_seq; /* entries per block_table row                */
  int32_t num_tokens;         /* prefill: T = cu_seqlens[B]; decode: unused */
  int32_t max_q_len;          /* prefill: upper bound of every chunk length
                                 cu_seqlens[b+1]-cu_seqlens[b]; decode: unused */
  int32_t num_ctas;           /* 0: library choice (one persistent CTA per
                                 SM); > 0 forces the grid size (testing)    */
} relattn_dims;

/*
 * Bytes of workspace a decode or prefill call with these sizes needs.  The
 * workspace holds the status word, the split-combine counters and the
 * partial softmax states of split-KV decode.  Returns 0 on invalid sizes.
 */
size_t relattn_workspace_size(const relattn_dims* dims,
                              const relattn_kv_cache* cache);

/* Zero-fill a workspace on `stream` (once, before its first use). */
int relattn_workspace_init(void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Paged decode: one query per sequence, attending to its own cached keys.
 *
 *   q          bf16 [B][Hq][d_qk]
 *   rel        fp32 [B][Hq][rel_extent]: the relative logits of each query
 *   kv_cache   the pool; must already hold each sequence's current token
 *   block_table int32 [B][max_blocks_per_seq]; only the entries of blocks
 *              holding a visible key are read
 *   seq_lens   int32 [B]: tokens in each sequence including the current one;
 *              the query sits at position seq_lens[b]-1.  Must lie in
 *              [1, max_blocks_per_seq*128], else RELATTN_DEV_BAD_LENGTH.
 *   window     W > 0: sliding window of W keys; W <= 0: global layer
 *   rel_extent distances covered by rel; must be a positive multiple of 4
 *   out        bf16 [B][Hq][d_v]
 *
 * Split-KV ("vLLM TML Inkling Support", section "Low-Latency Collectives and
 * Kernels": num_splits picked from batch and KV length): one persistent
 * kernel cuts the total window-aware key work of all sequences into equal
 * contiguous ranges, one per CTA, so the number of splits of each sequence
 * follows from batch, heads and lengths on the device.  A sequence cut by a
 * range boundary leaves partial softmax states in the workspace; the CTA that
 * finishes a sequence last merges them.  All query heads of one KV head are
 * packed into one tile, so each key/value is read once
 * ("Inkling 2 Small on vLLM", section "vLLM integration and optimisation":
 * six heads packed into one tile, KV read once).
 */
int relattn_decode(const void* q, const float* rel,
                   const relattn_kv_cache* kv_cache,
                   const int32_t* block_table, const int32_t* seq_lens,
                   int32_t window, int32_t rel_extent,
                   const relattn_dims* dims, void* out,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Multi-token decode: the verification step of speculative decoding.  Each
 * sequence has k query tokens -- the k newest, whose keys and values are
 * already in the cache -- and token i sits at position seq_lens[b] - k + i,
 * attending causally (and within the window) over the cache
 * ("vLLM TML Inkling Support", section "TML Inkling Model Architecture":
 * chained MTP heads propose up to 9 tokens per forward step; "Inkling 2
 * Small on vLLM", section "vLLM integration and optimisation": one kernel
 * for decode and verification, the heads of a KV group packed into one
 * tile).  relattn_decode is the k = 1 case.
 *
 *   q          bf16 [B][k][Hq][d_qk]
 *   rel        fp32 [B][k][Hq][rel_extent]: relative logits of each token
 *   seq_lens   int32 [B]: tokens in each sequence including all k query
 *              tokens.  Must lie in [k, max_blocks_per_seq*128], else
 *              RELATTN_DEV_BAD_LENGTH and that sequence's rows are zero.
 *   num_query_tokens  k, in [1, 16]; RELATTN_ERR_UNSUPPORTED otherwise
 *   out        bf16 [B][k][Hq][d_v]
 *   other arguments as for relattn_decode; the workspace size does not
 *   depend on k.
 *
 * The g heads of a KV head and up to 16 / g of the tokens share one tile and
 * one read of their keys; when more tokens than that share a KV head (and
 * g <= 8), up to 32 / g of them share a read, their rows split between two
 * tiles.  Larger k is cut into chunks of that many tokens, each reading the
 * keys its tokens see.
 */
int relattn_decode_multi(const void* q, const float* rel,
                         const relattn_kv_cache* kv_cache,
                         const int32_t* block_table, const int32_t* seq_lens,
                         int32_t num_query_tokens, int32_t window,
                         int32_t rel_extent, const relattn_dims* dims,
                         void* out, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Options of the *_ex entry points: the element types of rel and out, and an
 * optional gated output with a sink.  The plain entry points are the
 * defaults: fp32 rel, bf16 out, no sink, no gate.
 *
 *  - bf16 rel halves the bytes of the relative-logit input, which is most of
 *    a chunked prefill's traffic (fp32 [T][Hq][E]); rel is the product
 *    r @ rel_logits_proj of the layer's fused QKVR projection ("Inkling-Small
 *    on Gaudi 2", section "Attention with a relative bias"), which a bf16
 *    model produces in bf16.  Reading: the bias is the bf16 value widened
 *    exactly; everything else is unchanged.
 *  - fp32 out: the attention output kept in fp32, as the vLLM port of
 *    Inkling 2 Small does ("Inkling 2 Small on vLLM", section 准确率评估,
 *    accuracy evaluation).
 */
#define RELATTN_DTYPE_F32 0
#define RELATTN_DTYPE_BF16 1
#define RELATTN_DTYPE_E4M3 2

/*
 *  - sink / gate: the gated attention output of Inkling 2 ("Inkling 2 Small
 *    on vLLM", architecture table row for the attention output: a sigmoid
 *    gate on each head's output with a per-token attention sink).  Reading
 *    (no formula on the pages): sink[row][h] is one more logit in the
 *    softmax's normaliser, with no value, so the weights become
 *    exp(l_j) / (sum_j exp(l_j) + exp(sink)); gate[row][h] multiplies the
 *    head's output by 1 / (1 + exp(-gate)).  Both are fp32 device arrays of
 *    one value per query row and query head ([B][k][Hq] for decode, [T][Hq]
 *    for prefill), or NULL for none; the library reads them and owns
 *    neither.
 */
/*
 *  - kv: the element type of the KV cache.  0 or RELATTN_DTYPE_BF16: bf16.
 *    RELATTN_DTYPE_E4M3: FP8 e4m3 keys and values, one scale per cache, a
 *    key being k_scale times its e4m3 value and a value v_scale times its
 *    e4m3 value ("vLLM TML Inkling Support": FP8 global attention is a
 *    roadmap item; the format is this library's reading).  e4m3 caches are
 *    head-major, [num_blocks][num_kv_heads][128][d] (a token's head row is
 *    only 128 bytes; this keeps each block's rows of one head contiguous),
 *    and num_blocks * num_kv_heads * 128 must stay below 2^31.  Decode
 *    (one or several query tokens, any g) and prefill; d_v = 128
 *    (RELATTN_ERR_UNSUPPORTED otherwise).  The prefill quantises its new
 *    keys and values into the cache as relattn_cache_write does, then
 *    attends over the cache.  The kernels compute with f16 operands: every
 *    e4m3 value is exact in f16, and so is every bf16 q element of magnitude
 *    2^-14 .. 65504 (f16's normal range); smaller ones are rounded, larger
 *    ones overflow; P is f16.  k_scale and v_scale must be finite and > 0.
 */
/*
 *  - logit_scale: the log-position scale of the global layers, which
 *    multiplies q and the rel logits by a factor growing with the log of the
 *    position beyond 128K ("Inkling-Small on Gaudi 2", section "What was
 *    built").  Reading (no formula on the pages): one factor s per query
 *    token, an fp32 device array ([B][k] for decode, [T] for prefill) or
 *    NULL for none, and the logit of that token becomes
 *    s * (q . k / sqrt(d_qk) + rel); a sink logit is not scaled.  The model
 *    computes the factors (1 below 128K).  Each must be finite and > 0 (not
 *    checked: the library does not read device data on the host).
 */
typedef struct relattn_options {
  int32_t rel;       /* RELATTN_DTYPE_F32 or RELATTN_DTYPE_BF16 */
  int32_t out;       /* RELATTN_DTYPE_BF16 or RELATTN_DTYPE_F32 */
  const float* sink; /* NULL, or [rows][Hq] fp32 sink logits */
  const float* gate; /* NULL, or [rows][Hq] fp32 gate logits */
  int32_t kv;        /* 0 / RELATTN_DTYPE_BF16, or RELATTN_DTYPE_E4M3 */
  float k_scale;     /* e4m3 cache: key scale */
  float v_scale;     /* e4m3 cache: value scale */
  const float* logit_scale; /* NULL, or [rows] fp32 per-token logit factors */
} relattn_options;

/*
 * relattn_decode_multi with `options` (k = 1 is relattn_decode).  rel is
 * [B][k][Hq][rel_extent] of options->rel; out is [B][k][Hq][d_v] of
 * options->out; sink and gate, when given, are [B][k][Hq].  A bf16 rel needs
 * rel_extent a multiple of 8 (fp32: of 4): RELATTN_ERR_UNSUPPORTED
 * otherwise; an unknown type code is RELATTN_ERR_INVALID_ARG.  Same
 * workspace, errors and device status as relattn_decode.
 */
int relattn_decode_ex(const void* q, const void* rel, const relattn_options* options,
                      const relattn_kv_cache* kv_cache, const int32_t* block_table,
                      const int32_t* seq_lens, int32_t num_query_tokens, int32_t window,
                      int32_t rel_extent, const relattn_dims* dims, void* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Size of the library-owned scratch array used by relattn_decode_noalloc. */
#define RELATTN_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * Paged decode without a workspace, for callers that cannot allocate device
 * memory.  No counterpart on the pages; this is a convenience of the library.
 *
 * Some hosts own every device buffer themselves -- a serving engine that
 * hands a plugin only its inputs and outputs, or a runtime with a fixed
 * memory budget in which a foreign cudaMalloc (and the synchronisation it
 * implies) is not allowed -- and cannot provide the workspace relattn_decode
 * asks for.  This call takes the same arguments as relattn_decode without the
 * workspace and computes the same result with the same kernel; its split
 * state lives in one array of RELATTN_NOALLOC_SCRATCH_BYTES that the library
 * declares in device memory (held by every GPU that loads the library until
 * the process exits).  It allocates nothing and calls no allocating routine.
 *
 *  - Limit: if the split state for these sizes (relattn_workspace_size)
 *    exceeds RELATTN_NOALLOC_SCRATCH_BYTES, the call returns
 *    RELATTN_ERR_WORKSPACE and enqueues nothing.
 *  - The first call on a device looks up the array's device address (once,
 *    with that device current) and keeps it for the life of the process;
 *    make that first call before any stream capture on that device.  Calls
 *    must run in the device's primary context (the runtime's), and not after
 *    cudaDeviceReset, since either would leave the kept address stale.
 *  - Every call clears the status word and counters of the array on `stream`
 *    before its kernel, so no zero-filling is needed by the caller; the
 *    call's device status bits (RELATTN_DEV_*) stay in the array's status
 *    word until the next call, and relattn_decode_noalloc_status reads them.
 *  - All calls share the one array: calls whose work overlaps on the GPU
 *    (different streams without ordering between them) race and corrupt each
 *    other's results.  Order them on one stream.
 */
int relattn_decode_noalloc(const void* q, const float* rel,
                           const relattn_kv_cache* kv_cache,
                           const int32_t* block_table, const int32_t* seq_lens,
                           int32_t window, int32_t rel_extent,
                           const relattn_dims* dims, void* out, void* stream);

/*
 * Device status bits of the last relattn_decode_noalloc call on the current
 * device: the status word of the library's array, copied to host memory
 * after the work queued on `stream` (enqueue it on the stream of the calls).
 * Like relattn_read_status it synchronises `stream`, so it cannot be
 * captured in a graph.  Returns RELATTN_OK, RELATTN_ERR_INVALID_ARG (status
 * NULL) or RELATTN_ERR_CUDA.
 */
int relattn_decode_noalloc_status(uint32_t* status, void* stream);

/*
 * Chunked prefill with a cached prefix.
 *
 *   q          bf16 [T][Hq][d_qk]: the new tokens of all sequences, packed
 *   k, v       bf16 [T][Hkv][d_qk], [T][Hkv][d_v]: their keys and values
 *   rel        fp32 [T][Hq][rel_extent]
 *   cu_seqlens int32 [B+1]: new tokens of sequence b are rows
 *              cu_seqlens[b] .. cu_seqlens[b+1]-1 (cu_seqlens[0] = 0)
 *   cache      the pool (in-out): new token t of sequence b is first written
 *              to position ctx_lens[b]+t, then attends to positions
 *              0 .. ctx_lens[b]+t (windowed) -- the cached prefix and the
 *              chunk ("Inkling-Small on Gaudi 2", section "Attention with a
 *              relative bias": later chunks and prefix-cache hits prepend the
 *              cached context)
 *   block_table int32 [B][max_blocks_per_seq], covering ctx_lens[b] +
 *              chunk length positions
 *   ctx_lens   int32 [B]: cached prefix lengths
 *   window, rel_extent: as for relattn_decode
 *   out        bf16 [T][Hq][d_v]
 *
 * dims->num_tokens must equal cu_seqlens[B] and dims->max_q_len must bound
 * every chunk length (both host-side; nothing is read back).
 *
 * Work split: over a bf16 cache a work item is one 128-row query tile and two
 * query heads of one KV group, which share each read of their keys and
 * values ("Inkling 2 Small on vLLM", section "vLLM integration and
 * optimisation"); when the one-head items of a call would fit one wave of
 * CTAs (a latency-bound call) and no grid is forced, and over an e4m3 cache,
 * an item is one query tile and one head.  The results do not depend on the
 * split beyond rounding order.
 */
int relattn_prefill(const void* q, const void* k, const void* v,
                    const float* rel, const int32_t* cu_seqlens,
                    const relattn_kv_cache* cache,
                    const int32_t* block_table, const int32_t* ctx_lens,
                    int32_t window, int32_t rel_extent,
                    const relattn_dims* dims, void* out,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * relattn_prefill with `options`: rel [T][Hq][rel_extent] of options->rel,
 * out [T][Hq][d_v] of options->out, sink and gate (when given) [T][Hq],
 * logit_scale (when given) [T], and an e4m3 cache when options->kv says so
 * (see above).  A bf16 rel needs rel_extent a multiple of 8 (fp32: of 4):
 * RELATTN_ERR_UNSUPPORTED otherwise; an unknown type code is
 * RELATTN_ERR_INVALID_ARG.  Everything else as relattn_prefill.
 */
int relattn_prefill_ex(const void* q, const void* k, const void* v, const void* rel,
                       const relattn_options* options, const int32_t* cu_seqlens,
                       const relattn_kv_cache* kv_cache, const int32_t* block_table,
                       const int32_t* ctx_lens, int32_t window, int32_t rel_extent,
                       const relattn_dims* dims, void* out, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * Write new tokens' keys and values into the paged cache without attending:
 * the first step of relattn_prefill on its own, for callers that append
 * tokens themselves (a decode step's newest token, whose key and value
 * relattn_decode expects in the cache already) or that fill an e4m3 cache.
 * No counterpart on the pages beyond that step ("Inkling-Small on Gaudi 2",
 * section "Attention with a relative bias": the prefill writes the new keys
 * and values into the paged cache).
 *
 * Token t of sequence b (packed row cu_seqlens[b] + t, t < cu_seqlens[b+1] -
 * cu_seqlens[b]) goes to slot (ctx_lens[b] + t) % 128 of physical block
 * block_table[b][(ctx_lens[b] + t) / 128].  k [T][Hkv][d_qk] and v
 * [T][Hkv][d_v] are bf16 (16-byte aligned), T = dims->num_tokens; dims gives
 * batch, max_blocks_per_seq, num_tokens and max_q_len (the longest chunk);
 * num_q_heads is not read.  options may be NULL (a bf16 cache); otherwise
 * options->kv picks the cache's type and only kv, k_scale and v_scale are
 * read:
 *  - bf16: the values are copied (bit-exact);
 *  - e4m3 (head-major cache, d_v = 128): each key is stored as the e4m3 code
 *    of (key / k_scale), each value of (value / v_scale), the division in
 *    fp32 and the code the nearest e4m3 value with ties to the even code,
 *    magnitudes beyond 448 stored as +-448 (this library's reading: the
 *    pages name FP8 caches but no quantiser).
 * The workspace holds the status word (at least 256 bytes); a block id
 * outside the pool or an invalid length sets RELATTN_DEV_BAD_BLOCK_ID /
 * RELATTN_DEV_BAD_LENGTH and skips the token / sequence.  Asynchronous on
 * `stream`; nothing is allocated.  Returns RELATTN_OK, RELATTN_ERR_INVALID_ARG,
 * RELATTN_ERR_UNSUPPORTED (e4m3 with d_v != 128, more than 65535 sequences),
 * RELATTN_ERR_WORKSPACE or RELATTN_ERR_CUDA.
 */
int relattn_cache_write(const void* k, const void* v, const relattn_options* options,
                        const int32_t* cu_seqlens, const relattn_kv_cache* kv_cache,
                        const int32_t* block_table, const int32_t* ctx_lens,
                        const relattn_dims* dims, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * Read the device status word of a workspace into *status (synchronises
 * `stream`).  The word accumulates RELATTN_DEV_* bits until cleared with
 * relattn_workspace_init.
 */
int relattn_read_status(const void* workspace, uint32_t* status, void* stream);

/* Human-readable name of a return code. */
const char* relattn_status_string(int code);

/*
 * Test hook: replay the decode kernel's window-aware block walk and work
 * split without computing attention.  Each visited 64-key tile appends one
 * record of 6 int32 to `records` (device, capacity max_records records):
 *   { cta, sequence, kv_head, key_tile (first key / 64),
 *     logical_block, physical_block }
 * and *count (device int32, zero it first) counts the records.  The same
 * device code as relattn_decode picks the tiles.
 */
int relattn_debug_walk_decode(const int32_t* block_table,
                              const int32_t* seq_lens, int32_t window,
                              const relattn_kv_cache* cache,
                              const relattn_dims* dims, int32_t* records,
                              int32_t max_records, int32_t* count,
                              void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Test hook: relattn_debug_walk_decode for num_query_tokens tokens per
 * sequence and the cache type of options->kv (the other option fields are
 * not used; options may be NULL), with 8-int32 records per visited tile:
 *   { cta, sequence, first_token_of_chunk, kv_head, key_tile,
 *     physical_block, first_key, keys }
 * where the tile's keys first_key .. first_key + keys - 1 are the ones the
 * kernel brings: the whole 64-key tile, or with one query token over a bf16
 * cache, the 32-key half that holds the visible keys at an edge of the
 * range.  A chunk is the group of query tokens that share one pass over
 * their keys; its tokens start at first_token_of_chunk.
 */
int relattn_debug_walk_decode_ex(const int32_t* block_table, const int32_t* seq_lens,
                                 int32_t num_query_tokens, int32_t window,
                                 const relattn_options* options, const relattn_kv_cache* cache,
                                 const relattn_dims* dims, int32_t* records,
                                 int32_t max_records, int32_t* count, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Test hook: replay the work split and block walk of the prefill kernel whose
 * work items are a 128-row query tile and a pair of query heads of one KV
 * group (the kernel relattn_prefill runs over a bf16 cache unless the call
 * fits one wave of one-head items), with the same device code and the grid
 * that kernel gets.  Each (work item, key tile) visit appends
 * { sequence, first_row_of_query_tile (within the sequence), key_tile,
 *   logical_block, physical_block, first_head_of_item } (6 int32) to
 * `records`.
 */
int relattn_debug_walk_prefill(const int32_t* cu_seqlens,
                               const int32_t* ctx_lens,
                               const int32_t* block_table, int32_t window,
                               const relattn_kv_cache* cache,
                               const relattn_dims* dims, int32_t* records,
                               int32_t max_records, int32_t* count,
                               void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Test hook: relattn_debug_walk_prefill for the kernel that relattn_prefill_ex
 * runs with these options (options->rel and options->kv decide; the other
 * fields are not used; options may be NULL for the defaults): over a bf16
 * cache with a bf16 rel and d_v = 128, the kernel whose work items are a
 * 128-row query tile and ONE query head over 128-key tiles, whose records
 * are { sequence, first_row_of_query_tile, key_tile, logical_block,
 * physical_block, head } with key_tile counting 128-key tiles (it equals
 * logical_block); otherwise the two-heads kernel's records as above.  e4m3
 * caches: RELATTN_ERR_UNSUPPORTED.
 */
int relattn_debug_walk_prefill_ex(const int32_t* cu_seqlens, const int32_t* ctx_lens,
                                  const int32_t* block_table, int32_t window,
                                  const relattn_options* options,
                                  const relattn_kv_cache* cache, const relattn_dims* dims,
                                  int32_t* records, int32_t max_records, int32_t* count,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Test hook for failure detection: one thread waits on a shared-memory
 * barrier that nothing completes.  Every wait in the library's kernels has a
 * limit (about 2 s) after which it gives up, records
 * RELATTN_DEV_WAIT_TIMEOUT in the workspace's status word and lets the kernel
 * end; this call exercises that path on its own, so a test can see the
 * status bit and that the context stays usable.  Returns after enqueueing
 * (the kernel runs for about 2 s); RELATTN_ERR_WORKSPACE for a workspace
 * below 256 bytes or not 16-byte aligned.
 */
int relattn_debug_wait_timeout(void* workspace, size_t workspace_bytes, void* stream);

/*
 * Test hook for failure detection in the decode kernel: relattn_decode with
 * one change -- in every CTA the consumer warps treat the query wait of
 * their piece number `piece` (0 = the first piece of the CTA's range) as if
 * it had run past its limit.  They record RELATTN_DEV_WAIT_TIMEOUT and give
 * up the rest of their range, as after a real timeout: every split segment
 * that the rest of the range touches still receives the CTA's (empty)
 * partial and its arrival, so the workspace's split counters end at zero and
 * the next call on the same workspace is correct.  The CTA's producer warp
 * then finds no free stage and gives up after its own limit (about 2 s).
 * Output rows of the abandoned pieces are undefined.  RELATTN_ERR_INVALID_ARG
 * for piece < 0; otherwise arguments, errors and status as relattn_decode.
 */
int relattn_debug_decode_give_up(const void* q, const float* rel,
                                 const relattn_kv_cache* kv_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, int32_t window, int32_t rel_extent,
                                 const relattn_dims* dims, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t piece, void* stream);

/* ABI version of this header (major * 100 + minor). */
int relattn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RELATTN_H_ */
