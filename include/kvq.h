/*
 * kvq.h — C ABI of libkvq.so: low-bit KV-cache quantization (KIVI-style
 * asymmetric min–max codes, MixKVQ query-aware mixed-precision keys) and
 * fused decode attention over the packed cache, for one GB300 GPU (sm_103a).
 *
 * Sources, cited by page title and section:
 *  - "KIVI: KV cache axes" article: §1 decode attention s = qK^T/sqrt(D),
 *    p = softmax(s), o = pV; §2 group contract m = min, step =
 *    (max - m)/(2^b - 1), c = RNE((x - m)/step), x^ = m + step*c; §3 Key
 *    groups per channel over consecutive tokens, Value groups per token over
 *    consecutive channels; §4 residual buffer sealed in whole groups; §6 one
 *    global softmax over quantized history and residual; §7 byte accounting.
 *  - "MixKVQ: Query-Aware Mixed-Precision KV Cache Quantization for
 *    Long-Context Reasoning": salience A_d = I_d * S_d, three tiers
 *    BF16/UINT4/UINT2, residual R = 128 with lazy update, Algorithm 1
 *    (Prefill / Decoding / KeyQuant), GQA aggregation.
 *  - "PN-Mix" reproduction notes: Eq. 2 (clipped codes, constant-group
 *    branch), App. G (Key codes packed along tokens), the cache API shape
 *    (from_prefill / append / attention / storage; [batch, heads, tokens,
 *    head_dim]; query heads ordered by GQA group).
 *
 * Conventions for every call:
 *  - Device pointers are caller-owned, contiguous, on the current device and
 *    must stay valid until the stream work that uses them has finished.
 *  - Every call that takes a stream only enqueues work on it (asynchronous);
 *    none synchronizes except kvq_cache_status.
 *  - bf16 tensors are passed as kvq_bf16 (raw bf16 bit patterns).
 *  - Query head h reads KV head h / (Hq / Hkv) (heads ordered by GQA group).
 *  - Return value: KVQ_OK or one KVQ_ERR_* code; on error nothing was
 *    enqueued and the cache state is unchanged.  Data-dependent problems
 *    (non-finite input, an unrepresentable step) cannot be seen on the host
 *    without a sync; kernels record them as sticky flags in a device status
 *    word read by kvq_cache_status.
 *  - There is no CPU fallback: every computation runs in this library's
 *    CUDA kernels.
 *  - A kvq_cache handle is not thread-safe.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvq_bf16; /* raw bf16 bit pattern */

/* Fixed geometry of this implementation. */
#define KVQ_HEAD_DIM 128     /* D */
#define KVQ_K_GROUP 128      /* Key group: tokens per channel group        */
#define KVQ_V_GROUP 32       /* Value group: channels per token group      */
#define KVQ_RESIDUAL 128     /* R: residual capacity = flush granularity   */

/* Return codes. */
enum {
  KVQ_OK = 0,
  KVQ_ERR_ARG = 1,            /* NULL pointer, bad enum, negative size      */
  KVQ_ERR_SHAPE = 2,          /* unsupported geometry (D, bits, heads)      */
  KVQ_ERR_CAPACITY = 3,       /* quantized history would exceed max_tokens  */
  KVQ_ERR_RESIDUAL_FULL = 4,  /* append with 128 residual tokens: flush     */
  KVQ_ERR_RESIDUAL_NOT_FULL = 5, /* flush with fewer than 128 tokens        */
  KVQ_ERR_EMPTY = 6,          /* attention over a cache with no tokens      */
  KVQ_ERR_NOT_EMPTY = 7,      /* prefill into a cache that holds tokens     */
  KVQ_ERR_CUDA = 8,           /* a CUDA call or launch failed               */
  KVQ_ERR_WORKSPACE = 9,      /* workspace NULL or smaller than required    */
  KVQ_ERR_MODE = 10           /* call does not match the cache's key mode   */
};

/* Sticky device status flags (OR-ed), read by kvq_cache_status. */
enum {
  KVQ_FLAG_NONFINITE = 1,     /* a group held a NaN or infinity             */
  KVQ_FLAG_RANGE = 2,         /* (max - min)/(2^b - 1) not positive finite  */
  KVQ_FLAG_TIMEOUT = 4        /* a decode wait for staged data gave up; that
                                 call's output is invalid                   */
};

/* Key storage mode.  KVQ_K_KIVI is the KIVI article's streaming cache
 * ("KIVI: KV cache axes" §4–§7; MixKVQ's experimental setting G = 32, R =
 * 128): keys quantized per channel in groups of 32 tokens, sealed 128
 * tokens at a time (the key residual holds 0..127 tokens after every
 * append); values a FIFO residual of 128 tokens whose oldest token, once
 * the FIFO is full, leaves quantized per token in groups of 32 channels;
 * origins and steps kept in bf16 and computed in bf16 (every quantizer
 * operation an fp32 operation rounded to bf16; RNE codes, clipped; a
 * constant group keeps step 0).  k_bits = v_bits = 2 or 4; no sink window.
 * Appends seal keys themselves (kvq_flush_group returns MODE);
 * kvq_cache_lengths gives (quantized keys T_k, key residual r_K); with t =
 * T_k + r_K tokens, the values of the first max(0, t - 128) are quantized
 * and the last min(t, 128) sit in the FIFO.  The decode attends over all
 * t tokens with one softmax; each token's value comes from the side of the
 * value boundary it is on (§6). */
enum { KVQ_K_UNIFORM = 0, KVQ_K_MIXED = 1, KVQ_K_KIVI = 2, KVQ_K_PNMIX = 3 };

/* KVQ_K_PNMIX: PN-Mix H3/L1 keys (PN-Mix reproduction notes, Eq. 2, Eq. 6,
 * Eq. 7, App. G).  Once per prefill, kvq_pnmix_pairs scores every RoPE
 * channel pair of each (batch row, KV head) by Eq. 6 (mean pair norm of the
 * GQA group's prefill queries times that of the prefill keys) and keeps the
 * n_high_pairs highest (ties: the lower pair) at 3 bits; the other channels
 * take one bit with Eq. 7's midpoint correction.  Every 128-token key group
 * is quantized per channel: high channels by Eq. 2 (min-max, origin the
 * minimum, codes 0..7), low channels by Eq. 7 (scale s = (M - m)/2, offset
 * z = (3m + M)/4, code RNE((x - z)/s) clipped to 0..1), fp32 arithmetic
 * (each step rounded to fp32), fp32 offsets and scales.  Storage (App. G):
 * the codes' least significant bits over all channels (one bit each), then
 * the upper two bits of the high channels' codes.  Values as KVQ_K_UNIFORM
 * (v_bits per token over 32 channels).  k_bits is ignored; n_high_pairs is
 * a multiple of 16 in 0..64; no sink window.  The decode stores each
 * unit's channels with the selected pairs first (a fixed permutation of
 * the dot product), so the upper plane is dense. */
enum { KVQ_PAIRS_ADJACENT = 0, KVQ_PAIRS_SPLIT = 1 };

/* Channel tier ids (MixKVQ three-tier strategy). */
enum { KVQ_TIER_BF16 = 0, KVQ_TIER_UINT4 = 1, KVQ_TIER_UINT2 = 2 };

/*
 * Tier selection rule (kvq_channel_saliency, and a mixed cache's flushes).
 * In a mixed cache the record of a group has room for n_bf16 BF16 and
 * n_uint4 UINT4 channels; under THRESHOLD the channels are taken from the
 * largest A_d down, and a channel over its tier's room drops one tier.
 */
enum { KVQ_TIERS_RANK = 0, KVQ_TIERS_THRESHOLD = 1 };

typedef struct kvq_config {
  int batch;       /* B >= 1                                                */
  int kv_heads;    /* Hkv >= 1                                              */
  int head_dim;    /* D; must be KVQ_HEAD_DIM                               */
  int max_tokens;  /* capacity of the quantized history; multiple of 128    */
  int k_bits;      /* 2 or 4 (KVQ_K_UNIFORM, KVQ_K_KIVI); ignored for
                      KVQ_K_MIXED                                            */
  int v_bits;      /* 2 or 4                                                */
  int k_mode;      /* KVQ_K_UNIFORM, KVQ_K_MIXED or KVQ_K_KIVI              */
  int n_bf16;      /* KVQ_K_MIXED: BF16-tier channels per key group (RANK),
                      or at most that many (THRESHOLD)                      */
  int n_uint4;     /* KVQ_K_MIXED: UINT4-tier channels per key group (RANK),
                      or at most that many (THRESHOLD); the remaining
                      channels are UINT2                                    */
  int n_sink;      /* attention-sink window, 0..128: the sequence's first
                      n_sink tokens stay bf16 and are never quantized
                      (PN-Mix sink protection, N_s = 32; InnerQ's
                      high-precision window); 0 = none                      */
  int tier_mode;   /* KVQ_K_MIXED: KVQ_TIERS_RANK (0) or KVQ_TIERS_THRESHOLD */
  float tau_bf16;  /* THRESHOLD: A_d > tau_bf16 -> BF16 (MixKVQ tau_BF16)   */
  float tau_uint4; /* THRESHOLD: A_d > tau_uint4 -> UINT4 (tau_UINT4)       */
  int n_high_pairs;/* KVQ_K_PNMIX: channel pairs kept at 3 bits (multiple of
                      16, 0..D/2)                                            */
  int pair_layout; /* KVQ_K_PNMIX: KVQ_PAIRS_ADJACENT (pair i = channels 2i,
                      2i + 1, the paper's formula) or KVQ_PAIRS_SPLIT
                      (channels i, i + D/2, the Hugging Face Llama layout)  */
} kvq_config;

typedef struct kvq_tier_spec {
  int mode;         /* KVQ_TIERS_RANK or KVQ_TIERS_THRESHOLD                */
  int n_bf16;       /* RANK: channels with the largest A_d kept BF16        */
  int n_uint4;      /* RANK: the next channels stored UINT4                 */
  float tau_bf16;   /* THRESHOLD: A_d > tau_bf16 -> BF16                    */
  float tau_uint4;  /* THRESHOLD: tau_uint4 < A_d <= tau_bf16 -> UINT4      */
} kvq_tier_spec;

typedef struct kvq_cache kvq_cache; /* opaque */

/*
 * Device bytes one cache needs: the packed history (per (batch row, KV
 * head), max_tokens/128 group records of codes plus per-group origins
 * (bf16) and steps (fp32)), the bf16 residual windows [B][Hkv][128][D] for
 * K and V, the bf16 sink windows [B][Hkv][n_sink][D], and the status word.
 * KIVI article §7 gives the accounting.
 * Returns 0 for an invalid config.
 */
size_t kvq_cache_bytes(const kvq_config* cfg);

/*
 * Create a cache: the state MixKVQ Algorithm 1 keeps per layer (the packed
 * history, the full-precision residual; MixKVQ "system-level implementation
 * details": quantized store, BF16 outlier store, residual) and KIVI §4's
 * residual state machine.  dev_buf: NULL -> the library allocates kvq_cache_bytes
 * with cudaMallocAsync on s and frees it in kvq_cache_free; else a caller
 * buffer of buf_bytes >= kvq_cache_bytes (256-byte aligned), which the
 * caller keeps alive and frees after kvq_cache_free.  The cache starts
 * empty (no quantized tokens, empty residual, status 0).
 * Errors: ARG, SHAPE, CAPACITY (buf too small), CUDA.
 */
int kvq_cache_alloc(const kvq_config* cfg, void* dev_buf, size_t buf_bytes,
                    cudaStream_t s, kvq_cache** out);
/* Release a cache of kvq_cache_alloc (its own allocation freed on s; a
 * caller buffer is left to the caller).  Errors: ARG (NULL), CUDA. */
int kvq_cache_free(kvq_cache* cache, cudaStream_t s);

/* Host-side lengths (MixKVQ Algorithm 1's len(X_K_r) and the quantized
 * history; KIVI §4's boundaries): quantized history tokens and residual
 * tokens.  In KIVI mode the first is the sealed key tokens and the second
 * the key residual; the value FIFO holds min(total, 128) of the newest. */
int kvq_cache_lengths(const kvq_cache* cache, int* quantized_tokens,
                      int* residual_tokens);

/* Host-side length of the attention-sink window (0..n_sink). */
int kvq_cache_sink_tokens(const kvq_cache* cache, int* sink_tokens);

/* Empty the cache (lengths to 0, status word cleared on s): the state
 * before MixKVQ Algorithm 1's Prefill. */
int kvq_cache_reset(kvq_cache* cache, cudaStream_t s);

/*
 * MixKVQ Algorithm 1, Decoding, first step: append one token's key and
 * value (k_new, v_new: bf16 [B][Hkv][D]) to residual slot r; r += 1.  While
 * the attention-sink window holds fewer than n_sink tokens the token goes
 * there instead (the sequence's first tokens are the sinks).
 * Errors: ARG, RESIDUAL_FULL (r == 128: call kvq_flush_group first), CUDA.
 */
int kvq_append_residual(kvq_cache* cache, const kvq_bf16* k_new,
                        const kvq_bf16* v_new, cudaStream_t s);

/*
 * MixKVQ Algorithm 1, Decoding, "if len(X_K_r) == R": quantize the full
 * residual window as one Key group per (batch row, KV head, channel) over
 * its 128 tokens and one Value group per (token, 32 channels), append it to
 * the packed history and empty the residual.  KIVI article §2 contract,
 * PN-Mix Eq. 2 clipping and constant-group branch (step stored 0).
 * KVQ_K_MIXED: importance is I_d, fp32 [B][Hkv][D] (device), and the group's
 * tiers come from A_d = I_d * S_d with S_d at 2 bits (KeyQuant =
 * OutlierReserve + GroupQuant): RANK gives the n_bf16 largest A_d BF16 and
 * the next n_uint4 UINT4; THRESHOLD gives A_d > tau_bf16 BF16 and A_d >
 * tau_uint4 UINT4, from the largest A_d down, at most n_bf16 and n_uint4
 * (the channel ranking breaks ties by the lower index).  importance = NULL
 * in a mixed cache takes I_d from the online window (kvq_observe_query):
 * the running |q| sum / (query heads per KV head * steps observed since the
 * previous flush); the window then starts again.  Uniform caches take
 * importance = NULL.
 * Errors: ARG, MODE (importance given to a uniform cache), EMPTY (mixed
 * cache, importance NULL and no query observed), RESIDUAL_NOT_FULL,
 * CAPACITY, CUDA.  Flags: NONFINITE, RANGE.
 */
int kvq_flush_group(kvq_cache* cache, const float* importance, cudaStream_t s);

/*
 * MixKVQ online salience estimation (the running accumulator of query
 * magnitudes kept in the cache), with the workflow's window: I_d is the
 * mean |Q| of the queries of the current window, renewed every R tokens.
 * Add one decode step's query (q: bf16
 * [B][Hq][D], device, Hq a multiple of Hkv) to the mixed cache's running
 * sums, acc[b][kvh][d] += |q[b][h][d]| for the query heads h of the KV
 * group in ascending order (fp32, round to nearest).  Over a window of
 * steps this is the same sum, in the same order (token, then head), that
 * kvq_channel_saliency forms for I_d.  The window ends at the next
 * kvq_flush_group that takes its importance from it, and at
 * kvq_cache_reset.
 * Errors: ARG, MODE (uniform cache), SHAPE (Hq not a multiple of Hkv, or a
 * query head count other than the window's earlier steps), CUDA.  Flags:
 * NONFINITE (a non-finite query element).
 */
int kvq_observe_query(kvq_cache* cache, const kvq_bf16* q, int Hq, cudaStream_t s);

/*
 * MixKVQ Algorithm 1, Prefill: k, v bf16 [B][Hkv][L][D]; the first
 * s = min(L, n_sink) tokens go to the attention-sink window; of the other
 * L' = L - s, the first L' - (L' mod 128) are quantized into floor(L'/128)
 * groups exactly as kvq_flush_group does and the last L' mod 128 go to the
 * residual.  importance: as for kvq_flush_group.  L = 0 is allowed (no-op).
 * Errors: ARG, MODE, NOT_EMPTY, CAPACITY, CUDA.  Flags: NONFINITE, RANGE.
 */
int kvq_quantize_prefill(kvq_cache* cache, const kvq_bf16* k,
                         const kvq_bf16* v, int L, const float* importance,
                         cudaStream_t s);

/*
 * Workspace bytes kvq_decode_attention needs for Hq query heads at the
 * cache's capacity (split-K partials: per query head and split, the running
 * max, the normalizer and D accumulators, fp32).  0 on bad arguments.
 */
size_t kvq_decode_workspace_bytes(const kvq_cache* cache, int Hq);

/*
 * Fused decode attention (KIVI article §1 and §6; MixKVQ Algorithm 1 last
 * three lines): for each (b, h), s_t = q·k^_t / sqrt(D) over the
 * attention-sink tokens (bf16), the dequantized history and the residual
 * tokens, p = softmax over all of them together, o = sum_t p_t v^_t.  q: bf16 [B][Hq][D], Hq a multiple
 * of Hkv (at most 8 query heads per KV head); out: fp32 [B][Hq][D].
 * Uniform and mixed (MixKVQ) key caches alike: in a mixed group k^ is the
 * raw bf16 key on the BF16 tier and the dequantized code on the others.
 * ws: device scratch of >= kvq_decode_workspace_bytes(cache, Hq), not
 * aliased with any argument; its contents are overwritten.
 * Errors: ARG, SHAPE, EMPTY, WORKSPACE, CUDA.
 */
int kvq_decode_attention(const kvq_cache* cache, const kvq_bf16* q, int Hq,
                         float* out, void* ws, size_t ws_bytes, cudaStream_t s);

/*
 * One decode step of MixKVQ Algorithm 1 (Decoding: append the new token's
 * key and value, flush when the residual holds R = 128 tokens, then the
 * attention) in one call: the result equals kvq_append_residual, then
 * kvq_flush_group(importance) if the residual became full, then
 * kvq_decode_attention.  When neither a flush nor an append to the
 * attention-sink window is due, the decode kernel itself writes the token
 * into the residual, so the step is one decode launch and its combine.
 * k_new, v_new: bf16 [B][Hkv][D], 16-byte aligned; importance: as for
 * kvq_flush_group (NULL for uniform caches; NULL takes a mixed cache's
 * online window), used only when a flush happens; q, out, ws, ws_bytes: as
 * for kvq_decode_attention (ws sized by kvq_decode_workspace_bytes).
 * Errors: those of the three calls (RESIDUAL_FULL when the residual was
 * already full), checked before anything is enqueued where the call is
 * fused; the cache's lengths advance only on success.  As with the
 * separate calls, the lengths are host state that advances when the call
 * is enqueued: a captured stream graph replays the step for the lengths it
 * was captured at.
 */
int kvq_decode_step(kvq_cache* cache, const kvq_bf16* k_new, const kvq_bf16* v_new,
                    const float* importance, const kvq_bf16* q, int Hq, float* out,
                    void* ws, size_t ws_bytes, cudaStream_t s);

/*
 * Decode attention without any allocation (this entry point has no
 * counterpart on the pages; it exists for callers that cannot allocate).
 * Same inputs, output and errors as kvq_decode_attention, but the split-K
 * workspace is a fixed array of KVQ_STATIC_WORKSPACE_BYTES inside the
 * library's device memory instead of a caller buffer, and the call makes no
 * cudaMalloc, cudaFree or other allocating call.  It is meant for callers
 * that cannot allocate device memory when they decode: servers that reserve
 * all memory at start-up and forbid allocation on the request path, plain C
 * hosts without an allocator, replayed launch sequences.
 *  - Every GPU that loads the library holds the array until process exit.
 *  - The first call on a device looks the array's device address up once
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Call it with the cache's own device current (KVQ_ERR_ARG otherwise).
 *    The cached address belongs to that device's primary context: after a
 *    cudaDeviceReset (or anything else that destroys that context) the
 *    library must be reloaded before this entry point is used again.
 *  - All calls share the one array, so calls whose work overlaps on the GPU
 *    (other streams, other threads) race and corrupt each other's results;
 *    serialize them.  Each call rewrites every workspace entry it reads: a
 *    decode warp whose wait gave up (KVQ_FLAG_TIMEOUT) writes empty
 *    partials for the rows it leaves, so no earlier call's partial enters
 *    the merge, but that call's output is undefined (rows may be NaN).
 *  - The split of the token axis is reduced to fit the array.  Two partial
 *    slots per query row, 2*B*Hq*(D+2)*4 bytes, must fit (B*Hq <= 8065
 *    query rows); beyond that it returns KVQ_ERR_WORKSPACE.
 */
#define KVQ_STATIC_WORKSPACE_BYTES (8u << 20) /* 8 MiB per GPU */
int kvq_decode_attention_static(const kvq_cache* cache, const kvq_bf16* q,
                                int Hq, float* out, cudaStream_t s);

/*
 * Unquantized comparator (the 16-bit baseline of MixKVQ's and PN-Mix's
 * comparisons): the same decode attention over plain bf16 k, v
 * [B][Hkv][T][D] (T >= 1; k, v, q 16-byte aligned), same q/out
 * conventions.  ws: >= kvq_decode_bf16_workspace_bytes(B, Hkv, T, Hq) for
 * the current device (the split depends on its SM count; 0 on bad
 * arguments).  Errors: ARG, SHAPE, WORKSPACE, CUDA.
 */
size_t kvq_decode_bf16_workspace_bytes(int B, int Hkv, int T, int Hq);
int kvq_decode_bf16(const kvq_bf16* k, const kvq_bf16* v, int B, int Hkv,
                    int T, const kvq_bf16* q, int Hq, float* out, void* ws,
                    size_t ws_bytes, cudaStream_t s);

/*
 * MixKVQ salience: q_win bf16 [B][Hq][Lq][D] (query window), k_grp bf16
 * [B][Hkv][G][D] (key group, G tokens).  Per (b, kv head, d):
 *   I_d = (sum over tokens i ascending, then heads of the GQA group
 *          ascending, of |Q|, in fp32) / (n_rep * Lq)
 *   S_d = (max_t k - min_t k) / (2^sal_bits - 1)       (fp32)
 *   A_d = I_d * S_d                                     (fp32)
 * and tiers by spec: RANK orders channels by (A_d descending, d ascending)
 * and gives the first n_bf16 BF16, the next n_uint4 UINT4, the rest UINT2;
 * THRESHOLD applies A > tau_bf16 -> BF16, tau_uint4 < A <= tau_bf16 ->
 * UINT4, else UINT2.  I_out, A_out: fp32 [B][Hkv][D]; tiers_out: uint8
 * [B][Hkv][D]; any of the three may be NULL.
 * Errors: ARG, SHAPE, CUDA.  Non-finite inputs leave NaN in A_out and
 * UINT2 tiers (no cache to flag).
 */
int kvq_channel_saliency(const kvq_bf16* q_win, int Hq, int Lq,
                         const kvq_bf16* k_grp, int B, int Hkv, int G,
                         int sal_bits, const kvq_tier_spec* spec, float* I_out,
                         float* A_out, uint8_t* tiers_out, cudaStream_t s);

/* Synchronize s and return the cache's sticky KVQ_FLAG_* word. */
int kvq_cache_status(kvq_cache* cache, cudaStream_t s, int* status);

/*
 * Canonical export of the quantized history (device destination buffers),
 * for checking and debugging: the (codes, origin, step) of KIVI §2's group
 * contract on KIVI §3's axes (keys per channel along tokens, values per
 * token over channel groups), and MixKVQ's per-group tier layout
 * ("system-level implementation details").  T = quantized tokens, n = T/128.
 *  Key (uniform): codes uint8 [B][Hkv][n][D][128*k_bits/8] (each channel's
 *    128 codes LSB first along tokens), kmin bf16 [B][Hkv][n][D], kscale
 *    fp32 [B][Hkv][n][D].
 *  Value: codes uint8 [B][Hkv][T][D*v_bits/8] (LSB first along channels),
 *    vmin bf16 [B][Hkv][T][D/32], vscale fp32 [B][Hkv][T][D/32].
 *  Residual: k_r, v_r bf16 [B][Hkv][r][D] (may be NULL when r = 0).
 *  Key (mixed), per (b, kv head, group), at the record's room cb = n_bf16,
 *    c4 = n_uint4, c2 = D - cb - c4 (RANK) or D (THRESHOLD): counts uint8
 *    [..][2] (the group's own BF16 and UINT4 channel counts nb, n4; n2 =
 *    D - nb - n4; may be NULL), perm uint8 [..][D] (BF16, UINT4, UINT2
 *    channels, each ascending), raw bf16 [..][cb][128], c4 uint8
 *    [..][c4][64], m4 bf16 [..][c4], s4 fp32 [..][c4], c2 uint8
 *    [..][c2][32], m2 bf16 [..][c2], s2 fp32 [..][c2]; entries past the
 *    group's own count are zero.
 * With no quantized tokens nothing is copied and the buffers may be NULL.
 * Errors: ARG, MODE, CUDA.
 */
int kvq_export_k(const kvq_cache* cache, uint8_t* codes, kvq_bf16* kmin,
                 float* kscale, cudaStream_t s);
int kvq_export_v(const kvq_cache* cache, uint8_t* codes, kvq_bf16* vmin,
                 float* vscale, cudaStream_t s);
int kvq_export_residual(const kvq_cache* cache, kvq_bf16* k_r, kvq_bf16* v_r,
                        cudaStream_t s);
int kvq_export_k_mixed(const kvq_cache* cache, uint8_t* counts, uint8_t* perm, kvq_bf16* raw,
                       uint8_t* c4, kvq_bf16* m4, float* s4, uint8_t* c2,
                       kvq_bf16* m2, float* s2, cudaStream_t s);

/*
 * PN-Mix pair selection (PN-Mix reproduction notes, Eq. 6), once per
 * prefill, before kvq_quantize_prefill of a KVQ_K_PNMIX cache: for every
 * (b, KV head) and RoPE pair i (channels a, b of the config's layout),
 *   sigma_i = (1/Hg) sum_h (1/Lq) sum_t sqrt(q_a^2 + q_b^2)
 *             * (1/Lk) sum_t sqrt(k_a^2 + k_b^2),
 * over the GQA group's Hg = Hq / Hkv query heads (in order) of q (bf16
 * [B][Hq][Lq][D]) and the keys k (bf16 [B][Hkv][Lk][D]), every operation
 * fp32 rounded (sums in token order, then head order).  The n_high_pairs
 * largest sigma (ties: lower pair) become the 3-bit pairs; the cache keeps
 * the selection for every later flush.  sigma (fp32 [B][Hkv][D/2], device)
 * may be NULL.  k must be 16-byte aligned (its rows are copied in bulk).
 * Errors: ARG (also an unaligned k), SHAPE, MODE (not a PN-Mix cache),
 * NOT_EMPTY (the cache holds tokens), CUDA.  Flags: NONFINITE, TIMEOUT (a
 * bounded wait for a staged key chunk gave up: the selection is invalid).
 */
int kvq_pnmix_pairs(kvq_cache* cache, const kvq_bf16* q, int Hq, int Lq,
                    const kvq_bf16* k, int Lk, float* sigma, cudaStream_t s);

/*
 * Canonical export of a KVQ_K_PNMIX cache's keys, n = T/128 groups: codes
 * uint8 [B][Hkv][n][128][D] (one code per byte, token-major: 0..7 for the
 * high channels, 0..1 for the others), offset and scale fp32 [B][Hkv][n][D]
 * (origin m and step for the high channels, Eq. 7's z and s for the
 * others), high uint8 [B][Hkv][D] (1 for the channels of the selected
 * pairs; may be NULL).  Values: kvq_export_v.
 * Errors: ARG, MODE, CUDA.
 */
int kvq_export_pnmix(const kvq_cache* cache, uint8_t* codes, float* offset, float* scale,
                     uint8_t* high, cudaStream_t s);

/*
 * Canonical export of a KVQ_K_KIVI cache ("KIVI: KV cache axes" §4–§7), n =
 * T_k / 128 records, r_K key residual tokens, r_V = min(T_k + r_K, 128)
 * FIFO values (device destination buffers; the quantized ones may be NULL
 * when T_k = 0, k_res when r_K = 0):
 *  keys: k_codes uint8 [B][Hkv][n*4][D][32*bits/8] (per 32-token group and
 *    channel, the 32 codes LSB first along tokens), k_origin, k_step bf16
 *    [B][Hkv][n*4][D];
 *  values: v_codes uint8 [B][Hkv][n*128][D*bits/8] (LSB first along
 *    channels), v_origin, v_step bf16 [B][Hkv][n*128][D/32]; rows of tokens
 *    whose values are still in the FIFO are zero (the quantized values are
 *    the first T_k + r_K - r_V rows);
 *  k_res bf16 [B][Hkv][r_K][D]; v_res bf16 [B][Hkv][r_V][D], oldest first.
 * Errors: ARG, MODE (not a KIVI cache), CUDA.
 */
int kvq_export_kivi(const kvq_cache* cache, uint8_t* k_codes, kvq_bf16* k_origin,
                    kvq_bf16* k_step, uint8_t* v_codes, kvq_bf16* v_origin,
                    kvq_bf16* v_step, kvq_bf16* k_res, kvq_bf16* v_res, cudaStream_t s);

/*
 * The attention-sink window: k, v bf16 [B][Hkv][s][D] (s =
 * kvq_cache_sink_tokens; NULL allowed when s = 0).  Errors: ARG, CUDA.
 */
int kvq_export_sink(const kvq_cache* cache, kvq_bf16* k, kvq_bf16* v, cudaStream_t s);

/*
 * Failure-detection hook (no counterpart on the pages).  Every wait of a
 * decode warp for a record part it staged is bounded: after `polls` polls
 * of the barrier (default 2^20, restored by a negative value) the warp sets
 * KVQ_FLAG_TIMEOUT in the cache's status word, waits for its copy in flight
 * with the default limit (so no copy outlives the warp), writes empty
 * partials (weight 0) for the rows it leaves and returns; that call's
 * output is undefined.  polls = 0 makes every first wait give up at once,
 * which is how the tests exercise this path without a fault.  The setting
 * is process-wide and applies to launches enqueued after the call; it is
 * not meant for production use.  Returns the previous limit.
 */
int kvq_set_wait_limit(int polls);

/*
 * Measurement hook (no counterpart on the pages).  The next decode
 * attention call (kvq_decode_attention, kvq_decode_step or
 * kvq_decode_attention_static) records `ev` on its stream right after it
 * enqueues the split-K decode kernel and before it enqueues the combine
 * kernel, then forgets it; so an event recorded before the call and `ev`
 * bracket the decode kernel alone.  ev: an event of the caller's (created
 * with timing), owned by the caller; NULL cancels a pending one.  A call
 * that fails before its decode kernel is enqueued leaves the event pending.
 * The setting is process-wide, for benchmarks; it is not meant for
 * concurrent use.  Returns KVQ_OK.
 */
int kvq_set_decode_split_event(cudaEvent_t ev);

/* Human-readable name of a return code. */
const char* kvq_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
