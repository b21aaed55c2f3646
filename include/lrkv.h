/*
 * lrkv.h -- C ABI of the GB300 (sm_103a) library for attention over an
 * LRKV-compressed KV cache.
 *
 * The method ("Low-Rank Key Value Attention", O'Neill, Clancy, Matskevichus,
 * Reid, arXiv:2601.11471v3; slide deck of the same title):
 *   each head's key/value projection is W_h = W_shared + U_h B_h^T
 *   (Eqs. (2)-(3), frame "LRKV constrains differences between heads"), so per
 *   token and layer the cache holds a shared d_h-vector s plus one r-vector z_h
 *   per head, for keys and for values: 2(d_h + H r) elements (frame "Can heads
 *   share storage while keeping distinct K/V features?").  Decode never expands
 *   per-head keys or values; it evaluates the factored forms of Eqs. (6)-(7).
 *
 * Conventions shared by every entry point
 *   - All tensors are bf16 (IEEE binary16 brain-float bit patterns, uint16 in
 *     memory) unless stated, row-major, in DEVICE memory owned by the caller.
 *     The library allocates nothing and keeps no state between calls.
 *   - Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous: they validate on the host, enqueue kernels and return.
 *   - Host-detectable errors are returned before anything is launched; the
 *     calling thread can then read a one-line explanation from
 *     lrkv_last_error().  A launch failure returns LRKV_ERR_CUDA.
 *   - Errors only the device can see (an index read from device memory that is
 *     out of range, a bounded wait that expired) are OR-ed into the optional
 *     uint32 word `status_dev` (device memory, may be NULL) as LRKV_DEV_* bits;
 *     the offending access is skipped, never trapped.  Read the word after
 *     synchronising the stream.
 *   - Cache pages: the pools are indexed by physical block id b in
 *     [0, num_blocks); token slot = b * block_size + offset.
 *        sK     : [num_blocks][block_size][d_h + d_rope]   rows [s^K | k^R]
 *        sV     : [num_blocks][block_size][d_h]
 *        zK, zV : [num_blocks][block_size][H][r]
 *     (s = shared features K_s, V_s of Eq. (4); z_h = per-head latents R_h^K,
 *     R_h^V of Eq. (5); k^R = the optional decoupled positional key, below.)
 *     B_h^K, B_h^V are weights, not cache entries.
 *   - Decoupled positional key (d_rope > 0; "Low-Rank Key Value Attention",
 *     combination with MLA-style latent caches, whose decoupled rotary key is
 *     one d_rope-vector per token shared by all heads): every key row carries
 *     k^R = RoPE(x W^KR, pos) after s^K.  A query is then [q | q^R] (q^R already
 *     rotated by the caller), logits are q . (s^K + B_h^K z^K_h) + q^R . k^R, and
 *     the default scale is 1/sqrt(d_h + d_rope).  RoPE turns the pair (2i, 2i+1)
 *     of a d_rope-vector by the angle pos * rope_base^(-2i / d_rope).  Values
 *     carry no positional part.  d_rope == 0 is the plain method, bit for bit.
 *
 * Supported shapes (others return LRKV_ERR_UNSUPPORTED):
 *   block_size == 64, d_h in {64, 128}, r in {8, 16, 32} with r <= d_h,
 *   1 <= H <= 128, d a positive multiple of 8 (of 64 for the tensor-core append),
 *   d_rope in {0, 64}.  The decode calls with r = 32 and H >= 105 need H a multiple
 *   of 8: a stage of the scan then holds the latents of a group of heads, not of all.
 */
#ifndef LRKV_H
#define LRKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: lrkv_dims.num_splits and the layer-batched calls; 4: lrkv_prefill_fused,
 * lrkv_decode_partials and lrkv_decode_merge (no struct changed). */
#define LRKV_ABI_VERSION 4

typedef enum lrkv_status {
    LRKV_OK = 0,
    LRKV_ERR_INVALID_ARG = 1,   /* NULL or misaligned pointer, negative size, inconsistent arguments */
    LRKV_ERR_UNSUPPORTED = 2,   /* shape outside the supported set above */
    LRKV_ERR_WORKSPACE = 3,     /* workspace smaller than the *_workspace_bytes() figure */
    LRKV_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    LRKV_ERR_DEVICE_BOUNDS = 5, /* meaning of the LRKV_DEV_BAD_* bits, for lrkv_status_string */
    LRKV_ERR_TIMEOUT = 6        /* meaning of the LRKV_DEV_TIMEOUT bit, for lrkv_status_string */
} lrkv_status;

/* Bits kernels OR into *status_dev. */
#define LRKV_DEV_BAD_BLOCK 0x1u  /* a block_table entry needed by a call is outside [0, num_blocks) */
#define LRKV_DEV_BAD_SEQLEN 0x2u /* seq_len / q_start + Tq outside [1, max_blocks_per_seq * block_size]; that
                                    sequence's output rows are written as zeros */
#define LRKV_DEV_BAD_SLOT 0x4u   /* slot_mapping entry >= num_blocks * block_size (row skipped) */
#define LRKV_DEV_TIMEOUT 0x8u    /* a pipeline wait in a kernel gave up after its time limit (about 2 s) */

/* Model dimensions (frame "LRKV constrains differences between heads"). */
typedef struct lrkv_dims {
    int32_t H;           /* query heads */
    int32_t d_h;         /* head width */
    int32_t r;           /* residual rank of U_h B_h^T */
    int32_t d;           /* hidden size of the rows appended to the cache */
    int32_t block_size;  /* tokens per cache page; must be 64 */
    float softmax_scale; /* logit scale; 0 means 1/sqrt(d_h + d_rope) (frame "Compute logits ...") */
    int32_t d_rope;      /* width of the decoupled positional key shared by all heads; 0 = none */
    float rope_base;     /* RoPE base; 0 means 10000 (ignored when d_rope == 0) */
    int32_t num_splits;  /* decode only: how many equal contiguous pieces the batch's cached tokens
                            are cut into for the split-K scan (each piece is scanned by one CTA and
                            leaves one partial softmax state per sequence it touches); 0 = one per
                            SM (the default), else 1..65536.  Results agree across values up to
                            floating-point rounding. */
} lrkv_dims;

/* One layer's paged cache (device pointers, caller-owned, layout above). */
typedef struct lrkv_cache {
    void* sK;
    void* sV;
    void* zK;
    void* zV;
    int32_t num_blocks;
} lrkv_cache;

/* ABI version of the loaded library (LRKV_ABI_VERSION it was built with). */
int lrkv_abi_version(void);

/* Static description of a status code. */
const char* lrkv_status_string(lrkv_status s);

/* Explanation of the last non-OK status returned on the calling thread ("" if none). */
const char* lrkv_last_error(void);

/* Bytes of one cache page across the four pools: block_size * 2 * (2(d_h + H r) + d_rope).
 * Returns 0 for unsupported dims. */
size_t lrkv_cache_block_bytes(const lrkv_dims* dims);

/*
 * lrkv_append -- Eqs. (4)-(5): project n_tok hidden rows into the cache.
 *   Y = X W_cat, W_cat = [W_shared^K | W^KR | W_shared^V | U_1^K .. U_H^K | U_1^V .. U_H^V]
 *   (d x N, N = 2(d_h + H r) + d_rope; W^KR absent when d_rope == 0), accumulated
 *   in fp32; the d_rope columns of W^KR are then rotated at positions[t] (angle in
 *   double, sine and cosine in fp32 corrected to first order in double, products in
 *   double, result rounded to fp32: within ~1e-7 of the pair's magnitude of the exact
 *   rotation); everything is rounded to bf16
 *   (nearest, ties to even).  Row t is written to token slot slot_mapping[t]:
 *   columns [0, d_h + d_rope) -> sK, the next d_h -> sV, the next H r -> zK
 *   (head-major), the last H r -> zV.
 *   X            [n_tok][d]
 *   W_catT       [N][d]  (W_cat transposed: row c holds the weights of output column c)
 *   slot_mapping [n_tok] int32 (device); a negative entry skips the row,
 *                an entry >= num_blocks*block_size sets LRKV_DEV_BAD_SLOT and skips it.
 *   positions    [n_tok] int32 (device) token positions, >= 0; required when
 *                d_rope > 0, ignored (may be NULL) otherwise.
 *   n_tok == 0 is a no-op.  Small n_tok runs a bandwidth-bound kernel, large n_tok a
 *   tcgen05 tensor-core GEMM; both give bit-identical results whenever every fp32
 *   partial sum is exact.
 */
lrkv_status lrkv_append(const lrkv_dims* dims, const void* X, const void* W_catT, int32_t n_tok,
                        const int32_t* slot_mapping, const int32_t* positions, const lrkv_cache* cache,
                        uint32_t* status_dev, void* stream);

/* Workspace bytes lrkv_decode needs for `batch` sequences on the CURRENT device (for
 * lrkv_decode_layers pass num_layers * batch). */
size_t lrkv_decode_workspace_bytes(const lrkv_dims* dims, int32_t batch);

/*
 * lrkv_decode -- one decode step per sequence, factored form (Eqs. (6)-(7)):
 *   q~_h = q_h B_h^K;  score_t = (q_h . s^K_t + q~_h . z^K_{h,t}) * scale;
 *   a_h = softmax_t(score);  out_h = a_h V_s + (a_h R_h^V) (B_h^V)^T.
 *   The query attends to all seq_lens[b] cached tokens (positions 0..L-1; it is
 *   the newest position and is already in the cache).  Split over the sequence
 *   across the GPU's SMs, merged by log-sum-exp in a second kernel.  With a
 *   positional key the logit gains q^R . k^R_t (see the conventions above).
 *   q           [batch][H][d_h + d_rope]  ([q_h | q^R_h]; q~ uses the first d_h)
 *   BK, BV      [H][d_h][r]  (B_h^K, B_h^V)
 *   block_table [batch][max_blocks_per_seq] int32 (device)
 *   seq_lens    [batch] int32 (device)
 *   out         [batch][H][d_h]
 *   workspace   device scratch of >= lrkv_decode_workspace_bytes(dims, batch) bytes, 256-byte aligned.
 *   Capacity of one call: batch x max_blocks_per_seq x block_size below 2^34 tokens (times
 *   num_layers for lrkv_decode_layers); larger calls return LRKV_ERR_INVALID_ARG.
 */
lrkv_status lrkv_decode(const lrkv_dims* dims, const void* q, const void* BK, const void* BV,
                        const lrkv_cache* cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t batch, void* out, void* workspace,
                        size_t workspace_bytes, uint32_t* status_dev, void* stream);

/*
 * lrkv_decode_fused -- lrkv_decode with both absorptions moved into the caller's
 *   weights (the associativity of frame "Compute logits without expanding
 *   historical keys", step 1, and of Eq. (7), "reduce the latents to one r-vector,
 *   then map"): the query arrives with q~_h = x (W_h^Q B_h^K) already projected,
 *   and the output is returned before the residual up-projection, for an output
 *   projection with B_h^V folded into W^O.  Per sequence b and head h:
 *     score_t = ([q_h | q~_h] . [s^K_t | z^K_{h,t}]) * scale;  a_h = softmax_t(score)
 *     out_h   = [ sum_t a_t s^V_t  |  sum_t a_t z^V_{h,t} ]        (width d_h + r)
 *   i.e. single-head softmax attention over the concatenated features (with a
 *   positional key, [q_h | q^R_h | q~_h] . [s^K_t | k^R_t | z^K_{h,t}]).
 *   q           [batch][H][d_h + d_rope]   bf16
 *   q_tilde     [batch][H][r]     bf16, 16-byte aligned
 *   out         [batch][H][d_h + r] bf16 (nearest, ties to even from fp32)
 *   Everything else (cache, block_table, seq_lens, workspace, status, errors, the
 *   stream) is as for lrkv_decode; no B^K or B^V is read.  Unlike lrkv_decode, the
 *   call does not overlap the caller's previous kernel on the stream.
 */
lrkv_status lrkv_decode_fused(const lrkv_dims* dims, const void* q, const void* q_tilde, const lrkv_cache* cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                              uint32_t* status_dev, void* stream);

/*
 * lrkv_decode_partials / lrkv_decode_merge -- lrkv_decode cut at the log-sum-exp merge, for a
 *   sequence whose cached tokens are spread over several caches (e.g. one token range per
 *   device).  The online softmax of frame "Compute logits without expanding historical keys"
 *   is associative over any split of the tokens, and B_h^V is applied after the merge (Eq. (7):
 *   the latents are aggregated first), so each part only has to return, per (sequence, head),
 *   over its own tokens t:
 *     m   = max_t s_t,  s_t = ([q | q~] . [s^K_t | z^K_{h,t}]) * scale * log2(e)
 *     l   = sum_t 2^(s_t - m)
 *     acc = sum_t 2^(s_t - m) [s^V_t | z^V_{h,t}]                    (width d_h + r)
 *   and the merge of P parts is M = max_p m_p, w_p = 2^(m_p - M),
 *     out_h = (sum_p w_p acc_s,p + B_h^V sum_p w_p acc_z,p) / sum_p w_p l_p.
 *   lrkv_decode_partials: arguments as lrkv_decode (no B^V, no out); seq_lens[b] counts the
 *     tokens of sequence b held in THIS cache and may be 0 (an empty part: m = -inf, l = 0,
 *     acc = 0; no status bit).
 *     partials  [batch][H][d_h + r + 2] fp32: acc_s (d_h), acc_z (r), m, l
 *   lrkv_decode_merge: partials [num_parts][batch][H][d_h + r + 2] (the parts' outputs stacked,
 *     e.g. by an all-gather), BV as for lrkv_decode, out [batch][H][d_h] bf16 (nearest, ties to
 *     even).  A (sequence, head) that no part holds a token of gets zeros and
 *     LRKV_DEV_BAD_SEQLEN.  num_parts >= 1; 1 <= batch <= 65535 (0 is a no-op).
 *   Pointers 16-byte aligned, device memory, the caller's stream; errors as for lrkv_decode.
 */
lrkv_status lrkv_decode_partials(const lrkv_dims* dims, const void* q, const void* BK, const lrkv_cache* cache,
                                 const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t batch, float* partials, void* workspace, size_t workspace_bytes,
                                 uint32_t* status_dev, void* stream);
lrkv_status lrkv_decode_merge(const lrkv_dims* dims, int32_t num_parts, const float* partials, const void* BV,
                              int32_t batch, void* out, uint32_t* status_dev, void* stream);

/*
 * lrkv_decode_static_ws -- lrkv_decode without a caller workspace.  (The paper has
 *   no counterpart; this is a deployment convenience.)
 *   For callers that cannot allocate device memory: cudaMalloc/cudaFree can
 *   synchronise the whole device and stall other streams, some host frameworks
 *   own the GPU allocator and forbid foreign allocations, and some deployments fix
 *   their device-memory budget at start-up.  The scratch lives in a fixed array of
 *   LRKV_STATIC_WS_BYTES inside the library's device image, which every GPU that
 *   loads the library keeps until the process exits; this call allocates nothing.
 *   Arguments, layouts and results are those of lrkv_decode.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept per device together with
 *     the id of the context it was found in; after a device reset (a new context,
 *     which loads the library's device image afresh) the next call looks it up
 *     again, so make that call outside a stream capture too.
 *   - Returns LRKV_ERR_WORKSPACE (explained by lrkv_last_error()) when
 *     lrkv_decode_workspace_bytes(dims, batch) exceeds LRKV_STATIC_WS_BYTES.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents (nothing needs clearing: each call writes all scratch it reads).
 *     Calls whose kernels overlap on the GPU -- e.g. on two streams at once --
 *     race on it; serialise them.
 */
#define LRKV_STATIC_WS_BYTES ((size_t)16 << 20)
lrkv_status lrkv_decode_static_ws(const lrkv_dims* dims, const void* q, const void* BK, const void* BV,
                                  const lrkv_cache* cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t batch, void* out, uint32_t* status_dev,
                                  void* stream);

/* ======================================================================
 * Layer-batched calls: one launch of each kernel for several layers.
 *
 * A decode step of an L-layer model appends one row per sequence and attends over every
 * layer's cache.  Each layer has its own weights, cache pools, queries and outputs; the block
 * table and the lengths are the same for all layers.  When the queries of several layers are
 * known together (independent layers, or layers whose inputs are already computed), these
 * calls do the work of num_layers calls of lrkv_append / lrkv_decode in one launch per kernel,
 * with the whole batch's cached tokens of all layers divided evenly over the SMs -- many small
 * layers otherwise pay each kernel's fixed start-up and drain cost once per layer.
 *
 * Layer l's tensor is found at (layer 0's pointer) + l * stride, strides in bf16 elements
 * (multiples of 8, so every layer's tensors stay 16-byte aligned, and at least the size of
 * one layer's tensor: layers do not overlap).  The `cache` argument holds layer 0's pools
 * and num_blocks, the number of blocks of each layer's pools.
 * ====================================================================== */
typedef struct lrkv_layer_strides {
    int64_t X, W_catT;      /* lrkv_append_layers: hidden rows [n_tok][d], W_cat^T [N][d] */
    int64_t q, BK, BV, out; /* lrkv_decode_layers: [batch][H][d_h + d_rope], [H][d_h][r] (x2), [batch][H][d_h] */
    int64_t sK, sV, zK, zV; /* cache pools of both calls */
} lrkv_layer_strides;

/*
 * lrkv_append_layers -- lrkv_append of the same n_tok token slots (slot_mapping, positions)
 *   in num_layers layers: layer l's rows X_l W_cat,l go to layer l's pools.  Everything else
 *   as for lrkv_append; num_layers == 1 is lrkv_append (strides ignored, may be NULL).
 */
lrkv_status lrkv_append_layers(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* strides,
                               const void* X, const void* W_catT, int32_t n_tok, const int32_t* slot_mapping,
                               const int32_t* positions, const lrkv_cache* cache, uint32_t* status_dev,
                               void* stream);

/*
 * lrkv_decode_layers -- lrkv_decode of the same batch (block_table, seq_lens) in num_layers
 *   layers: out_l = decode(q_l, B^K_l, B^V_l, cache_l), Eqs. (6)-(7) per layer.  The workspace
 *   is lrkv_decode_workspace_bytes(dims, num_layers * batch) bytes.  Everything else as for
 *   lrkv_decode; num_layers == 1 is lrkv_decode (strides ignored, may be NULL).
 */
lrkv_status lrkv_decode_layers(const lrkv_dims* dims, int32_t num_layers, const lrkv_layer_strides* strides,
                               const void* q, const void* BK, const void* BV, const lrkv_cache* cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                               uint32_t* status_dev, void* stream);

/* Workspace bytes lrkv_prefill needs (0 today; kept so callers size it). */
size_t lrkv_prefill_workspace_bytes(const lrkv_dims* dims, int32_t batch, int32_t Tq);

/*
 * lrkv_prefill -- causal chunked prefill over the cache (Eqs. (6)-(7) with the
 *   causal mask of the softmax frame): query i of sequence b sits at absolute
 *   position p = q_start[b] + i and attends to cached tokens j <= p.  The chunk's
 *   own rows must already be in the cache (lrkv_append first).
 *   Logits use the concatenated width d_h + r: [q | q~] . [s^K | z^K_h]; the
 *   scale stays 1/sqrt(d_h) (the dot product is the same one), or 1/sqrt(d_h + d_rope)
 *   with a positional key (whose term q^R . k^R joins the logit).
 *   q        [batch][Tq][H][d_h + d_rope]
 *   q_start  [batch] int32 (device)
 *   out      [batch][Tq][H][d_h]
 */
lrkv_status lrkv_prefill(const lrkv_dims* dims, const void* q, const void* BK, const void* BV,
                         const lrkv_cache* cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* q_start, int32_t batch, int32_t Tq, void* out, void* workspace,
                         size_t workspace_bytes, uint32_t* status_dev, void* stream);

/*
 * lrkv_prefill_fused -- lrkv_prefill with both absorptions moved into the caller's
 *   weights, as lrkv_decode_fused does for one query (associativity of frame "Compute
 *   logits without expanding historical keys", step 1, and of Eq. (7)): query i of
 *   sequence b, at absolute position p = q_start[b] + i, arrives with q~_i = q_i B_h^K
 *   already projected, and head h returns
 *     out = [ sum_{j<=p} a_j s^V_j  |  sum_{j<=p} a_j z^V_{h,j} ]   (width d_h + r),
 *     a = softmax_{j<=p}(([q_i | q~_i] . [s^K_j | z^K_{h,j}]) * scale)
 *   (with a positional key, [q | q^R | q~] . [s^K | k^R | z^K_h]).
 *   q        [batch][Tq][H][d_h + d_rope]  bf16
 *   q_tilde  [batch][Tq][H][r]             bf16, 16-byte aligned
 *   out      [batch][Tq][H][d_h + r]       bf16 (nearest, ties to even from fp32)
 *   Everything else (cache, block_table, q_start, status, errors, the stream) is as
 *   for lrkv_prefill; no B^K or B^V is read and no workspace is needed.
 */
lrkv_status lrkv_prefill_fused(const lrkv_dims* dims, const void* q, const void* q_tilde, const lrkv_cache* cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* q_start,
                               int32_t batch, int32_t Tq, void* out, uint32_t* status_dev, void* stream);

/* ======================================================================
 * Training-time expanded projections ("Low-Rank Key Value Attention", frame
 * "Training learns the base and residuals together": the full per-head features
 * are materialised during training).  One projection -- keys or values alike:
 *   K_h = X W_h,  W_h = W_shared + U_h B_h^T                     (Eqs. (2)-(3))
 * with its factors' gradients by the chain rule.  Dims as above (d_rope must be
 * 0; block_size and softmax_scale are not used).  Layouts:
 *   X    [n_tok][d]
 *   W_T  [d_h + H r][d]   rows: W_shared^T (d_h rows), then U_1^T .. U_H^T (r rows each)
 *   B    [H][d_h][r]
 *   Y    [n_tok][d_h + H r]  = X W_T^T = [S | R_1 .. R_H], written by the forward
 *        (bf16), read by the backward
 *   K    [n_tok][H][d_h]   = S + R_h B_h^T
 * All products on the tensor cores with fp32 accumulation; S, R and the backward's
 * [G | dR] are rounded to bf16 between the steps; outputs bf16 (nearest even).
 * n_tok == 0 is a no-op.  Every row count, d and d_h + H r are as in the ABI
 * conventions (multiples of 8); r >= 8.
 * ====================================================================== */

/* Forward: Y and K. */
lrkv_status lrkv_train_forward(const lrkv_dims* dims, const void* X, const void* W_T, const void* B, int32_t n_tok,
                               void* Y, void* K, uint32_t* status_dev, void* stream);

/* Workspace bytes lrkv_train_backward needs for n_tok rows on the CURRENT device. */
size_t lrkv_train_workspace_bytes(const lrkv_dims* dims, int32_t n_tok);

/*
 * Backward for dK [n_tok][H][d_h]:
 *   dX   [n_tok][d]       = sum_h dK_h W_h^T
 *   dW_T [d_h + H r][d]   = [dW_shared^T ; dU_1^T ; ...] = [G | dR]^T X,
 *                          G = sum_h dK_h, dR_h = dK_h B_h
 *   dB   [H][d_h][r]      = dK_h^T R_h (split over tokens, partial sums added in a
 *                          fixed order)
 *   workspace >= lrkv_train_workspace_bytes(dims, n_tok) bytes, 256-byte aligned.
 */
lrkv_status lrkv_train_backward(const lrkv_dims* dims, const void* X, const void* W_T, const void* B, const void* Y,
                                const void* dK, int32_t n_tok, void* dX, void* dW_T, void* dB, void* workspace,
                                size_t workspace_bytes, uint32_t* status_dev, void* stream);

/* ======================================================================
 * Multi-head latent attention (second workload on the same skeleton).
 *
 * "Embeddings II: MLA & Architectural Choices" (weight absorption, decoupled RoPE,
 * the softmax denominator of the concatenated width), in the associative form of
 * "Low-Rank Key Value Attention", backup frame "MLA also admits associative
 * computation": per token and layer the cache holds one row [c_t | k^R_t] -- the
 * latent c_t = x_t W^DKV (d_c = 512) and the decoupled positional key
 * k^R_t = RoPE(x_t W^KR, t) (d_rope = 64), both shared by all heads:
 *        kv : [num_blocks][block_size][d_c + d_rope]   bf16
 * With W^UK_i folded into the query and W^UV_i into the output projection, head i
 * computes  logit_t = [q~_i | q^R_i] . [c_t | k^R_t] * scale  and returns
 * o_i = sum_t softmax(logit)_t c_t (width d_c, before W^UV_i).
 * Conventions (ownership, alignment, streams, errors, status bits) as above.
 * ====================================================================== */
typedef struct lrkv_mla_dims {
    int32_t H;           /* query heads, 1..128 */
    int32_t d_c;         /* latent width; must be 512 */
    int32_t d_rope;      /* positional key width; must be 64 */
    int32_t d_head;      /* per-head content width the absorbed dot product stands for (>= 1) */
    int32_t d;           /* hidden size of appended rows; a positive multiple of 8 */
    int32_t block_size;  /* tokens per cache page; must be 64 */
    float softmax_scale; /* 0 means 1/sqrt(d_head + d_rope) */
    float rope_base;     /* RoPE base; 0 means 10000 */
} lrkv_mla_dims;

/* Bytes of one cache page: block_size * 2 * (d_c + d_rope); 0 for unsupported dims. */
size_t lrkv_mla_cache_block_bytes(const lrkv_mla_dims* dims);

/*
 * lrkv_mla_append -- write n_tok cache rows: Y = X [W^DKV | W^KR] accumulated in fp32;
 *   the last d_rope columns are rotated at positions[t] (pair (2i, 2i+1) by the angle
 *   pos * rope_base^(-2i / d_rope), computed as for lrkv_append, result rounded to
 *   fp32); then bf16 (nearest, ties to even) into slot slot_mapping[t] of kv.
 *   X            [n_tok][d]
 *   W_T          [d_c + d_rope][d]  (row c holds the weights of output column c)
 *   slot_mapping [n_tok] int32 (device); negative skips the row, >= num_blocks*block_size
 *                sets LRKV_DEV_BAD_SLOT and skips it
 *   positions    [n_tok] int32 (device), >= 0
 */
lrkv_status lrkv_mla_append(const lrkv_mla_dims* dims, const void* X, const void* W_T, int32_t n_tok,
                            const int32_t* slot_mapping, const int32_t* positions, void* kv, int32_t num_blocks,
                            uint32_t* status_dev, void* stream);

/* Workspace bytes lrkv_mla_decode needs for `batch` sequences on the CURRENT device. */
size_t lrkv_mla_decode_workspace_bytes(const lrkv_mla_dims* dims, int32_t batch);

/*
 * lrkv_mla_decode -- one decode step per sequence over all seq_lens[b] cached tokens.
 *   q           [batch][H][d_c + d_rope]  ([q~_i | q^R_i], q^R rotated by the caller)
 *   kv          [num_blocks][block_size][d_c + d_rope]
 *   block_table [batch][max_blocks_per_seq] int32 (device)
 *   seq_lens    [batch] int32 (device)
 *   out         [batch][H][d_c] bf16 (nearest, ties to even from fp32)
 *   workspace   >= lrkv_mla_decode_workspace_bytes(dims, batch) bytes, 256-byte aligned
 *   Split over the sequence across pairs of CTAs (each pair divides the row's columns),
 *   merged by log-sum-exp in a second kernel.  A sequence with a length outside
 *   [1, max_blocks_per_seq * block_size] sets LRKV_DEV_BAD_SEQLEN and gets zero rows.
 *   The call does not overlap the caller's previous kernel on the stream.
 */
lrkv_status lrkv_mla_decode(const lrkv_mla_dims* dims, const void* q, const void* kv, int32_t num_blocks,
                            const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t batch, void* out, void* workspace, size_t workspace_bytes,
                            uint32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LRKV_H */
