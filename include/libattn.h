/*
 * libattn.h -- C ABI of libattn: masked exact attention with LSE output, LSE
 * merge of chunked attention, paged KV append and paged GQA decode, as
 * hand-written CUDA kernels for sm_103a (GB300).
 *
 * Conventions for every call
 * --------------------------
 * - Every data pointer is a DEVICE pointer on the current CUDA device; the
 *   caller allocates and frees every buffer (outputs and workspace included).
 *   The library never allocates, never frees, never synchronises, and only
 *   enqueues work on the stream it is given.  Calls on one stream run in
 *   order, so kv_append followed by paged_decode_attn on the same stream
 *   attends over the appended token.
 * - Arguments are validated on the host before anything is launched; a bad
 *   argument returns ATTN_ERR_INVALID_ARG (or ATTN_ERR_UNSUPPORTED for a
 *   valid but unimplemented shape/dtype) and enqueues nothing.
 * - A failed launch returns ATTN_ERR_CUDA.
 * - Errors found on the device (a block-table entry outside the cache, a
 *   position beyond the table, a pipeline wait that timed out) are OR-ed into
 *   a status word at the start of the caller's workspace and the offending
 *   work is skipped (never read out of bounds, never hang).  The word is
 *   sticky: read it with attn_check_device_status(), clear it with
 *   attn_reset_device_status().  A workspace must be zero-filled once before
 *   its first use.
 * - Tensors are described by attn_tensor: element strides, innermost
 *   dimension contiguous (stride 1).  Strides let the same call read the
 *   contiguous [B, H, P, D] layout and the packed [T, H, D] layout (viewed
 *   as [1, H, T, D] with strides {., D, H*D, 1}).
 * - Thread safety: calls hold no global mutable state on the host; two calls
 *   may run concurrently on different streams if their outputs and
 *   workspaces do not overlap.
 */
#ifndef LIBATTN_H
#define LIBATTN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* bad pointer, shape, stride or size       */
    ATTN_ERR_UNSUPPORTED = 2,    /* valid, but no kernel for this shape/dtype */
    ATTN_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed        */
    ATTN_ERR_TIMEOUT = 4,        /* device: a pipeline wait gave up          */
    ATTN_ERR_DEVICE_BOUNDS = 5,  /* device: table entry or position out of range */
    ATTN_ERR_WORKSPACE = 6       /* workspace NULL, misaligned or too small  */
} attn_status;

typedef enum attn_dtype { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype;

typedef struct attn_tensor {
    void *data;          /* device pointer to element [0,...,0]          */
    int32_t dtype;       /* attn_dtype                                   */
    int32_t ndim;        /* number of used entries in shape/stride       */
    int64_t shape[4];
    int64_t stride[4];   /* element strides; stride[ndim-1] must be 1    */
} attn_tensor;

/* A paged KV cache: K and V each [num_blocks, num_kv_heads, block_size,
 * head_dim], contiguous, bf16.  Token t of a sequence lives in physical
 * block block_table[t / block_size] at slot t % block_size ("LLM inference
 * memory accounting", section 15, paged KV cache). */
typedef struct attn_kv_cache {
    void *k;
    void *v;
    int32_t dtype;        /* ATTN_BF16 */
    int32_t block_size;   /* tokens per block; 16 is implemented */
    int64_t num_blocks;
    int32_t num_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
} attn_kv_cache;

/* Bytes of workspace each call needs (always a multiple of 256).  The first
 * 256 bytes hold the device status word. */
size_t attn_fwd_workspace_size(void);
/* Workspace that lets attn_fwd take its fastest path for this shape on the
 * current device (head_dim 64 or 128, bf16): the status word; for head_dim 64
 * the largest |k| element of every 128-key tile, one float per (batch, KV
 * head, tile), which bounds every score of the tile by |q|_1 max|k| and so lets
 * the kernel skip its softmax max pass wherever that bound rules out overflow
 * (used when B * Hq * Pq * Pk * D >= 2^36, where the extra pass over K pays);
 * and room for the partial results of query tiles whose key tiles are split
 * over several CTAs so that the last wave of CTAs fills the GPU (one SM's
 * worth of 256-row partials per SM, merged by the LSE rule).  attn_fwd /
 * attn_fwd_varlen accept any workspace of at least attn_fwd_workspace_size()
 * bytes and use what fits.  0 for a negative size. */
size_t attn_fwd_workspace_size_for(int32_t batch, int32_t kv_heads, int64_t num_keys, int32_t head_dim);
size_t kv_append_workspace_size(void);
size_t paged_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                   int32_t max_blocks, int32_t block_size,
                                   int32_t head_dim);

/*
 * attn_fwd -- exact masked scaled-dot-product attention with its softmax LSE.
 *
 * Defined by "MultiheadAttention fast path used 18 GB of VRAM" (TL;DR and the
 * fix that routes padded inputs through SDPA with an additive -inf mask) and
 * "[sglang] ROCm aiter ring attention" (section 1: the kernel also returns
 * the log-sum-exp so chunk results can be merged).  For every batch b, query
 * head h and query row i:
 *     s_j  = scale * <q[b,h,i,:], k[b,g,j,:]> + key_pad_mask[b, j]
 *     lse  = log(sum_j exp(s_j))                       (natural log)
 *     out  = sum_j exp(s_j - lse) * v[b,g,j,:]
 * with g = h / (Hq / Hkv) (grouped-query heads share a KV head).  The
 * Hq x Pq x Pk score matrix is never stored: extra device memory is the
 * output and LSE only.  A row whose keys are all masked yields out = 0 and
 * lse = -inf.
 *
 *   q    [B, Hq, Pq, D]   bf16 or f32 (strided view)
 *   k, v [B, Hkv, Pk, D]  same dtype as q
 *   key_pad_mask  float32 additive mask, row b at key_pad_mask + b*mask_stride_b,
 *                 Pk entries (0 keeps a key, -inf drops it; any finite value
 *                 is added as is).  NULL means no mask.  This is the additive
 *                 form: a boolean "True = padded" key_padding_mask must be
 *                 converted by the caller (True -> -inf).
 *   scale  multiplies q.k before the mask is added (usually 1/sqrt(D)).
 *   out  [B, Hq, Pq, D]   bf16 or f32 (strided view), written in full.
 *   lse  float32 [B, Hq, Pq] contiguous, or NULL.
 * Implemented: bf16 with D in {64, 128} on the tensor cores (fp32
 * accumulation and softmax); f32 with D <= 128, D % 4 == 0 on FP32 FMA (no
 * TF32).  Pq, Pk >= 0 (zero-size calls do nothing but validate).
 * Alignment: bf16 q/k/v base addresses and the strides of dims 0-2 must be
 * multiples of 16 bytes.
 */
attn_status attn_fwd(const attn_tensor *q, const attn_tensor *k, const attn_tensor *v,
                     const float *key_pad_mask, int64_t mask_stride_b, float scale,
                     const attn_tensor *out, float *lse,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_fwd_varlen -- attn_fwd with the key padding given as lengths.
 *
 * The same attention as attn_fwd, where batch row b attends to its first
 * key_lens[b] keys only (the padded tail of "MultiheadAttention fast path used
 * 18 GB of VRAM": padding is a suffix of each sequence's patches).  This is
 * exactly attn_fwd with an additive mask of 0 for keys < key_lens[b] and -inf
 * after, but no mask is read and KV tiles past the length are skipped.
 *   key_lens  int32 [B] device array; values are clamped to [0, Pk]; a row
 *             with 0 keys gives out = 0 and lse = -inf.
 * Other arguments, layouts and rules as attn_fwd.
 */
attn_status attn_fwd_varlen(const attn_tensor *q, const attn_tensor *k, const attn_tensor *v,
                            const int32_t *key_lens, float scale,
                            const attn_tensor *out, float *lse,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_key_padding_to_additive -- turn a boolean key_padding_mask into the
 * additive mask attn_fwd takes.
 *
 * "MultiheadAttention fast path used 18 GB of VRAM" (note on the mask
 * direction): nn.MultiheadAttention's key_padding_mask marks a key to IGNORE
 * with True, while SDPA's boolean attn_mask marks a key to KEEP with True;
 * passing one as the other silently corrupts the result.  The library only
 * takes the additive form; this converts the key_padding_mask convention:
 *   additive_mask[b*out_stride_b + j] = key_padding_mask[b*kpm_stride_b + j] ? -inf : 0
 *   key_padding_mask  uint8 [batch, num_keys] (non-zero = padded key), device
 *   additive_mask     float32 [batch, num_keys], device, caller-owned
 */
attn_status attn_key_padding_to_additive(const uint8_t *key_padding_mask, int64_t kpm_stride_b,
                                         int32_t batch, int64_t num_keys,
                                         float *additive_mask, int64_t out_stride_b,
                                         cudaStream_t stream);

/*
 * attn_lse_merge -- combine n attention results computed over disjoint KV
 * chunks of the same queries.
 *
 * Defined by "[sglang] ROCm aiter ring attention" (section 1): with partial
 * (out_i, lse_i), lse = log(sum_i exp(lse_i)) (evaluated with the maximum
 * subtracted) and out = sum_i exp(lse_i - lse) * out_i; the accuracy section
 * states that merging two chunks equals one call over all keys.  Partials
 * with lse_i = -inf carry weight 0; if all are -inf, out = 0, lse = -inf.
 *
 *   n       number of partials, 1 <= n <= 8
 *   outs    array of n tensors [B, H, P, D] (bf16 or f32, strided views)
 *   lses    array of n float32 pointers, each [B, H, P] contiguous
 *   out     [B, H, P, D] bf16 or f32; may alias outs[0] exactly (same
 *           data pointer and strides), must not overlap the other outs
 *   lse     float32 [B, H, P] contiguous, or NULL; must not overlap any lses[i]
 * D in {8, 16, ..., 64, 96, 128, 192, 256}; B, H <= 65535; bases and dim-0..2
 * strides 16-byte aligned.
 */
attn_status attn_lse_merge(int32_t n, const attn_tensor *outs, const float *const *lses,
                           const attn_tensor *out, float *lse, cudaStream_t stream);

/*
 * kv_append -- write one new token's K and V per sequence into the paged
 * cache ("KV cache in nanoVLM": after prefill, each decode step computes K/V
 * for the newest token only and adds it to the cache).
 *
 * For every sequence b: blk = block_table[b*bt_stride + pos[b]/block_size],
 * slot = pos[b] % block_size, and for every KV head g
 *     cache.k[blk, g, slot, :] = k_new[b, g, :],  cache.v likewise.
 * The copy is bit-exact.  pos[b] < 0 skips sequence b (an idle slot).
 * A position past the table (pos[b]/block_size >= max_blocks) or a block id
 * outside [0, num_blocks) sets ATTN_ERR_DEVICE_BOUNDS in the status word and
 * skips that sequence.
 *
 *   block_table  int32 [batch, >= max_blocks] (row stride bt_stride)
 *   pos          int32 [batch]
 *   k_new, v_new [batch, num_kv_heads, head_dim] bf16 (strided views)
 */
attn_status kv_append(const attn_kv_cache *cache, const int32_t *block_table, int64_t bt_stride,
                      int32_t max_blocks, const int32_t *pos,
                      const attn_tensor *k_new, const attn_tensor *v_new,
                      void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_decode_attn -- one query token per sequence attends over its paged
 * GQA cache ("KV cache in nanoVLM", attention step; "LLM inference memory
 * accounting", sections 11 and 15: query heads share KV heads, and the cache
 * is read through the block table).
 *
 * For every sequence b and query head h, with g = h / (Hq / Hkv) and
 * L = ctx_lens[b] (the appended token included):
 *     s_t = scale * <q[b,h,:], K[token t]>, t < L
 *     out[b,h,:] = sum_t softmax(s)_t * V[token t],  lse[b,h] = log sum_t exp(s_t)
 * where token t is read from block block_table[b*bt_stride + t/block_size],
 * slot t % block_size.  L = 0 gives out = 0, lse = -inf.  A context needing
 * more than max_blocks blocks, or a block id outside the cache, sets
 * ATTN_ERR_DEVICE_BOUNDS: the context is cut to the table and a block with a
 * bad id is left out (none of its slots is read), so that sequence's result
 * is not the attention over its whole context and must be discarded.
 * At head_dim 128 with at most 8 query heads per KV head the products run on
 * the tensor cores with the softmax weights rounded to bf16 before P.V (as
 * attn_fwd does); at head_dim 64 every step is fp32.
 *
 *   q       [batch, Hq, head_dim] bf16 (strided view)
 *   out     [batch, Hq, head_dim] bf16 or f32
 *   lse     float32 [batch, Hq] contiguous, or NULL
 *   workspace >= paged_decode_workspace_size(batch, Hq, max_blocks,
 *              block_size, head_dim) bytes: split-K partials, linear in
 *              the longest possible context, never quadratic, and one split
 *              count per (sequence, KV head): the CTA that finishes a
 *              (sequence, KV head) last merges its splits, so the call is a
 *              single launch.  Each call tags its counts with a generation
 *              of its own, so they need no clearing between calls, shapes
 *              or other uses of the buffer (only the status word must start
 *              at zero).  Calls that share a workspace must not overlap on
 *              the GPU.
 * Hq % Hkv == 0, Hq / Hkv <= 8.
 */
attn_status paged_decode_attn(const attn_tensor *q, const attn_kv_cache *cache,
                              const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                              const int32_t *ctx_lens, float scale,
                              const attn_tensor *out, float *lse,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_decode_attn_append -- kv_append and paged_decode_attn in one launch
 * ("KV cache in nanoVLM": each decode step computes the newest token's K/V,
 * adds it to the cache and attends with its query over the whole cache).
 *
 * The result equals kv_append(cache, block_table, pos, k_new, v_new) followed
 * by paged_decode_attn with ctx_lens[b] = pos[b] + 1, bit for bit in the
 * cache: the new token is written to block block_table[b][pos[b]/block_size],
 * slot pos[b] % block_size, and every query attends over tokens [0, pos[b]].
 * pos[b] < 0 leaves the cache alone and gives out = 0, lse = -inf.  A
 * position past the table or a bad block id sets ATTN_ERR_DEVICE_BOUNDS.
 *
 *   q            [batch, Hq, head_dim] bf16
 *   k_new, v_new [batch, Hkv, head_dim] bf16 (strided views)
 *   pos          int32 [batch]: the new token's position (tokens cached before it)
 *   workspace    as paged_decode_attn, same size for the same max_blocks
 * The appended slot must not be read by another sequence of the same call
 * (blocks shared between sequences are never appended to).
 */
attn_status paged_decode_attn_append(const attn_tensor *q, const attn_tensor *k_new, const attn_tensor *v_new,
                                     const attn_kv_cache *cache, const int32_t *block_table,
                                     int64_t bt_stride, int32_t max_blocks, const int32_t *pos,
                                     float scale, const attn_tensor *out, float *lse,
                                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_prefill_attn -- a chunk of T new tokens per sequence: write their K/V
 * into the paged cache and attend with their queries over the cache ("KV
 * cache in nanoVLM", prefill phase: the prompt is encoded in one pass and its
 * K/V fill the cache; "LLM inference memory accounting", section 20: a long
 * prompt may be prefilled chunk by chunk, which changes the schedule, not the
 * result).
 *
 * Sequence b holds start_pos[b] tokens before the chunk; chunk token i sits at
 * position p = start_pos[b] + i.  With k_new / v_new given, first
 *     cache.k[block_table[b][p/16], g, p % 16, :] = k_new[b, g, i, :]  (v likewise)
 * (both NULL: the chunk is already in the cache).  Then for every query head
 * h, with g = h / (Hq / Hkv), query i attends over the tokens t < n of KV
 * head g, read through the block table as in paged_decode_attn:
 *     n = p + 1                 causal = 1 (no token after its own position)
 *     n = start_pos[b] + T      causal = 0 (the whole chunk)
 *     out[b,h,i,:] = sum_t softmax(s)_t V[t],  lse[b,h,i] = log sum_t exp(s_t),
 *     s_t = scale * <q[b,h,i,:], K[t]>.
 * start_pos[b] < 0 or start_pos[b] + T > max_blocks * 16 sets
 * ATTN_ERR_DEVICE_BOUNDS, leaves that sequence's cache alone and writes its
 * outputs as out = 0, lse = -inf; a bad block id sets the same flag.
 *
 *   q, out       [batch, Hq, T, head_dim]; q bf16, out bf16 or f32 (strided views,
 *                16-byte aligned rows)
 *   k_new, v_new [batch, Hkv, T, head_dim] bf16, or both NULL
 *   start_pos    int32 [batch]
 *   lse          float32 [batch, Hq, T] contiguous, or NULL
 *   workspace    >= attn_fwd_workspace_size() bytes (the status word)
 * Cache head_dim 64 or 128.  Blocks of the chunk must not be shared with
 * another sequence of the same call.
 */
attn_status paged_prefill_attn(const attn_tensor *q, const attn_tensor *k_new, const attn_tensor *v_new,
                               const attn_kv_cache *cache, const int32_t *block_table, int64_t bt_stride,
                               int32_t max_blocks, const int32_t *start_pos, int32_t causal, float scale,
                               const attn_tensor *out, float *lse,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * An INT8 paged KV cache ("LLM inference memory accounting", section 18: BF16
 * KV held as INT8 halves the payload and adds scale metadata and a
 * dequantisation step).  K and V codes [num_blocks, num_kv_heads, block_size,
 * head_dim] int8 (contiguous), and one float32 scale per token row of K and of
 * V, [num_blocks, num_kv_heads, block_size] (contiguous): a row's value is
 * code * scale.  All four pointers 16-byte aligned.
 */
typedef struct attn_kv_cache_q8 {
    void *k;              /* int8 codes */
    void *v;
    float *k_scale;
    float *v_scale;
    int64_t num_blocks;
    int32_t block_size;   /* 16 */
    int32_t num_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
    int32_t reserved;     /* 0 */
} attn_kv_cache_q8;

/*
 * kv_append_q8 -- kv_append into an INT8 cache: for every sequence b (pos[b]
 * >= 0) and KV head g, the new token's K row x = k_new[b, g, :] (and likewise
 * V) is quantised with one scale per row, every step in float32:
 *     a = max_d |x_d|,  scale = a / 127,  code_d = clamp(rint(x_d / scale), -127, 127)
 * (IEEE division, rint rounding half to even; an all-zero row gets scale 0
 * and codes 0) and written to block block_table[b][pos[b]/16], slot pos[b] % 16.
 * Positions and block ids are checked as in kv_append.
 *   k_new, v_new [batch, Hkv, head_dim] bf16
 */
attn_status kv_append_q8(const attn_kv_cache_q8 *cache, const int32_t *block_table, int64_t bt_stride,
                         int32_t max_blocks, const int32_t *pos,
                         const attn_tensor *k_new, const attn_tensor *v_new,
                         void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_decode_attn_q8 -- paged_decode_attn over an INT8 cache: the same
 * definition applied to the dequantised rows (code * scale).  Reads about half
 * the bytes of the bf16 cache: 2 * head_dim + 8 bytes per token and KV head.
 * At head_dim 128 with at most 8 query heads per KV head the products run on
 * the tensor cores: q and the codes enter exactly as fp16, the softmax
 * weights (times the value scales, over a per-head reference) are rounded to
 * fp16, relative error <= 2^-11, and weights p * vs below 1e-30 are dropped
 * (p relative to the running max, so each moves an output by at most
 * 1e-30 * 127 / l, l >= 1); elsewhere every step is fp32.
 * Arguments, workspace size and error behaviour as paged_decode_attn.
 */
attn_status paged_decode_attn_q8(const attn_tensor *q, const attn_kv_cache_q8 *cache,
                                 const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                                 const int32_t *ctx_lens, float scale,
                                 const attn_tensor *out, float *lse,
                                 void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * paged_decode_attn_noalloc -- the same paged decode for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call; it
 * exists for this library's users.
 *
 * paged_decode_attn needs a workspace for its split-K partials.  A caller
 * that is handed only input and output buffers (a plugin inside a framework
 * that owns all device memory) or that must keep its device footprint fixed
 * and never call an allocator has nowhere to get one.  This call uses a
 * scratch array built into the library instead: 20 MiB per GPU, created when
 * the library's code is loaded onto that GPU and kept until the process
 * exits.  It allocates and frees nothing.  (With CUDA's lazy module loading,
 * the default, that load happens at the first use of the library's code on
 * the GPU, so the 20 MiB may leave the device's free memory during the first
 * call of this entry point there.)
 *
 *   Arguments and results are those of paged_decode_attn, without the
 *   workspace.  device_status (a device pointer, may be NULL) receives this
 *   call's status word: 0, or the bit (1 << ATTN_ERR_DEVICE_BOUNDS) when a
 *   block-table entry or context length was out of range.
 *   Returns ATTN_ERR_WORKSPACE when the call would need more than the 20 MiB
 *   scratch (batch * Hq * ceil(max_blocks*block_size/1024) * (head_dim+1) * 4
 *   bytes, plus 256); the 64-sequence, 32-head, head_dim 128 decode with
 *   contexts up to 8192 tokens needs 9.51 MB.
 *   The first call on each device looks up the scratch array's device
 *   address (with that device current) and remembers it with the id of the
 *   current context; make that first call before any stream capture.  After
 *   a device reset (a new context, into which the library's code is loaded
 *   again) the next call looks the address up again, so the same rule holds
 *   for the first call after a reset.
 *   `stream` must belong to the current device (the scratch is that
 *   device's): a stream of another device returns ATTN_ERR_INVALID_ARG.
 *   All calls on a device share the scratch.  The call clears the status
 *   word it needs zeroed on its stream; calls whose work overlaps on the GPU
 *   (other streams, other threads) race on the scratch and must be ordered by
 *   the caller.
 */
attn_status paged_decode_attn_noalloc(const attn_tensor *q, const attn_kv_cache *cache,
                                      const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                                      const int32_t *ctx_lens, float scale,
                                      const attn_tensor *out, float *lse,
                                      uint32_t *device_status, cudaStream_t stream);

/*
 * paged_decode_attn_append_q8 -- kv_append_q8 and paged_decode_attn_q8 in one
 * call ("KV cache in nanoVLM": the newest token's K/V join the cache and are
 * attended in the same step; "LLM inference memory accounting", section 18:
 * the INT8 cache).  The INT8 counterpart of paged_decode_attn_append:
 *   pos[b]          the new token's position (the context before it); the
 *                   result equals kv_append_q8(pos, k_new, v_new) followed by
 *                   paged_decode_attn_q8 with ctx_lens = pos + 1, the cache's
 *                   codes and scales bit for bit; pos < 0 marks an idle
 *                   sequence (nothing written, out = 0, lse = -inf)
 *   k_new, v_new    [batch, Hkv, head_dim] bf16, 16-byte aligned rows
 *   the rest        as paged_decode_attn_q8 (same workspace size)
 * Head dim 128 with Hq / Hkv in {1, 2, 4, 8} runs one decode launch (the
 * warp whose block holds the new slot quantises the rows) plus the split
 * merge; other shapes run kv_append_q8's kernel first.  Positions past the
 * table and bad block ids are reported as ATTN_ERR_DEVICE_BOUNDS in the
 * workspace status word, as for the two separate calls.
 */
attn_status paged_decode_attn_append_q8(const attn_tensor *q, const attn_tensor *k_new,
                                        const attn_tensor *v_new, const attn_kv_cache_q8 *cache,
                                        const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                                        const int32_t *pos, float scale, const attn_tensor *out, float *lse,
                                        void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Test/debug export: gather the paged cache of every (sequence, KV head) into
 * contiguous dst [batch, num_kv_heads, max_len, head_dim] (bf16), tokens
 * t < lens[b]; rows t >= lens[b] are left untouched.  Bit-exact.
 * which = 0 gathers K, 1 gathers V.  Same device-status rules as kv_append. */
attn_status paged_kv_gather(const attn_kv_cache *cache, int32_t which,
                            const int32_t *block_table, int64_t bt_stride, int32_t max_blocks,
                            const int32_t *lens, int32_t batch, int64_t max_len, void *dst,
                            void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Self-test of the device-side hang guard: launches one thread that waits on
 * a barrier phase nothing ever completes.  The wait gives up after
 * timeout_us microseconds (1 .. 1000000), ORs ATTN_ERR_TIMEOUT into the
 * workspace's status word and the kernel returns; the CUDA context stays
 * usable.  Every pipeline wait in the library's kernels uses the same guard
 * (with a 2 s limit). */
attn_status attn_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint32_t timeout_us,
                                       cudaStream_t stream);

/* Copy the workspace's status word to the host (synchronises `stream`).
 * Returns ATTN_OK or the lowest-numbered error recorded since the last reset;
 * *raw (if not NULL) receives the full bit set, bit e meaning status e. */
attn_status attn_check_device_status(const void *workspace, uint32_t *raw, cudaStream_t stream);

/* Clear the status word (enqueued on `stream`). */
attn_status attn_reset_device_status(void *workspace, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char *attn_status_string(attn_status status);

/* Library version as major*10000 + minor*100 + patch. */
int32_t attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_H */
