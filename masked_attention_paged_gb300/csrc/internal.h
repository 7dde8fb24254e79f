// internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel launchers.  Arguments reaching these functions are validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "libattn.h"

namespace attn {

struct View4 {
  void* data;
  int dtype;  // attn_dtype
  int64_t shape[4];
  int64_t stride[4];  // elements
};

struct AttnFwdArgs {
  int64_t B, Hq, Hkv, Pq, Pk, D;
  View4 q, k, v, out;
  const float* mask;  // [B, Pk] additive, row stride mask_stride; may be null
  int64_t mask_stride;
  const int32_t* key_lens;  // [B] valid keys per batch row (keys past it are padding); may be null
  float* key_bound;         // [B, Hkv, ceil(Pk/128)] largest |k| element per key tile, or null
  float* part_ws;           // room for split-unit partials (tensor-core path), or null
  size_t part_bytes;
  float scale;
  float* lse;         // [B, Hq, Pq] contiguous, may be null
  uint32_t* status;   // device status word
};

// bf16 inputs, D in {64, 128}: tcgen05 + TMA kernel
cudaError_t launch_attn_fwd_tc(const AttnFwdArgs& a, cudaStream_t stream);
// D = 128, no mask, no key lengths, scale > 0: the kernel on CTA pairs;
// cudaErrorNotSupported when the call or the device does not allow it
bool pair_kernel_applies(const AttnFwdArgs& a);
cudaError_t launch_attn_fwd_pair(const AttnFwdArgs& a, cudaStream_t stream);
// bf16 tensor map over a [B, H, P, D] view: box 64 columns x box_rows rows,
// 128-byte swizzle; slot[0..2] = coordinate slot of the row, head, batch
bool make_tile_map(CUtensorMap* map, int slot[3], const View4& t, int box_rows);
// merge the key parts of the split last-wave units of a tensor-core launch
// (256-row units, `split` parts each, normalised f32 rows + natural-log LSEs)
cudaError_t launch_split_merge(int D, bool out_bf16, const float* part_o, const float* part_lse, int split,
                               int full_units, int tail, int nq, int Hq, int Pq, const View4& out, float* lse,
                               cudaStream_t stream);
// f32 inputs, D <= 128, D % 4 == 0: FFMA kernel
cudaError_t launch_attn_fwd_simt(const AttnFwdArgs& a, cudaStream_t stream);
// Pk == 0: out = 0, lse = -inf
cudaError_t launch_attn_empty_keys(const AttnFwdArgs& a, cudaStream_t stream);
// a.key_bound[(b * Hkv + g) * tiles + j] = max |k| over keys [128 j, 128 j + 128) of (b, g)
cudaError_t launch_key_tile_bound(const AttnFwdArgs& a, cudaStream_t stream);
constexpr int kKeyTile = 128;  // keys per tile of the tensor-core kernel
constexpr int kMaxSplitRows = 256;  // query rows per tensor-core CTA
// streaming multiprocessors of the current device (cached per device)
int device_sm_count();
// bytes of split-unit partials the tensor-core kernel may need for head dim D
size_t split_partial_bytes(int D);

struct MergeArgs {
  int n;
  int64_t B, H, P, D;
  View4 outs[8];
  const float* lses[8];
  View4 out;
  float* lse;
};
cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t stream);

struct PagedCache {
  void* k;  // bf16, or int8 codes when k_scale is set
  void* v;
  const float* k_scale = nullptr;  // INT8 cache: float32 per token row [num_blocks, Hkv, block_size]
  const float* v_scale = nullptr;
  int64_t num_blocks;
  int block_size;
  int Hkv;
  int D;
};

struct AppendArgs {
  PagedCache cache;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* pos;
  int64_t B;
  View4 k_new, v_new;  // [B, Hkv, D] (shape[3] unused)
  uint32_t* status;
};
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);
// INT8 cache (a.cache.k_scale set): quantise and write the new token's rows
cudaError_t launch_kv_append_q8(const AppendArgs& a, cudaStream_t stream);

struct GatherArgs {
  PagedCache cache;
  int which;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* lens;
  int64_t B;
  int64_t max_len;
  void* dst;
  uint32_t* status;
};
cudaError_t launch_paged_gather(const GatherArgs& a, cudaStream_t stream);

struct DecodeArgs {
  PagedCache cache;
  View4 q;    // [B, Hq, D]
  View4 out;  // [B, Hq, D]
  float* lse; // [B, Hq] or null
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* ctx_lens;  // or, with k_new set, each sequence's new-token position
  View4 k_new, v_new;       // fused append: [B, Hkv, D]; data null for a plain decode
  int64_t B, Hq;
  float scale;
  void* partials;  // workspace after the status block
  int n_split;     // split slots per (sequence, head) in the partial buffer
  uint32_t gen;    // this call's generation, tags its split counts (never 0)
  uint32_t* status;
};
// tokens per split-K work unit of the paged decode
constexpr int kDecodeSplitTokens = 1024;
int decode_num_splits(int max_blocks, int block_size);
size_t decode_partial_bytes(int64_t B, int64_t Hq, int n_split, int D);
cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream);
// where the decode kernels' splits meet (decode_common.cuh): the partials and
// split counts in a.partials, and a.out / a.lse, which the last split of each
// (sequence, KV head) writes
struct SplitMerge;
SplitMerge decode_split_merge(const DecodeArgs& a, int D);
// INT8 cache, D = 128, 16-token blocks, Hq / Hkv in {1, 2, 4, 8}, no fused append:
// the tensor-core decode (decode_q8.cu) serves the call
bool paged_decode_q8_mma_supported(const DecodeArgs& a);
cudaError_t launch_paged_decode_q8_mma(const DecodeArgs& a, cudaStream_t stream);
// 4-D u8 tensor map over INT8 codes [num_blocks, Hkv, 16, 128] (contiguous):
// box = the 16 x 128 codes of one (block, head), 128-byte swizzle
bool make_code_cache_map(CUtensorMap* map, void* base, int64_t num_blocks, int Hkv);
// bf16 cache, D = 128, 16-token blocks, Hq / Hkv in {1, 2, 4, 8}: the tensor-core
// decode (decode_tc.cu) serves the call, fused append included
bool paged_decode_tc_supported(const DecodeArgs& a);
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, cudaStream_t stream);
// 4-D bf16 tensor map over one paged cache tensor [num_blocks, Hkv, 16, 128]
// (contiguous): box 64 columns x 16 rows of one (block, head), 128-byte swizzle
bool make_bf16_cache_map(CUtensorMap* map, void* base, int64_t num_blocks, int Hkv);

struct PrefillArgs {
  PagedCache cache;
  View4 q, out;        // [B, Hq, T, D]
  View4 k_new, v_new;  // [B, Hkv, T, D]; data null when the chunk is already cached
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* start_pos;  // [B] tokens cached before the chunk
  int causal;
  int64_t B, Hq, T;
  float scale;
  float* lse;  // [B, Hq, T] or null
  uint32_t* status;
};
// write the chunk's K/V to positions start_pos[b] + i of each sequence
cudaError_t launch_kv_append_chunk(const PrefillArgs& a, cudaStream_t stream);
// the chunk's queries over the paged cache (tcgen05 kernel, paged instance)
cudaError_t launch_paged_prefill_tc(const PrefillArgs& a, cudaStream_t stream);

// boolean key-padding mask (non-zero = padded) -> additive 0 / -inf
cudaError_t launch_padding_mask_to_additive(const uint8_t* kpm, int64_t kpm_stride, int64_t B, int64_t Pk,
                                            float* out, int64_t out_stride, cudaStream_t stream);

// one bounded mbarrier wait that nothing completes (exercises the timeout path)
cudaError_t launch_wait_timeout_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace attn
