// api.cu -- the extern "C" entry points of libattn: argument validation on the
// host (nothing is launched for a bad argument), workspace sizing, dispatch
// to the kernel launchers, and the device status word.
#include <math.h>
#include <string.h>

#include <atomic>

#include "internal.h"
#include "libattn.h"

namespace attn {
namespace {

constexpr size_t kStatusBytes = 256;  // head of every workspace: the status word

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int dtype) { return dtype == ATTN_BF16 ? 2 : 4; }

// Shape/stride sanity of a caller tensor: ndim, non-negative sizes, unit
// innermost stride, non-null data when non-empty.
attn_status check_tensor(const attn_tensor* t, int ndim) {
  if (t == nullptr || t->ndim != ndim) return ATTN_ERR_INVALID_ARG;
  if (t->dtype != ATTN_F32 && t->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  int64_t numel = 1;
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return ATTN_ERR_INVALID_ARG;
    numel *= t->shape[i];
  }
  if (numel > 0) {
    if (t->data == nullptr) return ATTN_ERR_INVALID_ARG;
    if (t->stride[ndim - 1] != 1) return ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < ndim - 1; ++i)
      if (t->stride[i] < 0) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

// 16-byte vector access: base and the outer strides keep 16-byte alignment.
bool vec16_ok(const attn_tensor* t) {
  const int eb = elem_bytes(t->dtype);
  if (!aligned(t->data, 16)) return false;
  for (int i = 0; i < t->ndim - 1; ++i)
    if ((t->stride[i] * eb) % 16 != 0 && t->shape[i] > 1) return false;
  return true;
}

View4 view(const attn_tensor* t) {
  View4 v;
  v.data = t->data;
  v.dtype = t->dtype;
  for (int i = 0; i < 4; ++i) {
    v.shape[i] = i < t->ndim ? t->shape[i] : 1;
    v.stride[i] = i < t->ndim ? t->stride[i] : 0;
  }
  return v;
}

attn_status check_workspace(void* ws, size_t bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256) || bytes < need) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

attn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

attn_status check_cache(const attn_kv_cache* c) {
  if (c == nullptr || c->k == nullptr || c->v == nullptr) return ATTN_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (c->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (c->block_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(c->k, 16) || !aligned(c->v, 16)) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status check_cache_q8(const attn_kv_cache_q8* c) {
  if (c == nullptr || c->k == nullptr || c->v == nullptr || c->k_scale == nullptr || c->v_scale == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (c->block_size != 16) return ATTN_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned(c->k, 16) || !aligned(c->v, 16) || !aligned(c->k_scale, 16) || !aligned(c->v_scale, 16))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

PagedCache paged_q8(const attn_kv_cache_q8* c) {
  PagedCache p;
  p.k = c->k;
  p.v = c->v;
  p.k_scale = c->k_scale;
  p.v_scale = c->v_scale;
  p.num_blocks = c->num_blocks;
  p.block_size = c->block_size;
  p.Hkv = c->num_kv_heads;
  p.D = c->head_dim;
  return p;
}

PagedCache paged(const attn_kv_cache* c) {
  PagedCache p;
  p.k = c->k;
  p.v = c->v;
  p.num_blocks = c->num_blocks;
  p.block_size = c->block_size;
  p.Hkv = c->num_kv_heads;
  p.D = c->head_dim;
  return p;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int32_t attn_version(void) { return 100; }

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
  }
  return "ATTN_UNKNOWN_STATUS";
}

size_t attn_fwd_workspace_size(void) { return kStatusBytes; }

// attn_fwd workspace: [status word][key-tile bounds (D = 64)][split-unit partials]
static size_t key_bound_bytes(int32_t batch, int32_t kv_heads, int64_t num_keys, int32_t head_dim) {
  if (head_dim != 64) return 0;  // the key-tile bounds serve the D = 64 kernel only
  const size_t tiles = static_cast<size_t>((num_keys + kKeyTile - 1) / kKeyTile);
  const size_t bytes = static_cast<size_t>(batch) * kv_heads * tiles * sizeof(float);
  return (bytes + 255) & ~size_t(255);
}

size_t attn_fwd_workspace_size_for(int32_t batch, int32_t kv_heads, int64_t num_keys, int32_t head_dim) {
  if (batch < 0 || kv_heads < 0 || num_keys < 0 || head_dim <= 0) return 0;
  if (head_dim != 64 && head_dim != 128) return kStatusBytes;  // no tensor-core kernel: the status word only
  const size_t parts = (split_partial_bytes(head_dim) + 255) & ~size_t(255);
  return kStatusBytes + key_bound_bytes(batch, kv_heads, num_keys, head_dim) + parts;
}
size_t kv_append_workspace_size(void) { return kStatusBytes; }

size_t paged_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks, int32_t block_size,
                                   int32_t head_dim) {
  if (batch < 0 || num_q_heads < 0 || max_blocks < 0 || block_size <= 0 || head_dim <= 0) return 0;
  const int ns = decode_num_splits(max_blocks, block_size);
  return kStatusBytes + decode_partial_bytes(batch, num_q_heads, ns, head_dim);
}

static attn_status attn_fwd_impl(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                                 const float* key_pad_mask, int64_t mask_stride_b, const int32_t* key_lens,
                                 float scale, const attn_tensor* out, float* lse, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  attn_status st;
  if ((st = check_tensor(q, 4)) != ATTN_OK) return st;
  if ((st = check_tensor(k, 4)) != ATTN_OK) return st;
  if ((st = check_tensor(v, 4)) != ATTN_OK) return st;
  if ((st = check_tensor(out, 4)) != ATTN_OK) return st;
  const int64_t B = q->shape[0], Hq = q->shape[1], Pq = q->shape[2], D = q->shape[3];
  const int64_t Hkv = k->shape[1], Pk = k->shape[2];
  if (k->shape[0] != B || k->shape[3] != D) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 4; ++i) {
    if (v->shape[i] != k->shape[i]) return ATTN_ERR_INVALID_ARG;
    if (out->shape[i] != q->shape[i]) return ATTN_ERR_INVALID_ARG;
  }
  if (D <= 0 || Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q->dtype != k->dtype || q->dtype != v->dtype) return ATTN_ERR_INVALID_ARG;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, attn_fwd_workspace_size())) != ATTN_OK) return st;
  if (key_pad_mask != nullptr && B > 1 && mask_stride_b < Pk) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535 || Pq > (int64_t(1) << 31) - 1 || Pk > (int64_t(1) << 31) - 1)
    return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || Pq == 0) return ATTN_OK;
  if (!vec16_ok(out)) return ATTN_ERR_INVALID_ARG;

  AttnFwdArgs a;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.Pq = Pq; a.Pk = Pk; a.D = D;
  a.q = view(q); a.k = view(k); a.v = view(v); a.out = view(out);
  a.mask = key_pad_mask;
  a.mask_stride = mask_stride_b;
  a.key_lens = key_lens;
  a.key_bound = nullptr;
  a.part_ws = nullptr;
  a.part_bytes = 0;
  a.scale = scale;
  a.lse = lse;
  a.status = static_cast<uint32_t*>(workspace);
  if (Pk == 0) return from_cuda(launch_attn_empty_keys(a, stream));

  if (q->dtype == ATTN_BF16) {
    if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
    if (!vec16_ok(q) || !vec16_ok(k) || !vec16_ok(v)) return ATTN_ERR_INVALID_ARG;
    // D = 64 with room in the workspace: per-tile key bounds first, which
    // let the kernel skip its softmax max pass on most tiles.  The extra pass
    // (one read of K and a launch) pays only on calls of a few hundred
    // microseconds and up: from B Hq Pq Pk D = 2^36 on.
    const double work = static_cast<double>(B) * Hq * static_cast<double>(Pq) * static_cast<double>(Pk) * D;
    const bool room = workspace_bytes >= attn_fwd_workspace_size_for(static_cast<int32_t>(B),
                                                                     static_cast<int32_t>(Hkv), Pk,
                                                                     static_cast<int32_t>(D));
    if (room) {
      const size_t kb = key_bound_bytes(static_cast<int32_t>(B), static_cast<int32_t>(Hkv), Pk,
                                        static_cast<int32_t>(D));
      a.part_ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes + kb);
      a.part_bytes = workspace_bytes - kStatusBytes - kb;
      if (D == 64 && work >= 68719476736.0) {
        a.key_bound = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
        if ((st = from_cuda(launch_key_tile_bound(a, stream))) != ATTN_OK) return st;
      }
    }
    return from_cuda(launch_attn_fwd_tc(a, stream));
  }
  if (D > 128 || D % 4 != 0) return ATTN_ERR_UNSUPPORTED;
  if (!vec16_ok(q) || !vec16_ok(k) || !vec16_ok(v)) return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_attn_fwd_simt(a, stream));
}

attn_status attn_fwd(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v, const float* key_pad_mask,
                     int64_t mask_stride_b, float scale, const attn_tensor* out, float* lse, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  return attn_fwd_impl(q, k, v, key_pad_mask, mask_stride_b, nullptr, scale, out, lse, workspace, workspace_bytes,
                       stream);
}

attn_status attn_fwd_varlen(const attn_tensor* q, const attn_tensor* k, const attn_tensor* v,
                            const int32_t* key_lens, float scale, const attn_tensor* out, float* lse,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (key_lens == nullptr) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, nullptr, 0, key_lens, scale, out, lse, workspace, workspace_bytes, stream);
}

attn_status attn_key_padding_to_additive(const uint8_t* key_padding_mask, int64_t kpm_stride_b, int32_t batch,
                                         int64_t num_keys, float* additive_mask, int64_t out_stride_b,
                                         cudaStream_t stream) {
  if (batch < 0 || num_keys < 0 || batch > 65535) return ATTN_ERR_INVALID_ARG;
  if (batch == 0 || num_keys == 0) return ATTN_OK;
  if (key_padding_mask == nullptr || additive_mask == nullptr) return ATTN_ERR_INVALID_ARG;
  if (batch > 1 && (kpm_stride_b < num_keys || out_stride_b < num_keys)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(additive_mask, 4)) return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_padding_mask_to_additive(key_padding_mask, kpm_stride_b, batch, num_keys, additive_mask,
                                                   out_stride_b, stream));
}

attn_status attn_lse_merge(int32_t n, const attn_tensor* outs, const float* const* lses, const attn_tensor* out,
                           float* lse, cudaStream_t stream) {
  if (n < 1 || n > 8 || outs == nullptr || lses == nullptr) return ATTN_ERR_INVALID_ARG;
  attn_status st;
  if ((st = check_tensor(out, 4)) != ATTN_OK) return st;
  const int64_t B = out->shape[0], H = out->shape[1], P = out->shape[2], D = out->shape[3];
  for (int i = 0; i < n; ++i) {
    if ((st = check_tensor(&outs[i], 4)) != ATTN_OK) return st;
    for (int d = 0; d < 4; ++d)
      if (outs[i].shape[d] != out->shape[d]) return ATTN_ERR_INVALID_ARG;
    if (outs[i].dtype != outs[0].dtype) return ATTN_ERR_INVALID_ARG;
  }
  // head dims with a merge kernel instance: 8..64 in steps of 8, 96, 128, 192, 256
  if (D % 8 != 0 || D > 256 || D <= 0 || (D > 64 && D != 96 && D != 128 && D != 192 && D != 256))
    return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (B * H * P == 0) return ATTN_OK;
  for (int i = 0; i < n; ++i) {
    if (lses[i] == nullptr || !aligned(lses[i], 4)) return ATTN_ERR_INVALID_ARG;
    if (!vec16_ok(&outs[i])) return ATTN_ERR_INVALID_ARG;
  }
  if (!vec16_ok(out)) return ATTN_ERR_INVALID_ARG;
  MergeArgs a;
  a.n = n;
  a.B = B; a.H = H; a.P = P; a.D = D;
  for (int i = 0; i < n; ++i) {
    a.outs[i] = view(&outs[i]);
    a.lses[i] = lses[i];
  }
  a.out = view(out);
  a.lse = lse;
  return from_cuda(launch_lse_merge(a, stream));
}

static attn_status kv_append_core(const PagedCache& pc, const int32_t* block_table, int64_t bt_stride,
                                  int32_t max_blocks, const int32_t* pos, const attn_tensor* k_new,
                                  const attn_tensor* v_new, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
  attn_status st;
  if ((st = check_tensor(k_new, 3)) != ATTN_OK) return st;
  if ((st = check_tensor(v_new, 3)) != ATTN_OK) return st;
  const int64_t B = k_new->shape[0];
  if (k_new->dtype != ATTN_BF16 || v_new->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i)
    if (v_new->shape[i] != k_new->shape[i]) return ATTN_ERR_INVALID_ARG;
  if (k_new->shape[1] != pc.Hkv || k_new->shape[2] != pc.D) return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, kv_append_workspace_size())) != ATTN_OK) return st;
  if (B == 0) return ATTN_OK;
  if (B > 0x7fffffff) return ATTN_ERR_UNSUPPORTED;
  if (block_table == nullptr || pos == nullptr || max_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (B > 1 && bt_stride < max_blocks) return ATTN_ERR_INVALID_ARG;
  if (!vec16_ok(k_new) || !vec16_ok(v_new)) return ATTN_ERR_INVALID_ARG;
  AppendArgs a;
  a.cache = pc;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks;
  a.pos = pos;
  a.B = B;
  a.k_new = view(k_new);
  a.v_new = view(v_new);
  a.status = static_cast<uint32_t*>(workspace);
  return from_cuda(pc.k_scale != nullptr ? launch_kv_append_q8(a, stream) : launch_kv_append(a, stream));
}

attn_status kv_append(const attn_kv_cache* cache, const int32_t* block_table, int64_t bt_stride,
                      int32_t max_blocks, const int32_t* pos, const attn_tensor* k_new, const attn_tensor* v_new,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache(cache)) != ATTN_OK) return st;
  return kv_append_core(paged(cache), block_table, bt_stride, max_blocks, pos, k_new, v_new, workspace,
                        workspace_bytes, stream);
}

attn_status kv_append_q8(const attn_kv_cache_q8* cache, const int32_t* block_table, int64_t bt_stride,
                         int32_t max_blocks, const int32_t* pos, const attn_tensor* k_new, const attn_tensor* v_new,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache_q8(cache)) != ATTN_OK) return st;
  return kv_append_core(paged_q8(cache), block_table, bt_stride, max_blocks, pos, k_new, v_new, workspace,
                        workspace_bytes, stream);
}

attn_status paged_kv_gather(const attn_kv_cache* cache, int32_t which, const int32_t* block_table,
                            int64_t bt_stride, int32_t max_blocks, const int32_t* lens, int32_t batch,
                            int64_t max_len, void* dst, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache(cache)) != ATTN_OK) return st;
  if (which != 0 && which != 1) return ATTN_ERR_INVALID_ARG;
  if (batch < 0 || max_len < 0) return ATTN_ERR_INVALID_ARG;
  if ((st = check_workspace(workspace, workspace_bytes, kv_append_workspace_size())) != ATTN_OK) return st;
  if (batch == 0 || max_len == 0) return ATTN_OK;
  if (block_table == nullptr || lens == nullptr || dst == nullptr || max_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if (batch > 1 && bt_stride < max_blocks) return ATTN_ERR_INVALID_ARG;
  if (!aligned(dst, 16) || batch > 65535 || (max_len + 15) / 16 > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  GatherArgs a;
  a.cache = paged(cache);
  a.which = which;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks;
  a.lens = lens;
  a.B = batch;
  a.max_len = max_len;
  a.dst = dst;
  a.status = static_cast<uint32_t*>(workspace);
  return from_cuda(launch_paged_gather(a, stream));
}

// Every decode call tags its split counts with a generation of its own, so a
// workspace needs no clearing between calls, shapes or other uses (zero is
// skipped: a zero-filled word then always belongs to no call).
static std::atomic<uint32_t> g_decode_gen{0};

static uint32_t next_decode_gen() {
  uint32_t g = g_decode_gen.fetch_add(1, std::memory_order_relaxed) + 1;
  if (g == 0) g = g_decode_gen.fetch_add(1, std::memory_order_relaxed) + 1;
  return g;
}

static attn_status paged_decode_impl(const attn_tensor* q, const attn_tensor* k_new, const attn_tensor* v_new,
                                     const PagedCache& pc, const int32_t* block_table, int64_t bt_stride,
                                     int32_t max_blocks, const int32_t* lens_or_pos, float scale,
                                     const attn_tensor* out, float* lse, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  const int32_t* ctx_lens = lens_or_pos;
  attn_status st;
  if ((st = check_tensor(q, 3)) != ATTN_OK) return st;
  if ((st = check_tensor(out, 3)) != ATTN_OK) return st;
  const int64_t B = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  for (int i = 0; i < 3; ++i)
    if (out->shape[i] != q->shape[i]) return ATTN_ERR_INVALID_ARG;
  if (q->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (D != pc.D) return ATTN_ERR_INVALID_ARG;
  if (Hq <= 0 || Hq % pc.Hkv != 0) return ATTN_ERR_INVALID_ARG;
  const int64_t G = Hq / pc.Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_ERR_UNSUPPORTED;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (max_blocks <= 0 || max_blocks > (1 << 24)) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || B * Hq > (int64_t(1) << 30)) return ATTN_ERR_UNSUPPORTED;
  const size_t need = paged_decode_workspace_size(static_cast<int32_t>(B), static_cast<int32_t>(Hq), max_blocks,
                                                  pc.block_size, pc.D);
  if ((st = check_workspace(workspace, workspace_bytes, need)) != ATTN_OK) return st;
  if (B == 0) return ATTN_OK;
  if (block_table == nullptr || ctx_lens == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B > 1 && bt_stride < max_blocks) return ATTN_ERR_INVALID_ARG;
  if (!vec16_ok(q)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(out->data, 8)) return ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < 2; ++i)
    if (out->stride[i] % 2 != 0 && out->shape[i] > 1) return ATTN_ERR_INVALID_ARG;
  const bool fused = k_new != nullptr || v_new != nullptr;
  if (fused) {
    if ((st = check_tensor(k_new, 3)) != ATTN_OK) return st;
    if ((st = check_tensor(v_new, 3)) != ATTN_OK) return st;
    if (k_new->dtype != ATTN_BF16 || v_new->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
      if (v_new->shape[i] != k_new->shape[i]) return ATTN_ERR_INVALID_ARG;
    if (k_new->shape[0] != B || k_new->shape[1] != pc.Hkv || k_new->shape[2] != D)
      return ATTN_ERR_INVALID_ARG;
    if (!vec16_ok(k_new) || !vec16_ok(v_new)) return ATTN_ERR_INVALID_ARG;
  }
  DecodeArgs a;
  a.cache = pc;
  a.q = view(q);
  a.k_new = fused ? view(k_new) : View4{};
  a.v_new = fused ? view(v_new) : View4{};
  a.out = view(out);
  a.lse = lse;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks;
  a.ctx_lens = ctx_lens;
  a.B = B;
  a.Hq = Hq;
  a.scale = scale;
  a.partials = static_cast<uint8_t*>(workspace) + kStatusBytes;
  a.n_split = decode_num_splits(max_blocks, pc.block_size);
  a.gen = next_decode_gen();
  a.status = static_cast<uint32_t*>(workspace);
  return from_cuda(launch_paged_decode(a, stream));
}

attn_status paged_decode_attn(const attn_tensor* q, const attn_kv_cache* cache, const int32_t* block_table,
                              int64_t bt_stride, int32_t max_blocks, const int32_t* ctx_lens, float scale,
                              const attn_tensor* out, float* lse, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache(cache)) != ATTN_OK) return st;
  return paged_decode_impl(q, nullptr, nullptr, paged(cache), block_table, bt_stride, max_blocks, ctx_lens, scale,
                           out, lse, workspace, workspace_bytes, stream);
}

attn_status paged_decode_attn_q8(const attn_tensor* q, const attn_kv_cache_q8* cache, const int32_t* block_table,
                                 int64_t bt_stride, int32_t max_blocks, const int32_t* ctx_lens, float scale,
                                 const attn_tensor* out, float* lse, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache_q8(cache)) != ATTN_OK) return st;
  return paged_decode_impl(q, nullptr, nullptr, paged_q8(cache), block_table, bt_stride, max_blocks, ctx_lens, scale,
                           out, lse, workspace, workspace_bytes, stream);
}

attn_status paged_decode_attn_append(const attn_tensor* q, const attn_tensor* k_new, const attn_tensor* v_new,
                                     const attn_kv_cache* cache, const int32_t* block_table, int64_t bt_stride,
                                     int32_t max_blocks, const int32_t* pos, float scale, const attn_tensor* out,
                                     float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (k_new == nullptr || v_new == nullptr) return ATTN_ERR_INVALID_ARG;
  attn_status st;
  if ((st = check_cache(cache)) != ATTN_OK) return st;
  return paged_decode_impl(q, k_new, v_new, paged(cache), block_table, bt_stride, max_blocks, pos, scale, out, lse,
                           workspace, workspace_bytes, stream);
}

attn_status paged_decode_attn_append_q8(const attn_tensor* q, const attn_tensor* k_new, const attn_tensor* v_new,
                                        const attn_kv_cache_q8* cache, const int32_t* block_table, int64_t bt_stride,
                                        int32_t max_blocks, const int32_t* pos, float scale, const attn_tensor* out,
                                        float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (k_new == nullptr || v_new == nullptr) return ATTN_ERR_INVALID_ARG;
  attn_status st;
  if ((st = check_cache_q8(cache)) != ATTN_OK) return st;
  return paged_decode_impl(q, k_new, v_new, paged_q8(cache), block_table, bt_stride, max_blocks, pos, scale, out,
                           lse, workspace, workspace_bytes, stream);
}

attn_status paged_prefill_attn(const attn_tensor* q, const attn_tensor* k_new, const attn_tensor* v_new,
                               const attn_kv_cache* cache, const int32_t* block_table, int64_t bt_stride,
                               int32_t max_blocks, const int32_t* start_pos, int32_t causal, float scale,
                               const attn_tensor* out, float* lse, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  attn_status st;
  if ((st = check_cache(cache)) != ATTN_OK) return st;
  if ((st = check_tensor(q, 4)) != ATTN_OK) return st;
  if ((st = check_tensor(out, 4)) != ATTN_OK) return st;
  const int64_t B = q->shape[0], Hq = q->shape[1], T = q->shape[2], D = q->shape[3];
  for (int i = 0; i < 4; ++i)
    if (out->shape[i] != q->shape[i]) return ATTN_ERR_INVALID_ARG;
  if (q->dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (D != cache->head_dim) return ATTN_ERR_INVALID_ARG;
  if (Hq <= 0 || Hq % cache->num_kv_heads != 0) return ATTN_ERR_INVALID_ARG;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (max_blocks <= 0 || max_blocks > (1 << 24)) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535 || T > (int64_t(1) << 30) || cache->num_blocks > 0x7fffffff)
    return ATTN_ERR_UNSUPPORTED;
  if ((k_new == nullptr) != (v_new == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (k_new != nullptr) {
    if ((st = check_tensor(k_new, 4)) != ATTN_OK) return st;
    if ((st = check_tensor(v_new, 4)) != ATTN_OK) return st;
    if (k_new->dtype != ATTN_BF16 || v_new->dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
    const int64_t want[4] = {B, cache->num_kv_heads, T, D};
    for (int i = 0; i < 4; ++i)
      if (k_new->shape[i] != want[i] || v_new->shape[i] != want[i]) return ATTN_ERR_INVALID_ARG;
  }
  if ((st = check_workspace(workspace, workspace_bytes, kStatusBytes)) != ATTN_OK) return st;
  if (B == 0 || T == 0) return ATTN_OK;
  if (block_table == nullptr || start_pos == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B > 1 && bt_stride < max_blocks) return ATTN_ERR_INVALID_ARG;
  if (!vec16_ok(q) || !vec16_ok(out)) return ATTN_ERR_INVALID_ARG;
  if (k_new != nullptr && (!vec16_ok(k_new) || !vec16_ok(v_new))) return ATTN_ERR_INVALID_ARG;
  PrefillArgs a;
  a.cache = paged(cache);
  a.q = view(q);
  a.out = view(out);
  a.k_new = k_new != nullptr ? view(k_new) : View4{};
  a.v_new = v_new != nullptr ? view(v_new) : View4{};
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.max_blocks = max_blocks;
  a.start_pos = start_pos;
  a.causal = causal;
  a.B = B;
  a.Hq = Hq;
  a.T = T;
  a.scale = scale;
  a.lse = lse;
  a.status = static_cast<uint32_t*>(workspace);
  if (k_new != nullptr && (st = from_cuda(launch_kv_append_chunk(a, stream))) != ATTN_OK) return st;
  return from_cuda(launch_paged_prefill_tc(a, stream));
}

attn_status attn_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t timeout_us,
                                       cudaStream_t stream) {
  attn_status st;
  if ((st = check_workspace(workspace, workspace_bytes, kStatusBytes)) != ATTN_OK) return st;
  if (timeout_us == 0 || timeout_us > 1000000u) return ATTN_ERR_INVALID_ARG;
  return from_cuda(launch_wait_timeout_selftest(static_cast<uint32_t*>(workspace),
                                                static_cast<uint64_t>(timeout_us) * 1000u, stream));
}

attn_status attn_check_device_status(const void* workspace, uint32_t* raw, cudaStream_t stream) {
  if (workspace == nullptr) return ATTN_ERR_WORKSPACE;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  if (raw != nullptr) *raw = word;
  for (int e = 1; e < 32; ++e)
    if (word & (1u << e)) return static_cast<attn_status>(e);
  return ATTN_OK;
}

attn_status attn_reset_device_status(void* workspace, cudaStream_t stream) {
  if (workspace == nullptr) return ATTN_ERR_WORKSPACE;
  return from_cuda(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), stream));
}

}  // extern "C"
