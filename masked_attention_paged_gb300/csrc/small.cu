// small.cu -- the bandwidth-bound kernels around the attention kernels:
//   kv_append       one token's K/V per sequence into the paged cache
//   paged_gather    paged cache -> contiguous copy (test/debug export)
//   lse_merge       n-way merge of chunk results through their LSE
//   empty_keys      out = 0, lse = -inf when there are no keys at all
// All moves are 16-byte vectors; append and gather are bit copies.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "q8_quant.cuh"
#include "internal.h"

namespace attn {
namespace {

// ---------------------------------------------------------------------------
// kv_append ("KV cache in nanoVLM": the decode step computes K/V of the newest
// token only and adds it to the cache).  One CTA per sequence; each thread
// moves 16 bytes of K and 16 bytes of V.
// ---------------------------------------------------------------------------
struct AppendParams {
  uint16_t* kc;
  uint16_t* vc;
  int64_t num_blocks;
  int block_size, Hkv, D;
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* pos;
  const uint16_t* kn;
  const uint16_t* vn;
  int64_t kn_stride[2], vn_stride[2];  // batch, head (elements)
  uint32_t* status;
};

__global__ void kv_append_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int pos = p.pos[b];
  if (pos < 0) return;  // idle sequence
  const int lb = pos / p.block_size;
  if (lb >= p.max_blocks) {
    if (threadIdx.x == 0) report(p.status, kStatusBounds);
    return;
  }
  const int blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + lb];
  if (blk < 0 || blk >= p.num_blocks) {
    if (threadIdx.x == 0) report(p.status, kStatusBounds);
    return;
  }
  const int slot = pos % p.block_size;
  const int vec_per_head = p.D / 8;
  for (int i = threadIdx.x; i < p.Hkv * vec_per_head; i += blockDim.x) {
    const int g = i / vec_per_head;
    const int c = (i % vec_per_head) * 8;
    const int64_t dst = ((static_cast<int64_t>(blk) * p.Hkv + g) * p.block_size + slot) * p.D + c;
    const uint4 kv = *reinterpret_cast<const uint4*>(p.kn + b * p.kn_stride[0] + g * p.kn_stride[1] + c);
    const uint4 vv = *reinterpret_cast<const uint4*>(p.vn + b * p.vn_stride[0] + g * p.vn_stride[1] + c);
    *reinterpret_cast<uint4*>(p.kc + dst) = kv;
    *reinterpret_cast<uint4*>(p.vc + dst) = vv;
  }
}

// ---------------------------------------------------------------------------
// kv_append_q8: quantise one new token's K and V rows per KV head (one warp per
// row pair) and write codes and scales.  Every step in float32 as the INT8
// definition reads: a = max |x|, scale = a / 127, code = clamp(rint(x / scale),
// -127, 127) with IEEE division and round-half-even (0 / 0 for a zero row).
// ---------------------------------------------------------------------------
struct AppendQ8Params {
  int8_t* kq;
  int8_t* vq;
  float* ks;
  float* vs;
  int64_t num_blocks;
  int Hkv, D;
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* pos;
  const uint16_t* kn;
  const uint16_t* vn;
  int64_t kn_stride[2], vn_stride[2];  // batch, head (elements)
  uint32_t* status;
};

template <int D>
__device__ __forceinline__ void quantise_row_q8(const uint16_t* src, int8_t* dst, float* scale_out, int lane) {
  constexpr int E = D / 32;  // elements per lane
  float x[E];
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = __uint_as_float(static_cast<uint32_t>(src[lane * E + e]) << 16);
  uint32_t packed;
  const float scale = quantise_lane_q8<E>(x, packed);
  if constexpr (E == 4) {
    *reinterpret_cast<uint32_t*>(dst + lane * 4) = packed;
  } else {
    *reinterpret_cast<uint16_t*>(dst + lane * 2) = static_cast<uint16_t>(packed);
  }
  if (lane == 0) *scale_out = scale;
}

template <int D>
__global__ void kv_append_q8_kernel(const AppendQ8Params p) {
  constexpr int kBS = 16;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = p.pos[b];
  if (pos < 0) return;  // idle sequence
  const int lb = pos / kBS;
  if (lb >= p.max_blocks) {
    if (threadIdx.x == 0) report(p.status, kStatusBounds);
    return;
  }
  const int blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + lb];
  if (blk < 0 || blk >= p.num_blocks) {
    if (threadIdx.x == 0) report(p.status, kStatusBounds);
    return;
  }
  const int slot = pos % kBS;
  for (int g = warp; g < p.Hkv; g += blockDim.x >> 5) {
    const int64_t row = (static_cast<int64_t>(blk) * p.Hkv + g) * kBS + slot;
    quantise_row_q8<D>(p.kn + b * p.kn_stride[0] + g * p.kn_stride[1], p.kq + row * D, p.ks + row, lane);
    quantise_row_q8<D>(p.vn + b * p.vn_stride[0] + g * p.vn_stride[1], p.vq + row * D, p.vs + row, lane);
  }
}

// ---------------------------------------------------------------------------
// kv_append_chunk: token i of sequence b's chunk (k_new[b, g, i, :]) goes to
// position start_pos[b] + i.  grid (vector tiles, B); 16-byte vectors, the
// dim chunk fastest, then the token, then the head, so consecutive threads
// read one head's rows of the chunk and write whole cache blocks.
// ---------------------------------------------------------------------------
struct ChunkAppendParams {
  uint16_t* kc;
  uint16_t* vc;
  int64_t num_blocks;
  int Hkv, D, T;
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* start_pos;
  const uint16_t* kn;
  const uint16_t* vn;
  int64_t kn_stride[3], vn_stride[3];  // batch, head, token (elements)
  uint32_t* status;
};

__global__ void kv_append_chunk_kernel(const ChunkAppendParams p) {
  constexpr int kBS = 16;
  const int b = blockIdx.y;
  const int start = p.start_pos[b];
  if (start < 0 || static_cast<int64_t>(start) + p.T > static_cast<int64_t>(p.max_blocks) * kBS) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(p.status, kStatusBounds);
    return;  // the whole sequence is skipped, as its attention is
  }
  const int vpr = p.D / 8;
  const int64_t n = static_cast<int64_t>(p.Hkv) * p.T * vpr;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % vpr);
    const int i = static_cast<int>((idx / vpr) % p.T);
    const int g = static_cast<int>(idx / (static_cast<int64_t>(vpr) * p.T));
    const int t = start + i;
    const int blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + t / kBS];
    if (blk < 0 || blk >= p.num_blocks) {
      report(p.status, kStatusBounds);
      continue;
    }
    const int64_t dst = ((static_cast<int64_t>(blk) * p.Hkv + g) * kBS + t % kBS) * p.D + c * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(p.kn + b * p.kn_stride[0] + g * p.kn_stride[1] +
                                                     i * p.kn_stride[2] + c * 8);
    const uint4 vv = *reinterpret_cast<const uint4*>(p.vn + b * p.vn_stride[0] + g * p.vn_stride[1] +
                                                     i * p.vn_stride[2] + c * 8);
    *reinterpret_cast<uint4*>(p.kc + dst) = kv;
    *reinterpret_cast<uint4*>(p.vc + dst) = vv;
  }
}

// ---------------------------------------------------------------------------
// paged_gather: dst[b, g, t, :] = cache[block_table[b][t / bs], g, t % bs, :]
// grid (token tiles of 16, Hkv, B); 16-byte vectors.
// ---------------------------------------------------------------------------
struct GatherParams {
  const uint16_t* cache;
  int64_t num_blocks;
  int block_size, Hkv, D;
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* lens;
  int64_t max_len;
  uint16_t* dst;
  uint32_t* status;
};

__global__ void paged_gather_kernel(const GatherParams p) {
  const int b = blockIdx.z, g = blockIdx.y;
  const int L = p.lens[b];
  const int vec = p.D / 8;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 16;
  for (int i = threadIdx.x; i < 16 * vec; i += blockDim.x) {
    const int64_t t = t0 + i / vec;
    if (t >= L || t >= p.max_len) continue;
    const int64_t lb = t / p.block_size;
    if (lb >= p.max_blocks) {
      report(p.status, kStatusBounds);
      continue;
    }
    const int blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + lb];
    if (blk < 0 || blk >= p.num_blocks) {
      report(p.status, kStatusBounds);
      continue;
    }
    const int c = (i % vec) * 8;
    const int64_t src = ((static_cast<int64_t>(blk) * p.Hkv + g) * p.block_size + t % p.block_size) * p.D + c;
    const int64_t dst = ((static_cast<int64_t>(b) * p.Hkv + g) * p.max_len + t) * p.D + c;
    *reinterpret_cast<uint4*>(p.dst + dst) = *reinterpret_cast<const uint4*>(p.cache + src);
  }
}

// ---------------------------------------------------------------------------
// lse_merge ("[sglang] ROCm aiter ring attention", section 1):
//   lse = M + log(sum_i exp(lse_i - M)),  out = sum_i exp(lse_i - lse) out_i
// Each group of D/8 threads owns one (b, h, p) row; rows are walked in the
// order of the contiguous LSE layout so the LSE reads coalesce.
// ---------------------------------------------------------------------------
struct MergeParams {
  int n;
  int64_t H, P, D, rows;
  const void* outs[8];
  int64_t ostride[8][3];
  const float* lses[8];
  int in_bf16;
  void* out;
  int64_t out_stride[3];
  int out_bf16;
  float* lse;
};

// 8 consecutive elements of a row as floats: 8 bf16 (16 bytes) or 8 f32 (32 bytes)
template <bool BF16>
__device__ __forceinline__ void load8(const void* base, int64_t off, float* v) {
  if constexpr (BF16) {
    const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
    v[0] = bf16lo_to_f32(w.x); v[1] = bf16hi_to_f32(w.x);
    v[2] = bf16lo_to_f32(w.y); v[3] = bf16hi_to_f32(w.y);
    v[4] = bf16lo_to_f32(w.z); v[5] = bf16hi_to_f32(w.z);
    v[6] = bf16lo_to_f32(w.w); v[7] = bf16hi_to_f32(w.w);
  } else {
    const float4* f = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    const float4 a = f[0], c = f[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
  }
}

// One CTA covers `rows` = 256 / (D/E) consecutive query rows of one (b, h); a
// row is D/E threads, each moving E consecutive elements of every partial
// (E = 16 where D allows it: 32 bytes of bf16 per partial and thread, which
// measured 18 % faster than 16 bytes on the chunked merge).  The partial
// count, the input type and E are template parameters, so a thread's loads go
// out back to back into exactly-sized registers, all before any result is
// needed.  The weights are computed in log2 units: w_i = 2^((lse_i - lse) * log2 e).
template <int NP, bool IN_BF16, int E>
__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeParams p, int vec, int rows) {
  const float kLog2e = 1.4426950408889634f;
  const int row_in_cta = static_cast<int>(threadIdx.x) / vec;
  const int64_t pp = static_cast<int64_t>(blockIdx.x) * rows + row_in_cta;
  if (row_in_cta >= rows || pp >= p.P) return;
  const int64_t hh = blockIdx.y, bb = blockIdx.z;
  const int c = (static_cast<int>(threadIdx.x) - row_in_cta * vec) * E;
  const int64_t r = (bb * p.H + hh) * p.P + pp;  // row of the contiguous LSE layout
  float l2[NP];
  float v[NP][E];
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    l2[i] = p.lses[i][r];
    const int64_t off = bb * p.ostride[i][0] + hh * p.ostride[i][1] + pp * p.ostride[i][2] + c;
#pragma unroll
    for (int q = 0; q < E / 8; ++q) load8<IN_BF16>(p.outs[i], off + 8 * q, &v[i][8 * q]);
  }
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < NP; ++i) {
    l2[i] *= kLog2e;
    M = fmaxf(M, l2[i]);
  }
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float lse = -INFINITY;
  if (M != -INFINITY) {
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NP; ++i) tot += fast_exp2(l2[i] - M);  // -inf -> 0
    const float lse2 = M + __log2f(tot);
    lse = lse2 * 0.6931471805599453f;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const float w = fast_exp2(l2[i] - lse2);
      if (w != 0.f) {  // a partial with no keys may hold anything
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, v[i][e], acc[e]);
      }
    }
  }
  const int64_t o = bb * p.out_stride[0] + hh * p.out_stride[1] + pp * p.out_stride[2] + c;
  if (p.out_bf16) {
#pragma unroll
    for (int q = 0; q < E / 8; ++q) {
      uint4 w;
      w.x = pack_bf16x2(acc[8 * q + 0], acc[8 * q + 1]);
      w.y = pack_bf16x2(acc[8 * q + 2], acc[8 * q + 3]);
      w.z = pack_bf16x2(acc[8 * q + 4], acc[8 * q + 5]);
      w.w = pack_bf16x2(acc[8 * q + 6], acc[8 * q + 7]);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o + 8 * q) = w;
    }
  } else {
    float4* f = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o);
#pragma unroll
    for (int q = 0; q < E / 4; ++q) f[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
  }
  if (p.lse != nullptr && c == 0) p.lse[r] = lse;
}

template <int NP>
cudaError_t launch_merge_np(const MergeParams& p, int e, dim3 grid, int threads, int vec, int rows,
                            cudaStream_t stream) {
  if (p.in_bf16) {
    if (e == 16)
      lse_merge_kernel<NP, true, 16><<<grid, threads, 0, stream>>>(p, vec, rows);
    else
      lse_merge_kernel<NP, true, 8><<<grid, threads, 0, stream>>>(p, vec, rows);
  } else {
    if (e == 16)
      lse_merge_kernel<NP, false, 16><<<grid, threads, 0, stream>>>(p, vec, rows);
    else
      lse_merge_kernel<NP, false, 8><<<grid, threads, 0, stream>>>(p, vec, rows);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// no keys: out = 0, lse = -inf
// ---------------------------------------------------------------------------
__global__ void empty_keys_kernel(void* out, int out_bf16, int64_t s0, int64_t s1, int64_t s2, int64_t H,
                                  int64_t P, int64_t D, float* lse) {
  const int64_t r = blockIdx.x;  // (b * H + h) * P + p
  const int64_t pp = r % P, hh = (r / P) % H, bb = r / (P * H);
  const int64_t o = bb * s0 + hh * s1 + pp * s2;
  for (int64_t d = threadIdx.x; d < D; d += blockDim.x) {
    if (out_bf16)
      static_cast<uint16_t*>(out)[o + d] = 0;
    else
      static_cast<float*>(out)[o + d] = 0.f;
  }
  if (lse != nullptr && threadIdx.x == 0) lse[r] = -INFINITY;
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  AppendParams p;
  p.kc = static_cast<uint16_t*>(a.cache.k);
  p.vc = static_cast<uint16_t*>(a.cache.v);
  p.num_blocks = a.cache.num_blocks;
  p.block_size = a.cache.block_size;
  p.Hkv = a.cache.Hkv;
  p.D = a.cache.D;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.pos = a.pos;
  p.kn = static_cast<const uint16_t*>(a.k_new.data);
  p.vn = static_cast<const uint16_t*>(a.v_new.data);
  p.kn_stride[0] = a.k_new.stride[0];
  p.kn_stride[1] = a.k_new.stride[1];
  p.vn_stride[0] = a.v_new.stride[0];
  p.vn_stride[1] = a.v_new.stride[1];
  p.status = a.status;
  const int threads = std::min(256, std::max(32, a.cache.Hkv * a.cache.D / 8));
  kv_append_kernel<<<static_cast<unsigned>(a.B), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_append_q8(const AppendArgs& a, cudaStream_t stream) {
  AppendQ8Params p;
  p.kq = static_cast<int8_t*>(a.cache.k);
  p.vq = static_cast<int8_t*>(a.cache.v);
  p.ks = const_cast<float*>(a.cache.k_scale);
  p.vs = const_cast<float*>(a.cache.v_scale);
  p.num_blocks = a.cache.num_blocks;
  p.Hkv = a.cache.Hkv;
  p.D = a.cache.D;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.pos = a.pos;
  p.kn = static_cast<const uint16_t*>(a.k_new.data);
  p.vn = static_cast<const uint16_t*>(a.v_new.data);
  p.kn_stride[0] = a.k_new.stride[0];
  p.kn_stride[1] = a.k_new.stride[1];
  p.vn_stride[0] = a.v_new.stride[0];
  p.vn_stride[1] = a.v_new.stride[1];
  p.status = a.status;
  const int threads = std::min(256, std::max(32, a.cache.Hkv * 32));
  if (a.cache.D == 128) {
    kv_append_q8_kernel<128><<<static_cast<unsigned>(a.B), threads, 0, stream>>>(p);
  } else if (a.cache.D == 64) {
    kv_append_q8_kernel<64><<<static_cast<unsigned>(a.B), threads, 0, stream>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_kv_append_chunk(const PrefillArgs& a, cudaStream_t stream) {
  ChunkAppendParams p;
  p.kc = static_cast<uint16_t*>(a.cache.k);
  p.vc = static_cast<uint16_t*>(a.cache.v);
  p.num_blocks = a.cache.num_blocks;
  p.Hkv = a.cache.Hkv;
  p.D = a.cache.D;
  p.T = static_cast<int>(a.T);
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.start_pos = a.start_pos;
  p.kn = static_cast<const uint16_t*>(a.k_new.data);
  p.vn = static_cast<const uint16_t*>(a.v_new.data);
  for (int i = 0; i < 3; ++i) {
    p.kn_stride[i] = a.k_new.stride[i];
    p.vn_stride[i] = a.v_new.stride[i];
  }
  p.status = a.status;
  const int64_t n = static_cast<int64_t>(p.Hkv) * p.T * (p.D / 8);
  const int64_t blocks = (n + 255) / 256;
  dim3 grid(static_cast<unsigned>(blocks < 4096 ? blocks : 4096), static_cast<unsigned>(a.B));
  kv_append_chunk_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_paged_gather(const GatherArgs& a, cudaStream_t stream) {
  GatherParams p;
  p.cache = static_cast<const uint16_t*>(a.which ? a.cache.v : a.cache.k);
  p.num_blocks = a.cache.num_blocks;
  p.block_size = a.cache.block_size;
  p.Hkv = a.cache.Hkv;
  p.D = a.cache.D;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.lens = a.lens;
  p.max_len = a.max_len;
  p.dst = static_cast<uint16_t*>(a.dst);
  p.status = a.status;
  dim3 grid(static_cast<unsigned>((a.max_len + 15) / 16), static_cast<unsigned>(a.cache.Hkv),
            static_cast<unsigned>(a.B));
  paged_gather_kernel<<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const MergeArgs& a, cudaStream_t stream) {
  MergeParams p;
  p.n = a.n;
  p.H = a.H;
  p.P = a.P;
  p.D = a.D;
  p.rows = a.B * a.H * a.P;
  for (int i = 0; i < a.n; ++i) {
    p.outs[i] = a.outs[i].data;
    p.ostride[i][0] = a.outs[i].stride[0];
    p.ostride[i][1] = a.outs[i].stride[1];
    p.ostride[i][2] = a.outs[i].stride[2];
    p.lses[i] = a.lses[i];
  }
  p.in_bf16 = a.outs[0].dtype == ATTN_BF16;
  p.out = a.out.data;
  p.out_stride[0] = a.out.stride[0];
  p.out_stride[1] = a.out.stride[1];
  p.out_stride[2] = a.out.stride[2];
  p.out_bf16 = a.out.dtype == ATTN_BF16;
  p.lse = a.lse;
  const int e = a.D % 16 == 0 ? 16 : 8;            // elements per thread
  const int vec = static_cast<int>(a.D / e);         // threads per row, <= 32
  if (a.H > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  const int rows = 256 / vec;
  const int threads = rows * vec;
  dim3 grid(static_cast<unsigned>((a.P + rows - 1) / rows), static_cast<unsigned>(a.H), static_cast<unsigned>(a.B));
  switch (a.n) {
    case 1: return launch_merge_np<1>(p, e, grid, threads, vec, rows, stream);
    case 2: return launch_merge_np<2>(p, e, grid, threads, vec, rows, stream);
    case 3: return launch_merge_np<3>(p, e, grid, threads, vec, rows, stream);
    case 4: return launch_merge_np<4>(p, e, grid, threads, vec, rows, stream);
    case 5: return launch_merge_np<5>(p, e, grid, threads, vec, rows, stream);
    case 6: return launch_merge_np<6>(p, e, grid, threads, vec, rows, stream);
    case 7: return launch_merge_np<7>(p, e, grid, threads, vec, rows, stream);
    case 8: return launch_merge_np<8>(p, e, grid, threads, vec, rows, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_empty_keys(const AttnFwdArgs& a, cudaStream_t stream) {
  const int64_t rows = a.B * a.Hq * a.Pq;
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  empty_keys_kernel<<<static_cast<unsigned>(rows), 64, 0, stream>>>(
      a.out.data, a.out.dtype == ATTN_BF16, a.out.stride[0], a.out.stride[1], a.out.stride[2], a.Hq, a.Pq, a.D,
      a.lse);
  return cudaGetLastError();
}

}  // namespace attn

// ---------------------------------------------------------------------------
// self-test of the bounded wait: one thread waits on an mbarrier phase that
// nothing completes; the wait must give up after `timeout_ns`, record
// ATTN_ERR_TIMEOUT in the status word and return.
// ---------------------------------------------------------------------------
namespace attn {
namespace {
__global__ void wait_timeout_selftest_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);  // never arrives
  __syncthreads();
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}
}  // namespace attn

// ---------------------------------------------------------------------------
// boolean key-padding mask -> additive mask ("MultiheadAttention fast path
// used 18 GB of VRAM", the note on mask direction: a key_padding_mask marks a
// padded key with True, which must become -inf; 0 keeps the key)
// ---------------------------------------------------------------------------
namespace attn {
namespace {
__global__ void padding_mask_to_additive_kernel(const uint8_t* kpm, int64_t kpm_stride, int64_t Pk, float* out,
                                                int64_t out_stride) {
  const int64_t b = blockIdx.y;
  for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < Pk;
       j += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[b * out_stride + j] = kpm[b * kpm_stride + j] ? -INFINITY : 0.0f;
}
}  // namespace

// ---------------------------------------------------------------------------
// key_tile_bound: the largest |k| element of each 128-key tile of bf16 K,
// one CTA per (tile, KV head, batch), 16-byte loads.
// ---------------------------------------------------------------------------
namespace {
__global__ void key_tile_bound_kernel(const uint16_t* __restrict__ k, int64_t s0, int64_t s1, int64_t s2, int Pk,
                                      int D, int Hkv, int tiles, float* __restrict__ bound) {
  const int j = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int key0 = j * kKeyTile;
  const int nkeys = min(kKeyTile, Pk - key0);
  const int vpr = D / 8;
  uint32_t mx2 = 0u;
  for (int i = threadIdx.x; i < nkeys * vpr; i += blockDim.x) {
    const int key = key0 + i / vpr, c = i % vpr;
    const uint4 w = *reinterpret_cast<const uint4*>(k + b * s0 + g * s1 + static_cast<int64_t>(key) * s2 + c * 8);
    mx2 = bf16x2_max_abs(mx2, w.x);
    mx2 = bf16x2_max_abs(mx2, w.y);
    mx2 = bf16x2_max_abs(mx2, w.z);
    mx2 = bf16x2_max_abs(mx2, w.w);
  }
  float m = fmaxf(bf16lo_to_f32(mx2), bf16hi_to_f32(mx2));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, part[w]);
    bound[(static_cast<int64_t>(b) * Hkv + g) * tiles + j] = m;
  }
}
}  // namespace

cudaError_t launch_key_tile_bound(const AttnFwdArgs& a, cudaStream_t stream) {
  const int tiles = static_cast<int>((a.Pk + kKeyTile - 1) / kKeyTile);
  dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(a.Hkv), static_cast<unsigned>(a.B));
  key_tile_bound_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(a.k.data), a.k.stride[0],
                                                  a.k.stride[1], a.k.stride[2], static_cast<int>(a.Pk),
                                                  static_cast<int>(a.D), static_cast<int>(a.Hkv), tiles,
                                                  a.key_bound);
  return cudaGetLastError();
}

cudaError_t launch_padding_mask_to_additive(const uint8_t* kpm, int64_t kpm_stride, int64_t B, int64_t Pk,
                                            float* out, int64_t out_stride, cudaStream_t stream) {
  const int64_t blocks = (Pk + 255) / 256;
  dim3 grid(static_cast<unsigned>(blocks < 1024 ? blocks : 1024), static_cast<unsigned>(B));
  padding_mask_to_additive_kernel<<<grid, 256, 0, stream>>>(kpm, kpm_stride, Pk, out, out_stride);
  return cudaGetLastError();
}
}  // namespace attn
