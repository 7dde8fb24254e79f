// attn_simt.cu -- masked exact attention with LSE for float32 inputs on the
// FP32 FMA pipes (no TF32: products and sums stay in fp32 so results meet a
// 1e-4 tolerance against the fp64 definition).
//
// Same definition as attn_fwd ("MultiheadAttention fast path used 18 GB of
// VRAM", SDPA with an additive -inf padding mask; "[sglang] ROCm aiter ring
// attention", section 1, LSE output), computed with the online softmax over
// 32- or 64-key tiles so that nothing quadratic in P is ever stored.
//
// A query row is owned by TPR threads, each holding 32 of its dimensions of q
// and of the running output; a K/V tile is staged in shared memory
// (each 32-float slice padded by 4 floats so the TPR slices fall in different
// banks) and read back as broadcasts.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kThreads = 128;
constexpr int kSlice = 32;            // dims per thread
constexpr int kSlicePad = kSlice + 4; // floats per slice in shared memory

struct SimtParams {
  const float* q;
  const float* k;
  const float* v;
  int64_t qs[3], ks[3], vs[3];  // b, h, row strides (elements); dim stride 1
  const float* mask;
  int64_t mask_stride;
  const int32_t* key_lens;  // per-batch valid keys, or null
  void* out;
  int64_t os[3];
  int out_bf16;
  float* lse;
  int Pq, Pk, D, Hq, group;
  float scale_log2;
};

template <int TPR>
__global__ void __launch_bounds__(kThreads) attn_fwd_simt_kernel(const SimtParams p) {
  constexpr int kRows = kThreads / TPR;
  constexpr int kRowFloats = TPR * kSlicePad;
  constexpr int kTileKeys = TPR == 4 ? 32 : 64;  // K + V tiles stay under 48 KB
  __shared__ __align__(16) float ks[kTileKeys * kRowFloats];
  __shared__ __align__(16) float vs[kTileKeys * kRowFloats];
  __shared__ float ms[kTileKeys];

  const int b = blockIdx.z, h = blockIdx.y;
  const int g = h / p.group;
  const int slice = threadIdx.x % TPR;
  const int row = blockIdx.x * kRows + threadIdx.x / TPR;
  const int d0 = slice * kSlice;
  const float kLog2e = 1.4426950408889634f;

  float q[kSlice], o[kSlice];
  {
    const float* qp = p.q + b * p.qs[0] + h * p.qs[1] + static_cast<int64_t>(row) * p.qs[2];
#pragma unroll
    for (int i = 0; i < kSlice; ++i) {
      const int d = d0 + i;
      q[i] = (row < p.Pq && d < p.D) ? qp[d] : 0.f;
      o[i] = 0.f;
    }
  }
  float m_run = -INFINITY, l_run = 0.f;
  const float* kbase = p.k + b * p.ks[0] + g * p.ks[1];
  const float* vbase = p.v + b * p.vs[0] + g * p.vs[1];
  const float* mrow = p.mask ? p.mask + b * p.mask_stride : nullptr;
  const int vec_per_row = TPR * kSlice / 4;
  int n_keys = p.Pk;  // keys of this batch row: all Pk, or its valid length
  if (p.key_lens != nullptr) {
    const int len = p.key_lens[b];
    n_keys = len < 0 ? 0 : (len < p.Pk ? len : p.Pk);
  }

  for (int k0 = 0; k0 < n_keys; k0 += kTileKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kTileKeys * vec_per_row; i += kThreads) {
      const int key = i / vec_per_row;
      const int d = (i % vec_per_row) * 4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (k0 + key < n_keys && d < p.D) {
        kv = *reinterpret_cast<const float4*>(kbase + static_cast<int64_t>(k0 + key) * p.ks[2] + d);
        vv = *reinterpret_cast<const float4*>(vbase + static_cast<int64_t>(k0 + key) * p.vs[2] + d);
      }
      const int off = key * kRowFloats + (d / kSlice) * kSlicePad + (d % kSlice);
      *reinterpret_cast<float4*>(ks + off) = kv;
      *reinterpret_cast<float4*>(vs + off) = vv;
    }
    if (threadIdx.x < kTileKeys) {
      const int key = k0 + threadIdx.x;
      ms[threadIdx.x] = key < n_keys ? (mrow ? mrow[key] * kLog2e : 0.f) : -INFINITY;
    }
    __syncthreads();

    float x[kTileKeys];
    float mt = -INFINITY;
#pragma unroll 8
    for (int j = 0; j < kTileKeys; ++j) {
      const float4* kr = reinterpret_cast<const float4*>(ks + j * kRowFloats + slice * kSlicePad);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kSlice / 4; ++i) {
        const float4 kv = kr[i];
        acc = fmaf(q[4 * i + 0], kv.x, acc);
        acc = fmaf(q[4 * i + 1], kv.y, acc);
        acc = fmaf(q[4 * i + 2], kv.z, acc);
        acc = fmaf(q[4 * i + 3], kv.w, acc);
      }
#pragma unroll
      for (int w = 1; w < TPR; w <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
      x[j] = fmaf(acc, p.scale_log2, ms[j]);
      mt = fmaxf(mt, x[j]);
    }
    const float m_new = fmaxf(m_run, mt);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);
    float rs = 0.f;
#pragma unroll
    for (int j = 0; j < kTileKeys; ++j) {
      x[j] = exp2f(x[j] - m_use);
      rs += x[j];
    }
    l_run = l_run * alpha + rs;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < kSlice; ++i) o[i] *= alpha;
#pragma unroll 8
    for (int j = 0; j < kTileKeys; ++j) {
      const float4* vr = reinterpret_cast<const float4*>(vs + j * kRowFloats + slice * kSlicePad);
      const float pj = x[j];
#pragma unroll
      for (int i = 0; i < kSlice / 4; ++i) {
        const float4 vv = vr[i];
        o[4 * i + 0] = fmaf(pj, vv.x, o[4 * i + 0]);
        o[4 * i + 1] = fmaf(pj, vv.y, o[4 * i + 1]);
        o[4 * i + 2] = fmaf(pj, vv.z, o[4 * i + 2]);
        o[4 * i + 3] = fmaf(pj, vv.w, o[4 * i + 3]);
      }
    }
  }

  if (row >= p.Pq) return;
  const bool empty = !(l_run > 0.f);
  const float inv_l = empty ? 0.f : 1.f / l_run;
  const int64_t ob = b * p.os[0] + h * p.os[1] + static_cast<int64_t>(row) * p.os[2];
#pragma unroll
  for (int i = 0; i < kSlice; i += 2) {
    const int d = d0 + i;
    if (d >= p.D) break;
    if (p.out_bf16) {
      // D % 4 == 0, so d and d + 1 are both in range
      *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(p.out) + ob + d) =
          pack_bf16x2(o[i] * inv_l, o[i + 1] * inv_l);
    } else {
      *reinterpret_cast<float2*>(static_cast<float*>(p.out) + ob + d) = make_float2(o[i] * inv_l, o[i + 1] * inv_l);
    }
  }
  if (p.lse != nullptr && slice == 0)
    p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Pq + row] =
        empty ? -INFINITY : (m_run + log2f(l_run)) * 0.6931471805599453f;
}

template <int TPR>
cudaError_t launch(const SimtParams& p, int64_t B, int64_t Hq, int64_t Pq, cudaStream_t stream) {
  constexpr int kRows = kThreads / TPR;
  dim3 grid(static_cast<unsigned>((Pq + kRows - 1) / kRows), static_cast<unsigned>(Hq), static_cast<unsigned>(B));
  attn_fwd_simt_kernel<TPR><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd_simt(const AttnFwdArgs& a, cudaStream_t stream) {
  SimtParams p;
  p.q = static_cast<const float*>(a.q.data);
  p.k = static_cast<const float*>(a.k.data);
  p.v = static_cast<const float*>(a.v.data);
  for (int i = 0; i < 3; ++i) {
    p.qs[i] = a.q.stride[i];
    p.ks[i] = a.k.stride[i];
    p.vs[i] = a.v.stride[i];
    p.os[i] = a.out.stride[i];
  }
  p.mask = a.mask;
  p.mask_stride = a.mask_stride;
  p.key_lens = a.key_lens;
  p.out = a.out.data;
  p.out_bf16 = a.out.dtype == ATTN_BF16;
  p.lse = a.lse;
  p.Pq = static_cast<int>(a.Pq);
  p.Pk = static_cast<int>(a.Pk);
  p.D = static_cast<int>(a.D);
  p.Hq = static_cast<int>(a.Hq);
  p.group = static_cast<int>(a.Hq / a.Hkv);
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  if (a.D <= 32) return launch<1>(p, a.B, a.Hq, a.Pq, stream);
  if (a.D <= 64) return launch<2>(p, a.B, a.Hq, a.Pq, stream);
  return launch<4>(p, a.B, a.Hq, a.Pq, stream);
}

}  // namespace attn
