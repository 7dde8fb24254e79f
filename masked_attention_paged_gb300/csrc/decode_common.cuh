// decode_common.cuh -- the end of every paged-decode CTA: combine the warps'
// online-softmax states, write the split's partial, and, in the CTA that
// completes a (sequence, KV head), merge that pair's splits into the output.
#pragma once

#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {

// Where the splits of a decode call meet.  A split is the CTA of one
// (sequence b, KV head gkv, 1024-token range); it writes its normalised
// output and log2 LSE for each query head h = gkv * G + hh to
//     o_part[((b * Hq + h) * n_split + split) * D + d],  lse_part[same slot]
// and counts itself in count[b * Hkv + gkv], a 64-bit word holding the
// call's generation (high half) and the splits done (low half).  Every call
// has a generation of its own, so a word from another call -- or whatever
// the workspace held -- reads as zero splits done: the counts need no
// initialisation and no reset.
struct SplitMerge {
  float* o_part;    // [B, Hq, n_split, D]
  float* lse_part;  // [B, Hq, n_split], log2 units
  unsigned long long* count;  // [B, Hkv] (generation << 32) | splits done
  uint32_t gen;     // this call's generation
  int n_split;
  int Hq, Hkv;
  void* out;        // [B, Hq, D] bf16 or f32, row strides os0 (batch), os1 (head) in elements
  int out_bf16;
  int64_t os0, os1;
  float* lse;       // [B, Hq] natural-log LSE, or null
};

// Each of the CTA's NW warps has left, per query head hh of the KV group, a
// record comb[(w * G + hh) * (D + 2) + ...] = {o[0..D) scaled to the warp's
// reference max, m (log2 units; -inf if the warp saw nothing), l}.  The
// warps are combined with the LSE rule of the ring-attention page and the
// split's partial is written as above; a split with nothing in it writes
// zeros and -inf.  Called by all NW * 32 threads after a barrier that
// publishes the records.
template <int D, int G, int NW>
__device__ __forceinline__ void decode_combine_warps(const float* comb, int gkv, int b, int split,
                                                     const SplitMerge& sm) {
  constexpr int kRec = D + 2;
  for (int x = threadIdx.x; x < G * D; x += NW * 32) {
    const int hh = x / D, d = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, comb[(w * G + hh) * kRec + D]);
    float lsum = 0.f, osum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float* rec = comb + (w * G + hh) * kRec;
        if (rec[D] == -INFINITY) continue;
        const float sc = fast_exp2(rec[D] - M);
        lsum = fmaf(sc, rec[D + 1], lsum);
        osum = fmaf(sc, rec[d], osum);
      }
    }
    const int h = gkv * G + hh;
    const int64_t slot = (static_cast<int64_t>(b) * sm.Hq + h) * sm.n_split + split;
    const bool empty = !(lsum > 0.f);
    sm.o_part[slot * D + d] = empty ? 0.f : osum / lsum;
    if (d == 0) sm.lse_part[slot] = empty ? -INFINITY : M + __log2f(lsum);
  }
}

// One warp merges the ns splits of (sequence b, query head h) with the LSE
// rule (log2 units): lane s holds split s's LSE (32 splits per pass), the
// max and the weights come from shuffles, and the outputs of up to 8 splits
// are loaded before any is used.  The partials come from other CTAs: they
// are read from L2 (ld.global.cg), never from a possibly stale L1 line.
template <int D>
__device__ __forceinline__ void decode_merge_head(const SplitMerge& sm, int b, int h, int ns, int lane) {
  constexpr int DPL = D / 32;  // dims per lane
  constexpr int kBatch = 8;    // splits whose outputs are in flight together
  const int64_t row = static_cast<int64_t>(b) * sm.Hq + h;
  const int64_t base = row * sm.n_split;
  const float ls0 = lane < ns ? __ldcg(sm.lse_part + base + lane) : -INFINITY;
  float M = ls0;
  for (int s0 = 32; s0 < ns; s0 += 32)
    if (s0 + lane < ns) M = fmaxf(M, __ldcg(sm.lse_part + base + s0 + lane));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  float acc[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < ns; s0 += 32) {
      const float ls = s0 == 0 ? ls0 : (s0 + lane < ns ? __ldcg(sm.lse_part + base + s0 + lane) : -INFINITY);
      const float w = ls == -INFINITY ? 0.f : fast_exp2(ls - M);
      wsum += w;
      const int n = min(32, ns - s0);
      for (int k0 = 0; k0 < n; k0 += kBatch) {
        float ov[kBatch][DPL];
        float wk[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          wk[u] = __shfl_sync(0xffffffffu, w, (k0 + u) & 31);
          const bool use = k0 + u < n && wk[u] > 0.f;  // a split with no weight may hold anything
          const float* op = sm.o_part + (base + s0 + k0 + u) * D + lane * DPL;
#pragma unroll
          for (int e = 0; e < DPL; ++e) ov[u][e] = use ? __ldcg(op + e) : 0.f;
          if (!use) wk[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wk[u], ov[u][e], acc[e]);
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
  }
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
  const int64_t ob = b * sm.os0 + h * sm.os1 + lane * DPL;
  if (sm.out_bf16) {
    uint16_t* dst = static_cast<uint16_t*>(sm.out) + ob;
#pragma unroll
    for (int e = 0; e < DPL; e += 2)
      *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  } else {
    float* dst = static_cast<float*>(sm.out) + ob;
#pragma unroll
    for (int e = 0; e < DPL; ++e) dst[e] = acc[e] * inv;
  }
  if (sm.lse != nullptr && lane == 0) sm.lse[row] = empty ? -INFINITY : (M + __log2f(wsum)) * 0.6931471805599453f;
}

// After decode_combine_warps: count this split in and, in the CTA that
// brings the count of (b, gkv) to ns (the splits that hold tokens), merge the
// splits of the group's G heads (warp w takes heads w, w + NW, ...).  Every
// CTA publishes its partial before its count (the fence), and the merging CTA
// fences again before it reads the others'.  A word of another generation,
// or one already at ns (the same generation replayed, as from a captured
// graph), starts the count afresh.  Called by all NW * 32 threads.
template <int D, int G, int NW>
__device__ __forceinline__ void decode_finish(const SplitMerge& sm, int gkv, int b, int ns) {
  __shared__ int s_last;
  __syncthreads();  // every thread of the CTA has written its part of the partial
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned long long* c = sm.count + static_cast<int64_t>(b) * sm.Hkv + gkv;
    const unsigned long long tag = static_cast<unsigned long long>(sm.gen) << 32;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c), now;
    for (;;) {
      const bool fresh = (old >> 32) == sm.gen && (old & 0xffffffffull) < static_cast<unsigned long long>(ns);
      now = fresh ? old + 1 : tag + 1;
      const unsigned long long seen = atomicCAS(c, old, now);
      if (seen == old) break;
      old = seen;
    }
    s_last = (now & 0xffffffffull) == static_cast<unsigned long long>(ns);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = warp; hh < G; hh += NW) decode_merge_head<D>(sm, b, gkv * G + hh, ns, lane);
}

// A sequence with no tokens: the CTA of its first split writes zeros and a
// -inf LSE for the group's heads (no split counts, nothing to merge).
template <int D, int G>
__device__ __forceinline__ void decode_write_empty(const SplitMerge& sm, int gkv, int b) {
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int hh = x / D, d = x % D;
    const int h = gkv * G + hh;
    const int64_t o = b * sm.os0 + h * sm.os1 + d;
    if (sm.out_bf16)
      static_cast<uint16_t*>(sm.out)[o] = 0;
    else
      static_cast<float*>(sm.out)[o] = 0.f;
    if (d == 0 && sm.lse != nullptr) sm.lse[static_cast<int64_t>(b) * sm.Hq + h] = -INFINITY;
  }
}

}  // namespace attn
