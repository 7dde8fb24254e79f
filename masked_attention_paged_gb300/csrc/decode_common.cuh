// decode_common.cuh -- the end of every paged-decode CTA: combine the warps'
// online-softmax states and write the split's partial for the split merge.
#pragma once

#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {

// Each of the CTA's NW warps has left, per query head hh of the KV group, a
// record comb[(w * G + hh) * (D + 2) + ...] = {o[0..D) scaled to the warp's
// reference max, m (log2 units; -inf if the warp saw nothing), l}.  The
// warps are combined with the LSE rule of the ring-attention page, and the
// split's normalised output and log2 LSE go to
//     o_part[((b * Hq + h) * n_split + split) * D + d],  lse_part[same slot]
// (h = gkv * G + hh); a split with nothing in it writes zeros and -inf.
// Called by all NW * 32 threads after a barrier that publishes the records.
template <int D, int G, int NW>
__device__ __forceinline__ void decode_combine_warps(const float* comb, int gkv, int b, int split, int Hq,
                                                     int n_split, float* o_part, float* lse_part) {
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
    const int64_t slot = (static_cast<int64_t>(b) * Hq + h) * n_split + split;
    const bool empty = !(lsum > 0.f);
    o_part[slot * D + d] = empty ? 0.f : osum / lsum;
    if (d == 0) lse_part[slot] = empty ? -INFINITY : M + __log2f(lsum);
  }
}

}  // namespace attn
