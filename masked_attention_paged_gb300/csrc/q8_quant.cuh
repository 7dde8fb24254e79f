// q8_quant.cuh -- the INT8 row quantiser of the paged KV cache ("LLM inference
// memory accounting", section 18: an INT8 cache stores codes plus scale
// metadata).  Shared by kv_append_q8 and the fused append of the INT8 decode,
// so both write the same bits.
#pragma once

#include <stdint.h>

namespace attn {

// One warp quantises one row; lane l holds its E elements (float32 values of
// the bf16 input).  scale = max|x| / 127 and code = clamp(rint(x / scale),
// -127, 127), every step in float32 with IEEE division and round-half-even;
// an all-zero row gives scale 0 and codes 0.  Returns the row's scale (the
// same in every lane); `packed` receives this lane's codes, element e in
// byte e.
template <int E>
__device__ __forceinline__ float quantise_lane_q8(const float (&x)[E], uint32_t& packed) {
  float a = 0.0f;
#pragma unroll
  for (int e = 0; e < E; ++e) a = fmaxf(a, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float scale = __fdiv_rn(a, 127.0f);
  packed = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float c = scale > 0.0f ? rintf(__fdiv_rn(x[e], scale)) : 0.0f;
    c = fminf(fmaxf(c, -127.0f), 127.0f);
    packed |= (static_cast<uint32_t>(static_cast<int32_t>(c)) & 0xffu) << (8 * e);
  }
  return scale;
}

}  // namespace attn
