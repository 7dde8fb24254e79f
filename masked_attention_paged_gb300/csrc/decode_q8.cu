// decode_q8.cu -- paged GQA decode over an INT8 KV cache on the tensor cores
// ("LLM inference memory accounting", section 18: an INT8 cache halves the
// KV bytes and adds per-token scales and a dequantisation step; "KV cache in
// nanoVLM": one query token per sequence attends over its cached K/V).
//
// Head dim 128, up to 8 query heads per KV head.  The FMA decode spends about
// eight instructions on every INT8 code (dequantise, then one fp32 multiply
// per query head), which leaves it issue-bound at half the bytes of the bf16
// cache.  Here both products run as mma.sync.m16n8k16 (fp16 in, fp32
// accumulate) and a code costs under one instruction:
//  * a code c is turned into the fp16 number 1152 + c by one LOP3 that puts
//    its byte (sign bit flipped, i.e. c + 128) under the exponent of 1024;
//    the 1152 it carries is removed afterwards: from the scores with the
//    per-head constant 1152 * sum(q), from the output with 1152 times the
//    sum of the weights, which a further MMA against a tile of ones yields in
//    the same rounding as the output;
//  * scores S = Q K^T with the query heads as the A rows (zero padded) and
//    the 16 tokens of a block as two n-tiles; the values go in transposed,
//    O^T = V^T W^T, where the weight fragment of a head is, register for
//    register, its score fragment: no shuffle moves it, and the output tile
//    is 128 dims x 8 heads;
//  * the key scale multiplies the score; the value scale multiplies the
//    softmax weight, w = p vs / ref, against a per-head reference that moves
//    lazily (up with the largest p vs of a block, down with the running max),
//    so the fp16 weights stay in [0, 2^8] whatever the scales are and O
//    accumulates straight in the MMA registers;
//  * each warp streams its blocks with two 4-D TMA loads per block (K and V
//    codes, 128-byte swizzle) plus two bulk copies of the row scales; tokens
//    are taken in the order n ^ ((n & 1) << 2) within each group of eight,
//    which makes every fragment load of K and of V free of bank conflicts.
// The CTA decomposition, the cross-warp combine and the split merge are those
// of the FMA decode: split s of 1024 tokens x KV head x sequence per CTA.
//
// Fused append ("KV cache in nanoVLM": the newest token's K/V join the cache
// and are attended in the same step): with k_new set, ctx_lens holds each
// sequence's new position, and the warp whose block holds it quantises the
// new K and V rows (the quantiser of kv_append_q8, so the bits are the same)
// once the block has landed, writes codes and scales over the slot's copy in
// shared memory and stores them to the cache.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "internal.h"
#include "q8_quant.cuh"

namespace attn {
namespace {

constexpr int kBS = 16;       // tokens per cache block
constexpr int kD = 128;       // head dim (one 128-byte code row per token)
constexpr int kWarps = 4;
constexpr int kQ8Stages = 3;  // per-warp buffer depth
constexpr int kCodeBytes = kBS * kD;  // one (block, head) of K or V codes
constexpr float kLazy = 8.0f;         // log2 headroom before a running max moves
constexpr float kBias = 1152.0f;      // value carried by the fp16 form of code 0
constexpr uint32_t kByteMask = 0x00FF00FFu;
constexpr uint32_t kHalfBits = 0x64806480u;  // exponent of 1024 in each half; 0x80 flips the code's sign bit

struct Q8MmaParams {
  CUtensorMap kmap;  // codes [num_blocks, Hkv, 16, 128] u8, box = one (block, head)
  CUtensorMap vmap;
  float* ks;  // [num_blocks, Hkv, 16]; written by the fused append only
  float* vs;
  uint8_t* kq;  // the code caches themselves (the fused append stores the new rows)
  uint8_t* vq;
  int64_t num_blocks;
  int Hkv;
  int Hq;
  const uint16_t* q;
  int64_t q_stride[2];  // batch, head
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* ctx_lens;  // or, with k_new set, each sequence's new-token position
  int len_add;              // 1 with a fused append
  const uint16_t* k_new;    // fused append: bf16 [B, Hkv, D] rows (null otherwise)
  const uint16_t* v_new;
  int64_t kn_stride[2], vn_stride[2];  // batch, head (elements)
  float scale_log2;
  SplitMerge sm;
  uint32_t* status;
};

// two codes (bytes 0 and 2 of x) as the fp16 pair (1152 + c0, 1152 + c2):
// bits under the mask take x with the sign bit flipped, the rest the exponent
__device__ __forceinline__ uint32_t codes_to_half2(uint32_t x) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(x), "n"(kByteMask), "n"(kHalfBits));
  return d;
}

template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "n"(SEL));
  return d;
}

// round-to-nearest-even f32 -> fp16 of two values; `lo` lands in bits 0..15
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// lo + hi of an fp16 pair (both exact in fp32)
__device__ __forceinline__ float half2_sum(uint32_t x) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
  return lo + hi;
}

// D (16x8, fp32) += A (16x16, fp16, rows g and g+8 in a0/a2 and a1/a3) * B (16x8)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ uint32_t word(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// token of position n (0..15) in the order the fragments use
__device__ __forceinline__ int tok_of(int n) { return n ^ ((n & 1) << 2); }

template <int G>
__global__ void __launch_bounds__(kWarps * 32, 4) paged_decode_q8_mma_kernel(const __grid_constant__ Q8MmaParams p) {
  static_assert(G >= 1 && G <= 8, "query heads per KV head");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled TMA tiles
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* codes = smem;                                                      // [warp][stage][K, V][2048]
  float* scl = reinterpret_cast<float*>(codes + kWarps * kQ8Stages * 2 * kCodeBytes);  // [warp][stage][K 16, V 16]
  uint64_t* bars = reinterpret_cast<uint64_t*>(scl + kWarps * kQ8Stages * 2 * kBS);
  // [warp][G][D + 2], used once every warp has left its block loop
  float* comb = reinterpret_cast<float*>(codes);
  static_assert(kWarps * 8 * (kD + 2) * 4 <= kWarps * kQ8Stages * 2 * kCodeBytes, "combine buffer fits");

  const int split = blockIdx.x, gkv = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2;  // fragment row: query head of the group (rows >= G are zero)
  const int t = lane & 3;   // fragment column pair
  const int L_req = p.ctx_lens[b] + p.len_add;
  int L = L_req < 0 ? 0 : L_req;
  if (L > p.max_blocks * kBS) {
    if (threadIdx.x == 0 && split == 0) report(p.status, kStatusBounds);
    L = p.max_blocks * kBS;
  }
  const int t_begin = split * kDecodeSplitTokens;
  if (t_begin >= L) {  // nothing of this sequence in this split
    if (split == 0) decode_write_empty<kD, G>(p.sm, gkv, b);
    return;
  }
  const int t_end = min(L, t_begin + kDecodeSplitTokens);
  const int nblk = (t_end - t_begin + kBS - 1) / kBS;
  const int lb0 = t_begin / kBS;
  // fused append: the new token is the last of the context (when it fits the
  // table); i_new is this warp's iteration over its block, or -1
  int i_new = -1;
  if (p.k_new != nullptr && L_req >= 1 && L_req == L && L - 1 >= t_begin) {
    const int rel = (L - 1) / kBS - lb0;
    if (rel % kWarps == warp) i_new = rel / kWarps;
  }

  uint8_t* wcodes = codes + warp * kQ8Stages * 2 * kCodeBytes;
  float* wscl = scl + warp * kQ8Stages * 2 * kBS;
  uint64_t* wbar = bars + warp * kQ8Stages;
  if (lane == 0) {
    for (int s = 0; s < kQ8Stages; ++s) mbar_init(&wbar[s], 1);
    if (warp == 0) {
      tma_prefetch_desc(&p.kmap);
      tma_prefetch_desc(&p.vmap);
    }
  }
  fence_mbar_init();
  __syncwarp();

  const int my_n = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
  int my_blk = -1;
  if (lane < my_n) {
    my_blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + lb0 + warp + kWarps * lane];
    if (my_blk < 0 || my_blk >= p.num_blocks) {
      report(p.status, kStatusBounds);
      my_blk = -1;
    }
  }
  auto issue = [&](int s, int blk) {
    if (blk < 0) {  // bad id: complete the phase without data; the block is skipped
      mbar_arrive(&wbar[s]);
      return;
    }
    uint8_t* dst = wcodes + s * 2 * kCodeBytes;
    float* sdst = wscl + s * 2 * kBS;
    const int64_t row = static_cast<int64_t>(blk) * p.Hkv + gkv;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&wbar[s], 2 * kCodeBytes + 2 * kBS * 4);
    tma_load_4d(dst, &p.kmap, &wbar[s], 0, 0, gkv, blk);
    tma_load_4d(dst + kCodeBytes, &p.vmap, &wbar[s], 0, 0, gkv, blk);
    bulk_load(sdst, p.ks + row * kBS, kBS * 4, &wbar[s]);
    bulk_load(sdst + kBS, p.vs + row * kBS, kBS * 4, &wbar[s]);
  };

  // ---- q of head g as fp16 A fragments.  K chunk c = 4 h + w of the QK
  // product takes dims d0 = 16 t + 64 h + 4 w .. d0 + 3 in this lane: the
  // k-slots (2t, 2t+1) hold dims (d0, d0+2), the slots (2t+8, 2t+9) dims
  // (d0+1, d0+3), matching the byte order codes_to_half2 produces.
  float qv[32];
  if (g < G) {
    const uint16_t* qrow = p.q + b * p.q_stride[0] + (gkv * G + g) * p.q_stride[1];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 w0 = *reinterpret_cast<const uint4*>(qrow + 16 * t + 64 * h);
      const uint4 w1 = *reinterpret_cast<const uint4*>(qrow + 16 * t + 64 * h + 8);
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        qv[16 * h + 2 * e] = bf16lo_to_f32(ws[e]);
        qv[16 * h + 2 * e + 1] = bf16hi_to_f32(ws[e]);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) qv[e] = 0.f;
  }
  // a power-of-two prescale keeps q inside the fp16 range (exact; the
  // scores take the factor back)
  float qmax = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) qmax = fmaxf(qmax, fabsf(qv[e]));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
  qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
  int qexp = 0;
  if (qmax >= 32768.f) qexp = static_cast<int>((__float_as_uint(qmax) >> 23) & 0xff) - 127 - 14;
  const float qpre = __uint_as_float(static_cast<uint32_t>(127 - qexp) << 23);
  const float sl = p.scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + qexp) << 23);
  uint32_t qa[8][2];
  float qsum = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const int e0 = 16 * (c >> 2) + 4 * (c & 3);
    qa[c][0] = pack_half2(qv[e0] * qpre, qv[e0 + 2] * qpre);
    qa[c][1] = pack_half2(qv[e0 + 1] * qpre, qv[e0 + 3] * qpre);
    // the sum of the rounded halves, as the MMA sees them
    qsum += half2_sum(qa[c][0]) + half2_sum(qa[c][1]);
  }
  qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
  qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
  const float corr = kBias * qsum;

  // the four tokens of this lane, in score-fragment order
  const int T[4] = {tok_of(2 * t), tok_of(2 * t + 1), 8 + tok_of(2 * t), 8 + tok_of(2 * t + 1)};
  // K fragment rows: token tok_of(g) of each n-tile
  const int krow = tok_of(g);

  // O^T = V^T W^T: m-tile mt holds dims 16 g + 2 mt (rows g) and 16 g + 2 mt + 1
  // (rows g + 8) of every head; the columns 2t, 2t+1 are this lane's heads
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  float z[4] = {0.f, 0.f, 0.f, 0.f};  // per head: the sum of the weights
  // softmax state of head g: running max (log2), partial sum of p over this
  // lane's tokens, and the value-weight reference: w = p vs / ref, with ref
  // shrunk by the same factor as p whenever m_run moves, so O keeps its scale
  float m_run = -INFINITY, l_part = 0.f, ref = 0.f, ref_inv = 0.f;

  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  bool ok = true;
  int issued = 0;
  for (int i = 0; i < kQ8Stages && i < my_n; ++i) {
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    if (lane == 0) issue(i, blk);
    issued = i + 1;
  }

  int s = 0;         // stage of block i
  uint32_t ph = 0;   // its phase parity
  for (int i = 0; i < my_n; ++i) {
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    const bool landed = mbar_wait(&wbar[s], ph, &abort_flag, p.status);
    if (!__all_sync(0xffffffffu, landed)) {
      ok = false;
      break;
    }
    if (blk >= 0) {
      uint8_t* kb = wcodes + s * 2 * kCodeBytes;
      uint8_t* vb = kb + kCodeBytes;
      float* ksb = wscl + s * 2 * kBS;
      float* vsb = ksb + kBS;
      const int tok0 = (lb0 + warp + kWarps * i) * kBS;
      if (i == i_new) {
        // the block has landed: quantise the new token's K and V rows and put
        // their codes and scales in place of whatever the slot held (lane l
        // holds dims 4l..4l+3, inside the row's 16-byte chunk l/4, which the
        // swizzle puts at chunk (l/4) ^ (slot % 8)); store them to the cache
        const int slot = (L - 1) % kBS;
        const int64_t row = (static_cast<int64_t>(blk) * p.Hkv + gkv) * kBS + slot;
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint16_t* src = w ? p.v_new + b * p.vn_stride[0] + gkv * p.vn_stride[1]
                                  : p.k_new + b * p.kn_stride[0] + gkv * p.kn_stride[1];
          const uint2 raw = *reinterpret_cast<const uint2*>(src + lane * 4);
          const float x[4] = {bf16lo_to_f32(raw.x), bf16hi_to_f32(raw.x), bf16lo_to_f32(raw.y),
                              bf16hi_to_f32(raw.y)};
          uint32_t packed;
          const float sc = quantise_lane_q8<4>(x, packed);
          *reinterpret_cast<uint32_t*>((w ? vb : kb) + slot * kD + ((((lane >> 2) ^ (slot & 7))) << 4) +
                                       (lane & 3) * 4) = packed;
          *reinterpret_cast<uint32_t*>((w ? p.vq : p.kq) + row * kD + lane * 4) = packed;
          if (lane == 0) {
            (w ? vsb : ksb)[slot] = sc;
            (w ? p.vs : p.ks)[row] = sc;
          }
        }
        __syncwarp();
      }

      // ---- S = Q K^T: n-tile j holds tokens 8 j + tok_of(n)
      float sacc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int tok = 8 * j + krow;
        const uint8_t* rowp = kb + tok * kD;
        const uint4 k0 = lds128(rowp + ((t ^ krow) << 4));
        const uint4 k1 = lds128(rowp + (((t + 4) ^ krow) << 4));
        float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t x = word(c < 4 ? k0 : k1, c & 3);
          mma_f16((c & 1) ? s2 : sacc[j], qa[c][0], 0u, qa[c][1], 0u, codes_to_half2(x), codes_to_half2(x >> 8));
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] += s2[e];
      }
      // scores in log2 units; the key scale multiplies the dot product with the codes
      float sc[4] = {sacc[0][0], sacc[0][1], sacc[1][0], sacc[1][1]};
      float vsc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sc[k] = (sc[k] - corr) * (ksb[T[k]] * sl);
        vsc[k] = vsb[T[k]];
      }
      if (tok0 + kBS > t_end) {  // slots past the context may hold anything (NaN scales too)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (tok0 + T[k] >= t_end) {
            sc[k] = -INFINITY;
            vsc[k] = 0.f;
          }
      }
      float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      if (bm > m_run + kLazy) {  // lazy: the reference max moves only by more than the margin
        const float alpha = fast_exp2(m_run - bm);  // 0 when m_run was -inf
        l_part *= alpha;
        // a reference shrunk to nothing is dropped (the next block sets a new
        // one); the weights it carried are below 1e-30 of any later block's
        ref *= alpha;
        if (!(ref > 1e-30f)) ref = 0.f;
        ref_inv = ref > 0.f ? 1.f / ref : 0.f;
        m_run = bm;
      }
      float pr[4], u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pr[k] = fast_exp2(sc[k] - m_run);
        u[k] = pr[k] * vsc[k];
      }
      l_part += (pr[0] + pr[1]) + (pr[2] + pr[3]);
      float um = fmaxf(fmaxf(u[0], u[1]), fmaxf(u[2], u[3]));
      um = fmaxf(um, __shfl_xor_sync(0xffffffffu, um, 1));
      um = fmaxf(um, __shfl_xor_sync(0xffffffffu, um, 2));
      // keep w = u / ref in [0, 2^8]: a larger block moves the reference and
      // rescales the output columns of its head (held by the lanes t = h / 2)
      // (weights below 1e-30 never set the reference: their reciprocal would
      // overflow, and next to l >= 1 they are nothing)
      const bool grow = um > fmaxf(ref * 256.f, 1e-30f);
      if (__any_sync(0xffffffffu, grow)) {
        const float gam = grow ? ref / um : 1.f;
        if (grow) {
          ref = um;
          ref_inv = 1.f / um;
        }
        const float f0 = __shfl_sync(0xffffffffu, gam, 8 * t), f1 = __shfl_sync(0xffffffffu, gam, 8 * t + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j][0] *= f0;
          o[j][1] *= f1;
          o[j][2] *= f0;
          o[j][3] *= f1;
        }
        z[0] *= f0;
        z[1] *= f1;
      }
      // the weights of head g are the B fragment of O^T = V^T W^T: k-slots
      // (2t, 2t+1) are tokens T[0], T[1]; (2t+8, 2t+9) are T[2], T[3]
      const uint32_t pb0 = pack_half2(u[0] * ref_inv, u[1] * ref_inv);
      const uint32_t pb1 = pack_half2(u[2] * ref_inv, u[3] * ref_inv);

      // ---- O^T += V^T W^T over the lane's 16-dim chunk g of tokens T[0..3]
      uint4 vr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) vr[k] = lds128(vb + T[k] * kD + ((g ^ (T[k] & 7)) << 4));
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t a = word(vr[0], w), bb = word(vr[1], w), c2 = word(vr[2], w), d2 = word(vr[3], w);
        const uint32_t ab_lo = prmt<0x5410u>(a, bb), ab_hi = prmt<0x7632u>(a, bb);
        const uint32_t cd_lo = prmt<0x5410u>(c2, d2), cd_hi = prmt<0x7632u>(c2, d2);
        // m-tile 2w: bytes 4w (rows g), 4w + 1 (rows g + 8); m-tile 2w + 1: bytes 4w + 2, 4w + 3
        mma_f16(o[2 * w], codes_to_half2(ab_lo), codes_to_half2(ab_lo >> 8), codes_to_half2(cd_lo),
                codes_to_half2(cd_lo >> 8), pb0, pb1);
        mma_f16(o[2 * w + 1], codes_to_half2(ab_hi), codes_to_half2(ab_hi >> 8), codes_to_half2(cd_hi),
                codes_to_half2(cd_hi >> 8), pb0, pb1);
      }
      // the sum of the weights as the MMA rounds them (A = ones)
      mma_f16(z, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u, pb0, pb1);
    }
    __syncwarp();
    if (i + kQ8Stages < my_n) {
      const int nb = __shfl_sync(0xffffffffu, my_blk, i + kQ8Stages);
      if (lane == 0) issue(s, nb);  // block i + kQ8Stages reuses stage s
      issued = i + kQ8Stages + 1;
    }
    if (++s == kQ8Stages) {
      s = 0;
      ph ^= 1u;
    }
  }
  if (!ok) {
    for (int i = (issued > kQ8Stages ? issued - kQ8Stages : 0); i < issued; ++i)
      drain_wait(&wbar[i % kQ8Stages], (i / kQ8Stages) & 1);
  }

  // ---- warp record per head: o (scaled to m_run), m_run, l
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  __syncthreads();  // the records overwrite the code buffers
  constexpr int kRec = kD + 2;
  if (g < G && t == 0) {
    float* rec = comb + (warp * G + g) * kRec;
    rec[kD] = (ok && m_run != -INFINITY) ? m_run : -INFINITY;
    rec[kD + 1] = ok ? l_part : 0.f;
  }
  // columns 2t, 2t+1: o = (O - 1152 Z) ref of that head (ref from lane 4 h)
  const float r0 = __shfl_sync(0xffffffffu, ref, 8 * t), r1 = __shfl_sync(0xffffffffu, ref, 8 * t + 4);
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    const int h = 2 * t + hc;
    if (h < G) {
      const float zb = kBias * z[hc], rr = hc ? r1 : r0;
      float* rec = comb + (warp * G + h) * kRec + 16 * g;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rec[2 * j] = (o[j][hc] - zb) * rr;
        rec[2 * j + 1] = (o[j][2 + hc] - zb) * rr;
      }
    }
  }
  __syncthreads();

  // ---- combine the warps, write this split's partial (normalised out, log2 LSE)
  decode_combine_warps<kD, G, kWarps>(comb, gkv, b, split, p.sm);
  decode_finish<kD, G, kWarps>(p.sm, gkv, b, (L + kDecodeSplitTokens - 1) / kDecodeSplitTokens);
}

constexpr size_t q8_mma_smem() {
  return 1024 + static_cast<size_t>(kWarps) * kQ8Stages * (2 * kCodeBytes + 2 * kBS * 4 + 8);
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, const Q8MmaParams& p, cudaStream_t stream) {
  auto kern = paged_decode_q8_mma_kernel<G>;
  const int smem = static_cast<int>(q8_mma_smem());
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.n_split), static_cast<unsigned>(a.cache.Hkv), static_cast<unsigned>(a.B));
  kern<<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// host side

bool paged_decode_q8_mma_supported(const DecodeArgs& a) {
  const int64_t G = a.cache.Hkv > 0 ? a.Hq / a.cache.Hkv : 0;
  return a.cache.k_scale != nullptr && a.cache.D == kD && a.cache.block_size == kBS &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_paged_decode_q8_mma(const DecodeArgs& a, cudaStream_t stream) {
  Q8MmaParams p = {};
  if (!make_code_cache_map(&p.kmap, a.cache.k, a.cache.num_blocks, a.cache.Hkv) ||
      !make_code_cache_map(&p.vmap, a.cache.v, a.cache.num_blocks, a.cache.Hkv))
    return cudaErrorInvalidValue;
  p.ks = const_cast<float*>(a.cache.k_scale);
  p.vs = const_cast<float*>(a.cache.v_scale);
  p.kq = static_cast<uint8_t*>(a.cache.k);
  p.vq = static_cast<uint8_t*>(a.cache.v);
  p.num_blocks = a.cache.num_blocks;
  p.Hkv = a.cache.Hkv;
  p.Hq = static_cast<int>(a.Hq);
  p.q = static_cast<const uint16_t*>(a.q.data);
  p.q_stride[0] = a.q.stride[0];
  p.q_stride[1] = a.q.stride[1];
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.ctx_lens = a.ctx_lens;
  p.len_add = a.k_new.data != nullptr ? 1 : 0;
  p.k_new = static_cast<const uint16_t*>(a.k_new.data);
  p.v_new = static_cast<const uint16_t*>(a.v_new.data);
  p.kn_stride[0] = a.k_new.stride[0];
  p.kn_stride[1] = a.k_new.stride[1];
  p.vn_stride[0] = a.v_new.stride[0];
  p.vn_stride[1] = a.v_new.stride[1];
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.sm = decode_split_merge(a, kD);
  p.status = a.status;
  cudaError_t e;
  switch (a.Hq / a.cache.Hkv) {
    case 1: e = launch_g<1>(a, p, stream); break;
    case 2: e = launch_g<2>(a, p, stream); break;
    case 4: e = launch_g<4>(a, p, stream); break;
    case 8: e = launch_g<8>(a, p, stream); break;
    default: return cudaErrorInvalidValue;
  }
  return e;
}

}  // namespace attn
