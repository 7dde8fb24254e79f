// decode.cu -- paged GQA decode: one query token per sequence attends over
// its paged KV cache ("KV cache in nanoVLM", the attention step of each
// decode iteration; "LLM inference memory accounting", sections 11 and 15:
// query heads share KV heads, and the cache is read through a block table).
//
// The work is HBM-bound (about 4 flops per KV byte), so this is an FMA
// kernel organised around the bytes:
//  * split-K over the context: CTA (split s, KV head g, sequence b) covers
//    tokens [1024 s, 1024 (s+1)) and all G = Hq/Hkv query heads of the group,
//    so every K/V byte is read from HBM once;
//  * each of the 4 warps walks every 4th 16-token block of the split; lane 0
//    streams the block's K and V (4 KB each at D = 128) with 1-D bulk copies
//    into a per-warp double buffer, the block ids prefetched from the table;
//  * lane l owns 8 consecutive dims (one 16-byte chunk) of a subset of the
//    block's tokens; dot products are reduced with a transposing shuffle
//    tree that leaves each lane a few (head, token) scores; the online
//    softmax keeps per-head running max/sum in log2 units with lazy rescale;
//  * the split's (output, LSE) goes to the workspace and a second kernel
//    merges the splits with the LSE rule of the ring-attention page.
// Fused append ("KV cache in nanoVLM": compute the new token's K/V, add it to
// the cache, attend): ctx_lens then holds each sequence's new-token position
// and the token itself is handed in.  Only the CTA whose split ends at that
// position reads its slot, so it substitutes the new K/V row into its copy of
// the block once the block has landed, and writes the row to the cache.
// INT8 cache ("LLM inference memory accounting", section 18): the block's
// codes (half the bytes) and its 16 per-token float32 scales of K and of V
// are streamed together; a score is the dot product with the codes times the
// key's scale, and a value row's scale is folded into its softmax weight.
#include <math.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "internal.h"

namespace attn {

int decode_num_splits(int max_blocks, int block_size) {
  const int64_t tokens = static_cast<int64_t>(max_blocks) * block_size;
  return static_cast<int>((tokens + kDecodeSplitTokens - 1) / kDecodeSplitTokens);
}

size_t decode_partial_bytes(int64_t B, int64_t Hq, int n_split, int D) {
  const size_t n = static_cast<size_t>(B) * Hq * n_split;
  // outputs, log2 LSEs, and one 8-byte split count per (sequence, KV head)
  // (Hq bounds Hkv), 8-byte aligned
  size_t bytes = n * D * sizeof(float) + n * sizeof(float);
  bytes = (bytes + 7) & ~size_t(7);
  bytes += static_cast<size_t>(B) * Hq * sizeof(unsigned long long);
  return (bytes + 255) & ~size_t(255);
}

SplitMerge decode_split_merge(const DecodeArgs& a, int D) {
  SplitMerge m;
  const size_t n = static_cast<size_t>(a.B) * a.Hq * a.n_split;
  m.o_part = static_cast<float*>(a.partials);
  m.lse_part = m.o_part + n * D;
  const size_t cnt_off = ((n * D + n) * sizeof(float) + 7) & ~size_t(7);
  m.count = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(a.partials) + cnt_off);
  m.gen = a.gen;
  m.n_split = a.n_split;
  m.Hq = static_cast<int>(a.Hq);
  m.Hkv = a.cache.Hkv;
  m.out = a.out.data;
  m.out_bf16 = a.out.dtype == ATTN_BF16;
  m.os0 = a.out.stride[0];
  m.os1 = a.out.stride[1];
  m.lse = a.lse;
  return m;
}

namespace {

constexpr int kBS = 16;                             // tokens per cache block
constexpr int kWarps = 4;
constexpr int kStages = 2;                          // per-warp buffer depth
constexpr float kLazyRescale = 8.0f;                // log2 units of headroom before a rescale

struct DecodeParams {
  const void* kc;  // bf16 or int8 codes
  const void* vc;
  const float* ks;  // INT8 cache: float32 scale per token row [num_blocks, Hkv, 16]
  const float* vs;
  int64_t num_blocks;
  int Hkv;
  const uint16_t* q;
  int64_t q_stride[2];  // batch, head
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* ctx_lens;
  int len_add;  // 1 with a fused append: ctx_lens holds the new token's position
  const uint16_t* k_new;  // fused append: [B, Hkv, D] rows (null otherwise)
  const uint16_t* v_new;
  int64_t kn_stride[2], vn_stride[2];  // batch, head
  float scale_log2;
  SplitMerge sm;
  uint32_t* status;
};

template <int D, int G, bool Q8>
struct Geo {
  static constexpr int CPR = D / 8;             // 16-byte chunks per token row = lanes per token set
  static constexpr int TS = 32 / CPR;           // token sets per warp
  static constexpr int TPL = kBS / TS;          // tokens per lane per block
  static constexpr int N = G * TPL;             // partial dot products per lane
  static constexpr int R = N >= CPR ? N / CPR : 1;  // scores a lane keeps after the reduce
  static constexpr int SHARE = N >= CPR ? 1 : CPR / N;  // lanes holding the same score
  static constexpr int HEAD_LANES = CPR / G;    // lanes of one token set holding one head
  static constexpr int EB = Q8 ? 1 : 2;         // bytes per element
  static constexpr int BLOCK_BYTES = kBS * D * EB;
  static constexpr int SCALE_BYTES = Q8 ? kBS * 4 : 0;  // one block's row scales, K or V
  static constexpr int STAGE_BYTES = 2 * BLOCK_BYTES + 2 * SCALE_BYTES;
};

// 8 consecutive elements of a row as floats: 8 bf16 (16 bytes) or 8 int8 codes (8 bytes)
template <bool Q8>
__device__ __forceinline__ void load8(const uint8_t* src, float f[8]) {
  if constexpr (Q8) {
    // code b -> the float 2^23 + (b + 128) (its byte placed in a mantissa
    // whose unit is 1), minus 2^23 + 128: exact, and on the full-rate integer
    // and FMA pipes rather than the conversion unit
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    const uint32_t x0 = w.x ^ 0x80808080u, x1 = w.y ^ 0x80808080u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[e] = __uint_as_float(__byte_perm(x0, 0x4B000000u, 0x7540u | e)) - 8388736.0f;
      f[4 + e] = __uint_as_float(__byte_perm(x1, 0x4B000000u, 0x7540u | e)) - 8388736.0f;
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    f[0] = bf16lo_to_f32(w.x); f[1] = bf16hi_to_f32(w.x); f[2] = bf16lo_to_f32(w.y); f[3] = bf16hi_to_f32(w.y);
    f[4] = bf16lo_to_f32(w.z); f[5] = bf16hi_to_f32(w.z); f[6] = bf16lo_to_f32(w.w); f[7] = bf16hi_to_f32(w.w);
  }
}

template <int D, int G, bool Q8>
__global__ void __launch_bounds__(kWarps * 32) paged_decode_kernel(const DecodeParams p) {
  using Gm = Geo<D, G, Q8>;
  extern __shared__ __align__(128) uint8_t smem[];
  // per warp: kStages x {K block, V block[, K scales, V scales]}
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * Gm::STAGE_BYTES);
  float* comb = reinterpret_cast<float*>(bars + kWarps * kStages);  // [kWarps][G][D + 2]

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cl = lane % Gm::CPR;  // chunk column
  const int ts = lane / Gm::CPR;  // token set
  const int L_req = p.ctx_lens[b] + p.len_add;
  int L = L_req < 0 ? 0 : L_req;
  if (L > p.max_blocks * kBS) {
    if (threadIdx.x == 0 && split == 0) report(p.status, kStatusBounds);
    L = p.max_blocks * kBS;
  }
  const int t_begin = split * kDecodeSplitTokens;
  if (t_begin >= L) {  // nothing of this sequence in this split
    if (split == 0) decode_write_empty<D, G>(p.sm, g, b);
    return;
  }
  const int t_end = min(L, t_begin + kDecodeSplitTokens);
  const int nblk = (t_end - t_begin + kBS - 1) / kBS;
  const int lb0 = t_begin / kBS;
  // fused append: the new token is the last of the context (when it fits the
  // table); i_new is this warp's iteration over its block, or -1
  int i_new = -1;
  if (!Q8 && p.k_new != nullptr && L_req >= 1 && L_req == L && L - 1 >= t_begin) {
    const int rel = (L - 1) / kBS - lb0;
    if (rel % kWarps == warp) i_new = rel / kWarps;
  }

  uint8_t* wbuf = smem + warp * kStages * Gm::STAGE_BYTES;
  uint64_t* wbar = bars + warp * kStages;
  if (lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&wbar[s], 1);
  fence_mbar_init();
  __syncwarp();

  // this warp's blocks: i-th is lb0 + warp + kWarps*i; lane i prefetches its id
  const int my_n = nblk > warp ? (nblk - warp + kWarps - 1) / kWarps : 0;
  int my_blk = -1;
  if (lane < my_n) {
    my_blk = p.bt[static_cast<int64_t>(b) * p.bt_stride + lb0 + warp + kWarps * lane];
    if (my_blk < 0 || my_blk >= p.num_blocks) {
      report(p.status, kStatusBounds);
      my_blk = -1;
    }
  }
  // lane 0: start the copy of this warp's i-th block (its id already broadcast)
  auto issue = [&](int i, int blk) {
    const int s = i % kStages;
    if (blk < 0) {  // bad id: complete the phase without data; the block is skipped
      mbar_arrive(&wbar[s]);
      return;
    }
    uint8_t* dst = wbuf + s * Gm::STAGE_BYTES;
    const int64_t row = static_cast<int64_t>(blk) * p.Hkv + g;  // (block, KV head) slab
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&wbar[s], Gm::STAGE_BYTES);
    bulk_load(dst, static_cast<const uint8_t*>(p.kc) + row * Gm::BLOCK_BYTES, Gm::BLOCK_BYTES, &wbar[s]);
    bulk_load(dst + Gm::BLOCK_BYTES, static_cast<const uint8_t*>(p.vc) + row * Gm::BLOCK_BYTES, Gm::BLOCK_BYTES,
              &wbar[s]);
    if constexpr (Q8) {
      bulk_load(dst + 2 * Gm::BLOCK_BYTES, p.ks + row * kBS, Gm::SCALE_BYTES, &wbar[s]);
      bulk_load(dst + 2 * Gm::BLOCK_BYTES + Gm::SCALE_BYTES, p.vs + row * kBS, Gm::SCALE_BYTES, &wbar[s]);
    }
  };

  // q of this lane's 8 dims for every head of the group, pre-scaled to log2 units
  float qf[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const int h = g * G + hh;
    const uint4 w = *reinterpret_cast<const uint4*>(p.q + b * p.q_stride[0] + h * p.q_stride[1] + cl * 8);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      qf[hh][2 * e] = bf16lo_to_f32(wv[e]) * p.scale_log2;
      qf[hh][2 * e + 1] = bf16hi_to_f32(wv[e]) * p.scale_log2;
    }
  }
  // q as packed pairs: every dot product and output update below takes two
  // fp32 lanes per fma.rn.f32x2
  uint64_t q2[G][4];
#pragma unroll
  for (int hh = 0; hh < G; ++hh)
#pragma unroll
    for (int e = 0; e < 4; ++e) q2[hh][e] = f2_pack(qf[hh][2 * e], qf[hh][2 * e + 1]);
  float o[G][8];
  float m_run[G];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m_run[hh] = -INFINITY;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[hh][e] = 0.f;
  }
  // after the reduce this lane keeps scores idx = k + R * (cl / SHARE), k < R,
  // of the list idx = head * TPL + i (token TS * i + ts of the block)
  const int my_idx0 = Gm::R * (cl / Gm::SHARE);
  const int my_head = my_idx0 / Gm::TPL;
  const bool counts_sum = (cl % Gm::SHARE) == 0;  // one of the lanes sharing a score adds it
  float l_part = 0.f;

  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  bool ok = true;
  int issued = 0;
  // prologue: every lane takes part in the broadcast, lane 0 issues
  for (int i = 0; i < kStages && i < my_n; ++i) {
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    if (lane == 0) issue(i, blk);
    issued = i + 1;
  }

  for (int i = 0; i < my_n; ++i) {
    const int s = i % kStages;
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    const bool landed = mbar_wait(&wbar[s], (i / kStages) & 1, &abort_flag, p.status);
    if (!__all_sync(0xffffffffu, landed)) {  // leave together: the shuffles below need every lane
      ok = false;
      break;
    }
    if (blk >= 0) {
      uint8_t* kb = wbuf + s * Gm::STAGE_BYTES;
      uint8_t* vb = kb + Gm::BLOCK_BYTES;
      const float* ksb = reinterpret_cast<const float*>(kb + 2 * Gm::BLOCK_BYTES);  // Q8 only
      const float* vsb = ksb + kBS;
      if (i == i_new) {
        // the block has landed: put the new token's row in place of whatever
        // the slot held, and store it to the cache (lanes [0, CPR) carry K's
        // 16-byte chunks, lanes [CPR, 2 CPR) V's)
        const int slot = (L - 1) % kBS;
        if (lane < 2 * Gm::CPR) {
          const bool is_v = lane >= Gm::CPR;
          const int c = lane % Gm::CPR;
          const uint16_t* src = is_v ? p.v_new + b * p.vn_stride[0] + g * p.vn_stride[1]
                                     : p.k_new + b * p.kn_stride[0] + g * p.kn_stride[1];
          const uint4 w = *reinterpret_cast<const uint4*>(src + c * 8);
          *reinterpret_cast<uint4*>((is_v ? vb : kb) + slot * (D * 2) + c * 16) = w;
          uint16_t* cache = static_cast<uint16_t*>(const_cast<void*>(is_v ? p.vc : p.kc));
          const int64_t off = (static_cast<int64_t>(blk) * p.Hkv + g) * (kBS * D) + slot * D + c * 8;
          *reinterpret_cast<uint4*>(cache + off) = w;
        }
        __syncwarp();
      }
      const int tok0 = (lb0 + warp + kWarps * i) * kBS;  // first token of the block

      // partial dot products over this lane's 8 dims
      float acc[Gm::N];
#pragma unroll
      for (int i2 = 0; i2 < Gm::TPL; ++i2) {
        const int t = Gm::TS * i2 + ts;
        float kf[8];
        load8<Q8>(kb + t * (D * Gm::EB) + cl * 8 * Gm::EB, kf);
        const uint64_t k2[4] = {f2_pack(kf[0], kf[1]), f2_pack(kf[2], kf[3]), f2_pack(kf[4], kf[5]),
                                f2_pack(kf[6], kf[7])};
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          uint64_t a2 = ffma2(q2[hh][0], k2[0], 0ull);
#pragma unroll
          for (int e = 1; e < 4; ++e) a2 = ffma2(q2[hh][e], k2[e], a2);
          float lo, hi;
          f2_unpack(a2, lo, hi);
          acc[hh * Gm::TPL + i2] = lo + hi;
        }
      }
      // transposing reduce over the CPR lanes of a token set: each stage
      // halves the list a lane carries and sums it with its partner's half
#pragma unroll
      for (int st = 0; (Gm::CPR >> (st + 1)) >= 1; ++st) {
        const int mask = Gm::CPR >> (st + 1);
        const int cur = Gm::N >> st;
        if (cur > 1) {
          const int half = cur >> 1;
          const bool upper = (cl & mask) != 0;
#pragma unroll
          for (int k = 0; k < half; ++k) {
            const float send = upper ? acc[k] : acc[k + half];
            const float keep = upper ? acc[k + half] : acc[k];
            acc[k] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
          }
        } else {
          acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], mask);
        }
      }
      // scores kept by this lane; tokens past the context are masked
      float sc[Gm::R];
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < Gm::R; ++k) {
        const int idx = my_idx0 + k;
        const int t = Gm::TS * (idx % Gm::TPL) + ts;
        // INT8: the dot product with the codes times the key row's scale
        sc[k] = (tok0 + t < t_end) ? (Q8 ? acc[k] * ksb[t] : acc[k]) : -INFINITY;
        mx = fmaxf(mx, sc[k]);
      }
      // block max of each head: lanes of the head within the token set, then across token sets
#pragma unroll
      for (int m = 1; m < Gm::HEAD_LANES; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
#pragma unroll
      for (int m = Gm::CPR; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      float m_mine = 0.f, alpha_mine = 1.f;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float mb = __shfl_sync(0xffffffffu, mx, hh * Gm::HEAD_LANES);
        // lazy rescale: move the reference max only when the block exceeds it by a margin
        if (mb > m_run[hh] + kLazyRescale || (m_run[hh] == -INFINITY && mb != -INFINITY)) {
          const float alpha = fast_exp2(m_run[hh] - mb);  // 0 when m_run was -inf
#pragma unroll
          for (int e = 0; e < 8; ++e) o[hh][e] *= alpha;
          if (hh == my_head) alpha_mine = alpha;
          m_run[hh] = mb;
        }
        if (hh == my_head) m_mine = m_run[hh];
      }
      l_part *= alpha_mine;
      float pk[Gm::R];
#pragma unroll
      for (int k = 0; k < Gm::R; ++k) {
        pk[k] = (sc[k] == -INFINITY) ? 0.f : fast_exp2(sc[k] - m_mine);
        if (counts_sum) l_part += pk[k];
      }
      // every lane needs p of its own tokens for all heads
      float pv[G][Gm::TPL];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
#pragma unroll
        for (int i2 = 0; i2 < Gm::TPL; ++i2) {
          const int idx = hh * Gm::TPL + i2;
          const int src = ts * Gm::CPR + (idx / Gm::R) * Gm::SHARE;
          pv[hh][i2] = __shfl_sync(0xffffffffu, pk[idx % Gm::R], src);
        }
      }
#pragma unroll
      for (int i2 = 0; i2 < Gm::TPL; ++i2) {
        const int t = Gm::TS * i2 + ts;
        if (tok0 + t >= t_end) continue;  // slots past the context may hold anything (even NaN)
        float vf[8];
        load8<Q8>(vb + t * (D * Gm::EB) + cl * 8 * Gm::EB, vf);
        const float vsc = Q8 ? vsb[t] : 1.0f;  // INT8: the value row's scale joins its weight
        const uint64_t v2[4] = {f2_pack(vf[0], vf[1]), f2_pack(vf[2], vf[3]), f2_pack(vf[4], vf[5]),
                                f2_pack(vf[6], vf[7])};
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float w = Q8 ? pv[hh][i2] * vsc : pv[hh][i2];
          const uint64_t w2 = f2_pack(w, w);
#pragma unroll
          for (int e = 0; e < 4; ++e) f2_unpack(ffma2(w2, v2[e], f2_pack(o[hh][2 * e], o[hh][2 * e + 1])), o[hh][2 * e], o[hh][2 * e + 1]);
        }
      }
    }
    __syncwarp();
    if (i + kStages < my_n) {
      const int nb = __shfl_sync(0xffffffffu, my_blk, i + kStages);
      if (lane == 0) issue(i + kStages, nb);
      issued = i + kStages + 1;
    }
  }
  if (!ok) {
    // let copies still in flight land before the shared memory is released
    for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
      drain_wait(&wbar[i % kStages], (i / kStages) & 1);
  }

  // ---- warp totals: sum over the lanes of a head, and over token sets
#pragma unroll
  for (int m = 1; m < Gm::HEAD_LANES; m <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, m);
#pragma unroll
  for (int m = Gm::CPR; m < 32; m <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, m);
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
#pragma unroll
      for (int m = Gm::CPR; m < 32; m <<= 1) o[hh][e] += __shfl_xor_sync(0xffffffffu, o[hh][e], m);
    }
  }
  constexpr int kRec = D + 2;  // per (warp, head): o[D], m, l
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const float lh = __shfl_sync(0xffffffffu, l_part, hh * Gm::HEAD_LANES);
    float* rec = comb + (warp * G + hh) * kRec;
    if (ts == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) rec[cl * 8 + e] = o[hh][e];
    }
    if (lane == 0) {
      rec[D] = ok ? m_run[hh] : -INFINITY;
      rec[D + 1] = ok ? lh : 0.f;
    }
  }
  __syncthreads();

  // ---- combine the warps and write this split's partial (normalised out, log2 LSE)
  decode_combine_warps<D, G, kWarps>(comb, g, b, split, p.sm);
  decode_finish<D, G, kWarps>(p.sm, g, b, (L + kDecodeSplitTokens - 1) / kDecodeSplitTokens);
}

template <int D, int G, bool Q8>
cudaError_t launch_decode(const DecodeArgs& a, const DecodeParams& p, cudaStream_t stream) {
  using Gm = Geo<D, G, Q8>;
  const int smem = kWarps * kStages * Gm::STAGE_BYTES + kWarps * kStages * 8 + kWarps * G * (D + 2) * 4;
  auto kern = paged_decode_kernel<D, G, Q8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.n_split), static_cast<unsigned>(a.cache.Hkv), static_cast<unsigned>(a.B));
  kern<<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, bool Q8>
cudaError_t launch_decode_d(const DecodeArgs& a, const DecodeParams& p, cudaStream_t stream) {
  switch (a.Hq / a.cache.Hkv) {
    case 1: return launch_decode<D, 1, Q8>(a, p, stream);
    case 2: return launch_decode<D, 2, Q8>(a, p, stream);
    case 4: return launch_decode<D, 4, Q8>(a, p, stream);
    case 8: return launch_decode<D, 8, Q8>(a, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// host side

cudaError_t launch_paged_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (paged_decode_tc_supported(a)) return launch_paged_decode_tc(a, stream);
  if (paged_decode_q8_mma_supported(a)) return launch_paged_decode_q8_mma(a, stream);
  if (a.cache.k_scale != nullptr && a.k_new.data != nullptr) {
    // this kernel appends to a bf16 cache only: an INT8 cache gets its new
    // rows from kv_append_q8 first (ctx_lens holds the new positions)
    AppendArgs ap;
    ap.cache = a.cache;
    ap.block_table = a.block_table;
    ap.bt_stride = a.bt_stride;
    ap.max_blocks = a.max_blocks;
    ap.pos = a.ctx_lens;
    ap.B = a.B;
    ap.k_new = a.k_new;
    ap.v_new = a.v_new;
    ap.status = a.status;
    const cudaError_t e = launch_kv_append_q8(ap, stream);
    if (e != cudaSuccess) return e;
  }
  DecodeParams p;
  p.kc = a.cache.k;
  p.vc = a.cache.v;
  p.ks = a.cache.k_scale;
  p.vs = a.cache.v_scale;
  p.num_blocks = a.cache.num_blocks;
  p.Hkv = a.cache.Hkv;
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
  p.sm = decode_split_merge(a, static_cast<int>(a.cache.D));
  p.status = a.status;
  const bool q8 = a.cache.k_scale != nullptr;
  if (a.cache.D == 64) return q8 ? launch_decode_d<64, true>(a, p, stream) : launch_decode_d<64, false>(a, p, stream);
  if (a.cache.D == 128)
    return q8 ? launch_decode_d<128, true>(a, p, stream) : launch_decode_d<128, false>(a, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
