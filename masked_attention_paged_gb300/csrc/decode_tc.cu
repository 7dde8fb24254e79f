// decode_tc.cu -- paged GQA decode over a bf16 KV cache on the tensor cores
// ("KV cache in nanoVLM": the query of the newest token attends over the
// cached K/V; "LLM inference memory accounting", sections 11 and 15: query
// heads share KV heads, and the cache is read through a block table).
//
// Head dim 128, up to 8 query heads per KV head.  The work is HBM-bound, so
// the aim is to spend as few instructions per KV byte as possible: both
// products run as mma.sync.m16n8k16 (bf16 in, fp32 accumulate), and the K
// and V operands come out of shared memory ready-made:
//  * each warp streams its 16-token blocks with four 2-D boxes of the paged
//    tensor map (64 columns x 16 rows of K and of V, 128-byte swizzle);
//  * S = Q K^T with the query heads as the A rows (zero padded) and the 16
//    tokens as two n-tiles; `ldmatrix` hands each lane its K fragment
//    (a token's consecutive dims), conflict-free through the swizzle;
//  * O^T = V^T P^T: `ldmatrix.trans` hands each lane its V^T fragment (two
//    tokens of one dim), and the weight fragment of a head is, register for
//    register, its score fragment; the output tile is 128 dims x 8 heads;
//  * online softmax per head in log2 units with the lazy rescale of the FMA
//    decode (the reference max moves only by more than 8); P is rounded to
//    bf16, as in the tensor-core attention kernel.
// Fused append ("KV cache in nanoVLM": compute the new token's K/V, add it to
// the cache, attend): ctx_lens then holds each sequence's new-token position;
// the warp whose block holds that slot writes the new rows over the slot's
// copy in shared memory once the block has landed, and stores them to the
// cache.  The CTA decomposition, the cross-warp combine and the split merge
// are those of the FMA decode: split s of 1024 tokens x KV head x sequence.
#include <cuda.h>
#include <math.h>

#include "common.cuh"
#include "decode_common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kBS = 16;      // tokens per cache block
constexpr int kD = 128;      // head dim
constexpr int kWarps = 4;
constexpr int kTcStages = 2;  // per-warp buffer depth
constexpr int kHalfBytes = kBS * 128;      // one 64-column box of a block: 16 rows x 128 bytes
constexpr int kRowsBytes = 2 * kHalfBytes;  // K (or V) of one (block, head)
constexpr float kLazy = 8.0f;               // log2 headroom before the running max moves

struct TcDecodeParams {
  CUtensorMap kmap;  // [num_blocks, Hkv, 16, 128] bf16, box 64 columns x 16 rows
  CUtensorMap vmap;
  uint16_t* kc;      // the caches themselves (fused append stores the new rows)
  uint16_t* vc;
  int64_t num_blocks;
  int Hkv;
  int Hq;
  const uint16_t* q;
  int64_t q_stride[2];  // batch, head
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* ctx_lens;
  int len_add;              // 1 with a fused append: ctx_lens holds the new token's position
  const uint16_t* k_new;    // fused append: [B, Hkv, D] rows (null otherwise)
  const uint16_t* v_new;
  int64_t kn_stride[2], vn_stride[2];  // batch, head
  float scale_log2;
  SplitMerge sm;
  uint32_t* status;
};

// D (16x8, fp32) += A (16x16, bf16) * B (16x8, bf16)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// four 8x8 b16 matrices; lane l supplies the address of row l % 8 of matrix l / 8
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// byte offset of 16-byte chunk `ch` (0..15, 8 dims each) of token row `tok`
// in a block's 128-byte-swizzled image: [half][16 rows][8 chunks]
__device__ __forceinline__ uint32_t sw_off(int tok, int ch) {
  return static_cast<uint32_t>((ch >> 3) * kHalfBytes + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4));
}


template <int G>
__global__ void __launch_bounds__(kWarps * 32, 3) paged_decode_tc_kernel(const __grid_constant__ TcDecodeParams p) {
  static_assert(G >= 1 && G <= 8, "query heads per KV head");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled TMA boxes
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = smem;  // [warp][stage][K, V][2 halves][16 rows][128 bytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles + kWarps * kTcStages * 2 * kRowsBytes);
  // [warp][G][D + 2], used once every warp has left its block loop
  float* comb = reinterpret_cast<float*>(tiles);
  static_assert(kWarps * 8 * (kD + 2) * 4 <= kWarps * kTcStages * 2 * kRowsBytes, "combine buffer fits");

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

  uint8_t* wtiles = tiles + warp * kTcStages * 2 * kRowsBytes;
  uint64_t* wbar = bars + warp * kTcStages;
  if (lane == 0) {
    for (int s = 0; s < kTcStages; ++s) mbar_init(&wbar[s], 1);
    if (warp == 0) {
      tma_prefetch_desc(&p.kmap);
      tma_prefetch_desc(&p.vmap);
    }
  }
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
  auto issue = [&](int s, int blk) {
    if (blk < 0) {  // bad id: complete the phase without data; the block is skipped
      mbar_arrive(&wbar[s]);
      return;
    }
    uint8_t* dst = wtiles + s * 2 * kRowsBytes;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(&wbar[s], 2 * kRowsBytes);
    tma_load_4d(dst, &p.kmap, &wbar[s], 0, 0, gkv, blk);
    tma_load_4d(dst + kHalfBytes, &p.kmap, &wbar[s], 64, 0, gkv, blk);
    tma_load_4d(dst + kRowsBytes, &p.vmap, &wbar[s], 0, 0, gkv, blk);
    tma_load_4d(dst + kRowsBytes + kHalfBytes, &p.vmap, &wbar[s], 64, 0, gkv, blk);
  };

  // q of head g as bf16 A fragments: k-chunk c (dims 16c..16c+15) takes dims
  // (16c + 2t, +1) in register 0 and (16c + 8 + 2t, +1) in register 1
  uint32_t qa[8][2];
#pragma unroll
  for (int c = 0; c < 8; ++c) qa[c][0] = qa[c][1] = 0u;
  if (g < G) {
    const uint16_t* qrow = p.q + b * p.q_stride[0] + (gkv * G + g) * p.q_stride[1];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      qa[c][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * c + 2 * t);
      qa[c][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * c + 8 + 2 * t);
    }
  }
  // the lane's four tokens of a block, in score-fragment order
  const int T[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
  // ldmatrix row addresses (byte offsets in a block image), lane-constant:
  // K: matrix l / 8 = 8-dim chunk 2c + l / 8 of token 8j + l % 8
  // V^T: matrix l / 8 = chunk 2 mt + (l / 8) % 2 of token 8 (l / 16) + l % 8
  const int mi = lane >> 3, mr = lane & 7;

  // O^T = V^T P^T: m-tile mt holds dims 16 mt + g (rows g) and 16 mt + 8 + g
  // (rows g + 8) of every head; the columns 2t, 2t+1 are this lane's heads
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
  float m_run = -INFINITY, l_part = 0.f;  // softmax state of head g (log2 units)

  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  bool ok = true;
  int issued = 0;
  for (int i = 0; i < kTcStages && i < my_n; ++i) {
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    if (lane == 0) issue(i, blk);
    issued = i + 1;
  }

  int s = 0;        // stage of block i
  uint32_t ph = 0;  // its phase parity
  for (int i = 0; i < my_n; ++i) {
    const int blk = __shfl_sync(0xffffffffu, my_blk, i);
    const bool landed = mbar_wait(&wbar[s], ph, &abort_flag, p.status);
    if (!__all_sync(0xffffffffu, landed)) {  // leave together: the shuffles below need every lane
      ok = false;
      break;
    }
    if (blk >= 0) {
      uint8_t* kb = wtiles + s * 2 * kRowsBytes;
      uint8_t* vb = kb + kRowsBytes;
      const int tok0 = (lb0 + warp + kWarps * i) * kBS;  // first token of the block
      if (i == i_new) {
        // the block has landed: put the new token's rows in place of whatever
        // the slot held, and store them to the cache (lanes 0-15 carry K's
        // 16-byte chunks, lanes 16-31 V's)
        const int slot = (L - 1) % kBS;
        const bool is_v = lane >= 16;
        const int ch = lane & 15;
        const uint16_t* src = is_v ? p.v_new + b * p.vn_stride[0] + gkv * p.vn_stride[1]
                                   : p.k_new + b * p.kn_stride[0] + gkv * p.kn_stride[1];
        const uint4 w = *reinterpret_cast<const uint4*>(src + ch * 8);
        *reinterpret_cast<uint4*>((is_v ? vb : kb) + sw_off(slot, ch)) = w;
        uint16_t* cache = is_v ? p.vc : p.kc;
        const int64_t off = (static_cast<int64_t>(blk) * p.Hkv + gkv) * (kBS * kD) + slot * kD + ch * 8;
        *reinterpret_cast<uint4*>(cache + off) = w;
      }
      const int r0 = t_end - tok0;  // valid rows of the block
      if (r0 < kBS) {
        // V rows past the context may hold anything (even NaN), and 0 * NaN
        // is not 0 in the MMA: zero them
        for (int c = lane; c < (kBS - r0) * 16; c += 32)
          *reinterpret_cast<uint4*>(vb + sw_off(r0 + c / 16, c & 15)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();

      // ---- S = Q K^T: n-tile j holds tokens 8j .. 8j+7
      float sacc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[j][e] = 0.f;
#pragma unroll
      for (int c = 0; c < 8; c += 2) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t kf[4];  // b0, b1 of k-chunk c, then of c + 1
          ldsm_x4(smem_u32(kb + sw_off(8 * j + mr, 2 * c + mi)), kf);
          mma_bf16(sacc[j], qa[c][0], 0u, qa[c][1], 0u, kf[0], kf[1]);
          mma_bf16(sacc[j], qa[c + 1][0], 0u, qa[c + 1][1], 0u, kf[2], kf[3]);
        }
      }
      float sc[4] = {sacc[0][0] * p.scale_log2, sacc[0][1] * p.scale_log2, sacc[1][0] * p.scale_log2,
                     sacc[1][1] * p.scale_log2};
      if (r0 < kBS) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (T[k] >= r0) sc[k] = -INFINITY;
      }
      float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
      // lazy rescale: the reference max moves only when a block exceeds it by
      // a margin; the output columns of head h are held by the lanes t = h / 2
      const bool move = bm > m_run + kLazy;
      if (__any_sync(0xffffffffu, move)) {
        float alpha = 1.f;
        if (move) {
          alpha = fast_exp2(m_run - bm);  // 0 when m_run was -inf
          l_part *= alpha;
          m_run = bm;
        }
        const float f0 = __shfl_sync(0xffffffffu, alpha, 8 * t), f1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          o[j][0] *= f0;
          o[j][1] *= f1;
          o[j][2] *= f0;
          o[j][3] *= f1;
        }
      }
      float pr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) pr[k] = fast_exp2(sc[k] - m_run);  // -inf -> 0
      l_part += (pr[0] + pr[1]) + (pr[2] + pr[3]);
      // the weights of head g are the B fragment of O^T = V^T P^T
      const uint32_t pb0 = pack_bf16x2(pr[0], pr[1]);
      const uint32_t pb1 = pack_bf16x2(pr[2], pr[3]);

      // ---- O^T += V^T P^T
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t va[4];  // dims 16mt + g / + 8 + g of tokens (2t, 2t+1), then (2t+8, 2t+9)
        ldsm_x4_trans(smem_u32(vb + sw_off(8 * (mi >> 1) + mr, 2 * mt + (mi & 1))), va);
        mma_bf16(o[mt], va[0], va[1], va[2], va[3], pb0, pb1);
      }
    }
    __syncwarp();
    if (i + kTcStages < my_n) {
      const int nb = __shfl_sync(0xffffffffu, my_blk, i + kTcStages);
      if (lane == 0) issue(s, nb);  // block i + kTcStages reuses stage s
      issued = i + kTcStages + 1;
    }
    if (++s == kTcStages) {
      s = 0;
      ph ^= 1u;
    }
  }
  if (!ok) {
    // let copies still in flight land before the shared memory is reused
    for (int i = (issued > kTcStages ? issued - kTcStages : 0); i < issued; ++i)
      drain_wait(&wbar[i % kTcStages], (i / kTcStages) & 1);
  }

  // ---- warp record per head: o (scaled to m_run), m_run, l
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 1);
  l_part += __shfl_xor_sync(0xffffffffu, l_part, 2);
  __syncthreads();  // the records overwrite the tile buffers
  constexpr int kRec = kD + 2;
  if (g < G && t == 0) {
    float* rec = comb + (warp * G + g) * kRec;
    rec[kD] = (ok && m_run != -INFINITY) ? m_run : -INFINITY;
    rec[kD + 1] = ok ? l_part : 0.f;
  }
  // columns 2t, 2t+1: dims 16 mt + g (registers 0, 1) and 16 mt + 8 + g (2, 3)
#pragma unroll
  for (int hc = 0; hc < 2; ++hc) {
    const int h = 2 * t + hc;
    if (h < G) {
      float* rec = comb + (warp * G + h) * kRec + g;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        rec[16 * mt] = o[mt][hc];
        rec[16 * mt + 8] = o[mt][2 + hc];
      }
    }
  }
  __syncthreads();

  // ---- combine the warps, write this split's partial (normalised out, log2 LSE)
  decode_combine_warps<kD, G, kWarps>(comb, gkv, b, split, p.sm);
  decode_finish<kD, G, kWarps>(p.sm, gkv, b, (L + kDecodeSplitTokens - 1) / kDecodeSplitTokens);
}

constexpr size_t tc_decode_smem() {
  return 1024 + static_cast<size_t>(kWarps) * kTcStages * (2 * kRowsBytes + 8);
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, const TcDecodeParams& p, cudaStream_t stream) {
  auto kern = paged_decode_tc_kernel<G>;
  const int smem = static_cast<int>(tc_decode_smem());
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.n_split), static_cast<unsigned>(a.cache.Hkv), static_cast<unsigned>(a.B));
  kern<<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// host side

bool paged_decode_tc_supported(const DecodeArgs& a) {
  const int64_t G = a.cache.Hkv > 0 ? a.Hq / a.cache.Hkv : 0;
  return a.cache.k_scale == nullptr && a.cache.D == kD && a.cache.block_size == kBS &&
         (G == 1 || G == 2 || G == 4 || G == 8);
}

cudaError_t launch_paged_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  TcDecodeParams p = {};
  if (!make_bf16_cache_map(&p.kmap, a.cache.k, a.cache.num_blocks, a.cache.Hkv) ||
      !make_bf16_cache_map(&p.vmap, a.cache.v, a.cache.num_blocks, a.cache.Hkv))
    return cudaErrorInvalidValue;
  p.kc = static_cast<uint16_t*>(a.cache.k);
  p.vc = static_cast<uint16_t*>(a.cache.v);
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
