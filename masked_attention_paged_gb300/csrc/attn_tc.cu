// attn_tc.cu -- masked exact attention with LSE on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA), bf16 inputs, fp32 accumulation and softmax.
//
// What it computes ("MultiheadAttention fast path used 18 GB of VRAM", the
// SDPA route with an additive -inf padding mask; "[sglang] ROCm aiter ring
// attention", section 1, the LSE the merge needs): for each query row
//   s_j = scale * q.k_j + mask_j,  out = sum_j softmax(s)_j v_j,  lse = log sum_j e^{s_j}
// without ever storing the score matrix: one 128 x 128 score tile per query
// tile lives in tensor memory at a time and is folded into the running output
// with the online-softmax rescale.
//
// CTA = two 128-row query tiles (A and B) of one (batch, head) sharing every
// K/V tile; 3 warpgroups:
//   warp 0      TMA producer: Q_A and Q_B once, then K_j / V_j tiles into a
//               ring of shared-memory stages (128-byte swizzle; 4-D tensor maps
//               so the same code reads [B,H,P,D] and packed [T,H,D] layouts).
//   warp 1      allocates all 512 TMEM columns; lane 0 issues tcgen05.mma for
//               tile A, lane 0 of warp 3 for tile B:
//                 S_t = Q_t K_j^T  (M=128, N=128, K=D, both operands in smem)
//                 O_t += P_t V_j   (M=128, N=D, K=128, P from TMEM, V in smem)
//               so the tensor pipe works on one tile while the other tile's
//               softmax runs; completion is signalled with tcgen05.commit ->
//               mbarrier, and a K/V stage is released after both issuers'
//               commits.
//   warp 2      stages each key tile's mask and a has-masked-keys flag.
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: thread r owns
//               row r (TMEM lane r).  It reads its S row from TMEM, adds the
//               mask, keeps the running max/sum in log2 units, writes P as
//               bf16 pairs back into the first 64 columns of the same S
//               region (the MMA that reads P precedes, in issue order, the
//               next S MMA that overwrites it), rescales O in TMEM only when
//               its reference max moves by more than kRescaleMargin, and
//               finally normalises O and writes out / lse.
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,256+D), O_B after it.
//
// Paged instances (PAGED) serve chunked prefill over a paged KV cache ("KV
// cache in nanoVLM", prefill phase; "LLM inference memory accounting",
// sections 15 and 20): the queries are a chunk of T new tokens at positions
// start + i of their sequence, and each 128-key tile is gathered from eight
// 16-token cache blocks through the block table, one 16-row TMA box per
// block at its row offset (the 128-byte swizzle repeats every 8 rows, so the
// tile's shared-memory image is the same as a 128-row load).  Keys past a
// row's limit (its own position when causal, the sequence end otherwise) are
// selected to -inf rather than masked by addition, so whatever an unfilled
// cache slot holds never reaches the softmax; V rows past the CTA's last key
// are zeroed in shared memory before the last PV, as P = 0 times a NaN would
// not be 0.
//
// Every wait is bounded (common.cuh): a hang turns into ATTN_ERR_TIMEOUT in
// the caller's status word and the CTA winds down and frees its TMEM.
#include <cuda.h>
#include <math.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kBM = 128;       // query rows per tile (two tiles per CTA)
constexpr int kBN = 128;       // keys per KV tile
constexpr int kThreads = 384;  // 3 warpgroups
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
constexpr int kBoxBytes = kBM * 128;  // one 64-column (128-byte) box of 128 rows
// A row's reference max (log2 units) only moves when the tile max exceeds it
// by more than this; P then stays below 2^8, well inside bf16 and fp32 range.
constexpr float kRescaleMargin = 8.0f;

template <int D, bool SEP = (D == 64)>
struct Cfg {
  // SEP (D = 64 only): P in its own TMEM columns (S_A, S_B 128 columns each,
  // O_A, O_B 64 each, P_A, P_B 64 each = 512): the next S can then be issued
  // as soon as the softmax has read the current one, and each softmax
  // warpgroup runs tile after tile without waiting for its PV; the max pass
  // is skipped only where precomputed key bounds certify a tile.  Otherwise
  // P is written over the first half of its S region, and the softmax
  // exponentiates optimistically and redoes a tile whose row sums fail.
  static_assert(D == 64 || !SEP, "P apart from S needs D = 64");
  static constexpr bool kSepP = SEP;
  // With P apart from S each tile gets its own MMA-issuing warp; with P over
  // S one warp issues both tiles in the order PV_A, S_A', PV_B, S_B', which
  // keeps each tile's PV -> next-S chain short.
  static constexpr bool kTwoIssuers = kSepP;
  // setmaxnreg split of the 168 registers per thread the CTA is launched
  // with (384 x 168 = 64512): 128 x kRegsCtl + 256 x kRegsSoft must not
  // exceed it.  At D = 64 the two MMA issuers sit on the critical path and
  // spilled at 88 (measured: 104 / 200 is 3 % faster than 88 / 208).
  static constexpr int kRegsCtl = kSepP ? 104 : 88;
  static constexpr int kRegsSoft = kSepP ? 200 : 208;
  static_assert(128 * kRegsCtl + 256 * kRegsSoft <= 384 * 168, "register split exceeds the launch allocation");
  static constexpr uint32_t kColP0 = 256 + 2 * D;  // P_A, P_B (kSepP only)
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBM * D * 2;
  static constexpr int kStages = (D == 64) ? 4 : 2;
  static constexpr uint32_t kColO0 = 256;
  static constexpr int kOffQ = 0;  // Q_A, Q_B
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffMask = kOffV + kStages * kTileBytes;  // [2 buf][kBN] floats, log2 units
  static constexpr int kOffBar = kOffMask + 2 * kBN * 4;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + slack to align the base to 1024
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t s_free[2], o_done[2];   // kSepP: S read out by the softmax; PV done
  uint64_t m_full[2], m_empty[2];  // mask tile staging (warp 2 -> softmax warps)
  uint64_t o_final[2];
  uint64_t first_p;                // tile A's issuer has seen its first P (completes once)
  int m_flag[2];                   // tile has a masked key (or keys past Pk)
  float kmax[2];                   // largest |k| element of the tile (score bound)
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Barriers) <= 512, "barrier block outgrew its shared-memory slot");

struct TmaCoordMap {
  // which tensor-map coordinate slot (1..3) carries the row, head and batch index
  int slot_p, slot_h, slot_b;
};

struct TcParams {
  int Pq, Pk, Hq, group;
  float scale_log2;
  int scale_positive;  // max of raw scores == max of scaled scores
  const float* mask;
  int64_t mask_stride;
  const int32_t* key_lens;  // per-batch valid keys, or null (all Pk)
  const float* key_bound;   // [B, Hkv, key_tiles] largest |k| element per 128-key tile, or null
  int key_tiles;
  // Non-paged grids are 1-D over units (query-tile pair, head, batch), the
  // pair fastest.  The first full_units CTAs take one unit each; the rest
  // take one of `split` parts of the KV tiles of the remaining units, so the
  // last wave fills every SM.  A part writes its rows (normalised, f32) and
  // LSE (natural log) to part_o / part_lse for split_merge_kernel.
  int nq;  // query-tile pairs per (batch, head)
  int full_units;
  int split;
  float* part_o;    // [units past full_units][split][2 kBM][D]
  float* part_lse;  // [units past full_units][split][2 kBM]
  // PAGED: cache read through the block table
  const int32_t* bt;
  int64_t bt_stride;
  int max_blocks;
  int num_blocks;
  const int32_t* start_pos;  // [B] tokens cached before the chunk
  int causal;
  void* out;
  int64_t out_stride[3];  // b, h, row (elements)
  float* lse;
  uint32_t* status;
  TmaCoordMap cq, ck, cv;
};

// Which (query-tile pair, head, batch) a CTA works on, and which KV part.
struct UnitIdx {
  int h, b, q0;
  int part;   // >= 0: index of this CTA's KV part of a split unit
  int prow0;  // first row of that part in part_o / part_lse
};

template <bool PAGED>
__device__ __forceinline__ UnitIdx unit_index(const TcParams& prm, unsigned bx, unsigned by, unsigned bz,
                                              unsigned gx) {
  UnitIdx u;
  u.part = -1;
  u.prow0 = 0;
  if constexpr (PAGED) {
    u.h = static_cast<int>(by);
    u.b = static_cast<int>(bz);
    // causal: the longest query tiles (latest positions) first
    u.q0 = static_cast<int>(prm.causal ? gx - 1 - bx : bx) * (2 * kBM);
  } else {
    int unit = static_cast<int>(bx);
    if (unit >= prm.full_units) {
      const int r = unit - prm.full_units;
      unit = prm.full_units + r / prm.split;
      u.part = r % prm.split;
      u.prow0 = r * (2 * kBM);
    }
    u.q0 = (unit % prm.nq) * (2 * kBM);
    u.h = (unit / prm.nq) % prm.Hq;
    u.b = unit / (prm.nq * prm.Hq);
  }
  return u;
}

// The CTA index read through an opaque move, so that a unit decoded from it
// is recomputed where it is needed rather than kept live in registers.
__device__ __forceinline__ unsigned cta_x() {
  unsigned x;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(x));
  return x;
}

__device__ __forceinline__ void coords(const TmaCoordMap& m, int p, int h, int b, int& c1, int& c2, int& c3) {
  c1 = m.slot_p == 1 ? p : (m.slot_h == 1 ? h : b);
  c2 = m.slot_p == 2 ? p : (m.slot_h == 2 ? h : b);
  c3 = m.slot_p == 3 ? p : (m.slot_h == 3 ? h : b);
}

template <int D, bool OUT_BF16, bool PAGED, bool SEP>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const TcParams prm) {
  using C = Cfg<D, SEP>;
  // With P apart from S the softmax skips the max pass on tiles where a
  // bound certifies that no exponential can overflow (see the stager)
  constexpr bool kCert = C::kSepP && !PAGED;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kOffBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const UnitIdx ui = unit_index<PAGED>(prm, blockIdx.x, blockIdx.y, blockIdx.z, gridDim.x);
  const int h = ui.h, b = ui.b, q0 = ui.q0;
  const int g = h / prm.group;
  // keys of this batch row: all Pk, or its valid length (tiles past it are skipped)
  int n_keys = prm.Pk;
  int start = 0;  // PAGED: position of the chunk's first token
  if constexpr (PAGED) {
    start = prm.start_pos[b];
    const int64_t seq_len = static_cast<int64_t>(start) + prm.Pq;
    if (start < 0 || seq_len > static_cast<int64_t>(prm.max_blocks) * 16) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) report(prm.status, kStatusBounds);
      n_keys = 0;  // the sequence is written as zeros
    } else {
      // the last key any row of this CTA may see
      n_keys = prm.causal ? start + min(q0 + 2 * kBM, prm.Pq) : static_cast<int>(seq_len);
    }
  } else if (prm.key_lens != nullptr) {
    const int len = prm.key_lens[b];
    n_keys = len < 0 ? 0 : (len < prm.Pk ? len : prm.Pk);
  }
  // this CTA's key tiles: [kv0, kv0 + nkv), all of them unless it is a part
  int kv0 = 0;
  int nkv = (n_keys + kBN - 1) / kBN;
  if (ui.part >= 0) {
    const int per = (nkv + prm.split - 1) / prm.split;
    kv0 = min(nkv, ui.part * per);
    nkv = min(nkv, kv0 + per) - kv0;
  }
  volatile int* abort = &bars->abort;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], C::kTwoIssuers ? 2 : 1);  // one commit per MMA issuer
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], C::kTwoIssuers ? 2 : 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->m_full[t], 1);
      mbar_init(&bars->m_empty[t], 8);
      mbar_init(&bars->s_free[t], 4);
      mbar_init(&bars->o_done[t], 1);
    }
    mbar_init(&bars->o_final[0], 1);
    mbar_init(&bars->o_final[1], 1);
    mbar_init(&bars->first_p, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  // Register budget: launched at 168 per thread (384 x 168 = 64512).  At
  // D = 128 the producer/MMA/mask warpgroup gives up 80 per thread (10240)
  // and the two softmax warpgroups take 40 (2 x 128 x 40 = 10240); at D = 64
  // 64 and 32 (8192 each way).
  if (warp < 4) regs_dec<C::kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int c1, c2, c3;
      mbar_arrive_expect_tx(&bars->q_full, 2 * C::kTileBytes);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        coords(prm.cq, q0 + t * kBM, h, b, c1, c2, c3);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(smem + C::kOffQ + t * C::kTileBytes + x * kBoxBytes, &tm_q, &bars->q_full, x * 64, c1, c2,
                      c3);
      }
    }
    int k_issued = 0, v_issued = 0;
    if constexpr (PAGED) {
      // the whole warp streams K/V: lane i < 8 owns logical block 8j + i of
      // key tile j (its two 64-column boxes of K and of V), so one
      // warp-instruction issues a half of every block; the ids are read one
      // tile ahead.  Blocks wholly past the CTA's last key are not loaded,
      // nor is a bad block id.
      constexpr int kBlk = kBN / 16;
      constexpr int kBlockBytes = 16 * D * 2;
      const int32_t* bt_row = prm.bt + static_cast<int64_t>(b) * prm.bt_stride + kv0 * kBlk;
      auto block_id = [&](int j) {
        const int nb = min(kBlk, (n_keys - (kv0 + j) * kBN + 15) / 16);
        return (j < nkv && lane < nb) ? bt_row[j * kBlk + lane] : -1;
      };
      int id_next = block_id(0);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        int id = id_next;
        id_next = block_id(j + 1);
        if (lane < kBlk && id != -1 && (id < 0 || id >= prm.num_blocks)) {
          report(prm.status, kStatusBounds);
          id = -1;
        }
        if (id >= 0 && lane >= kBlk) id = -1;
        const int n_ok = __popc(__ballot_sync(0xffffffffu, id >= 0));
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->k_empty[s], ph ^ 1, abort, prm.status))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[s], n_ok * kBlockBytes);
        __syncwarp();
        if (id >= 0)
#pragma unroll
          for (int x = 0; x < C::kBoxes; ++x)
            tma_load_4d(smem + C::kOffK + s * C::kTileBytes + x * kBoxBytes + lane * 2048, &tm_k, &bars->k_full[s],
                        x * 64, 0, g, id);
        k_issued = j + 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_empty[s], ph ^ 1, abort, prm.status))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->v_full[s], n_ok * kBlockBytes);
        __syncwarp();
        if (id >= 0)
#pragma unroll
          for (int x = 0; x < C::kBoxes; ++x)
            tma_load_4d(smem + C::kOffV + s * C::kTileBytes + x * kBoxBytes + lane * 2048, &tm_v, &bars->v_full[s],
                        x * 64, 0, g, id);
        v_issued = j + 1;
      }
    } else if (lane == 0) {
      int c1, c2, c3;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        if (!mbar_wait(&bars->k_empty[s], ph ^ 1, abort, prm.status)) break;
        mbar_arrive_expect_tx(&bars->k_full[s], C::kTileBytes);
        coords(prm.ck, (kv0 + j) * kBN, g, b, c1, c2, c3);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(smem + C::kOffK + s * C::kTileBytes + x * kBoxBytes, &tm_k, &bars->k_full[s], x * 64,
                      c1, c2, c3);
        k_issued = j + 1;
        if (!mbar_wait(&bars->v_empty[s], ph ^ 1, abort, prm.status)) break;
        mbar_arrive_expect_tx(&bars->v_full[s], C::kTileBytes);
        coords(prm.cv, (kv0 + j) * kBN, g, b, c1, c2, c3);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_4d(smem + C::kOffV + s * C::kTileBytes + x * kBoxBytes, &tm_v, &bars->v_full[s], x * 64,
                      c1, c2, c3);
        v_issued = j + 1;
      }
    }
    if (lane == 0) {
      if (*abort) {
        // let every copy still in flight land before the CTA exits
        drain_wait(&bars->q_full, 0);
        for (int j = (k_issued > C::kStages ? k_issued - C::kStages : 0); j < k_issued; ++j)
          drain_wait(&bars->k_full[j % C::kStages], (j / C::kStages) & 1);
        for (int j = (v_issued > C::kStages ? v_issued - C::kStages : 0); j < v_issued; ++j)
          drain_wait(&bars->v_full[j % C::kStages], (j / C::kStages) & 1);
      }
    }
  } else if (warp == 1 || (C::kTwoIssuers && warp == 3)) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, false, true);
      auto issue_s = [&](int t, int j) {  // S_t = Q_t K_j^T
        const uint32_t qa = smem_u32(smem + C::kOffQ) + t * C::kTileBytes;
        const uint32_t k_addr = smem_u32(smem + C::kOffK + (j % C::kStages) * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;  // 16 dims = 32 bytes of a 128-byte row
          umma_bf16_ss(tmem + col_s(t), sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                       idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int j) {  // O_t += P_t V_j, P_t in TMEM
        const uint32_t v_addr = smem_u32(smem + C::kOffV + (j % C::kStages) * C::kTileBytes);
        const uint32_t p_tmem = tmem + (C::kSepP ? C::kColP0 + t * 64 : col_s(t));
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // 16 keys = 8 TMEM columns of packed P; V is MN-major (d contiguous):
          // 16 keys = two 8-row groups (SBO), next 64-column box of d at LBO
          umma_bf16_ts(tmem + C::kColO0 + t * D, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024),
                       idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort, prm.status) && nkv > 0 &&
                mbar_wait(&bars->k_full[0], 0, abort, prm.status);
      if constexpr (C::kTwoIssuers) {
        // warp 1 issues every MMA of query tile A, warp 3 every MMA of tile B,
        // so each tile's chain waits only on its own softmax warpgroup:
        // S_t(j+1) as soon as the softmax has read S_t(j), PV_t(j) once P_t(j)
        // is written
        const int t = warp == 1 ? 0 : 1;
        // Tile B starts once tile A's first P is written.  Started together,
        // the two tiles run in lockstep: both softmax warpgroups compute at
        // once while the tensor pipe idles, then both wait for their next S.
        // Half a step apart, one tile's MMAs overlap the other's softmax.
        // The wait is on a barrier of its own, which completes once: by the
        // time it runs, p_full[0] may have moved on by a phase or two, and a
        // parity wait on it would then wait for a later phase while tile A
        // needs this issuer's commits to free its K/V stages.
        if (ok && t == 1) ok = mbar_wait(&bars->first_p, 0, abort, prm.status);
        if (ok) {
          tc_fence_after();
          issue_s(t, 0);
          umma_commit(&bars->s_full[t]);
          umma_commit(&bars->k_empty[0]);
        }
        for (int j = 0; ok && j < nkv; ++j) {
          const int s = j % C::kStages;
          const int j1 = j + 1;
          const int s1 = j1 % C::kStages;
          if (j1 < nkv) {
            if (!mbar_wait(&bars->k_full[s1], (j1 / C::kStages) & 1, abort, prm.status) ||
                !mbar_wait(&bars->s_free[t], j & 1, abort, prm.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, j1);
            umma_commit(&bars->s_full[t]);
            umma_commit(&bars->k_empty[s1]);
          }
          if (!mbar_wait(&bars->p_full[t], j & 1, abort, prm.status) ||
              !mbar_wait(&bars->v_full[s], (j / C::kStages) & 1, abort, prm.status)) {
            ok = false;
            break;
          }
          if (t == 0 && j == 0) mbar_arrive(&bars->first_p);
          tc_fence_after();
          issue_pv(t, j);
          umma_commit(&bars->o_done[t]);
          umma_commit(&bars->v_empty[s]);
        }
        // completes when every MMA of this tile has: O_t is final
        umma_commit(&bars->o_final[t]);
        drain_wait(&bars->o_final[t], 0);
      } else {
        // one issuer, order PV_A(j), S_A(j+1), PV_B(j), S_B(j+1): P_t(j) sits
        // in S_t's columns and S_t(j+1) follows the PV_t(j) that reads it
        // (one thread's MMAs execute in issue order)
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          umma_commit(&bars->s_full[0]);
          issue_s(1, 0);
          umma_commit(&bars->s_full[1]);
          umma_commit(&bars->k_empty[0]);
        }
        for (int j = 0; ok && j < nkv; ++j) {
          const int s = j % C::kStages;
          const int j1 = j + 1;
          const int s1 = j1 % C::kStages;
          if (!mbar_wait(&bars->p_full[0], j & 1, abort, prm.status) ||
              !mbar_wait(&bars->v_full[s], (j / C::kStages) & 1, abort, prm.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, j);
          if (j1 < nkv) {
            if (!mbar_wait(&bars->k_full[s1], (j1 / C::kStages) & 1, abort, prm.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, j1);
            umma_commit(&bars->s_full[0]);
          }
          if (!mbar_wait(&bars->p_full[1], j & 1, abort, prm.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, j);
          umma_commit(&bars->v_empty[s]);
          if (j1 < nkv) {
            issue_s(1, j1);
            umma_commit(&bars->s_full[1]);
            umma_commit(&bars->k_empty[s1]);
          }
        }
        // completes when every MMA above has: O_A and O_B are final
        umma_commit(&bars->o_final[0]);
        umma_commit(&bars->o_final[1]);
        drain_wait(&bars->o_final[1], 0);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ mask stager
    // Each 128-key tile's additive mask, in log2 units (-inf past Pk), goes
    // to a double-buffered shared array with a flag telling whether any of
    // its keys is masked; both softmax warpgroups read it.
    const float kLog2e = 1.4426950408889634f;
    const float* mrow = prm.mask ? prm.mask + static_cast<int64_t>(b) * prm.mask_stride : nullptr;
    float* mbuf = reinterpret_cast<float*>(smem + C::kOffMask);
    // paged instances have no mask tensor: the softmax applies the row limits
    for (int j = 0; j < (PAGED ? 0 : nkv); ++j) {
      const int s = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->m_empty[s], ((j >> 1) & 1) ^ 1, abort, prm.status))) break;
      float v[4];
      bool any = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = (kv0 + j) * kBN + lane * 4 + e;
        v[e] = key >= n_keys ? -INFINITY : (mrow ? mrow[key] * kLog2e : 0.0f);
        any |= v[e] != 0.0f;
      }
      *reinterpret_cast<float4*>(mbuf + s * kBN + lane * 4) = make_float4(v[0], v[1], v[2], v[3]);
      any = __any_sync(0xffffffffu, any);
      if (lane == 0) bars->m_flag[s] = any || !prm.scale_positive;
      if constexpr (kCert) {
        // The largest |k| element of K_j, precomputed (+inf without it):
        // every score of the tile obeys |q.k| <= |q|_1 max|k|, which lets the
        // softmax skip its max pass.
        if (lane == 0)
          bars->kmax[s] = prm.key_bound != nullptr
                              ? prm.key_bound[(static_cast<int64_t>(b) * (prm.Hq / prm.group) + g) * prm.key_tiles +
                                              kv0 + j]
                              : INFINITY;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->m_full[s]);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    regs_inc<C::kRegsSoft>();
    const int t = (warp >> 2) - 1;            // query tile 0 (A) or 1 (B)
    const int quarter = warp & 3;             // TMEM lanes this warp may touch
    const int row = quarter * 32 + lane;      // row within the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_col = col_s(t);
    const uint32_t o_col = C::kColO0 + t * D;
    // P as bf16 pairs (key 2i in the low half): its own region (D = 64) or the
    // first 64 columns of S_t (D = 128)
    const uint32_t p_col = C::kSepP ? C::kColP0 + t * 64 : s_col;
    const float* mbuf = reinterpret_cast<const float*>(smem + C::kOffMask);
    float m_run = -INFINITY;  // reference max, log2 units
    float l_run = 0.0f;       // running sum of 2^(x - m_run)
    bool ok = true;
    // kCert: L1 norm of this row's query (rows past Pq were zero-filled)
    float q_l1 = 0.0f;
    if constexpr (kCert) {
      if (nkv > 0 && __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort, prm.status))) {
        const uint8_t* qt = smem + C::kOffQ + t * C::kTileBytes;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {  // 128-byte swizzled row: chunk ch sits at ch ^ (row % 8)
          const uint4 w = *reinterpret_cast<const uint4*>(qt + row * 128 + ((ch ^ (row & 7)) << 4));
          q_l1 += (fabsf(bf16lo_to_f32(w.x)) + fabsf(bf16hi_to_f32(w.x))) +
                  (fabsf(bf16lo_to_f32(w.y)) + fabsf(bf16hi_to_f32(w.y))) +
                  (fabsf(bf16lo_to_f32(w.z)) + fabsf(bf16hi_to_f32(w.z))) +
                  (fabsf(bf16lo_to_f32(w.w)) + fabsf(bf16hi_to_f32(w.w)));
        }
      }
    }
    // PAGED: keys [0, row_lim) are this row's (its own position when causal)
    int row_lim = n_keys;
    if constexpr (PAGED) {
      if (prm.causal) row_lim = min(n_keys, start + q0 + t * kBM + row + 1);
    }

    for (int j = 0; j < nkv; ++j) {
      const int mb_i = j & 1;
      // wait outcomes are made warp-uniform: tcgen05.ld/st need the whole warp
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, abort, prm.status) &&
                                       (PAGED || mbar_wait(&bars->m_full[mb_i], (j >> 1) & 1, abort, prm.status)))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
      // D = 128: the first half of the scores first; the second half is
      // loaded while the fast path exponentiates the first
      constexpr int kFirstLd = C::kSepP ? 4 : 2;
#pragma unroll
      for (int c = 0; c < kFirstLd; ++c) tmem_ld32(tmem + lane_addr + s_col + c * 32, sr[c]);
      // keys of this tile the row may see: [0, lim)
      const int lim = row_lim - (kv0 + j) * kBN;
      const bool masked_tile = PAGED ? __any_sync(0xffffffffu, lim < kBN) || !prm.scale_positive
                                     : bars->m_flag[mb_i] != 0;
#pragma unroll
      for (int c = 0; c < kFirstLd; ++c) tmem_wait_ld(sr[c]);
#pragma unroll
      for (int c = kFirstLd; c < 4; ++c) tmem_ld32(tmem + lane_addr + s_col + c * 32, sr[c]);
      bool second_pending = kFirstLd < 4;
      auto finish_ld = [&]() {
        if (second_pending) {
#pragma unroll
          for (int c = kFirstLd; c < 4; ++c) tmem_wait_ld(sr[c]);
          second_pending = false;
        }
      };
#define SV(c) __uint_as_float(sr[(c) >> 5][(c) & 31])
      if constexpr (C::kSepP) {  // S is in registers: the next S may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[t]);
      }

      float alpha = 1.0f;
      float rs = 0.0f;
      bool done = false;
      // P apart from S: the weights as bf16 pairs, packed before the wait for
      // PV_t(j-1) that frees P's columns
      uint32_t pws[C::kSepP ? 4 : 1][16];
      // Fast path: exponentiate against the current reference max without a
      // max pass.  P over S: every term is <= 2^64 exactly when the row sum
      // is, which keeps the sums far from fp32 overflow; if some row fails,
      // the warp reloads S (its columns are intact until P is written over
      // them) and takes the full path below.  P apart from S (S's columns are
      // handed back right after the load, so nothing could be reloaded): the
      // path is taken only where |s| <= |q|_1 max|k| certifies every term to
      // be <= 2^60.
      bool try_fast;
      if constexpr (kCert) {
        const float bound = q_l1 * bars->kmax[mb_i] * prm.scale_log2;  // scale > 0 on unmasked tiles
        try_fast = !masked_tile && __all_sync(0xffffffffu, m_run != -INFINITY && bound - m_run <= 60.0f);
      } else {
        // paged tiles with keys past a row's limit take it too, the keys
        // selected to -inf before the exponential
        try_fast = !C::kSepP && (PAGED || !masked_tile) && __all_sync(0xffffffffu, m_run != -INFINITY);
      }
      if (try_fast) {
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.0f;
        const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
        const uint64_t ng2 = f2_pack(-m_run, -m_run);
        // two keys per packed fma / add; sums in 8 partial accumulators;
        // LIMIT: keys at or past the row's limit give 0
        auto fast_loop = [&](auto limit_c) {
          [[maybe_unused]] constexpr bool LIMIT = decltype(limit_c)::value;
          if constexpr (C::kSepP) {
            // P in its own columns, written once PV_t(j-1) has read the last
            // tile's: the weights wait in registers, packed as bf16 pairs
#pragma unroll
            for (int c = 0; c < kBN; c += 2) {
              float x0, x1;
              f2_unpack(ffma2(f2_pack(SV(c), SV(c + 1)), sc2, ng2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              pws[c >> 5][(c & 31) >> 1] = pack_bf16x2(p0, p1);
              const int a = (c >> 1) & 3;
              uint64_t acc = f2_pack(rsum[a], rsum[4 + a]);
              f2_unpack(fadd2(acc, f2_pack(p0, p1)), rsum[a], rsum[4 + a]);
            }
          } else {
            // P over S: each 32-key chunk of P goes to TMEM as soon as it is
            // computed (chunk c lands on columns 16c..16c+15, whose scores
            // are already in registers), while the scores stay in registers
            // so that a failed check below can redo the tile from them
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              if (c == kFirstLd) finish_ld();
              uint32_t pw[16];
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const int key = c * 32 + i;
                float x0, x1;
                f2_unpack(ffma2(f2_pack(SV(key), SV(key + 1)), sc2, ng2), x0, x1);
                if constexpr (LIMIT) {
                  x0 = key < lim ? x0 : -INFINITY;
                  x1 = key + 1 < lim ? x1 : -INFINITY;
                }
                const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                pw[i >> 1] = pack_bf16x2(p0, p1);
                const int a = (i >> 1) & 3;
                uint64_t acc = f2_pack(rsum[a], rsum[4 + a]);
                f2_unpack(fadd2(acc, f2_pack(p0, p1)), rsum[a], rsum[4 + a]);
              }
              tmem_st16(tmem + lane_addr + p_col + c * 16, pw);
            }
          }
        };
        if (PAGED && masked_tile)
          fast_loop(std::integral_constant<bool, PAGED>());
        else
          fast_loop(std::integral_constant<bool, false>());
        rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) + ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
        if (kCert || __all_sync(0xffffffffu, rs <= 18446744073709551616.0f)) {  // 2^64; false for NaN
          done = true;
        } else {
          // the scores are intact in registers; the P just stored is written
          // over again below, after these stores have landed
          tmem_wait_st();
        }
      }
      if (!done) {
        finish_ld();
        // tile max in log2 units: 8 independent chains of 3-input max
        float mx[8];
        if (!masked_tile) {
          // no masked key: the max of the raw scores, scaled once (scale > 0)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(SV(2 * i), SV(2 * i + 1));
#pragma unroll
          for (int c = 16; c < kBN; c += 2) mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], SV(c), SV(c + 1));
        } else if constexpr (PAGED) {
          // logits, keys past the row's limit selected to -inf, in place
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            const float x = c < lim ? SV(c) * prm.scale_log2 : -INFINITY;
            sr[c >> 5][c & 31] = __float_as_uint(x);
            mx[(c >> 1) & 7] = fmaxf(mx[(c >> 1) & 7], x);
          }
        } else {
          // logits with the additive mask, in place
          const float4* mb = reinterpret_cast<const float4*>(mbuf + mb_i * kBN);
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
          for (int c4 = 0; c4 < kBN / 4; ++c4) {
            const float4 mv = mb[c4];
            const float x0 = fmaf(SV(4 * c4), prm.scale_log2, mv.x);
            const float x1 = fmaf(SV(4 * c4 + 1), prm.scale_log2, mv.y);
            const float x2 = fmaf(SV(4 * c4 + 2), prm.scale_log2, mv.z);
            const float x3 = fmaf(SV(4 * c4 + 3), prm.scale_log2, mv.w);
            sr[c4 >> 3][(4 * c4) & 31] = __float_as_uint(x0);
            sr[c4 >> 3][(4 * c4 + 1) & 31] = __float_as_uint(x1);
            sr[c4 >> 3][(4 * c4 + 2) & 31] = __float_as_uint(x2);
            sr[c4 >> 3][(4 * c4 + 3) & 31] = __float_as_uint(x3);
            mx[(2 * c4) & 7] = fmax3(mx[(2 * c4) & 7], x0, x1);
            mx[(2 * c4 + 1) & 7] = fmax3(mx[(2 * c4 + 1) & 7], x2, x3);
          }
        }
        float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        if (!masked_tile) mt *= prm.scale_log2;
        // lazy reference max: move it only when the tile exceeds it by the margin
        if (mt > m_run + kRescaleMargin || (m_run == -INFINITY && mt != -INFINITY)) {
          alpha = fast_exp2(m_run - mt);  // 0 when nothing was unmasked before
          m_run = mt;
        }
        const float m_sub = (m_run == -INFINITY) ? 0.0f : m_run;
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.0f;
        auto chunk_out = [&](int c) {
          uint32_t pw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pw[i] = pack_bf16x2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
          tmem_st16(tmem + lane_addr + p_col + c * 16, pw);
        };
        // D = 128 stores P 32 keys at a time as they are exponentiated (each
        // chunk's values die once in TMEM); D = 64 first exponentiates the whole
        // row, giving PV_t(j-1) time to finish before it must wait for it
        constexpr bool kChunked = !C::kSepP;
        const float neg = -m_sub;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (!masked_tile) {
            const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2), ng2 = f2_pack(neg, neg);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              f2_unpack(ffma2(f2_pack(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), sc2, ng2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              sr[c][i] = __float_as_uint(p0);
              sr[c][i + 1] = __float_as_uint(p1);
              const int a = (i >> 1) & 3;
              uint64_t acc = f2_pack(rsum[a], rsum[4 + a]);
              f2_unpack(fadd2(acc, f2_pack(p0, p1)), rsum[a], rsum[4 + a]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float pv = fast_exp2(__uint_as_float(sr[c][i]) - m_sub);  // -inf -> 0
              sr[c][i] = __float_as_uint(pv);
              rsum[i & 7] += pv;
            }
          }
          if constexpr (kChunked) chunk_out(c);
        }
        rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) + ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
        if constexpr (!kChunked) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pws[c][i] = pack_bf16x2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
          // P_t and O_t are free once PV_t(j-1) has completed
          if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], (j - 1) & 1, abort, prm.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_st16(tmem + lane_addr + p_col + c * 16, pws[c]);
        }
      } else if constexpr (C::kSepP) {
        // fast path passed: P goes to its own columns once PV_t(j-1) has read
        // them (over S, P is in TMEM already)
        if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], (j - 1) & 1, abort, prm.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(tmem + lane_addr + p_col + c * 16, pws[c]);
      }
#undef SV
      __syncwarp();
      if (!PAGED && lane == 0) mbar_arrive(&bars->m_empty[mb_i]);  // this warp is done with the mask tile
      l_run = l_run * alpha + rs;

      // O_t is stable here: PV_t(j-1) has completed (o_done, or the commit
      // behind s_full when P shares S's columns)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + o_col + c * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_addr + o_col + c * 32, o);
        }
      }
      if constexpr (PAGED) {
        // last tile: V rows past the CTA's last key were not loaded (or hold
        // whatever the cache's unfilled slots hold); zero them before PV reads
        // them.  Both softmax warpgroups write the same zeros.  The stage is
        // not refilled before this warpgroup's p_full below.
        const int r0 = n_keys - (kv0 + j) * kBN;
        if (j == nkv - 1 && r0 < kBN) {
          const int s = j % C::kStages;
          if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[s], (j / C::kStages) & 1, abort, prm.status))) {
            ok = false;
            break;
          }
          uint8_t* vst = smem + C::kOffV + s * C::kTileBytes;
          const int nchunk = (kBN - r0) * 8;  // 16-byte chunks of the rows past r0, per box
#pragma unroll
          for (int x = 0; x < C::kBoxes; ++x)
            for (int c = row; c < nchunk; c += kBM)
              *reinterpret_cast<uint4*>(vst + x * kBoxBytes + (r0 + c / 8) * 128 + (c % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async_smem();  // the generic-proxy stores before the MMA's async-proxy reads
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t]);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && nkv > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_final[t], 0, abort, prm.status));
      tc_fence_after();
    }
    // the unit again, from the CTA index (cheaper than keeping it live)
    const UnitIdx ue = unit_index<PAGED>(prm, PAGED ? blockIdx.x : cta_x(), blockIdx.y, blockIdx.z, gridDim.x);
    const int part = ue.part;
    const int qi = ue.q0 + t * kBM + row;
    const bool empty = !(l_run > 0.0f);
    const float inv_l = empty ? 0.0f : 1.0f / l_run;
    const int64_t prow = ue.prow0 + t * kBM + row;  // part rows: normalised f32 partials
    const int64_t obase = part >= 0 ? prow * D
                                    : static_cast<int64_t>(ue.b) * prm.out_stride[0] +
                                          static_cast<int64_t>(ue.h) * prm.out_stride[1] +
                                          static_cast<int64_t>(qi) * prm.out_stride[2];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (ok && nkv > 0) {
        tmem_ld32(tmem + lane_addr + o_col + c * 32, o);
        tmem_wait_ld(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (qi < prm.Pq && ok && part >= 0) {
        float4* dst = reinterpret_cast<float4*>(prm.part_o + obase + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(o[4 * i + 0]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                               __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
      } else if (qi < prm.Pq && ok) {
        if constexpr (OUT_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(prm.out) + obase + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l);
            dst[i] = w;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(prm.out) + obase + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i + 0]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                 __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
        }
      }
    }
    if (qi < prm.Pq && ok && (part >= 0 || prm.lse != nullptr)) {
      const float lse2 = empty ? -INFINITY : (m_run + __log2f(l_run));
      if (part >= 0)
        prm.part_lse[prow] = lse2 * 0.6931471805599453f;
      else
        prm.lse[(static_cast<int64_t>(ue.b) * prm.Hq + ue.h) * prm.Pq + qi] = lse2 * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the KV parts of each split unit: per query row, the LSE rule of the
// ring-attention page (out = sum_c exp(lse_c - lse) out_c) over its `split`
// (<= 8) normalised partials.  One warp per row: lane c holds part c's LSE,
// the max and the weights come from shuffles, and every part's row is
// loaded before any is used.
template <int D, bool OUT_BF16>
__global__ void split_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int split,
                                   int full_units, int tail, int nq, int Hq, int Pq, void* out, int64_t os0,
                                   int64_t os1, int64_t os2, float* lse) {
  constexpr int E = D / 32;
  constexpr int kMaxParts = 8;
  const int w = static_cast<int>((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= tail * 2 * kBM) return;
  const int u = w / (2 * kBM), r = w % (2 * kBM);
  const int unit = full_units + u;
  const int qi = (unit % nq) * (2 * kBM) + r;
  if (qi >= Pq) return;
  const int h = (unit / nq) % Hq, b = unit / (nq * Hq);
  const float l_mine =
      lane < split ? part_lse[static_cast<int64_t>(u * split + lane) * (2 * kBM) + r] : -INFINITY;
  float M = l_mine;
#pragma unroll
  for (int m = 4; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));
  M = __shfl_sync(0xffffffffu, M, 0);  // lanes 0-7 hold the parts
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (M != -INFINITY) {
    const float w_mine = l_mine == -INFINITY ? 0.0f : expf(l_mine - M);
    float ov[kMaxParts][E];
    float wk[kMaxParts];
#pragma unroll
    for (int c = 0; c < kMaxParts; ++c) {
      wk[c] = __shfl_sync(0xffffffffu, w_mine, c);
      const bool use = c < split && wk[c] > 0.0f;  // a part with no keys may hold anything
      const int64_t prow = static_cast<int64_t>(u * split + c) * (2 * kBM) + r;
#pragma unroll
      for (int e = 0; e < E; ++e) ov[c][e] = use ? part_o[prow * D + lane * E + e] : 0.0f;
      if (!use) wk[c] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < kMaxParts; ++c) {
      wsum += wk[c];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wk[c], ov[c][e], acc[e]);
    }
  }
  const bool empty = !(wsum > 0.0f);
  const float inv = empty ? 0.0f : 1.0f / wsum;
  const int64_t ob = static_cast<int64_t>(b) * os0 + static_cast<int64_t>(h) * os1 + static_cast<int64_t>(qi) * os2 +
                     lane * E;
  if constexpr (OUT_BF16) {
    uint16_t* dst = static_cast<uint16_t*>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  } else {
    float* dst = static_cast<float*>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) dst[e] = acc[e] * inv;
  }
  if (lse != nullptr && lane == 0)
    lse[(static_cast<int64_t>(b) * Hq + h) * Pq + qi] = empty ? -INFINITY : M + logf(wsum);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The slots of make_tile_map, as attn_tc_kernel reads them.
bool make_map(CUtensorMap* map, TmaCoordMap* cm, const View4& t) {
  int slot[3];
  if (!make_tile_map(map, slot, t, kBM)) return false;
  cm->slot_p = slot[0];
  cm->slot_h = slot[1];
  cm->slot_b = slot[2];
  return true;
}

// A 4-D bf16 tensor map over one paged cache tensor [num_blocks, Hkv, 16, D]
// (contiguous): dims (D, slot, head, block), box 64 columns x 16 slots of one
// head of one block, 128-byte swizzle.
bool make_cache_map(CUtensorMap* map, void* base, int64_t num_blocks, int Hkv, int D) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), 16, static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(16) * D * 2,
                                 static_cast<cuuint64_t>(Hkv) * 16 * D * 2};
  const cuuint32_t box[4] = {64, 16, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// A 4-D bf16 tensor map over a [B, H, P, D] view whose row/head/batch
// strides may come in any order (contiguous or packed [T, H, D]).  The
// three outer dimensions are ordered by increasing stride; slot[0], slot[1]
// and slot[2] receive the coordinate slot (1..3) that carries the row, the
// head and the batch index.  Box: 64 columns x box_rows rows, 128-byte
// swizzle, zero fill outside the tensor.
bool make_tile_map(CUtensorMap* map, int slot[3], const View4& t, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  struct Dim {
    int64_t size, stride;
    int which;  // 0 = row (P), 1 = head, 2 = batch
  } d[3] = {{t.shape[2], t.stride[2], 0}, {t.shape[1], t.stride[1], 1}, {t.shape[0], t.stride[0], 2}};
  // a dimension of extent 1 has no meaningful stride: give it a valid one
  for (auto& x : d)
    if (x.size <= 1) x.stride = int64_t(1) << 30;
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (d[j].stride < d[i].stride || (d[j].stride == d[i].stride && d[j].which < d[i].which)) {
        Dim tmp = d[i];
        d[i] = d[j];
        d[j] = tmp;
      }
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(t.shape[3]), 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {64, 1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 3; ++i) {
    dims[i + 1] = static_cast<cuuint64_t>(d[i].size < 1 ? 1 : d[i].size);
    strides[i] = static_cast<cuuint64_t>(d[i].stride) * 2;
    slot[d[i].which] = i + 1;
    if (d[i].which == 0) box[i + 1] = static_cast<cuuint32_t>(box_rows);
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, t.data, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_bf16_cache_map(CUtensorMap* map, void* base, int64_t num_blocks, int Hkv) {
  return make_cache_map(map, base, num_blocks, Hkv, 128);
}

bool make_code_cache_map(CUtensorMap* map, void* base, int64_t num_blocks, int Hkv) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[4] = {128, 16, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {128, 16 * 128, static_cast<cuuint64_t>(Hkv) * 16 * 128};
  const cuuint32_t box[4] = {128, 16, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

// The setmaxnreg split (the control warpgroup down to Cfg::kRegsCtl
// registers, the two softmax warpgroups up to kRegsSoft) must fit in the
// registers the launch gives the CTA (threads x registers per thread as
// compiled); a split that asks for more would wait forever, so a kernel
// compiled with fewer is never launched.
template <int D, bool SEP, typename Kern>
bool register_split_fits(Kern kern) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return false;
  return 128 * Cfg<D, SEP>::kRegsCtl + 256 * Cfg<D, SEP>::kRegsSoft <= fa.numRegs * kThreads;
}

template <int D, bool OUT_BF16, bool SEP>
cudaError_t launch_tc(const AttnFwdArgs& a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  TcParams p = {};
  if (!make_map(&mq, &p.cq, a.q) || !make_map(&mk, &p.ck, a.k) || !make_map(&mv, &p.cv, a.v))
    return cudaErrorInvalidValue;
  p.Pq = static_cast<int>(a.Pq);
  p.Pk = static_cast<int>(a.Pk);
  p.Hq = static_cast<int>(a.Hq);
  p.group = static_cast<int>(a.Hq / a.Hkv);
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.scale_positive = p.scale_log2 > 0.0f;
  p.mask = a.mask;
  p.mask_stride = a.mask_stride;
  p.key_lens = a.key_lens;
  p.key_bound = a.key_bound;
  p.key_tiles = static_cast<int>((a.Pk + kBN - 1) / kBN);
  p.out = a.out.data;
  p.out_stride[0] = a.out.stride[0];
  p.out_stride[1] = a.out.stride[1];
  p.out_stride[2] = a.out.stride[2];
  p.lse = a.lse;
  p.status = a.status;
  // One CTA per unit (query-tile pair, head, batch); when the units end in a
  // partial wave, the units of that wave are each split into parts over
  // their KV tiles so that the last wave fills the SMs, and merged after.
  const int64_t nq = (a.Pq + 2 * kBM - 1) / (2 * kBM);
  const int64_t units = nq * a.Hq * a.B;
  if (units > 0x7fffffff / 8) return cudaErrorInvalidValue;
  p.nq = static_cast<int>(nq);
  p.full_units = static_cast<int>(units);
  p.split = 1;
  p.part_o = a.part_ws;
  p.part_lse = nullptr;
  const int sms = device_sm_count();
  const int64_t tail = sms > 0 ? units % sms : 0;
  if (a.part_ws != nullptr && units > sms && tail > 0 && tail <= sms / 2) {
    const int64_t kv_tiles = (a.Pk + kBN - 1) / kBN;
    int split = static_cast<int>(sms / tail);
    split = split > 8 ? 8 : split;
    if (split > kv_tiles / 2) split = static_cast<int>(kv_tiles / 2);
    const size_t rows = static_cast<size_t>(tail) * split * (2 * kBM);
    if (split >= 2 && rows * (D + 1) * sizeof(float) <= a.part_bytes) {
      p.full_units = static_cast<int>(units - tail);
      p.split = split;
      p.part_lse = a.part_ws + rows * D;
    }
  }
  auto kern = attn_fwd_tc_kernel<D, OUT_BF16, false, SEP>;
  static const bool regs_fit = register_split_fits<D, SEP>(kern);
  if (!regs_fit) return cudaErrorInvalidConfiguration;
  const int smem = Cfg<D, SEP>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t ctas = p.full_units + (units - p.full_units) * p.split;
  kern<<<static_cast<unsigned>(ctas), kThreads, smem, stream>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.split == 1) return e;
  return launch_split_merge(D, OUT_BF16, p.part_o, p.part_lse, p.split, p.full_units,
                            static_cast<int>(units - p.full_units), p.nq, p.Hq, p.Pq, a.out, a.lse, stream);
}

template <int D, bool OUT_BF16>
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  TcParams p = {};
  if (!make_map(&mq, &p.cq, a.q) || !make_cache_map(&mk, a.cache.k, a.cache.num_blocks, a.cache.Hkv, D) ||
      !make_cache_map(&mv, a.cache.v, a.cache.num_blocks, a.cache.Hkv, D))
    return cudaErrorInvalidValue;
  p.Pq = static_cast<int>(a.T);
  p.Pk = 0;
  p.Hq = static_cast<int>(a.Hq);
  p.group = static_cast<int>(a.Hq / a.cache.Hkv);
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.scale_positive = p.scale_log2 > 0.0f;
  p.bt = a.block_table;
  p.bt_stride = a.bt_stride;
  p.max_blocks = a.max_blocks;
  p.num_blocks = static_cast<int>(a.cache.num_blocks);
  p.start_pos = a.start_pos;
  p.causal = a.causal;
  p.out = a.out.data;
  p.out_stride[0] = a.out.stride[0];
  p.out_stride[1] = a.out.stride[1];
  p.out_stride[2] = a.out.stride[2];
  p.lse = a.lse;
  p.status = a.status;
  auto kern = attn_fwd_tc_kernel<D, OUT_BF16, true, (D == 64)>;
  static const bool regs_fit = register_split_fits<D, (D == 64)>(kern);
  if (!regs_fit) return cudaErrorInvalidConfiguration;
  const int smem = Cfg<D, (D == 64)>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>((a.T + 2 * kBM - 1) / (2 * kBM)), static_cast<unsigned>(a.Hq),
            static_cast<unsigned>(a.B));
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

int device_sm_count() {
  static std::atomic<int> counts[64] = {};  // per device; any thread may fill an entry (same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

size_t split_partial_bytes(int D) {
  // at most one SM's worth of part CTAs per SM, each 2 kBM rows of D + 1 floats
  const size_t sms = static_cast<size_t>(device_sm_count());
  return sms * (2 * kBM) * (static_cast<size_t>(D) + 1) * sizeof(float);
}

cudaError_t launch_split_merge(int D, bool out_bf16, const float* part_o, const float* part_lse, int split,
                               int full_units, int tail, int nq, int Hq, int Pq, const View4& out, float* lse,
                               cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(tail) * (2 * kBM) * 32;
  const unsigned blocks = static_cast<unsigned>((threads + 255) / 256);
  const int64_t s0 = out.stride[0], s1 = out.stride[1], s2 = out.stride[2];
  if (D == 64 && out_bf16)
    split_merge_kernel<64, true><<<blocks, 256, 0, stream>>>(part_o, part_lse, split, full_units, tail, nq, Hq, Pq,
                                                             out.data, s0, s1, s2, lse);
  else if (D == 64)
    split_merge_kernel<64, false><<<blocks, 256, 0, stream>>>(part_o, part_lse, split, full_units, tail, nq, Hq, Pq,
                                                              out.data, s0, s1, s2, lse);
  else if (D == 128 && out_bf16)
    split_merge_kernel<128, true><<<blocks, 256, 0, stream>>>(part_o, part_lse, split, full_units, tail, nq, Hq,
                                                              Pq, out.data, s0, s1, s2, lse);
  else if (D == 128)
    split_merge_kernel<128, false><<<blocks, 256, 0, stream>>>(part_o, part_lse, split, full_units, tail, nq, Hq,
                                                               Pq, out.data, s0, s1, s2, lse);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_tc(const AttnFwdArgs& a, cudaStream_t stream) {
  const bool bf16_out = a.out.dtype == ATTN_BF16;
  if (pair_kernel_applies(a)) {
    // D = 128 without a mask: the CTA-pair kernel, where the device can
    // hold its clusters
    const cudaError_t e = launch_attn_fwd_pair(a, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  if (a.D == 64) {
    // with key bounds: P apart from S and the certified max-free tiles;
    // without: P over S and the optimistic tiles
    if (a.key_bound != nullptr)
      return bf16_out ? launch_tc<64, true, true>(a, stream) : launch_tc<64, false, true>(a, stream);
    return bf16_out ? launch_tc<64, true, false>(a, stream) : launch_tc<64, false, false>(a, stream);
  }
  if (a.D == 128) return bf16_out ? launch_tc<128, true, false>(a, stream) : launch_tc<128, false, false>(a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_paged_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  const bool bf16_out = a.out.dtype == ATTN_BF16;
  if (a.cache.D == 64) return bf16_out ? launch_prefill<64, true>(a, stream) : launch_prefill<64, false>(a, stream);
  if (a.cache.D == 128)
    return bf16_out ? launch_prefill<128, true>(a, stream) : launch_prefill<128, false>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attn
