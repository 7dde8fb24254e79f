// attn_pair.cu -- attention at head_dim 128 on CTA pairs: the tensor cores of
// two SMs multiply as one (tcgen05 cta_group::2, M = 256).
//
// What it computes: the same as attn_tc.cu ("MultiheadAttention fast path
// used 18 GB of VRAM", the SDPA route; "[sglang] ROCm aiter ring attention",
// section 1, the LSE), for calls with no mask tensor, no key lengths and a
// positive scale -- every key in [0, Pk) counts:
//   s_j = scale * q.k_j,  out = sum_j softmax(s)_j v_j,  lse = log sum_j e^{s_j}
// one 128 x 128 score tile per query tile at a time, in tensor memory.
//
// A cluster of two CTAs takes 256 query rows of one (batch, head), as one CTA
// of attn_tc.cu does.  CTA r of the pair holds query tile r (rows 128 r ..)
// and, of every 128-key K/V tile, the half that the pair's products assign to
// it: keys [64 r, 64 r + 64) of K and value dims [64 r, 64 r + 64) of V.  Two
// threads of CTA 0 issue every product for both:
//   S = Q K^T   (M = 256 rows over the pair, N = 128 keys, K = 128 dims)
//   O += P V    (M = 256, N = 128 dims, K = 128 keys, P from each CTA's TMEM)
// and each CTA finds its own 128 rows of S and O in its own TMEM.  Each K/V
// tile is still read once per 256 query rows, but a CTA stages and the
// products read only half of it, and with one query tile per CTA the tensor
// memory holds three score buffers per tile: the next two score tiles are
// computed while the softmax works on the current one.
//
// Per CTA, 256 threads:
//   warps 0, 3  TMA producers: Q_r once and this CTA's halves of K_j (warp
//               0), of V_j (warp 3), each into a ring of its own.
//   warp 1      TMEM: all 512 columns, allocated by the two CTAs together.
//   warps 2, 1  in CTA 0, lane 0 issues every S product (warp 2) and every
//               PV product (warp 1) of the pair, and signals completions to
//               both CTAs' barriers (multicast commit); in CTA 1, lane 0
//               arrives on CTA 0's copy barriers as each of CTA 1's copies
//               lands (Q and K, V), so that CTA 0's barrier completes when
//               both halves are there.
//   warps 4-7   softmax: thread r owns query row r (TMEM lane r), as in
//               attn_tc.cu (optimistic max-free tiles, redone when a row sum
//               fails; lazy rescale of O), P written as bf16 pairs over the
//               first 64 columns of its S buffer; each warp then arrives on
//               CTA 0's p_full.
// TMEM columns: S/P buffers [0,128), [128,256), [256,384); O [384,512).
//
// Every wait is bounded: a hang turns into ATTN_ERR_TIMEOUT, the abort is
// raised in both CTAs, in-flight copies and MMAs are drained, and the pair
// meets at a cluster barrier before the tensor memory is freed.
#include <cuda.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace attn {
namespace {

constexpr int kRows = 128;      // query rows per CTA
constexpr int kKeys = 128;      // keys per K/V tile
constexpr int kD = 128;         // head dim
constexpr int kThreads = 256;
constexpr int kStages = 4;      // K/V ring
constexpr int kSBuf = 3;        // score buffers
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 384;
constexpr float kRescaleMargin = 8.0f;  // as attn_tc.cu: P stays below 2^8

constexpr int kQBox = kRows * 128;        // 64-column box of 128 rows
constexpr int kKHalfBox = (kKeys / 2) * 128;  // 64-column box of 64 key rows
constexpr int kHalfBytes = 16384;          // a CTA's half of a K or V tile
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kQBox;
constexpr int kOffV = kOffK + kStages * kHalfBytes;
constexpr int kOffBar = kOffV + kStages * kHalfBytes;
constexpr int kSmemBytes = kOffBar + 512 + 1024;  // + slack to align the base to 1024

struct Bars {
  // this CTA's copies landed; in CTA 0 also CTA 1's (its relay arrives)
  uint64_t q_full;
  uint64_t k_full[kStages], v_full[kStages];
  uint64_t k_empty[kStages], v_empty[kStages];  // the pair's products are done with the stage
  uint64_t s_full[kSBuf];                       // score buffer holds the next tile
  uint64_t p_full[kSBuf];                       // CTA 0: P written by both CTAs' softmax warps
  uint64_t o_done[kSBuf];                       // the PV product reading buffer b has completed
  uint64_t o_final;                             // every PV product has completed
  uint64_t s_final;                             // every S product has completed
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block outgrew its shared-memory slot");

struct PairParams {
  int Pq, Pk, Hq, group;
  float scale_log2;
  int nq;          // 256-row query blocks per (batch, head)
  int full_units;  // clusters [0, full_units) take one unit each
  int split;       // the rest take one of `split` key parts of a unit
  float* part_o;   // [units past full_units][split][256][128]
  float* part_lse;
  void* out;
  int64_t out_stride[3];  // b, h, row (elements)
  float* lse;
  uint32_t* status;
  int slot_q[3], slot_k[3], slot_v[3];  // tensor-map coordinate slot of (row, head, batch)
};

struct Unit {
  int h, b, q0, part, prow0;
};

__device__ __forceinline__ Unit pair_unit(const PairParams& p, int cl) {
  Unit u;
  u.part = -1;
  u.prow0 = 0;
  int unit = cl;
  if (unit >= p.full_units) {
    const int r = unit - p.full_units;
    unit = p.full_units + r / p.split;
    u.part = r % p.split;
    u.prow0 = r * (2 * kRows);
  }
  u.q0 = (unit % p.nq) * (2 * kRows);
  u.h = (unit / p.nq) % p.Hq;
  u.b = unit / (p.nq * p.Hq);
  return u;
}

__device__ __forceinline__ void map_coords(const int (&slot)[3], int row, int h, int b, int& c1, int& c2, int& c3) {
  c1 = slot[0] == 1 ? row : (slot[1] == 1 ? h : b);
  c2 = slot[0] == 2 ? row : (slot[1] == 2 ? h : b);
  c3 = slot[0] == 3 ? row : (slot[1] == 3 ? h : b);
}

// ---------------------------------------------------------------------------
// cluster and CTA-pair primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
// the shared::cluster address of the same location in CTA `rank`
__device__ __forceinline__ uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// every thread of both CTAs
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on a barrier of the other CTA.  Default (CTA-scope) release: what
// the arrive publishes is tensor memory written before a
// tcgen05.fence::before_thread_sync, or a copy the barrier's transaction
// count already covered -- not generic stores that the other CTA reads.
// (Release at cluster scope measured twice the per-step time.)
__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void store_remote(uint32_t cluster_addr, int v) {
  asm volatile("st.relaxed.cluster.shared::cluster.s32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ bool try_wait_bar(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// The waits of this kernel: bounded, and a timeout raises the abort in both
// CTAs.  Default (CTA-scope) acquire, as for the arrives above; the tensor
// core operations after a wait are ordered by tcgen05.fence::after_thread_sync.
struct Ctx {
  volatile int* abort;
  uint32_t peer_abort;  // the other CTA's abort flag
  uint32_t* status;
};

__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, const Ctx& cx) {
  if (try_wait_bar(bar, parity, 0u)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (try_wait_bar(bar, parity, 200000u)) return true;
    if (*cx.abort) return false;
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      *cx.abort = 1;
      store_remote(cx.peer_abort, 1);
      report(cx.status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void pdrain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!try_wait_bar(bar, parity, 200000u)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
  }
}

__device__ __forceinline__ void tmem_alloc2(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D (+)= A B over the pair: A's rows 128 r .. in CTA r (shared memory, or TMEM
// for mma2_ts), B's N range split between the CTAs at the same shared-memory
// offset, D's rows 128 r .. in CTA r's TMEM
__device__ __forceinline__ void mma2_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// one arrival on the barrier at this offset in both CTAs once every product
// this thread has issued is complete
__device__ __forceinline__ void commit2(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

template <bool OUT_BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PairParams prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();
  const Unit ui = pair_unit(prm, static_cast<int>(cluster_index()));
  const int h = ui.h, b = ui.b, q0 = ui.q0;
  const int g = h / prm.group;
  // this pair's key tiles: [kv0, kv0 + nkv), all of them unless it is a part
  const int n_keys = prm.Pk;
  int kv0 = 0;
  int nkv = (n_keys + kKeys - 1) / kKeys;
  if (ui.part >= 0) {
    const int per = (nkv + prm.split - 1) / prm.split;
    kv0 = min(nkv, ui.part * per);
    nkv = min(nkv, kv0 + per) - kv0;
  }
  const Ctx cx{&bars->abort, peer_addr(&bars->abort, rank ^ 1u), prm.status};

  if (threadIdx.x == 0) {
    // CTA 0's copy barriers also count the arrival of CTA 1's relay
    const uint32_t copies = rank == 0 ? 2 : 1;
    mbar_init(&bars->q_full, copies);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], copies);
      mbar_init(&bars->v_full[s], copies);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 8);  // four softmax warps in each CTA
    }
    for (int i = 0; i < kSBuf; ++i) mbar_init(&bars->o_done[i], 1);
    mbar_init(&bars->o_final, 1);
    mbar_init(&bars->s_final, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc2(&bars->tmem_base, kTmemCols);
    tmem_relinquish2();
  }
  // both CTAs' barriers are initialised before either touches the other's
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ producers
    // warp 0: Q once, then the K halves; warp 3: the V halves.  Two rings,
    // so that neither copy waits for the other's stage to be released.
    const bool is_k = warp == 0;
    int issued = 0;
    if (lane == 0 && nkv > 0) {  // a part with no key tiles loads nothing
      int c1, c2, c3;
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_arrive_expect_tx(&bars->q_full, 2 * kQBox);
        map_coords(prm.slot_q, q0 + static_cast<int>(rank) * kRows, h, b, c1, c2, c3);
        for (int x = 0; x < 2; ++x) tma_load_4d(smem + kOffQ + x * kQBox, &tm_q, &bars->q_full, x * 64, c1, c2, c3);
      } else {
        tma_prefetch_desc(&tm_v);
      }
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        const int key0 = (kv0 + j) * kKeys;
        uint64_t* full = is_k ? &bars->k_full[s] : &bars->v_full[s];
        if (!pwait(is_k ? &bars->k_empty[s] : &bars->v_empty[s], ph ^ 1, cx)) break;
        mbar_arrive_expect_tx(full, kHalfBytes);
        if (is_k) {
          map_coords(prm.slot_k, key0 + static_cast<int>(rank) * (kKeys / 2), g, b, c1, c2, c3);
          for (int x = 0; x < 2; ++x)
            tma_load_4d(smem + kOffK + s * kHalfBytes + x * kKHalfBox, &tm_k, full, x * 64, c1, c2, c3);
        } else {
          map_coords(prm.slot_v, key0, g, b, c1, c2, c3);
          tma_load_4d(smem + kOffV + s * kHalfBytes, &tm_v, full, static_cast<int>(rank) * 64, c1, c2, c3);
        }
        issued = j + 1;
      }
      if (*cx.abort) {
        // let every copy into this CTA's shared memory land before it exits
        if (is_k) pdrain(&bars->q_full, 0);
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
          pdrain(is_k ? &bars->k_full[j % kStages] : &bars->v_full[j % kStages], (j / kStages) & 1);
      }
    }
  } else if (rank == 0 && (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------ MMA issuers
    // warp 2 issues every S product, warp 1 every PV product.  S(j) goes to
    // buffer j % 3, which PV(j - 3) reads P(j - 3) from: products of two
    // threads run in no fixed order, so S(j) waits for PV(j - 3) to complete
    // (the buffer's o_done) -- three tiles ahead of the softmax, off its path.
    if (lane == 0 && warp == 2) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(2 * kRows, kKeys, false, false);
      const uint32_t q_addr = smem_u32(smem + kOffQ);
      bool ok = nkv > 0 && pwait(&bars->q_full, 0, cx);
      for (int j = 0; ok && j < nkv; ++j) {
        const int buf = j % kSBuf;
        const int s = j % kStages;
        if (!pwait(&bars->k_full[s], (j / kStages) & 1, cx) ||
            (j >= kSBuf && !pwait(&bars->o_done[buf], ((j - kSBuf) / kSBuf) & 1, cx))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + kOffK + s * kHalfBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {  // 16 dims = 32 bytes of a 128-byte row
          const uint32_t qa = q_addr + (kk >> 2) * kQBox + (kk & 3) * 32;
          const uint32_t ka = k_addr + (kk >> 2) * kKHalfBox + (kk & 3) * 32;
          mma2_ss(tmem + buf * 128, sdesc_sw128(qa, 16, 1024), sdesc_sw128(ka, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        commit2(&bars->s_full[buf]);
        commit2(&bars->k_empty[s]);
      }
      // every S product complete before the pair may wind down
      commit2(&bars->s_final);
      pdrain(&bars->s_final, 0);
    } else if (lane == 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(2 * kRows, kD, false, true);
      bool ok = nkv > 0;
      for (int j = 0; ok && j < nkv; ++j) {
        const int buf = j % kSBuf;
        const int s = j % kStages;
        if (!pwait(&bars->p_full[buf], (j / kSBuf) & 1, cx) || !pwait(&bars->v_full[s], (j / kStages) & 1, cx)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_u32(smem + kOffV + s * kHalfBytes);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          // 16 keys = 8 TMEM columns of packed P; V is MN-major (d
          // contiguous), this CTA's 64 dims one 128-byte row per key
          mma2_ts(tmem + kColO, tmem + buf * 128 + kk * 8, sdesc_sw128(v_addr + kk * 2048, kHalfBytes, 1024),
                  idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        commit2(&bars->o_done[buf]);
        commit2(&bars->v_empty[s]);
      }
      // completes when every PV product has: O is final in both CTAs
      commit2(&bars->o_final);
      pdrain(&bars->o_final, 0);
    }
  } else if (rank == 1 && (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------ relays
    // warp 2: Q and the K halves, warp 1: the V halves of this CTA
    const bool is_k = warp == 2;
    if (lane == 0 && nkv > 0) {
      bool ok = !is_k || pwait(&bars->q_full, 0, cx);
      if (ok && is_k) arrive_remote(peer_addr(&bars->q_full, 0));
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % kStages;
        if (!pwait(is_k ? &bars->k_full[s] : &bars->v_full[s], (j / kStages) & 1, cx)) break;
        arrive_remote(peer_addr(is_k ? &bars->k_full[s] : &bars->v_full[s], 0));
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;         // TMEM lanes this warp may touch
    const int row = quarter * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float m_run = -INFINITY;  // reference max, log2 units
    float l_run = 0.0f;       // running sum of 2^(x - m_run)
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int buf = j % kSBuf;
      const uint32_t s_col = buf * 128;
      // wait outcomes are made warp-uniform: tcgen05.ld/st need the whole warp
      if (!__all_sync(0xffffffffu, pwait(&bars->s_full[buf], (j / kSBuf) & 1, cx))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
      // the first half of the scores first; the second half is loaded while
      // the fast path exponentiates the first
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_ld32(tmem + lane_addr + s_col + c * 32, sr[c]);
      // keys of this tile that exist: [0, lim) (the tail of the last tile
      // was zero-filled by the copy and must not count)
      const int lim = n_keys - (kv0 + j) * kKeys;
      const bool limited = lim < kKeys;
#pragma unroll
      for (int c = 0; c < 2; ++c) tmem_wait_ld(sr[c]);
#pragma unroll
      for (int c = 2; c < 4; ++c) tmem_ld32(tmem + lane_addr + s_col + c * 32, sr[c]);
      bool second_pending = true;
      auto finish_ld = [&]() {
        if (second_pending) {
#pragma unroll
          for (int c = 2; c < 4; ++c) tmem_wait_ld(sr[c]);
          second_pending = false;
        }
      };
#define SV(c) __uint_as_float(sr[(c) >> 5][(c) & 31])
      float alpha = 1.0f;
      float rs = 0.0f;
      bool done = false;
      // Fast path: exponentiate against the current reference max without a
      // max pass.  Every term is <= 2^64 exactly when the row sum is, which
      // keeps the sums far from fp32 overflow; if some row fails, the warp
      // takes the full path below from the scores still in registers.
      if (__all_sync(0xffffffffu, m_run != -INFINITY)) {
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.0f;
        const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2);
        const uint64_t ng2 = f2_pack(-m_run, -m_run);
        auto fast_loop = [&](auto limit_c) {
          constexpr bool LIMIT = decltype(limit_c)::value;
          // each 32-key chunk of P goes to TMEM as soon as it is computed
          // (chunk c lands on columns 16c..16c+15, whose scores are already
          // in registers)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c == 2) finish_ld();
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
            tmem_st16(tmem + lane_addr + s_col + c * 16, pw);
          }
        };
        if (limited)
          fast_loop(std::integral_constant<bool, true>());
        else
          fast_loop(std::integral_constant<bool, false>());
        rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) + ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
        if (__all_sync(0xffffffffu, rs <= 18446744073709551616.0f)) {  // 2^64; false for NaN
          done = true;
        } else {
          // the P just stored is written over again below, after these
          // stores have landed
          tmem_wait_st();
        }
      }
      if (!done) {
        finish_ld();
        // tile max in log2 units: 8 independent chains of 3-input max
        float mx[8];
        if (!limited) {
          // the max of the raw scores, scaled once (scale > 0)
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = fmaxf(SV(2 * i), SV(2 * i + 1));
#pragma unroll
          for (int c = 16; c < kKeys; c += 2) mx[(c >> 1) & 7] = fmax3(mx[(c >> 1) & 7], SV(c), SV(c + 1));
        } else {
          // logits, keys past the end selected to -inf, in place
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const float x = c < lim ? SV(c) * prm.scale_log2 : -INFINITY;
            sr[c >> 5][c & 31] = __float_as_uint(x);
            mx[(c >> 1) & 7] = fmaxf(mx[(c >> 1) & 7], x);
          }
        }
        float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
        if (!limited) mt *= prm.scale_log2;
        // lazy reference max: move it only when the tile exceeds it by the margin
        if (mt > m_run + kRescaleMargin || (m_run == -INFINITY && mt != -INFINITY)) {
          alpha = fast_exp2(m_run - mt);  // 0 when nothing was seen before
          m_run = mt;
        }
        const float m_sub = (m_run == -INFINITY) ? 0.0f : m_run;
        float rsum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rsum[i] = 0.0f;
        const float neg = -m_sub;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pw[16];
          if (!limited) {
            const uint64_t sc2 = f2_pack(prm.scale_log2, prm.scale_log2), ng2 = f2_pack(neg, neg);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              f2_unpack(ffma2(f2_pack(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), sc2, ng2), x0, x1);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              pw[i >> 1] = pack_bf16x2(p0, p1);
              const int a = (i >> 1) & 3;
              uint64_t acc = f2_pack(rsum[a], rsum[4 + a]);
              f2_unpack(fadd2(acc, f2_pack(p0, p1)), rsum[a], rsum[4 + a]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float p0 = fast_exp2(__uint_as_float(sr[c][i]) - m_sub);  // -inf -> 0
              const float p1 = fast_exp2(__uint_as_float(sr[c][i + 1]) - m_sub);
              pw[i >> 1] = pack_bf16x2(p0, p1);
              rsum[i & 7] += p0;
              rsum[(i + 1) & 7] += p1;
            }
          }
          tmem_st16(tmem + lane_addr + s_col + c * 16, pw);
        }
        rs = ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3])) + ((rsum[4] + rsum[5]) + (rsum[6] + rsum[7]));
      }
#undef SV
      l_run = l_run * alpha + rs;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // O is rescaled once PV(j-1) has completed (and before this warp's
        // p_full lets PV(j) start).  Its buffer's barrier is at most one
        // phase behind: PV(j-4), the previous product on it, completed
        // before S(j-1), which this warp has already read.
        const int pb = (j - 1) % kSBuf;
        if (!__all_sync(0xffffffffu, pwait(&bars->o_done[pb], ((j - 1) / kSBuf) & 1, cx))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + kColO + c * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_addr + kColO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&bars->p_full[buf]);
        else
          arrive_remote(peer_addr(&bars->p_full[buf], 0));
      }
    }

    // ---------------------------------------------------------- epilogue
    if (ok && nkv > 0) {
      ok = __all_sync(0xffffffffu, pwait(&bars->o_final, 0, cx));
      tc_fence_after();
    }
    const int qi = q0 + static_cast<int>(rank) * kRows + row;
    const bool empty = !(l_run > 0.0f);
    const float inv_l = empty ? 0.0f : 1.0f / l_run;
    const int64_t prow = ui.prow0 + static_cast<int>(rank) * kRows + row;  // part rows: normalised f32
    const int64_t obase = ui.part >= 0 ? prow * kD
                                       : static_cast<int64_t>(b) * prm.out_stride[0] +
                                             static_cast<int64_t>(h) * prm.out_stride[1] +
                                             static_cast<int64_t>(qi) * prm.out_stride[2];
#pragma unroll
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t o[32];
      if (ok && nkv > 0) {
        tmem_ld32(tmem + lane_addr + kColO + c * 32, o);
        tmem_wait_ld(o);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0u;
      }
      if (qi < prm.Pq && ok && ui.part >= 0) {
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
    if (qi < prm.Pq && ok && (ui.part >= 0 || prm.lse != nullptr)) {
      const float lse2 = empty ? -INFINITY : (m_run + __log2f(l_run));
      if (ui.part >= 0)
        prm.part_lse[prow] = lse2 * 0.6931471805599453f;
      else
        prm.lse[(static_cast<int64_t>(b) * prm.Hq + h) * prm.Pq + qi] = lse2 * 0.6931471805599453f;
    }
  }

  // neither CTA leaves (nor frees the tensor memory) while the other may
  // still arrive on its barriers or the pair's products may still read it
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem, kTmemCols);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

// clusters of two that fit on the device at once (cached per device; 0 when
// none do, and the caller falls back to the one-CTA kernel)
template <typename Kern>
int pair_slots(Kern kern) {
  static std::atomic<int> slots[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = slots[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = -1;
    }
    if (n <= 0) n = -1;
    slots[dev].store(n, std::memory_order_relaxed);
  }
  return n > 0 ? n : 0;
}

template <bool OUT_BF16>
cudaError_t launch_pair(const AttnFwdArgs& a, cudaStream_t stream) {
  auto kern = attn_fwd_pair_kernel<OUT_BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int slots = pair_slots(kern);
  if (slots == 0) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  PairParams p = {};
  if (!make_tile_map(&mq, p.slot_q, a.q, kRows) || !make_tile_map(&mk, p.slot_k, a.k, kKeys / 2) ||
      !make_tile_map(&mv, p.slot_v, a.v, kKeys))
    return cudaErrorInvalidValue;
  p.Pq = static_cast<int>(a.Pq);
  p.Pk = static_cast<int>(a.Pk);
  p.Hq = static_cast<int>(a.Hq);
  p.group = static_cast<int>(a.Hq / a.Hkv);
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.out = a.out.data;
  p.out_stride[0] = a.out.stride[0];
  p.out_stride[1] = a.out.stride[1];
  p.out_stride[2] = a.out.stride[2];
  p.lse = a.lse;
  p.status = a.status;
  // One cluster per unit (256 query rows of a head and batch); when the
  // units end in a partial wave of clusters, each unit of that wave is split
  // into parts over its key tiles so that the last wave fills the device,
  // and the parts are merged after.
  const int64_t nq = (a.Pq + 2 * kRows - 1) / (2 * kRows);
  const int64_t units = nq * a.Hq * a.B;
  if (units > 0x7fffffff / 16) return cudaErrorInvalidValue;
  p.nq = static_cast<int>(nq);
  p.full_units = static_cast<int>(units);
  p.split = 1;
  p.part_o = a.part_ws;
  p.part_lse = nullptr;
  const int64_t tail = units % slots;
  if (a.part_ws != nullptr && units > slots && tail > 0 && tail <= slots / 2) {
    const int64_t kv_tiles = (a.Pk + kKeys - 1) / kKeys;
    int split = static_cast<int>(slots / tail);
    split = split > 8 ? 8 : split;
    if (split > kv_tiles / 2) split = static_cast<int>(kv_tiles / 2);
    const size_t rows = static_cast<size_t>(tail) * split * (2 * kRows);
    if (split >= 2 && rows * (kD + 1) * sizeof(float) <= a.part_bytes) {
      p.full_units = static_cast<int>(units - tail);
      p.split = split;
      p.part_lse = a.part_ws + rows * kD;
    }
  }
  const int64_t clusters = p.full_units + (units - p.full_units) * p.split;
  kern<<<static_cast<unsigned>(2 * clusters), kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.split == 1) return e;
  return launch_split_merge(kD, OUT_BF16, p.part_o, p.part_lse, p.split, p.full_units,
                            static_cast<int>(units - p.full_units), p.nq, p.Hq, p.Pq, a.out, a.lse, stream);
}

}  // namespace

bool pair_kernel_applies(const AttnFwdArgs& a) {
  return a.D == 128 && a.mask == nullptr && a.key_lens == nullptr && a.scale > 0.0f && a.Pk > 0;
}

cudaError_t launch_attn_fwd_pair(const AttnFwdArgs& a, cudaStream_t stream) {
  if (!pair_kernel_applies(a)) return cudaErrorNotSupported;
  return a.out.dtype == ATTN_BF16 ? launch_pair<true>(a, stream) : launch_pair<false>(a, stream);
}

}  // namespace attn
