// attn_bwd_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) backward pass of DFlash
// block attention for the Kimi K3 MLA head dims (bf16; d_nope = 128, d_rope =
// 64 head-shared, d_v = 128).
//
// Gradients of L = sum dout . out (the forward of KimiK3DFlashAttention on the
// DFlash Kimi K3 draft page, whose draft is trained), per head, with P the
// softmax weights recomputed from the forward's lse and D = dout . out:
//   S = Q K^T,  dP = dO V^T,  dS = P (dP - D)
//   dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO
// Two kernels, each one CTA per tile, 352 threads: warp 0 issues TMA loads,
// warp 1 owns TMEM and issues S (S^T) and the accumulating MMAs, warp 10
// issues dP (dP^T), warps 2..9 do the elementwise work and the epilogue.  The
// elementwise warps are two per TMEM lane quarter (one TMEM lane = one row per
// thread); the two split each tile's 64 columns in halves, so that two warps per
// sub-partition hide each other's latency.  An N = 64 score MMA costs nearly as
// many cycles as an N = 128 one from a single issuing thread; from two threads
// the two streams interleave, and a score buffer is complete once both have
// committed to it.
//
// bwd_dq_tc: a 128-row query tile; Q and dO stay in shared memory and 64-key
// tiles of K and V stream through a three-stage ring.  Per key tile j:
//   S_j = Q K_j^T, dP_j = dO V_j^T   SS MMAs, M = 128, N = 64   (TMEM, two buffers)
//   dS_j (bf16) over S_j's columns once read                    (elementwise warps)
//   dQ += dS_j K_j                   TS MMAs, N = 192: K_j read MN-major over its
//                                    three 64-column panels
// Warp 1 issues S_{j+1} before dQ_j, and warp 10 issues dP_{j+1} once the
// elementwise warps are done with tile j - 1, so the tensor pipe works on the
// next tile while the elementwise warps work on this one.
// TMEM: S buffers [0,64) [64,128), dP buffers [128,192) [192,256), dQ [256,448).
//
// bwd_dkdv_tc: a 128-key tile; K and V stay in shared memory and 64-row tiles
// of Q and dO stream through a three-stage ring.  Per query tile j:
//   S^T_j = K Q_j^T, dP^T_j = V dO_j^T   SS MMAs, M = 128 keys, N = 64 rows
//   P^T_j, dS^T_j (bf16) over S^T_j's columns once read            (elementwise)
//   dV += P^T_j dO_j  (N = 128),  dK += dS^T_j Q_j  (N = 192)       TS MMAs
// S^T has two buffers and dP^T one: warp 10 issues dP^T_{j+1} once the
// elementwise warps have read dP^T_j.  TMEM: S^T [0,64) [64,128), dP^T [128,192),
// dV [192,320), dK [320,512).  The rope columns of dK are this head's share of
// the head-shared k_rope gradient and are added into an fp32 accumulator.
// Column ownership: the two warps of a lane quarter read 32 columns each of a
// 64-column score buffer and write their bf16 results only over their own 32
// columns (a warp's packed results would otherwise land on columns its
// partner has not read yet).  Packed column of key/row r: 32 (r / 32) +
// (r % 32) / 2, plus 16 for dS^T; a 16-wide MMA k-step ks starts at packed
// column 32 (ks / 2) + 8 (ks % 2).
//
// Key (dq) and query (dkdv) tiles that no row-key pair of the CTA's tile sees
// are skipped, by the anchored rule or the dense mask's 128 x 128 tile
// classes.  Every mbarrier wait is bounded; one that runs past its budget
// records DFLASH_ERR_TIMEOUT and the CTA winds down.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

using tc::Ctl;
using tc::kWaitBudgetNs;
using tc::range_bits;

constexpr int kDn = 128, kDr = 64, kDqk = 192, kDv = 128;
constexpr int kThreads = 352;           // warps 0..9 and a second MMA-issuing warp (warp 10)
constexpr uint32_t kElemThreads = 256;  // warps 2..9
constexpr uint32_t kStages = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kP128 = 128 * 128;  // panel: 128 rows x 64 bf16, 128-byte swizzled
constexpr uint32_t kP64 = 64 * 128;    // panel: 64 rows x 64 bf16
constexpr uint32_t kStageBytes = 5 * kP64;  // dq: K (3 panels) + V (2); dkdv: Q (3) + dO (2)
constexpr uint32_t kOffFixed = 0;           // dq: Q (3 x 128 rows) + dO (2); dkdv: K (3) + V (2)
constexpr uint32_t kOffStage = 5 * kP128;
constexpr uint32_t kOffCols = kOffStage + kStages * kStageBytes;  // dkdv: per-warp column data
// Epilogue staging in the idle stage ring: bytes per staged row (the row's bf16
// results + 16 of padding, so that the 32 lanes' row writes spread over the banks).
constexpr uint32_t kStgRow = 336;    // dkdv: 320 (dv + 32 columns of dk_nope, or 96 columns of dk_nope)
constexpr uint32_t kStgRowDq = 208;  // dq: 192 (96 columns)
static_assert(8 * 32 * kStgRow <= kStages * kStageBytes, "epilogue staging fits in the stage ring");
constexpr uint32_t kColWords = 5 * 32;                             // per warp: lse2, D, ctx, nlo, nhi
constexpr uint32_t kOffBar = kOffCols + 8 * kColWords * 4;

enum {
  BAR_FIXED = 0,                          // Q+dO (dq) or K+V (dkdv) landed
  BAR_FULL = 1,                           // kStages: stage landed
  BAR_EMPTY = BAR_FULL + kStages,         // kStages: stage free
  BAR_SP = BAR_EMPTY + kStages,           // 2: scores of buffer b computed (S and dP: two commits)
  BAR_DS = BAR_SP + 2,                    // 2: bf16 operands of buffer b written (256 arrivals)
  BAR_DPFREE = BAR_DS + 2,                // dkdv: dP^T read (256 arrivals)
  BAR_DONE = BAR_DPFREE + 1,              // all accumulating MMAs completed
  BAR_DRAIN = BAR_DONE + 1,
  BAR_DRAIN2 = BAR_DRAIN + 1,             // the second MMA issuer's drain
  kNumBars = BAR_DRAIN2 + 1
};
constexpr uint32_t kOffSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffSlot + 4;
// Tile table (dq: key tiles, dkdv: query tiles): two bit arrays, need and full.
constexpr int kFlagTiles = 16384;  // tiles the table covers
constexpr uint32_t kFlagWords = kFlagTiles / 32;
constexpr uint32_t kOffFlags = (kOffAbort + 4 + 15) & ~15u;
constexpr uint32_t kSmemBytes = kOffFlags + 2 * kFlagWords * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kIdScore = ptx::idesc_bf16_f32(128, 64, 0, 0);  // both K-major
constexpr uint32_t kIdN192 = ptx::idesc_bf16_f32(128, 192, 0, 1);  // B MN-major, three panels
constexpr uint32_t kIdN128 = ptx::idesc_bf16_f32(128, 128, 0, 1);  // B MN-major, two panels

struct BwdTcArgs {
  AttnParams p;
  const float* lse;
  const float* D;
  const void* dout;
  void* dq;
  void* dkn;
  void* dvo;
  float* dkr_acc;
  const int* tile_amax;  // [B, ceil(Q/64)] largest anchor of each 64-row query tile
  const int* tile_amin;  // [B, ceil(Q/64)] smallest anchor of each 64-row query tile
  int nqt64;
  int mask_vec;  // dense: 16-byte mask loads allowed
  int group;     // (batch row, head) pairs per scheduling group
};

// CTA order.  CTAs are dispatched in linear block order; the grid is 1-D over
// groups of `group` (batch row, head) pairs, and inside a group over tile levels
// longest first with the pairs fastest.  Inside a group the longest tiles start
// first (tails are filled by short ones); the group keeps the K/V streams that
// are live at once few enough to stay in L2.  group = 0 keeps the plain order
// (tiles fastest, in index order), which measured faster with dense masks.
// Returns (level, pair); level 0 is the longest tile.
__device__ __forceinline__ int2 cta_place(int group, int ntiles, int zh, bool last_first) {
  const long long L = blockIdx.x;
  if (group == 0) {
    const int tile = (int)(L % ntiles);
    return make_int2(last_first ? ntiles - 1 - tile : tile, (int)(L / ntiles));
  }
  const long long per = (long long)group * ntiles;
  const int grp = (int)(L / per);
  const int g0 = grp * group, gsz = min(group, zh - g0);
  const int r = (int)(L - grp * per);
  return make_int2(r / gsz, g0 + r % gsz);
}

__device__ __forceinline__ int clamp_anchor(const AttnParams& p, long long idx) {
  int a = p.anchors[idx];
  if (a < 0 || a > p.S) {
    record_error(p.err, DFLASH_ERR_INVALID);
    a = a < 0 ? 0 : p.S;
  }
  return a;
}

// Any visible (row, key) pair between query rows [r0, r1) and keys [k0, k1)?
// amax: the largest anchor of those rows (anchored).
__device__ __forceinline__ bool pair_needed(const BwdTcArgs& a, int b, int r0, int r1, int k0, int k1, int amax) {
  const AttnParams& p = a.p;
  if (p.mode == kDense)
    return p.classes[((long long)b * p.nqt + r0 / kTileM) * p.nkt + k0 / kTileN] != DFLASH_TILE_SKIP;
  if (k0 < p.S && k0 < amax) return true;
  const int u0 = p.S + (r0 / p.bs) * p.bs;
  const int u1 = p.S + min(((r1 - 1) / p.bs + 1) * p.bs, p.Q);
  return k0 < u1 && k1 > u0;
}

// The tile table of a CTA: bit i of need says that some (row, key) pair of
// tile i is visible, bit i of full that every pair is.  The table covers the
// first n tiles of the axis; eval(i) works out tile i's flags (bit 0 need, bit
// 1 full) for the tiles past it.  Built once per CTA by all its warps (32 tiles
// per ballot), so that the roles find the next tile they need with a bit scan
// instead of a load per tile.
template <typename Eval>
struct TileTable {
  uint32_t* need;
  uint32_t* full;
  int n, total;
  Eval eval;
  __device__ void build() const {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int base = 32 * warp; base < n; base += blockDim.x) {
      const int i = base + lane;
      const uint32_t f = i < n ? eval(i) : 0u;
      const uint32_t nb = __ballot_sync(0xffffffffu, f & 1u), fb = __ballot_sync(0xffffffffu, (f & 2u) != 0u);
      if (lane == 0) {
        need[base >> 5] = nb;
        full[base >> 5] = fb;
      }
    }
  }
  // First needed tile after t (total when none is left).
  __device__ int next(int t) const {
    for (int i = t + 1; i < n; i = (i | 31) + 1) {
      const uint32_t w = need[i >> 5] >> (i & 31);
      if (w) return i + __ffs(w) - 1;
    }
    for (int i = max(t + 1, n); i < total; ++i)
      if (eval(i) & 1u) return i;
    return total;
  }
  __device__ bool is_full(int i) const { return i < n ? (full[i >> 5] >> (i & 31)) & 1u : (eval(i) & 2u) != 0u; }
};
template <typename Eval>
__device__ __forceinline__ TileTable<Eval> tile_table(uint8_t* base, int n, int total, int cap, Eval eval) {
  uint32_t* need = reinterpret_cast<uint32_t*>(base + kOffFlags);
  return TileTable<Eval>{need, need + kFlagWords, min(min(n, kFlagTiles), cap), total, eval};
}

struct Smem {
  uint8_t* base;
  uint32_t sbase;
  Ctl ctl;
  uint32_t* tmem_slot;
};

__device__ __forceinline__ Smem setup_smem(uint8_t* raw, const AttnParams& p) {
  Smem s;
  s.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.sbase = ptx::smem_u32(s.base);
  s.ctl.bar0 = s.sbase + kOffBar;
  s.ctl.abort = reinterpret_cast<volatile int*>(s.base + kOffAbort);
  s.ctl.err = p.err;
  s.ctl.budget = p.wait_ns;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.base + kOffSlot);
  return s;
}

// Thread 0, first: the barriers (sp_commits: MMA commits that complete a score
// buffer, two since S and dP come from two issuing threads) and the tensor maps.
__device__ __forceinline__ void init_barriers(const Smem& s, const CUtensorMap* m0, const CUtensorMap* m1,
                                              const CUtensorMap* m2, const CUtensorMap* m3, const CUtensorMap* m4,
                                              uint32_t sp_commits) {
  ptx::mbar_init(s.ctl.bar(BAR_FIXED), 1);
  for (uint32_t i = 0; i < kStages; ++i) {
    ptx::mbar_init(s.ctl.bar(BAR_FULL + i), 1);
    ptx::mbar_init(s.ctl.bar(BAR_EMPTY + i), 1);
  }
  for (int i = 0; i < 2; ++i) {
    ptx::mbar_init(s.ctl.bar(BAR_SP + i), sp_commits);
    ptx::mbar_init(s.ctl.bar(BAR_DS + i), kElemThreads);
  }
  ptx::mbar_init(s.ctl.bar(BAR_DPFREE), kElemThreads);
  ptx::mbar_init(s.ctl.bar(BAR_DONE), 1);
  ptx::mbar_init(s.ctl.bar(BAR_DRAIN), 1);
  ptx::mbar_init(s.ctl.bar(BAR_DRAIN2), 1);
  *s.ctl.abort = 0;
  ptx::fence_mbar_init();
  ptx::fence_proxy_async_smem();
  ptx::prefetch_tmap(m0);
  ptx::prefetch_tmap(m1);
  ptx::prefetch_tmap(m2);
  ptx::prefetch_tmap(m3);
  ptx::prefetch_tmap(m4);
}

// All threads, after the tile table is built: TMEM, and the barrier that
// publishes the barriers' initialisation and the table.
__device__ __forceinline__ void init_common(const Smem& s) {
  const int warp = threadIdx.x >> 5;
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(s.tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
}

// The MMA thread's last act: wait (bounded) until every MMA it issued has
// completed, so that TMEM can be released.
__device__ __forceinline__ void drain(const Smem& s, int bar = BAR_DRAIN) {
  ptx::tc_commit(s.ctl.bar(bar));
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(s.ctl.bar(bar), 0)) {
    if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
      record_error(s.ctl.err, DFLASH_ERR_TIMEOUT);
      break;
    }
  }
}

// The TMA thread's last act (also after a timeout): every load it issued -- the
// fixed tiles and at most the last kStages stages -- lands before the CTA exits,
// since a copy still in flight would write into shared memory the CTA no longer
// owns.
__device__ __forceinline__ void loads_landed(const Smem& s, uint32_t stages_issued) {
  s.ctl.wait_landed(BAR_FIXED, 0);
  for (uint32_t i = stages_issued > kStages ? stages_issued - kStages : 0u; i < stages_issued; ++i)
    s.ctl.wait_landed(BAR_FULL + i % kStages, (i / kStages) & 1u);
}

__device__ __forceinline__ void teardown(const Smem& s, uint32_t tmem) {
  ptx::tc_fence_before();
  __syncthreads();
  if ((threadIdx.x >> 5) == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Dense mask term in base-2 units (the forward's clamp of huge finite values).
__device__ __forceinline__ float mask2(float mk) { return mk == -INFINITY ? -INFINITY : fmaxf(mk * kLog2e, -3.0e38f); }

// ============================================================================ dq
template <bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ BwdTcArgs a, const __grid_constant__ CUtensorMap tmQ,
                     const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmKn,
                     const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const AttnParams& p = a.p;
  const Smem s = setup_smem(smem_raw, p);
  const Ctl& ctl = s.ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The last query tiles first: under sorted anchors they see the most context.
  const int nqt128 = (p.Q + 127) / 128;
  const int2 pl = cta_place(a.group, nqt128, p.H * p.B, true);
  const int t = nqt128 - 1 - pl.x, h = pl.y % p.H, b = pl.y / p.H;
  const int S = p.S, Q = p.Q, K = S + Q;
  const int r0 = t * 128, r1 = min(r0 + 128, Q);
  const int nkt = (K + 63) / 64;
  int amax = 0;
  if (!DENSE) {
    const long long ti = (long long)b * a.nqt64 + 2 * t;
    amax = a.tile_amax[ti];
    if (r0 + 64 < Q) amax = max(amax, a.tile_amax[ti + 1]);
  }
  // Per 64-key tile: bit 0 = some (row, key) pair of this query tile and it is
  // visible, bit 1 (dense) = its mask tile is all 0.
  auto tile_flags = [&](int kt) -> uint32_t {
    const uint32_t need = pair_needed(a, b, r0, r1, kt * 64, min(kt * 64 + 64, K), amax) ? 1u : 0u;
    if (!DENSE) return need;
    return need | (p.classes[((long long)b * p.nqt + t) * p.nkt + (kt * 64) / kTileN] == DFLASH_TILE_FULL ? 2u : 0u);
  };
  const uint32_t sQ = s.sbase + kOffFixed, sDO = sQ + 3 * kP128, sSt = s.sbase + kOffStage;
  if (threadIdx.x == 0) {
    init_barriers(s, &tmQ, &tmDO, &tmKn, &tmKr, &tmV, 2);
    // the resident Q and dO need no tile table: they load while it is built
    const int qrow = (int)((long long)b * Q + r0);
    ptx::mbar_arrive_expect_tx(ctl.bar(BAR_FIXED), 5 * kP128);
    for (int pn = 0; pn < 3; ++pn) ptx::tma_load_3d(sQ + pn * kP128, &tmQ, ctl.bar(BAR_FIXED), 64 * pn, h, qrow);
    for (int pn = 0; pn < 2; ++pn) ptx::tma_load_3d(sDO + pn * kP128, &tmDO, ctl.bar(BAR_FIXED), 64 * pn, h, qrow);
  }
  const auto tiles = tile_table(s.base, nkt, nkt, p.flag_tiles, tile_flags);
  tiles.build();

  init_common(s);  // its barrier publishes the barriers and the flags
  const uint32_t tmem = *s.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA
      uint32_t j = 0;
      // (timeout test: the stalled CTA's key tiles never arrive)
      for (int kt = tiles.next(-1); kt < nkt && (int)blockIdx.x != p.stall_cta; kt = tiles.next(kt)) {
        const uint32_t st = j % kStages;
        if (!ctl.wait(BAR_EMPTY + st, ((j / kStages) & 1u) ^ 1u)) break;
        const uint32_t fb = ctl.bar(BAR_FULL + st), dst = sSt + st * kStageBytes;
        const int krow = (int)((long long)b * K + kt * 64);
        ptx::mbar_arrive_expect_tx(fb, kStageBytes);
        ptx::tma_load_3d(dst, &tmKn, fb, 0, h, krow);
        ptx::tma_load_3d(dst + kP64, &tmKn, fb, 64, h, krow);
        ptx::tma_load_2d(dst + 2 * kP64, &tmKr, fb, 0, krow);
        ptx::tma_load_3d(dst + 3 * kP64, &tmV, fb, 0, h, krow);
        ptx::tma_load_3d(dst + 4 * kP64, &tmV, fb, 64, h, krow);
        ++j;
      }
      loads_landed(s, j);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA
      const uint64_t dQd = ptx::smem_desc(sQ, 16, 1024);
      const uint64_t dStK = ptx::smem_desc(sSt, 16, 1024);   // stage, K-major (B of S and dP)
      const uint64_t dStN = ptx::smem_desc(sSt, kP64, 1024);  // stage, MN-major (B of dQ)
      bool ok = ctl.wait(BAR_FIXED, 0);
      auto issue_scores = [&](uint32_t jj) -> bool {
        const uint32_t st = jj % kStages;
        if (!ctl.wait(BAR_FULL + st, (jj / kStages) & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t dS = tmem + 64u * (jj & 1u);
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks) {
          const uint32_t pn = ks >> 2, sub = (ks & 3) * 32;
          ptx::mma_ss(dS, dQd + ((pn * kP128 + sub) >> 4), dStK + ((st * kStageBytes + pn * kP64 + sub) >> 4),
                      kIdScore, ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_SP + (jj & 1u)));
        return true;
      };
      auto issue_dq = [&](uint32_t jj) -> bool {
        const uint32_t st = jj % kStages;
        if (!ctl.wait(BAR_DS + (jj & 1u), (jj >> 1) & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t aS = tmem + 64u * (jj & 1u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)  // 16 keys: 8 packed columns of dS, two 1024-byte row groups of K
          ptx::mma_ts(tmem + 256u, aS + 32u * (ks >> 1) + 8u * (ks & 1), dStN + ((st * kStageBytes + ks * 2048u) >> 4),
                      kIdN192, jj > 0 || ks > 0);
        ptx::tc_commit(ctl.bar(BAR_EMPTY + st));
        return true;
      };
      uint32_t j = 0;
      for (int kt = tiles.next(-1); ok && kt < nkt; kt = tiles.next(kt)) {
        ok = issue_scores(j);
        if (ok && j > 0) ok = issue_dq(j - 1);
        ++j;
      }
      if (ok && j > 0) ok = issue_dq(j - 1);
      if (ok) ptx::tc_commit(ctl.bar(BAR_DONE));
      drain(s);
    }
  } else if (warp == 10) {
    if (lane == 0) {
      // ------------------------------------------------------ second MMA issuer: dP
      const uint64_t dDOd = ptx::smem_desc(sDO, 16, 1024);
      const uint64_t dStK = ptx::smem_desc(sSt, 16, 1024);
      bool ok = ctl.wait(BAR_FIXED, 0);
      uint32_t j = 0;
      for (int kt = tiles.next(-1); ok && kt < nkt; kt = tiles.next(kt)) {
        const uint32_t st = j % kStages;
        if (!ctl.wait(BAR_FULL + st, (j / kStages) & 1u)) break;
        // dP buffer j & 1 is free once the elementwise warps are done with tile j - 2
        if (j > 1 && !ctl.wait(BAR_DS + (j & 1u), ((j - 2) >> 1) & 1u)) break;
        ptx::tc_fence_after();
        const uint32_t dP = tmem + 128u + 64u * (j & 1u);
#pragma unroll
        for (int ks = 0; ks < kDv / 16; ++ks) {
          const uint32_t pn = ks >> 2, sub = (ks & 3) * 32;
          ptx::mma_ss(dP, dDOd + ((pn * kP128 + sub) >> 4),
                      dStK + ((st * kStageBytes + (3 + pn) * kP64 + sub) >> 4), kIdScore, ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_SP + (j & 1u)));
        ++j;
      }
      drain(s, BAR_DRAIN2);
    }
  } else {
    // ------------------------------------------------------------------ elementwise + epilogue
    const int quad = warp & 3;
    const uint32_t half = (uint32_t)(warp - 2) >> 2;  // which 32 of the tile's 64 keys
    const int row = quad * 32 + lane;
    const int i = r0 + row;
    const bool row_ok = i < Q;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    const long long li = ((long long)b * p.H + h) * Q + i;
    const float lse2 = row_ok ? a.lse[li] * kLog2e : 0.f;
    const float Di = row_ok ? a.D[li] : 0.f;
    int ctx = 0, nlo = 0, nhi = 0;
    const __nv_bfloat16* mrow = nullptr;
    if (DENSE) {
      mrow = static_cast<const __nv_bfloat16*>(p.mask) + ((long long)b * Q + (row_ok ? i : 0)) * (long long)K;
    } else if (row_ok) {
      ctx = clamp_anchor(p, (long long)b * p.nb + i / p.bs);
      const int blk = i / p.bs;
      nlo = S + blk * p.bs;
      nhi = S + min(blk * p.bs + p.bs, Q);
    }
    uint32_t j = 0;
    bool ok = true;
    for (int kt = tiles.next(-1); kt < nkt; kt = tiles.next(kt)) {
      const int k0 = kt * 64 + 32 * (int)half;  // this warp's first key
      uint32_t vis = 0;
      bool full_tile = false;  // dense: an all-0 mask tile needs no mask reads
      if (row_ok) {
        if (DENSE) {
          vis = (uint32_t)range_bits(0, K - k0);
          full_tile = tiles.is_full(kt);
        } else {
          vis = (uint32_t)((range_bits(0, ctx - k0) | range_bits(nlo - k0, nhi - k0)) & range_bits(0, K - k0));
        }
      }
      // warp-uniform outcome: the warp's lanes leave the loop together
      if (!__all_sync(0xffffffffu, ctl.wait(BAR_SP + (j & 1u), (j >> 1) & 1u))) {
        ok = false;
        break;
      }
      float mk[32];
      if (DENSE) {
        if (full_tile) {
#pragma unroll
          for (int c = 0; c < 32; ++c) mk[c] = 0.f;
        } else if (a.mask_vec && k0 + 32 <= K) {
          const uint4* mp = reinterpret_cast<const uint4*>(mrow + k0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 w = __ldg(mp + v4);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              mk[v4 * 8 + 2 * u] = __uint_as_float(ws[u] << 16);
              mk[v4 * 8 + 2 * u + 1] = __uint_as_float(ws[u] & 0xFFFF0000u);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int k = k0 + c;
            mk[c] = (row_ok && k < K) ? __bfloat162float(mrow[k]) : -INFINITY;
          }
        }
      }
      ptx::tc_fence_after();
      const uint32_t cS = tmem + lane_off + 64u * (j & 1u), cP = tmem + lane_off + 128u + 64u * (j & 1u);
      uint32_t sx[32], px[32];
      // nothing between the asynchronous TMEM loads and their wait
      ptx::tmem_ld32(cS + 32u * half, sx);
      ptx::tmem_ld32(cP + 32u * half, px);
      ptx::tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float g[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float x = __uint_as_float(sx[c + e]);
          const float m2 = DENSE ? mask2(mk[c + e]) : 0.f;
          const bool v = ((vis >> (c + e)) & 1u) && m2 != -INFINITY;
          const float pr = v ? ptx::ex2(fmaf(x, c2, m2) - lse2) : 0.f;
          g[e] = pr * (__uint_as_float(px[c + e]) - Di);
        }
        pk[c / 2] = ptx::pack_bf16x2(g[0], g[1]);
      }
      ptx::tmem_st16(cS + 32u * half, pk);  // dS (bf16 pairs) over this warp's S columns, already read
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ctl.bar(BAR_DS + (j & 1u)));
      ++j;
    }
    // ---- epilogue: dq = scale * dQ (bf16); each warp of a lane quarter writes 96 of the 192 columns.
    // The rows of a warp lie H * 384 bytes apart in dq: the results are staged in
    // the idle stage ring and written row by row (12 lanes to a row's 192 bytes).
    if (ok && j > 0 && !__all_sync(0xffffffffu, ctl.wait(BAR_DONE, 0))) ok = false;
    if (ok) {
      ptx::tc_fence_after();
      uint8_t* stg = s.base + kOffStage + (uint32_t)(warp - 2) * 32u * kStgRowDq;
#pragma unroll 1
      for (int cc = 96 * (int)half; cc < 96 * (int)half + 96; cc += 32) {
        uint32_t o[32], pk[16];
        if (j > 0) {
          ptx::tmem_ld32(tmem + lane_off + 256u + cc, o);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          pk[e / 2] = ptx::pack_bf16x2(__uint_as_float(o[e]) * p.scale, __uint_as_float(o[e + 1]) * p.scale);
        uint4* dst = reinterpret_cast<uint4*>(stg + lane * kStgRowDq + (cc - 96 * (int)half) * 2);
#pragma unroll
        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
      __syncwarp();
      constexpr int kPieces = 96 / 8;  // 16-byte pieces of a row's 96 columns
      for (int idx = lane; idx < 32 * kPieces; idx += 32) {
        const int r = idx / kPieces, pc = idx % kPieces;
        const int ir = r0 + quad * 32 + r;
        if (ir >= Q) continue;
        __nv_bfloat16* g = static_cast<__nv_bfloat16*>(a.dq) + (((long long)b * Q + ir) * p.H + h) * (long long)kDqk;
        *reinterpret_cast<uint4*>(g + 96 * (int)half + 8 * pc) =
            *reinterpret_cast<const uint4*>(stg + r * kStgRowDq + 16 * pc);
      }
    }
  }
  teardown(s, tmem);
}

// ============================================================================ dk, dv
template <bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ BwdTcArgs a, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmKn,
                       const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  const AttnParams& p = a.p;
  const Smem s = setup_smem(smem_raw, p);
  const Ctl& ctl = s.ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The first key tiles first: under sorted anchors the most query rows see them.
  const int2 pl = cta_place(a.group, (p.S + p.Q + 127) / 128, p.H * p.B, false);
  const int kt = pl.x, h = pl.y % p.H, b = pl.y / p.H;
  const int S = p.S, Q = p.Q, K = S + Q;
  const int k0 = kt * 128, k1 = min(k0 + 128, K);
  const int nqt = a.nqt64;
  // Per 64-row query tile: bit 0 = some (row, key) pair of it and this key tile
  // is visible, bit 1 = every pair is.
  auto tile_flags = [&](int t) -> uint32_t {
    const long long ti = (long long)b * nqt + t;
    const bool whole = t * 64 + 64 <= Q;
    if (DENSE) {
      const uint8_t c = p.classes[((long long)b * p.nqt + (t * 64) / kTileM) * p.nkt + kt];
      return (c != DFLASH_TILE_SKIP ? 1u : 0u) | (whole && k1 <= K && c == DFLASH_TILE_FULL ? 2u : 0u);
    }
    const int amax = a.tile_amax[ti], amin = a.tile_amin[ti];
    return (pair_needed(a, b, t * 64, min(t * 64 + 64, Q), k0, k1, amax) ? 1u : 0u) |
           (whole && k1 <= S && k1 <= amin ? 2u : 0u);
  };
  const uint32_t sK = s.sbase + kOffFixed, sV = sK + 3 * kP128, sSt = s.sbase + kOffStage;
  if (threadIdx.x == 0) {
    init_barriers(s, &tmQ, &tmDO, &tmKn, &tmKr, &tmV, 2);
    // the resident K and V need no tile table: they load while it is built
    const int krow = (int)((long long)b * K + k0);
    ptx::mbar_arrive_expect_tx(ctl.bar(BAR_FIXED), 5 * kP128);
    ptx::tma_load_3d(sK, &tmKn, ctl.bar(BAR_FIXED), 0, h, krow);
    ptx::tma_load_3d(sK + kP128, &tmKn, ctl.bar(BAR_FIXED), 64, h, krow);
    ptx::tma_load_2d(sK + 2 * kP128, &tmKr, ctl.bar(BAR_FIXED), 0, krow);
    ptx::tma_load_3d(sV, &tmV, ctl.bar(BAR_FIXED), 0, h, krow);
    ptx::tma_load_3d(sV + kP128, &tmV, ctl.bar(BAR_FIXED), 64, h, krow);
  }
  const auto tiles = tile_table(s.base, nqt, nqt, p.flag_tiles, tile_flags);
  tiles.build();

  init_common(s);  // its barrier publishes the barriers and the flags
  const uint32_t tmem = *s.tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA
      uint32_t j = 0;
      // (timeout test: the stalled CTA's query tiles never arrive)
      for (int t = tiles.next(-1); t < nqt && (int)blockIdx.x != p.stall_cta; t = tiles.next(t)) {
        const uint32_t st = j % kStages;
        if (!ctl.wait(BAR_EMPTY + st, ((j / kStages) & 1u) ^ 1u)) break;
        const uint32_t fb = ctl.bar(BAR_FULL + st), dst = sSt + st * kStageBytes;
        const int qrow = (int)((long long)b * Q + t * 64);
        ptx::mbar_arrive_expect_tx(fb, kStageBytes);
        for (int pn = 0; pn < 3; ++pn) ptx::tma_load_3d(dst + pn * kP64, &tmQ, fb, 64 * pn, h, qrow);
        for (int pn = 0; pn < 2; ++pn) ptx::tma_load_3d(dst + (3 + pn) * kP64, &tmDO, fb, 64 * pn, h, qrow);
        ++j;
      }
      loads_landed(s, j);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA
      const uint64_t dKd = ptx::smem_desc(sK, 16, 1024), dVd = ptx::smem_desc(sV, 16, 1024);
      const uint64_t dStK = ptx::smem_desc(sSt, 16, 1024);   // Q/dO stage, K-major (B of S^T, dP^T)
      const uint64_t dStN = ptx::smem_desc(sSt, kP64, 1024);  // MN-major (B of dK, dV)
      bool ok = ctl.wait(BAR_FIXED, 0);
      auto wait_stage = [&](uint32_t jj) -> bool {
        if (!ctl.wait(BAR_FULL + jj % kStages, (jj / kStages) & 1u)) return false;
        ptx::tc_fence_after();
        return true;
      };
      auto issue_st = [&](uint32_t jj) {
        const uint32_t st = jj % kStages;
#pragma unroll
        for (int ks = 0; ks < kDqk / 16; ++ks) {
          const uint32_t pn = ks >> 2, sub = (ks & 3) * 32;
          ptx::mma_ss(tmem + 64u * (jj & 1u), dKd + ((pn * kP128 + sub) >> 4),
                      dStK + ((st * kStageBytes + pn * kP64 + sub) >> 4), kIdScore, ks > 0);
        }
      };
      auto issue_acc = [&](uint32_t jj) -> bool {
        const uint32_t st = jj % kStages;
        if (!ctl.wait(BAR_DS + (jj & 1u), (jj >> 1) & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t aP = tmem + 64u * (jj & 1u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {  // 16 query rows per k-step
          const uint32_t boff = (st * kStageBytes + ks * 2048u) >> 4;
          const uint32_t acol = aP + 32u * (ks >> 1) + 8u * (ks & 1);
          ptx::mma_ts(tmem + 192u, acol, dStN + boff + ((3 * kP64) >> 4), kIdN128, jj > 0 || ks > 0);
          ptx::mma_ts(tmem + 320u, acol + 16u, dStN + boff, kIdN192, jj > 0 || ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_EMPTY + st));
        return true;
      };
      // S^T and the accumulating MMAs; warp 10 issues dP^T, so that the two
      // streams of MMAs interleave and neither waits on the other's barrier.
      uint32_t j = 0;
      for (int t = tiles.next(-1); ok && t < nqt; t = tiles.next(t)) {
        if (!wait_stage(j)) {
          ok = false;
          break;
        }
        issue_st(j);
        ptx::tc_commit(ctl.bar(BAR_SP + (j & 1u)));
        if (j > 0 && !issue_acc(j - 1)) {
          ok = false;
          break;
        }
        ++j;
      }
      if (ok && j > 0) ok = issue_acc(j - 1);
      if (ok) ptx::tc_commit(ctl.bar(BAR_DONE));
      drain(s);
    }
  } else if (warp == 10) {
    if (lane == 0) {
      // ------------------------------------------------------ second MMA issuer: dP^T
      const uint64_t dVd = ptx::smem_desc(sV, 16, 1024);
      const uint64_t dStK = ptx::smem_desc(sSt, 16, 1024);
      bool ok = ctl.wait(BAR_FIXED, 0);
      uint32_t j = 0;
      for (int t = tiles.next(-1); ok && t < nqt; t = tiles.next(t)) {
        const uint32_t st = j % kStages;
        if (!ctl.wait(BAR_FULL + st, (j / kStages) & 1u)) break;
        // dP^T has one buffer: the elementwise warps must have read dP^T(j-1)
        if (j > 0 && !ctl.wait(BAR_DPFREE, (j - 1) & 1u)) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kDv / 16; ++ks) {
          const uint32_t pn = ks >> 2, sub = (ks & 3) * 32;
          ptx::mma_ss(tmem + 128u, dVd + ((pn * kP128 + sub) >> 4),
                      dStK + ((st * kStageBytes + (3 + pn) * kP64 + sub) >> 4), kIdScore, ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_SP + (j & 1u)));
        ++j;
      }
      drain(s, BAR_DRAIN2);
    }
  } else {
    // ------------------------------------------------------------------ elementwise + epilogue
    const int quad = warp & 3;
    const uint32_t half = (uint32_t)(warp - 2) >> 2;  // which 32 of the query tile's 64 rows
    const int krow_local = quad * 32 + lane;
    const int k = k0 + krow_local;
    const bool key_ok = k < K;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    // this warp's copy of its 32 query rows' data: lse2, D, ctx, nlo, nhi
    float* cl = reinterpret_cast<float*>(s.base + kOffCols) + (warp - 2) * kColWords;
    float* cD = cl + 32;
    int* cctx = reinterpret_cast<int*>(cl + 64);
    int* cnlo = cctx + 32;
    int* cnhi = cnlo + 32;
    // The per-row data of the next query tile is loaded one tile ahead, so that its
    // memory latency overlaps this tile's work.
    struct RowData {
      float l, d;
      int ctx, lo, hi;
    };
    auto load_row = [&](int t) {
      RowData r{0.f, 0.f, 0, 0, 0};
      const int i = t * 64 + 32 * (int)half + lane;
      if (t < nqt && i < Q) {
        const long long li = ((long long)b * p.H + h) * Q + i;
        r.l = a.lse[li] * kLog2e;
        r.d = a.D[li];
        if (!DENSE) {
          r.ctx = clamp_anchor(p, (long long)b * p.nb + i / p.bs);
          const int blk = i / p.bs;
          r.lo = S + blk * p.bs;
          r.hi = S + min(blk * p.bs + p.bs, Q);
        }
      }
      return r;
    };
    uint32_t j = 0;
    bool ok = true;
    int t = tiles.next(-1);
    RowData nxt = load_row(t);
    for (; t < nqt;) {
      const int t_after = tiles.next(t);
      const int r0 = t * 64 + 32 * (int)half;  // this warp's first query row
      // every (row, key) pair of the 64 x 128 tile visible: no per-pair mask
      const bool full_tile = tiles.is_full(t);
      __syncwarp();
      cl[lane] = nxt.l;
      cD[lane] = nxt.d;
      cctx[lane] = nxt.ctx;
      cnlo[lane] = nxt.lo;
      cnhi[lane] = nxt.hi;
      __syncwarp();
      nxt = load_row(t_after);
      // the warp's 32 rows' lse (base 2) and D, in registers for the element loop
      float nl[32], dd[32];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const float4 x4 = reinterpret_cast<const float4*>(cl)[v];
        const float4 d4 = reinterpret_cast<const float4*>(cD)[v];
        nl[4 * v] = -x4.x;
        nl[4 * v + 1] = -x4.y;
        nl[4 * v + 2] = -x4.z;
        nl[4 * v + 3] = -x4.w;
        dd[4 * v] = d4.x;
        dd[4 * v + 1] = d4.y;
        dd[4 * v + 2] = d4.z;
        dd[4 * v + 3] = d4.w;
      }
      // anchored: which of the warp's 32 rows see this thread's key, as a bit mask
      // worked out before the scores arrive (one short loop, so that the element
      // loop below carries no per-element selection code)
      // (16-byte loads of four rows' bounds, no branches: rows past Q were staged
      // with empty ranges)
      uint32_t vmask = 0xffffffffu;
      if (!DENSE && !full_tile) {
        vmask = 0u;
        if (key_ok) {
          const int4* c4 = reinterpret_cast<const int4*>(cctx);
          const int4* l4 = reinterpret_cast<const int4*>(cnlo);
          const int4* h4 = reinterpret_cast<const int4*>(cnhi);
#pragma unroll 2
          for (int v = 0; v < 8; ++v) {
            const int4 c = c4[v], lo = l4[v], hi = h4[v];
            const uint32_t b0 = (uint32_t)((k < c.x) | ((k >= lo.x) & (k < hi.x)));
            const uint32_t b1 = (uint32_t)((k < c.y) | ((k >= lo.y) & (k < hi.y)));
            const uint32_t b2 = (uint32_t)((k < c.z) | ((k >= lo.z) & (k < hi.z)));
            const uint32_t b3 = (uint32_t)((k < c.w) | ((k >= lo.w) & (k < hi.w)));
            vmask |= (b0 | (b1 << 1) | (b2 << 2) | (b3 << 3)) << (4 * v);
          }
        }
      }
      // dense, partial tile: the warp's 32 rows' mask values at this thread's key
      // (bf16 pairs), loaded before the scores arrive
      uint32_t mpk[16];
      if (DENSE && !full_tile) {
        const uint16_t* mk = static_cast<const uint16_t*>(p.mask) + (long long)b * Q * K + k;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const uint32_t lo = key_ok && r0 + c < Q ? mk[(long long)(r0 + c) * K] : 0xFF80u;
          const uint32_t hi = key_ok && r0 + c + 1 < Q ? mk[(long long)(r0 + c + 1) * K] : 0xFF80u;
          mpk[c / 2] = lo | (hi << 16);
        }
      }
      if (!__all_sync(0xffffffffu, ctl.wait(BAR_SP + (j & 1u), (j >> 1) & 1u))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t cS = tmem + lane_off + 64u * (j & 1u);
      uint32_t sx[32], px[32];
      // tcgen05.ld writes its registers asynchronously: nothing may come between
      // the loads and the wait, or the compiler could copy registers not yet written
      ptx::tmem_ld32(cS + 32u * half, sx);
      ptx::tmem_ld32(tmem + lane_off + 128u + 32u * half, px);
      ptx::tmem_wait_ld();
      // this warp's columns of dP^T(j) are in registers: dP^T(j+1) may overwrite them
      ptx::tc_fence_before();
      ptx::mbar_arrive(ctl.bar(BAR_DPFREE));
      uint32_t pkP[16], pkG[16];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float pr[2], g[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = c + e;
          const float x = __uint_as_float(sx[col]);
          float arg;
          bool vis;
          if (!DENSE) {
            arg = fmaf(x, c2, nl[col]);
            vis = (vmask >> col) & 1u;
          } else if (full_tile) {
            arg = fmaf(x, c2, nl[col]);
            vis = true;
          } else {
            const uint32_t w = mpk[col / 2];
            const float m2 = mask2(__uint_as_float((col & 1) ? (w & 0xFFFF0000u) : (w << 16)));
            vis = m2 != -INFINITY;
            arg = fmaf(x, c2, m2) + nl[col];
          }
          pr[e] = vis ? ptx::ex2(arg) : 0.f;
          g[e] = pr[e] * (__uint_as_float(px[col]) - dd[col]);
        }
        pkP[c / 2] = ptx::pack_bf16x2(pr[0], pr[1]);
        pkG[c / 2] = ptx::pack_bf16x2(g[0], g[1]);
      }
      ptx::tmem_st16(cS + 32u * half, pkP);        // P^T, then dS^T, over this warp's 32 S^T columns
      ptx::tmem_st16(cS + 32u * half + 16u, pkG);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ctl.bar(BAR_DS + (j & 1u)));
      ++j;
      t = t_after;
    }
    // ---- epilogue: dv, dk_nope (bf16), rope share of dk added into the fp32 accumulator.
    // TMEM columns 192.. hold dV (128) then dK (192): ten 32-column chunks, five per warp.
    // A thread holds one key row, and the rows of a warp lie H * 256 bytes apart
    // in dv and dk_nope: the bf16 results are staged in the idle stage ring and
    // written row by row, 16 lanes to a 256-byte row, so that a store covers two
    // rows instead of 32.
    if (ok && j > 0 && !__all_sync(0xffffffffu, ctl.wait(BAR_DONE, 0))) ok = false;
    if (ok) {
      ptx::tc_fence_after();
      uint8_t* stg = s.base + kOffStage + (uint32_t)(warp - 2) * 32u * kStgRow;
      const long long kk = (long long)b * K + (key_ok ? k : 0);
      float4* racc = reinterpret_cast<float4*>(a.dkr_acc + kk * (long long)kDr);
#pragma unroll 1
      for (int cc = 160 * (int)half; cc < 160 * (int)half + 160; cc += 32) {
        uint32_t o[32];
        if (j > 0) {
          ptx::tmem_ld32(tmem + lane_off + 192u + cc, o);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0u;
        }
        if (cc < kDv + kDn) {
          const float sc = cc < kDv ? 1.f : p.scale;
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            pk[e / 2] = ptx::pack_bf16x2(__uint_as_float(o[e]) * sc, __uint_as_float(o[e + 1]) * sc);
          // staged row: half 0 [dv 0..127 | dk_nope 0..31], half 1 [dk_nope 32..127]
          uint4* dst = reinterpret_cast<uint4*>(stg + lane * kStgRow + (cc - 160 * (int)half) * 2);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        } else if (j > 0 && key_ok) {
          const int d0 = cc - kDv - kDn;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            atomicAdd(racc + d0 / 4 + v,
                      make_float4(__uint_as_float(o[4 * v]) * p.scale, __uint_as_float(o[4 * v + 1]) * p.scale,
                                  __uint_as_float(o[4 * v + 2]) * p.scale, __uint_as_float(o[4 * v + 3]) * p.scale));
        }
      }
      __syncwarp();
      // staged bytes [soff, soff + 16 * pieces) of each row -> columns gcol.. of out
      auto put = [&](uint32_t soff, int pieces, void* out, int ld, int gcol) {
        for (int idx = lane; idx < 32 * pieces; idx += 32) {
          const int r = idx / pieces, pc = idx % pieces;
          const int kr = k0 + quad * 32 + r;
          if (kr >= K) continue;
          __nv_bfloat16* g = static_cast<__nv_bfloat16*>(out) + (((long long)b * K + kr) * p.H + h) * (long long)ld;
          *reinterpret_cast<uint4*>(g + gcol + 8 * pc) = *reinterpret_cast<const uint4*>(stg + r * kStgRow + soff + 16 * pc);
        }
      };
      if (half == 0) {
        put(0, kDv / 8, a.dvo, kDv, 0);
        put(2 * kDv, 4, a.dkn, kDn, 0);
      } else {
        put(0, (kDn - 32) / 8, a.dkn, kDn, 32);
      }
    }
  }
  teardown(s, tmem);
}

}  // namespace

bool bwd_tc_supported(int dn, int dr, int dv) { return dn == kDn && dr == kDr && dv == kDv; }

namespace {
// A second stream per host thread and device, with the fork and join events.
// They are created on first use and kept for the life of the process (a
// cudaDeviceReset by the caller invalidates them: later backward calls on that
// thread then fail with DFLASH_ERR_CUDA).
struct Fork {
  bool ok;
  cudaStream_t aux;
  cudaEvent_t join;
};
Fork fork_stream(cudaStream_t stream) {
  struct Aux {
    int dev = -1;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
  };
  constexpr int kMaxDev = 64;
  static thread_local Aux aux[kMaxDev];
  Fork f{false, nullptr, nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return f;
  Aux& x = aux[dev];
  if (x.dev != dev) {
    if (cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess)
      return f;
    x.dev = dev;
  }
  if (cudaEventRecord(x.fork, stream) != cudaSuccess || cudaStreamWaitEvent(x.s, x.fork, 0) != cudaSuccess)
    return f;
  f.ok = true;
  f.aux = x.s;
  f.join = x.join;
  return f;
}
cudaError_t join_stream(const Fork& f, cudaStream_t stream) {
  cudaError_t e = cudaEventRecord(f.join, f.aux);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, f.join, 0);
  return e;
}
}  // namespace

cudaError_t launch_attn_bwd_tc(const AttnParams& p, const float* lse, const void* dout, void* dq, void* dkn,
                               void* dv, const float* D, float* dkr_acc, const int* tile_amax64,
                               const int* tile_amin64, cudaStream_t stream) {
  BwdTcArgs a;
  a.p = p;
  a.lse = lse;
  a.D = D;
  a.dout = dout;
  a.dq = dq;
  a.dkn = dkn;
  a.dvo = dv;
  a.dkr_acc = dkr_acc;
  a.tile_amax = tile_amax64;
  a.tile_amin = tile_amin64;
  a.nqt64 = (p.Q + 63) / 64;
  a.mask_vec = 0;
  if (p.mode == kDense) a.mask_vec = (((uintptr_t)p.mask & 15u) == 0) && ((p.S + p.Q) % 8 == 0);
  const long long q_rows = (long long)p.B * p.Q, kv_rows = (long long)p.B * (p.S + p.Q);
  CUtensorMap q128, do128, kn64, kr64, v64, q64, do64, kn128, kr128, v128;
  if (!make_map_3d(&q128, p.q, q_rows, p.H, kDqk, 128) || !make_map_3d(&do128, dout, q_rows, p.H, kDv, 128) ||
      !make_map_3d(&kn64, p.kn, kv_rows, p.H, kDn, 64) || !make_map_2d(&kr64, p.kr, kv_rows, kDr, 64) ||
      !make_map_3d(&v64, p.v, kv_rows, p.H, kDv, 64) || !make_map_3d(&q64, p.q, q_rows, p.H, kDqk, 64) ||
      !make_map_3d(&do64, dout, q_rows, p.H, kDv, 64) || !make_map_3d(&kn128, p.kn, kv_rows, p.H, kDn, 128) ||
      !make_map_2d(&kr128, p.kr, kv_rows, kDr, 128) || !make_map_3d(&v128, p.v, kv_rows, p.H, kDv, 128))
    return cudaErrorInvalidValue;
  const bool dense = p.mode == kDense;
  auto kdq = dense ? bwd_dq_tc_kernel<true> : bwd_dq_tc_kernel<false>;
  auto kkv = dense ? bwd_dkdv_tc_kernel<true> : bwd_dkdv_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes)) != cudaSuccess)
    return e;
  // Scheduling groups of about three waves of CTAs each.
  const int nsm = sm_count() > 0 ? sm_count() : 148;
  const int zh = p.H * p.B;
  auto group_for = [&](int ntiles) {
    const long long ng = std::max(1LL, ((long long)zh * ntiles + 3LL * nsm / 2) / (3LL * nsm));  // groups, rounded
    return (int)((zh + ng - 1) / ng);
  };
  // dq and dk/dv are independent: dq runs on a second stream (forked from and
  // joined back into the caller's), so that each grid's last, partial wave of
  // CTAs is filled by the other's.
  const Fork fk = fork_stream(stream);
  if (!fk.ok) return cudaErrorUnknown;
  if (p.Q > 0) {
    const int nq = (p.Q + 127) / 128;
    a.group = dense ? 0 : group_for(nq);
    kdq<<<(unsigned)((long long)zh * nq), kThreads, kSmemBytes, fk.aux>>>(a, q128, do128, kn64, kr64, v64);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int nk = (p.S + p.Q + 127) / 128;
  a.group = dense ? 0 : group_for(nk);
  kkv<<<(unsigned)((long long)zh * nk), kThreads, kSmemBytes, stream>>>(a, q64, do64, kn128, kr128, v128);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return join_stream(fk, stream);
}

}  // namespace dflash
