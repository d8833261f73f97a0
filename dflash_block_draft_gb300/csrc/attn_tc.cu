// attn_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) DFlash block attention, sm_103a.
//
// Shapes: bf16 q/k/v with d_nope = 128, d_rope = 64 (head-shared rope key),
// d_v = 128 -- the Kimi K3 MLA head layout of the DFlash draft
// (nemo_automodel.components.speculative.dflash.draft_kimi_k3 page:
// KimiK3DFlashAttention, one K/V per query head; module docstring: the
// qk_rope slice is a head-shared extension of the key, no rotary).
//
// One work item = (segment, pair of adjacent 128-row query tiles, head).  The
// two query tiles ("halves" 0 and 1) share every K/V tile the item loads.  Per
// item the kernel walks the 128-key tiles of [context | noise] that the
// schedule marks FULL or PARTIAL for either half (anchored rule, or the dense
// mask's tile classes) and keeps an online softmax per query row:
//   S_i  = Q_i,nope K_nope^T + Q_i,rope K_rope^T    tcgen05 SS MMAs into TMEM (fp32)
//   P_i  = exp2(S_i * scale * log2 e - m)           softmax warpgroup i, one row per thread
//   O_i += P_i V                                    tcgen05 TS MMAs, P_i (bf16) read from TMEM
//   out = O / l,  lse = (m + log2 l) ln 2
//
// Warp roles (384 threads): warp 0 issues TMA loads, warp 1 owns TMEM, warps 1
// and 2 issue the MMAs of halves 0 and 1 (warp 3 idle), warps 4..7 and 8..11
// are the softmax/epilogue warpgroups of halves 0 and 1.  The first warpgroup
// gives registers back (setmaxnreg 120) so that the softmax warpgroups get 192
// registers a thread: 128*120 + 256*192 = 384*168, the launch budget.  Each
// half's MMAs go out from its own thread in the order
//   QK_i(j) [softmax_i(j)] PV_i(j) QK_i(j+1) ...
// PV_i(j) goes out in two parts: keys 0-63 as soon as the softmax has written
// that half of P (so it runs during the softmax of keys 64-127), then keys
// 64-127 and QK_i(j+1) back to back.  The QKs of the two halves take turns
// (QK_0(j), QK_1(j), QK_0(j+1), ...), so S_1 lands one QK after S_0 and the
// two softmax warpgroups run staggered rather than in step; left free, the
// two issue streams interleave MMA by MMA and both S land together.  Turns on
// whole groups (PV and QK) would let one half's softmax overlap all of the
// other half's MMAs, but then the ring must hold two key tiles per half, more
// than fits next to the two Q tiles.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512);
// P_i (bf16 pairs) overwrites the first 64 columns of S_i once they are read,
// and QK_i(j+1) is issued only after PV_i(j), which the tensor pipe runs in order.
// Shared memory: both Q tiles (96 KB) and a ring of eight 16 KB panels through
// which each key tile streams as five panels, all in the 128-byte-swizzled
// layout TMA writes: K (nope 0-63, nope 64-127, rope) then V (v 0-63,
// v 64-127).  PV runs as N = 128 MMAs, which need the two V panels adjacent;
// for the one tile in eight whose V pair would wrap around the ring's end, the
// tile's panels are stored V first (see v_first).
// The grid is persistent (one CTA per SM); items are dealt in a snake order over
// a longest-first list (query tiles with the most context first).
// Every mbarrier wait is bounded; a wait that runs past its budget records
// DFLASH_ERR_TIMEOUT, raises a CTA abort flag and the CTA winds down.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBM = 128, kBN = 128;
constexpr uint32_t kPanel = kBM * 128;    // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kQBytes = 3 * kPanel;  // per half: nope 0-63, nope 64-127, rope
constexpr uint32_t kRing = 8;             // ring panels
constexpr uint32_t kPanelsPerTile = 5;    // K: 3, V: 2
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = 2 * kQBytes;
constexpr uint32_t kOffBar = kOffRing + kRing * kPanel;

enum {
  BAR_Q_FULL = 0,
  BAR_Q_EMPTY = 1,
  BAR_RING_FULL = 2,                       // kRing
  BAR_RING_EMPTY = BAR_RING_FULL + kRing,  // kRing
  BAR_S_FULL = BAR_RING_EMPTY + kRing,     // 2 (per half)
  BAR_P_LO = BAR_S_FULL + 2,               // 2: P of keys 0-63 written
  BAR_P_HI = BAR_P_LO + 2,                 // 2: P of keys 64-127 written
  BAR_PV_LO = BAR_P_HI + 2,                // 2: PV of keys 0-63 completed
  BAR_QK_TURN = BAR_PV_LO + 2,             // 2: QK_i(g) issued
  BAR_O_FULL = BAR_QK_TURN + 2,            // 2
  BAR_DRAIN = BAR_O_FULL + 2,
  kNumBars = BAR_DRAIN + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;  // S_i at kColS + 128 i, O_i at kColO + 128 i

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
// Register split between the control warpgroup and the softmax warpgroups.
// (104 / 200 removes the anchored softmax's few spilled words, but measured
// about 1 % slower on GB300 than 120 / 192.)
template <bool DENSE>
struct RegSplit {
  static constexpr uint32_t ctl = 120, softmax = 192;
  static_assert(128 * ctl + 256 * softmax == kThreads * kLaunchRegs, "register split");
};
using tc::kWaitBudgetNs;
using tc::Ctl;
using tc::PrepCtx;
using tc::kPrepFull;
using tc::kPrepAnchored;
using tc::kPrepDense;
using tc::kPrepNone;
using tc::max64;
using tc::mask64;

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, kDv, 0, 1);  // P from TMEM, V MN-major (both panels)

// Ring placement of key tile g (counted over the CTA's whole run): its panels
// are ring slots (5g .. 5g+4) mod 8.  Normally K takes the first three and V the
// last two; when those two would be slots 7 and 0, V takes the first two
// instead, so that V always occupies two adjacent slots.
__device__ __forceinline__ bool v_first(uint32_t g) { return (g * kPanelsPerTile + 3u) % kRing == kRing - 1u; }
__device__ __forceinline__ uint32_t k_panel0(uint32_t g) { return g * kPanelsPerTile + (v_first(g) ? 2u : 0u); }
__device__ __forceinline__ uint32_t v_panel0(uint32_t g) { return g * kPanelsPerTile + (v_first(g) ? 0u : 3u); }

struct TcArgs {
  AttnParams p;
  int segments;
  int nqt;      // query tiles per segment (max over segments for ragged)
  int npair;    // ceil(nqt / 2)
  int n_items;  // npair * segments * H
  int mask_vec; // dense: mask rows are 16-byte aligned
  int out_v8;   // out is 32-byte aligned: rows are written with 32-byte stores
  int cls_v16;  // dense: every row of tile classes starts 16-byte aligned
};

struct Item {
  int ok;
  int z, h;
  Seg sg;
  int r0[2], r1[2];
  int amin[2], amax[2];
  bool has[2];
  int nkt;
  const uint8_t* cls[2];
  int ctx_end, noise_begin, noise_end;  // anchored: the pair's non-SKIP tiles are [0,ctx_end) U [noise_begin,noise_end)
};

// DENSE: the kernel reads tile classes of a dense mask (else the anchored rule).
template <bool DENSE>
__device__ __forceinline__ Item decode_item(const TcArgs& a, int idx) {
  Item it;
  const AttnParams& p = a.p;
  const int zh = a.segments * p.H;
  const int pair = a.npair - 1 - idx / zh;  // longest (latest) query tiles first
  const int rem = idx % zh;
  it.z = rem / p.H;
  it.h = rem % p.H;
  it.sg = resolve_segment(p, it.z);
  it.ok = it.sg.ok;
  if (!it.ok) return it;
  const int S = it.sg.S, Qn = it.sg.Q;
  it.nkt = (S + Qn + kBN - 1) / kBN;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = 2 * pair + i;
    it.r0[i] = t * kBM;
    it.has[i] = it.r0[i] < Qn;
    it.r1[i] = min(it.r0[i] + kBM, Qn);
    it.cls[i] = nullptr;
    it.amin[i] = S;
    it.amax[i] = 0;
    if (!it.has[i]) continue;
    if (DENSE) {
      it.cls[i] = p.classes + ((long long)it.z * p.nqt + t) * p.nkt;
    } else {
      // The tile's anchors, eight independent loads at a time (a load-use chain
      // per anchor would cost one memory latency each).
      const int j0 = it.r0[i] / p.bs, j1 = (it.r1[i] - 1) / p.bs;
      const int* ap = p.anchors + it.sg.anc0;
      for (int jb = j0; jb <= j1; jb += 8) {
        int an[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) an[u] = __ldg(ap + min(jb + u, j1));
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = an[u] < 0 ? 0 : (an[u] > S ? S : an[u]);
          it.amin[i] = min(it.amin[i], c);
          it.amax[i] = max(it.amax[i], c);
        }
      }
    }
  }
  it.ok = it.has[0];
  if (it.ok && !DENSE) {
    // Context keys some row sees: k < max anchor.  Noise keys some row sees: the
    // blocks of the pair's rows, [blk(first row) * bs, (blk(last row) + 1) * bs) within Q.
    const int amax = max(it.amax[0], it.has[1] ? it.amax[1] : 0);
    const int last = it.has[1] ? it.r1[1] : it.r1[0];
    const int u0 = (it.r0[0] / p.bs) * p.bs;
    const int u1 = min(((last - 1) / p.bs + 1) * p.bs, Qn);
    it.ctx_end = (min(amax, S) + kBN - 1) / kBN;
    it.noise_begin = (S + u0) / kBN;
    it.noise_end = (S + u1 + kBN - 1) / kBN;
  }
  return it;
}

// Next key tile after kt that either half needs (it.nkt when none is left).
template <bool DENSE>
__device__ __forceinline__ int next_tile(const TcArgs& a, const Item& it, int kt) {
  ++kt;
  if (!DENSE) {
    if (kt < it.ctx_end) return kt;
    kt = max(kt, it.noise_begin);
    return kt < it.noise_end ? kt : it.nkt;
  }
  // SKIP is 0, so a run of skipped tiles is a run of zero bytes in both halves'
  // class rows: look at 16 tiles per load once the index is 16-aligned (a tile
  // at a time would cost one dependent load per skipped tile).
  const uint8_t* c0 = it.cls[0];
  const uint8_t* c1 = it.has[1] ? it.cls[1] : it.cls[0];
  for (; kt < it.nkt && (!a.cls_v16 || (kt & 15)); ++kt)
    if ((__ldg(c0 + kt) | __ldg(c1 + kt)) != DFLASH_TILE_SKIP) return kt;
  for (; kt + 16 <= it.nkt; kt += 16) {
    const uint4 w0 = __ldg(reinterpret_cast<const uint4*>(c0 + kt));
    const uint4 w1 = __ldg(reinterpret_cast<const uint4*>(c1 + kt));
    const uint32_t w[4] = {w0.x | w1.x, w0.y | w1.y, w0.z | w1.z, w0.w | w1.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (w[u]) return kt + 4 * u + (__ffs(w[u]) - 1) / 8;
  }
  for (; kt < it.nkt; ++kt)
    if ((__ldg(c0 + kt) | __ldg(c1 + kt)) != DFLASH_TILE_SKIP) return kt;
  return it.nkt;
}

// Class of tile kt for the query tile of one half, from that half's scalars.
template <bool DENSE>
__device__ __forceinline__ int half_class(const TcArgs& a, const Seg& sg, bool has, int r0, int r1, int amin,
                                          int amax, const uint8_t* cls, int kt) {
  if (!has) return DFLASH_TILE_SKIP;
  if (DENSE) return cls[kt];
  return anchored_tile_class(sg.S, sg.Q, a.p.bs, r0, r1, amin, amax, kt);
}

// Item index of this CTA's round k (snake order over the longest-first list).
__device__ __forceinline__ int item_of_round(int k) {
  const int G = gridDim.x;
  return k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
}

template <bool DENSE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap tmQ,
                   const __grid_constant__ CUtensorMap tmKn, const __grid_constant__ CUtensorMap tmKr,
                   const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& p = a.p;

  Ctl ctl;
  ctl.bar0 = sbase + kOffBar;
  ctl.abort = reinterpret_cast<volatile int*>(smem + kOffAbort);
  ctl.err = p.err;
  ctl.budget = p.wait_ns;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ctl.bar(BAR_Q_FULL), 1);
    ptx::mbar_init(ctl.bar(BAR_Q_EMPTY), 2);  // both MMA issuers
    for (uint32_t s = 0; s < kRing; ++s) {
      ptx::mbar_init(ctl.bar(BAR_RING_FULL + s), 1);
      ptx::mbar_init(ctl.bar(BAR_RING_EMPTY + s), 2);  // both MMA issuers
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ctl.bar(BAR_S_FULL + i), 1);
      ptx::mbar_init(ctl.bar(BAR_P_LO + i), 128);
      ptx::mbar_init(ctl.bar(BAR_P_HI + i), 128);
      ptx::mbar_init(ctl.bar(BAR_PV_LO + i), 1);
      ptx::mbar_init(ctl.bar(BAR_QK_TURN + i), 1);
      ptx::mbar_init(ctl.bar(BAR_O_FULL + i), 1);
    }
    ptx::mbar_init(ctl.bar(BAR_DRAIN), 2);  // both MMA issuers
    *ctl.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmKn);
    ptx::prefetch_tmap(&tmKr);
    ptx::prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t ring = sbase + kOffRing;
  if (warp < 4) ptx::setmaxnreg_dec<RegSplit<DENSE>::ctl>();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pc = 0, n_items = 0;  // ring panel counter, items loaded
      bool stop = false;
      for (int k = 0; !stop && k * (int)gridDim.x < a.n_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= a.n_items) continue;
        const Item it = decode_item<DENSE>(a, idx);
        if (!it.ok) continue;
        if (n_items > 0 && !ctl.wait(BAR_Q_EMPTY, (n_items - 1) & 1u)) break;
        ptx::mbar_arrive_expect_tx(ctl.bar(BAR_Q_FULL), 2 * kQBytes);
        for (int i = 0; i < 2; ++i) {
          const int qrow = (int)(it.sg.q0 + it.r0[i]);
          for (int pn = 0; pn < 3; ++pn)
            ptx::tma_load_3d(sbase + kOffQ + i * kQBytes + pn * kPanel, &tmQ, ctl.bar(BAR_Q_FULL), 64 * pn, it.h,
                             qrow);
        }
        ++n_items;
        if ((int)blockIdx.x == p.stall_cta) break;  // timeout test: this item's key tiles never arrive
        for (int kt = next_tile<DENSE>(a, it, -1); kt < it.nkt && !stop; kt = next_tile<DENSE>(a, it, kt)) {
          const int krow = (int)(it.sg.kv0 + (long long)kt * kBN);
          const bool vf = v_first(pc / kPanelsPerTile);
          for (uint32_t pn = 0; pn < kPanelsPerTile; ++pn, ++pc) {
            const uint32_t s = pc % kRing;
            if (!ctl.wait(BAR_RING_EMPTY + s, ((pc / kRing) & 1u) ^ 1u)) {
              stop = true;
              break;
            }
            const uint32_t dst = ring + s * kPanel;
            const uint32_t fb = ctl.bar(BAR_RING_FULL + s);
            ptx::mbar_arrive_expect_tx(fb, kPanel);
            // role: 0, 1 k_nope halves; 2 k_rope; 3, 4 v halves
            const uint32_t role = vf ? (pn < 2 ? pn + 3 : pn - 2) : pn;
            if (role < 2) ptx::tma_load_3d(dst, &tmKn, fb, 64 * role, it.h, krow);
            else if (role == 2) ptx::tma_load_2d(dst, &tmKr, fb, 0, krow);
            else ptx::tma_load_3d(dst, &tmV, fb, 64 * (role - 3), it.h, krow);
          }
        }
      }
      // Wind-down (also after a timeout): every load this thread issued lands
      // before the CTA exits, since a copy still in flight would write into
      // shared memory the CTA no longer owns.  The last kRing panels and the
      // last Q load are the only ones that can still be outstanding.
      for (uint32_t i = pc > kRing ? pc - kRing : 0u; i < pc; ++i)
        ctl.wait_landed(BAR_RING_FULL + i % kRing, (i / kRing) & 1u);
      if (n_items > 0) ctl.wait_landed(BAR_Q_FULL, (n_items - 1) & 1u);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the MMAs of half 0, warp 2 those of half 1, each in its own
    // order  PV_i(j-1) QK_i(j) PV_i(j) QK_i(j+1) ...  so that a late softmax of one
    // half never holds back the other half's MMAs.  Ring panels and the Q buffer
    // are released when both halves have committed (their barriers count 2).
    if (lane == 0) {
      const int i = warp - 1;
      uint32_t g = 0, n_items = 0;  // global tile counter, items started
      auto panel_ready = [&](uint32_t pcx) -> bool {
        return ctl.wait(BAR_RING_FULL + pcx % kRing, (pcx / kRing) & 1u);
      };
      auto release = [&](uint32_t pcx) { ptx::tc_commit(ctl.bar(BAR_RING_EMPTY + pcx % kRing)); };
      // Descriptors are built once; a k-step only adds its byte offset >> 4 to the
      // start-address field (every operand lies below 256 KB, so the 14-bit field
      // never carries).
      const uint64_t dq = ptx::smem_desc(sbase + kOffQ + i * kQBytes, 16, 1024);
      const uint64_t dRingK = ptx::smem_desc(ring, 16, 1024);
      const uint64_t dRingV = ptx::smem_desc(ring, kPanel, 1024);
      const uint32_t d_s = tmem + kColS + 128u * i;  // S_i; P_i aliases its head
      const uint32_t d_o = tmem + kColO + 128u * i;
      auto issue_qk = [&](uint32_t gg) {
        const uint32_t s0 = k_panel0(gg);
#pragma unroll
        for (int ks = 0; ks < (kDn + kDr) / 16; ++ks) {
          const uint32_t pn = (uint32_t)(ks >> 2), sub = (uint32_t)(ks & 3) * 32u;
          const uint32_t kslot = (s0 + pn) % kRing;
          ptx::mma_ss(d_s, dq + ((pn * kPanel + sub) >> 4), dRingK + ((kslot * kPanel + sub) >> 4), kIdescQK, ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_S_FULL + i));
      };
      auto issue_pv = [&](uint32_t gg, bool first, int ks0) {
        const uint64_t dv = dRingV + (((v_panel0(gg) % kRing) * kPanel) >> 4);
#pragma unroll
        for (int ks = ks0; ks < ks0 + kBN / 32; ++ks) {
          // 16 keys: 8 packed P columns; V rows: two 1024-byte groups of 8 keys;
          // the 128 output columns span both V panels (LBO = one panel)
          ptx::mma_ts(d_o, d_s + (uint32_t)ks * 8u, dv + (((uint32_t)ks * 2048u) >> 4), kIdescPV,
                      !(first && ks == 0));
        }
      };
      // Waits for tile gg's V panels and P_i (the panels are normally in place long
      // before P_i, so that the MMAs go out right after P_i arrives).
      auto pv_ready = [&](uint32_t gg) -> bool {
        const uint32_t vp = v_panel0(gg);
        return panel_ready(vp) && panel_ready(vp + 1) && ctl.wait(BAR_P_LO + i, gg & 1u);
      };
      // PV of keys 0-63, then (once the softmax has written it) of keys 64-127.
      auto pv_issue = [&](uint32_t gg, bool first) -> bool {
        const uint32_t vp = v_panel0(gg);
        issue_pv(gg, first, 0);
        ptx::tc_commit(ctl.bar(BAR_PV_LO + i));
        if (!ctl.wait(BAR_P_HI + i, gg & 1u)) return false;
        ptx::tc_fence_after();
        issue_pv(gg, false, kBN / 32);
        release(vp);
        release(vp + 1);
        return true;
      };
      bool stop = false;
      for (int k = 0; !stop && k * (int)gridDim.x < a.n_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= a.n_items) continue;
        const Item it = decode_item<DENSE>(a, idx);
        if (!it.ok) continue;
        if (!ctl.wait(BAR_Q_FULL, n_items & 1u)) break;
        ++n_items;
        int kt = next_tile<DENSE>(a, it, -1);
        if (kt >= it.nkt) {  // nothing visible for this pair of query tiles
          ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));
          continue;
        }
        bool first_tile = true, first_pv = true;
        for (;;) {
          const int kn = next_tile<DENSE>(a, it, kt);
          const uint32_t kp = k_panel0(g);  // first K panel of tile g
          // The K panels never wait on this half's PV of tile g-1: the ring slots they
          // reuse were freed by MMAs of tiles g-2 and earlier, or by QK of tile g-1.
          if (!panel_ready(kp) || !panel_ready(kp + 1) || !panel_ready(kp + 2) || (!first_tile && !pv_ready(g - 1))) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          if (!first_tile) {
            if (!pv_issue(g - 1, first_pv)) {
              stop = true;
              break;
            }
            first_pv = false;
          }
          // QK of half 1 after QK of half 0 of the same tile, QK of half 0 after QK of
          // half 1 of the previous tile: S_1 lands one QK after S_0, so the two
          // softmax warpgroups start apart instead of together.
          if (i == 1 ? !ctl.wait(BAR_QK_TURN + 0, g & 1u) : (g > 0 && !ctl.wait(BAR_QK_TURN + 1, (g - 1) & 1u))) {
            stop = true;
            break;
          }
          issue_qk(g);
          ptx::mbar_arrive(ctl.bar(BAR_QK_TURN + i));
          release(kp);
          release(kp + 1);
          release(kp + 2);
          first_tile = false;
          ++g;
          if (kn >= it.nkt) break;
          kt = kn;
        }
        if (stop) break;
        ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));  // every QK of this half has been issued
        if (!pv_ready(g - 1)) break;  // PV of the item's last tile
        ptx::tc_fence_after();
        if (!pv_issue(g - 1, first_pv)) break;
        ptx::tc_commit(ctl.bar(BAR_O_FULL + i));
      }
      // Drain: every MMA this thread issued has finished before TMEM is released.
      ptx::tc_commit(ctl.bar(BAR_DRAIN));
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(ctl.bar(BAR_DRAIN), 0)) {
        if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
          record_error(ctl.err, DFLASH_ERR_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue (warps 4..11)
    ptx::setmaxnreg_inc<RegSplit<DENSE>::softmax>();
    const int half = (warp - 4) >> 2;  // query tile of the pair
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_col = tmem + lane_off + kColS + 128u * half;
    const uint32_t o_col = tmem + lane_off + kColO + 128u * half;
    const float c2 = p.scale_log2;
    uint32_t g = 0, n_full = 0;
    bool stop = false;
    for (int k = 0; !stop && k * (int)gridDim.x < a.n_items; ++k) {
      const int idx = item_of_round(k);
      if (idx >= a.n_items) continue;
      const Item it = decode_item<DENSE>(a, idx);
      if (!it.ok) continue;
      // this half's scalars (selected, so that the item's arrays stay in registers)
      const bool h_has = half ? it.has[1] : it.has[0];
      const int h_r0 = half ? it.r0[1] : it.r0[0], h_r1 = half ? it.r1[1] : it.r1[0];
      const int h_amin = half ? it.amin[1] : it.amin[0], h_amax = half ? it.amax[1] : it.amax[0];
      const uint8_t* h_cls = half ? it.cls[1] : it.cls[0];
      const int i = h_r0 + row;
      const bool row_ok = h_has && i < h_r1;
      const int S = it.sg.S, Qn = it.sg.Q, K = S + Qn;
      // The row's output and lse addresses, resolved once (fewer live registers
      // across the tile loop).
      uint4* out_dst = row_ok ? reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                         ((it.sg.q0 + i) * p.H + it.h) * (long long)kDv)
                              : nullptr;
      float* lse_dst = row_ok && p.lse ? p.lse + it.sg.lse0 + (long long)it.h * it.sg.lse_hs + i : nullptr;
      int ctx_lim = 0, nlo = 0, nhi = 0;
      const __nv_bfloat16* mrow = nullptr;
      if (DENSE) {
        mrow = static_cast<const __nv_bfloat16*>(p.mask) + ((long long)it.z * p.Q + (row_ok ? i : 0)) * (long long)K;
      } else if (row_ok) {
        ctx_lim = row_anchor(p, it.sg, i);
        const int blk = i / p.bs;
        nlo = S + blk * p.bs;
        nhi = S + min(blk * p.bs + p.bs, Qn);
      }
      float m_used = -INFINITY, l = 0.f;
      bool any_tile = false;
      int kt = next_tile<DENSE>(a, it, -1);
      int cls = kt < it.nkt ? half_class<DENSE>(a, it.sg, h_has, h_r0, h_r1, h_amin, h_amax, h_cls, kt) : 0;
      while (kt < it.nkt) {
        any_tile = true;
        // With a dense mask the next tile and its class are loads of tile-class
        // bytes: they are looked up before the wait for this tile's scores, so that
        // their latency overlaps the wait instead of following this tile (the
        // anchored schedule is arithmetic and is evaluated after the tile).
        int kn = 0, cls_n = 0;
        if (DENSE) {
          kn = next_tile<DENSE>(a, it, kt);
          cls_n = kn < it.nkt ? half_class<DENSE>(a, it.sg, h_has, h_r0, h_r1, h_amin, h_amax, h_cls, kn) : 0;
        }
        const int k0 = kt * kBN;
        // How this row treats the tile: plain scores, anchored mask, dense mask, or
        // nothing.  A FULL tile that runs past the segment's last key still needs the
        // per-key test: the columns past S+Q hold the next segment's keys.
        int kind;
        if (!row_ok || cls == DFLASH_TILE_SKIP) kind = kPrepNone;
        else if (cls == DFLASH_TILE_FULL && k0 + kBN <= K) kind = kPrepFull;
        else kind = DENSE ? kPrepDense : kPrepAnchored;
        const PrepCtx pc{ctx_lim - k0, nlo - k0, nhi - k0, mrow ? mrow + k0 : nullptr, K - k0,
                         a.mask_vec != 0, c2};
        if (kind == kPrepDense) {
          // The row's 256 mask bytes of this tile go to L1 while S is computed.
          const char* mp = reinterpret_cast<const char*>(pc.mask);
          const int span = min(K - k0, kBN) * 2;
          ptx::prefetch_l1(mp);
          ptx::prefetch_l1(mp + min(128, span - 1));
          ptx::prefetch_l1(mp + span - 1);
        }
        // Waits feeding warp-collective TMEM accesses are made warp-uniform: a
        // timeout seen by one lane stops the whole warp.
        if (!__all_sync(0xffffffffu, ctl.wait(BAR_S_FULL + half, g & 1u))) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        // One TMEM read per 64-column half.  p = exp2(x - m) uses the running
        // reference m (base-2 units) and is packed to bf16 pairs (lower key in the
        // low half) over the first 64 columns of S, which are already read.  Only
        // when a half's maximum exceeds m by more than 2^8 -- always on the row's
        // first visible scores, rarely afterwards -- does m move; everything built
        // with the old m is then scaled by alpha = exp2(m_old - m_new): O and l.
        // P of keys 0-63 is handed to the MMA issuer as soon as it is written, so
        // that PV of those keys runs while the second half is computed; a rescale
        // in the second half therefore waits for that PV and scales O after it.
        // (At the first half, PV of the previous tile has completed: it was
        // issued before this tile's QK.)
        const bool scaled = kind == kPrepDense;  // dense scores are already in base-2 units
        const float cm = scaled ? 1.f : c2;
        float2 lsum = make_float2(0.f, 0.f);
        // The anchored kernel keeps one copy of the half's code (a smaller
        // instruction-cache footprint: the unrolled loop measured 2 % slower); with
        // a dense mask the unrolled form lets the second half's mask loads start early.
#pragma unroll(DENSE ? 2 : 1)
        for (int hh = 0; hh < 2; ++hh) {
          float x[64];
          ptx::tmem_ld32(s_col + 64u * hh, reinterpret_cast<uint32_t*>(x));
          ptx::tmem_ld32(s_col + 64u * hh + 32u, reinterpret_cast<uint32_t*>(x) + 32);
          ptx::tmem_wait_ld();
          mask64<DENSE>(x, kind, 64 * hh, pc);
          const float mh = max64(x) * cm;
          const bool raise = mh > m_used + 8.0f;  // also when m is still -inf and this half sees a key
          const bool scale_o = raise && m_used != -INFINITY;
          // O is rescaled by whole warps (TMEM loads and stores are warp-collective):
          // lanes whose reference did not move scale by 1.
          if (__any_sync(0xffffffffu, scale_o)) {
            const float alpha = scale_o ? ptx::ex2(m_used - mh) : 1.f;
            // the second half: O may still be taking PV of keys 0-63 (P written
            // with the old reference); scale O once that has completed
            if (hh == 1 && !__all_sync(0xffffffffu, ctl.wait(BAR_PV_LO + half, g & 1u))) stop = true;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < kDv; cc += 32) {
              uint32_t o[32];
              ptx::tmem_ld32(o_col + cc, o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              ptx::tmem_st32(o_col + cc, o);
            }
            ptx::tmem_wait_st();
            l *= alpha;
            lsum.x *= alpha;
            lsum.y *= alpha;
          }
          if (raise) m_used = mh;
          const float msub = m_used == -INFINITY ? 0.f : m_used;
          const float2 mul2 = make_float2(cm, cm), neg2 = make_float2(-msub, -msub);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float2 arg = __ffma2_rn(make_float2(x[c], x[c + 1]), mul2, neg2);
            const float2 pp = make_float2(ptx::ex2(arg.x), ptx::ex2(arg.y));
            lsum = __fadd2_rn(lsum, pp);
            pk[c / 2] = ptx::pack_bf16x2(pp.x, pp.y);
          }
          ptx::tmem_st32(s_col + 32u * hh, pk);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(ctl.bar((hh == 0 ? BAR_P_LO : BAR_P_HI) + half));
        }
        if (stop) break;
        l += lsum.x + lsum.y;
        ++g;
        if (!DENSE) {
          kn = next_tile<DENSE>(a, it, kt);
          cls_n = kn < it.nkt ? half_class<DENSE>(a, it.sg, h_has, h_r0, h_r1, h_amin, h_amax, h_cls, kn) : 0;
        }
        kt = kn;
        cls = cls_n;
      }
      if (stop) break;
      // ---- epilogue: out = O / l (bf16, round to nearest even), lse = (m + log2 l) ln 2
      uint32_t ob[kDv / 2];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (any_tile) {
        if (!__all_sync(0xffffffffu, ctl.wait(BAR_O_FULL + half, n_full & 1u))) break;
        ++n_full;
        ptx::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kDv; cc += 32) {
          uint32_t o[32];
          ptx::tmem_ld32(o_col + cc, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            ob[(cc + e) / 2] = ptx::pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kDv / 2; ++e) ob[e] = 0u;
      }
      if (row_ok) {
        uint4* dst = out_dst;
        if (a.out_v8) {
          // a row is 256 contiguous bytes: eight 32-byte stores (a sector each)
#pragma unroll
          for (int v = 0; v < kDv / 16; ++v) ptx::st_global_v8(dst + 2 * v, ob + 8 * v);
        } else {
#pragma unroll
          for (int v = 0; v < kDv / 8; ++v) dst[v] = make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]);
        }
        if (lse_dst) *lse_dst = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool make_map_3d(CUtensorMap* m, const void* base, long long rows, int heads, int width, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * heads};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d_box(CUtensorMap* m, const void* base, const unsigned long long dims[3],
                     const unsigned long long strides_bytes[2], const unsigned box[3]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, const void* base, long long rows, int width, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool tc_supported(int dn, int dr, int dv) { return dn == kDn && dr == kDr && dv == kDv; }

cudaError_t launch_attn_tc(const AttnParams& p, int segments, int nqt, long long q_rows, long long kv_rows,
                           cudaStream_t stream) {
  TcArgs a;
  a.p = p;
  a.segments = segments;
  a.nqt = nqt;
  a.npair = (nqt + 1) / 2;
  a.n_items = a.npair * segments * p.H;
  a.mask_vec = 0;
  if (p.mode == kDense) a.mask_vec = (((uintptr_t)p.mask & 15u) == 0) && ((p.S + p.Q) % 8 == 0);
  a.out_v8 = ((uintptr_t)p.out & 31u) == 0;
  // class rows are nkt bytes apart from a 16-byte aligned base (the workspace)
  a.cls_v16 = p.mode == kDense && ((uintptr_t)p.classes & 15u) == 0 && p.nkt % 16 == 0;
  if (a.n_items <= 0) return cudaSuccess;
  CUtensorMap mq, mkn, mkr, mv;
  if (!make_map_3d(&mq, p.q, q_rows, p.H, kDn + kDr, kBM) || !make_map_3d(&mkn, p.kn, kv_rows, p.H, kDn, kBN) ||
      !make_map_2d(&mkr, p.kr, kv_rows, kDr, kBN) || !make_map_3d(&mv, p.v, kv_rows, p.H, kDv, kBN))
    return cudaErrorInvalidValue;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  // The setmaxnreg split assumes the kernel launches with exactly kLaunchRegs
  // registers per thread; any other count would make setmaxnreg.inc wait forever.
  auto kernel = p.mode == kDense ? attn_tc_kernel<true> : attn_tc_kernel<false>;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || fa.numRegs != kLaunchRegs)
    return cudaErrorInvalidConfiguration;
  const int grid = a.n_items < nsm ? a.n_items : nsm;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, mq, mkn, mkr, mv);
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
