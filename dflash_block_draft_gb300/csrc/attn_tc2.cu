// attn_tc2.cu -- DFlash block attention on CTA pairs (tcgen05 cta_group::2), sm_103a.
//
// The same operation, shapes and online softmax as attn_tc.cu (bf16, d_nope =
// 128, d_rope = 64 head-shared, d_v = 128; nemo_automodel.components.
// speculative.dflash.draft_kimi_k3 page, KimiK3DFlashAttention), computed by
// clusters of two CTAs whose tensor cores run each MMA together:
//   S_i  = Q_i K^T   M = 256 rows (128 in each CTA), N = 128 keys; each CTA
//                    holds 64 of the keys (B is split along N)
//   O_i += P_i V     M = 256 rows, A = P_i from each CTA's TMEM; each CTA holds
//                    64 of the 128 value columns for all 128 keys
// A work item is (segment, four adjacent 128-row query tiles, head).  CTA c of
// the pair owns query tiles 4q + 2i + c for halves i = 0, 1, so one pair MMA
// covers two adjacent query tiles.  Because each CTA stores only half of every
// K/V tile (40 KB), three key tiles fit in flight next to the two Q tiles, and
// the two halves can take turns on the tensor pipe: one half's MMAs run while
// the other half's softmax works.
//
// Roles (384 threads per CTA, as in attn_tc.cu):
//   warp 0        TMA producer (each CTA loads its own Q tiles and K/V halves)
//   warp 1        even CTA: TMEM owner and MMA issuer of half 0;
//                 odd CTA: forwards its load completions to the even CTA
//   warp 2        even CTA: MMA issuer of half 1
//   warps 4..11   softmax and epilogue of halves 0 and 1 for this CTA's rows
// Barriers that the MMAs complete (S, O, ring slots, Q) receive multicast
// commits in both CTAs; the even CTA's issuers wait for the odd CTA's loads and
// P through arrivals on the even CTA's barriers.
// Every wait is bounded: a timeout records DFLASH_ERR_TIMEOUT and raises the
// abort flag of both CTAs, which then wind down.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

using tc::Ctl;
using tc::kPrepAnchored;
using tc::kPrepDense;
using tc::kPrepFull;
using tc::kPrepNone;
using tc::kWaitBudgetNs;
using tc::mask64;
using tc::max64;
using tc::PrepCtx;

constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBM = 128, kBN = 128;
constexpr uint32_t kPanel = 128 * 128;      // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kHalfPanel = 64 * 128;   // 64 rows x 128 bytes
constexpr uint32_t kQBytes = 3 * kPanel;    // per half: nope 0-63, nope 64-127, rope
constexpr uint32_t kKBytes = 3 * kHalfPanel;  // this CTA's 64 keys: nope 0-63, nope 64-127, rope
constexpr uint32_t kVBytes = kPanel;          // 128 keys x this CTA's 64 value columns
constexpr uint32_t kSlotBytes = kKBytes + kVBytes;
constexpr uint32_t kSlots = 3;  // key tiles in flight
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = 2 * kQBytes;
constexpr uint32_t kOffBar = kOffRing + kSlots * kSlotBytes;

enum {
  BAR_Q_FULL = 0,
  BAR_Q_EMPTY = 1,
  BAR_K_FULL = 2,                    // kSlots
  BAR_V_FULL = BAR_K_FULL + kSlots,  // kSlots
  BAR_EMPTY = BAR_V_FULL + kSlots,   // kSlots
  BAR_S_FULL = BAR_EMPTY + kSlots,   // 2 (per half)
  BAR_P_FULL = BAR_S_FULL + 2,       // 2, even CTA
  BAR_O_FULL = BAR_P_FULL + 2,       // 2
  BAR_TURN = BAR_O_FULL + 2,         // 2, even CTA
  BAR_DRAIN = BAR_TURN + 2,
  kNumBars = BAR_DRAIN + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffRing % 1024 == 0 && kSlotBytes % 1024 == 0 && kKBytes % 1024 == 0, "128-byte swizzle alignment");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;  // S_i at kColS + 128 i, O_i at kColO + 128 i

constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168;
constexpr uint32_t kCtlRegs = 120, kSoftmaxRegs = 192;
static_assert(128 * kCtlRegs + 256 * kSoftmaxRegs == kThreads * kLaunchRegs, "register split");

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(2 * kBM, kBN, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(2 * kBM, kDv, 0, 1);  // P from TMEM, V MN-major

struct Tc2Args {
  AttnParams p;
  int segments;
  int nqt;      // query tiles per segment (max over segments for ragged)
  int nquad;    // ceil(nqt / 4)
  int n_items;  // nquad * segments * H
  int mask_vec; // dense: mask rows are 16-byte aligned
  int out_v8;   // out is 32-byte aligned: rows are written with 32-byte stores
};

struct Item {
  int ok;
  int z, h;
  Seg sg;
  int nkt;
  int r0[2], r1[2];        // this CTA's query tile of each half
  int amin[2], amax[2];
  bool has[2];
  const uint8_t* cls[2];
  const uint8_t* ucls[4];  // dense: tile classes of the item's four query tiles (null: no such tile)
  int ctx_end, noise_begin, noise_end;  // anchored: the item's non-SKIP tiles are [0,ctx_end) U [noise_begin,noise_end)
};

// min/max of the clipped anchors of the blocks of query rows [r0, r1)
__device__ __forceinline__ void anchor_range(const AttnParams& p, const Seg& sg, int r0, int r1, int& amin,
                                             int& amax) {
  const int j0 = r0 / p.bs, j1 = (r1 - 1) / p.bs;
  const int* ap = p.anchors + sg.anc0;
  for (int jb = j0; jb <= j1; jb += 8) {
    int an[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) an[u] = __ldg(ap + min(jb + u, j1));
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = an[u] < 0 ? 0 : (an[u] > sg.S ? sg.S : an[u]);
      amin = min(amin, c);
      amax = max(amax, c);
    }
  }
}

// DENSE: the kernel reads tile classes of a dense mask (else the anchored rule).
template <bool DENSE>
__device__ __forceinline__ Item decode_item(const Tc2Args& a, int idx, uint32_t rank) {
  Item it;
  const AttnParams& p = a.p;
  const int zh = a.segments * p.H;
  const int quad = a.nquad - 1 - idx / zh;  // longest (latest) query tiles first
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
    const int t = 4 * quad + 2 * i + (int)rank;
    it.r0[i] = t * kBM;
    it.has[i] = it.r0[i] < Qn;
    it.r1[i] = min(it.r0[i] + kBM, Qn);
    it.cls[i] = nullptr;
    it.amin[i] = S;
    it.amax[i] = 0;
    if (!it.has[i]) continue;
    if (DENSE) it.cls[i] = p.classes + ((long long)it.z * p.nqt + t) * p.nkt;
    else anchor_range(p, it.sg, it.r0[i], it.r1[i], it.amin[i], it.amax[i]);
  }
  const int q_first = 4 * quad * kBM;
  it.ok = q_first < Qn;
  if (!it.ok) return it;
  const int q_last = min(q_first + 4 * kBM, Qn);  // rows [q_first, q_last) of the item
  if (DENSE) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = 4 * quad + j;
      it.ucls[j] = t * kBM < Qn ? p.classes + ((long long)it.z * p.nqt + t) * p.nkt : nullptr;
    }
  } else {
    // Context keys some row of the item sees: k < max anchor.  Noise keys: the
    // blocks of the item's rows.
    int umin = S, umax = 0;
    anchor_range(p, it.sg, q_first, q_last, umin, umax);
    const int u0 = (q_first / p.bs) * p.bs;
    const int u1 = min(((q_last - 1) / p.bs + 1) * p.bs, Qn);
    it.ctx_end = (min(umax, S) + kBN - 1) / kBN;
    it.noise_begin = (S + u0) / kBN;
    it.noise_end = (S + u1 + kBN - 1) / kBN;
  }
  return it;
}

// Next key tile after kt that some row of the item needs (it.nkt when none is left).
template <bool DENSE>
__device__ __forceinline__ int next_tile(const Tc2Args& a, const Item& it, int kt) {
  ++kt;
  if (!DENSE) {
    if (kt < it.ctx_end) return kt;
    kt = max(kt, it.noise_begin);
    return kt < it.noise_end ? kt : it.nkt;
  }
  for (; kt < it.nkt; ++kt) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (it.ucls[j] && it.ucls[j][kt] != DFLASH_TILE_SKIP) return kt;
  }
  return it.nkt;
}

template <bool DENSE>
__device__ __forceinline__ int half_class(const Tc2Args& a, const Seg& sg, bool has, int r0, int r1, int amin,
                                          int amax, const uint8_t* cls, int kt) {
  if (!has) return DFLASH_TILE_SKIP;
  if (DENSE) return cls[kt];
  return anchored_tile_class(sg.S, sg.Q, a.p.bs, r0, r1, amin, amax, kt);
}

// Item index of this cluster in its k-th pass over the grid (snake order over the longest-first list).
__device__ __forceinline__ int item_of_round(int k) {
  const int G = (int)gridDim.x >> 1, c = (int)blockIdx.x >> 1;
  return k * G + ((k & 1) ? (G - 1 - c) : c);
}

template <bool DENSE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc2_kernel(const __grid_constant__ Tc2Args a, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmKn, const __grid_constant__ CUtensorMap tmKr,
                    const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& p = a.p;
  const uint32_t rank = ptx::cluster_rank();
  const bool lead = rank == 0;
  const int G = (int)gridDim.x >> 1;  // clusters

  Ctl ctl;
  ctl.bar0 = sbase + kOffBar;
  ctl.abort = reinterpret_cast<volatile int*>(smem + kOffAbort);
  ctl.err = p.err;
  ctl.peer_abort = ptx::mapa(sbase + kOffAbort, rank ^ 1u);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    const uint32_t from_peer = lead ? 2u : 1u;  // even CTA: its own producer + the odd CTA's forwarder
    ptx::mbar_init(ctl.bar(BAR_Q_FULL), from_peer);
    ptx::mbar_init(ctl.bar(BAR_Q_EMPTY), 2);  // both MMA issuers
    for (uint32_t s = 0; s < kSlots; ++s) {
      ptx::mbar_init(ctl.bar(BAR_K_FULL + s), from_peer);
      ptx::mbar_init(ctl.bar(BAR_V_FULL + s), from_peer);
      ptx::mbar_init(ctl.bar(BAR_EMPTY + s), 2);  // both MMA issuers
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ctl.bar(BAR_S_FULL + i), 1);
      ptx::mbar_init(ctl.bar(BAR_P_FULL + i), 8);  // one arrival per softmax warp of either CTA
      ptx::mbar_init(ctl.bar(BAR_O_FULL + i), 1);
      ptx::mbar_init(ctl.bar(BAR_TURN + i), 1);
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
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t ring = sbase + kOffRing;
  if (warp < 4) ptx::setmaxnreg_dec<kCtlRegs>();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t g = 0, n_items = 0;  // key tiles loaded, items loaded
      bool stop = false;
      for (int k = 0; !stop && k * G < a.n_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= a.n_items) continue;
        const Item it = decode_item<DENSE>(a, idx, rank);
        if (!it.ok) continue;
        if (n_items > 0 && !ctl.wait_cluster(BAR_Q_EMPTY, (n_items - 1) & 1u)) break;
        ptx::mbar_arrive_expect_tx(ctl.bar(BAR_Q_FULL), 2 * kQBytes);
        for (int i = 0; i < 2; ++i) {
          const int qrow = (int)(it.sg.q0 + it.r0[i]);
          for (int pn = 0; pn < 3; ++pn)
            ptx::tma_load_3d(sbase + kOffQ + i * kQBytes + pn * kPanel, &tmQ, ctl.bar(BAR_Q_FULL), 64 * pn, it.h,
                             qrow);
        }
        ++n_items;
        for (int kt = next_tile<DENSE>(a, it, -1); kt < it.nkt; kt = next_tile<DENSE>(a, it, kt), ++g) {
          const uint32_t s = g % kSlots;
          if (!ctl.wait_cluster(BAR_EMPTY + s, ((g / kSlots) & 1u) ^ 1u)) {
            stop = true;
            break;
          }
          const uint32_t dst = ring + s * kSlotBytes;
          const int krow = (int)(it.sg.kv0 + (long long)kt * kBN);
          const uint32_t kb = ctl.bar(BAR_K_FULL + s), vb = ctl.bar(BAR_V_FULL + s);
          ptx::mbar_arrive_expect_tx(kb, kKBytes);
          const int krow_c = krow + 64 * (int)rank;  // this CTA's 64 keys
          ptx::tma_load_3d(dst, &tmKn, kb, 0, it.h, krow_c);
          ptx::tma_load_3d(dst + kHalfPanel, &tmKn, kb, 64, it.h, krow_c);
          ptx::tma_load_2d(dst + 2 * kHalfPanel, &tmKr, kb, 0, krow_c);
          ptx::mbar_arrive_expect_tx(vb, kVBytes);
          ptx::tma_load_3d(dst + kKBytes, &tmV, vb, 64 * (int)rank, it.h, krow);  // this CTA's 64 value columns
        }
      }
    }
  } else if (warp == 1 && !lead) {
    // ------------------------------------------------------------ odd CTA: load forwarder
    // The even CTA's issuers may use a Q tile or ring slot only once this CTA's
    // half of it has landed too: pass each completion on, in load order.
    if (lane == 0) {
      const uint32_t remote0 = ptx::mapa(ctl.bar(0), 0u);  // barrier 0 of the even CTA
      auto forward = [&](int b) { ptx::mbar_arrive_remote(remote0 + 8u * (uint32_t)b); };
      uint32_t g = 0, n_items = 0;
      bool stop = false;
      for (int k = 0; !stop && k * G < a.n_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= a.n_items) continue;
        const Item it = decode_item<DENSE>(a, idx, rank);
        if (!it.ok) continue;
        if (!ctl.wait_cluster(BAR_Q_FULL, n_items & 1u)) break;
        forward(BAR_Q_FULL);
        ++n_items;
        for (int kt = next_tile<DENSE>(a, it, -1); kt < it.nkt; kt = next_tile<DENSE>(a, it, kt), ++g) {
          const uint32_t s = g % kSlots, ph = (g / kSlots) & 1u;
          if (!ctl.wait_cluster(BAR_K_FULL + s, ph)) {
            stop = true;
            break;
          }
          forward(BAR_K_FULL + (int)s);
          if (!ctl.wait_cluster(BAR_V_FULL + s, ph)) {
            stop = true;
            break;
          }
          forward(BAR_V_FULL + (int)s);
        }
      }
    }
  } else if (lead && (warp == 1 || warp == 2)) {
    // ------------------------------------------------------------ even CTA: MMA issuers
    // Issuer i runs  QK_i(j) [softmax_i(j)] PV_i(j) QK_i(j+1) ...  and the two
    // issuers take turns group by group ([PV_i(j-1)] QK_i(j), then the other
    // half's group), so the tensor pipe alternates between the halves.
    if (lane == 0) {
      const int i = warp - 1;
      uint32_t g = 0, n_items = 0, ev = 0;  // key tiles, items started, MMA groups issued
      // Descriptors are built once; a k-step only adds its byte offset >> 4 to the
      // start-address field (every operand lies below 256 KB, so the field never carries).
      const uint64_t dq = ptx::smem_desc(sbase + kOffQ + i * kQBytes, 16, 1024);
      const uint64_t dRing = ptx::smem_desc(ring, 16, 1024);
      const uint32_t d_s = tmem + kColS + 128u * i;  // S_i; P_i aliases its head
      const uint32_t d_o = tmem + kColO + 128u * i;
      auto issue_qk = [&](uint32_t gg) {
        const uint32_t slot = (gg % kSlots) * kSlotBytes;
#pragma unroll
        for (int ks = 0; ks < (kDn + kDr) / 16; ++ks) {
          const uint32_t pn = (uint32_t)(ks >> 2), sub = (uint32_t)(ks & 3) * 32u;
          ptx::mma_ss_pair(d_s, dq + ((pn * kPanel + sub) >> 4), dRing + ((slot + pn * kHalfPanel + sub) >> 4),
                           kIdescQK, ks > 0);
        }
        ptx::tc_commit_pair(ctl.bar(BAR_S_FULL + i));
      };
      auto issue_pv = [&](uint32_t gg, bool first) {
        const uint32_t vslot = (gg % kSlots) * kSlotBytes + kKBytes;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          // 16 keys: 8 packed P columns; V rows: two 1024-byte groups of 8 keys
          ptx::mma_ts_pair(d_o, d_s + (uint32_t)ks * 8u, dRing + ((vslot + (uint32_t)ks * 2048u) >> 4), kIdescPV,
                           !(first && ks == 0));
        }
        ptx::tc_commit_pair(ctl.bar(BAR_EMPTY + gg % kSlots));  // K and V of tile gg are no longer read
      };
      auto take_turn = [&]() -> bool {
        if (i == 0) return ev == 0 || ctl.wait_cluster(BAR_TURN + 0, (ev - 1u) & 1u);
        return ctl.wait_cluster(BAR_TURN + 1, ev & 1u);
      };
      auto pass_turn = [&]() {
        ptx::mbar_arrive(ctl.bar(BAR_TURN + (i ^ 1)));
        ++ev;
      };
      auto pv_ready = [&](uint32_t gg) -> bool {
        return ctl.wait_cluster(BAR_V_FULL + gg % kSlots, (gg / kSlots) & 1u) &&
               ctl.wait_cluster(BAR_P_FULL + i, gg & 1u);
      };
      bool stop = false;
      for (int k = 0; !stop && k * G < a.n_items; ++k) {
        const int idx = item_of_round(k);
        if (idx >= a.n_items) continue;
        const Item it = decode_item<DENSE>(a, idx, rank);
        if (!it.ok) continue;
        if (!ctl.wait_cluster(BAR_Q_FULL, n_items & 1u)) break;
        ++n_items;
        int kt = next_tile<DENSE>(a, it, -1);
        if (kt >= it.nkt) {  // nothing visible for this item
          ptx::tc_commit_pair(ctl.bar(BAR_Q_EMPTY));
          continue;
        }
        bool first_tile = true, first_pv = true;
        for (;;) {
          const int kn = next_tile<DENSE>(a, it, kt);
          if (!ctl.wait_cluster(BAR_K_FULL + g % kSlots, (g / kSlots) & 1u) || (!first_tile && !pv_ready(g - 1)) ||
              !take_turn()) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          if (!first_tile) {
            issue_pv(g - 1, first_pv);
            first_pv = false;
          }
          issue_qk(g);
          pass_turn();
          first_tile = false;
          ++g;
          if (kn >= it.nkt) break;
          kt = kn;
        }
        if (stop) break;
        ptx::tc_commit_pair(ctl.bar(BAR_Q_EMPTY));  // every QK of this half has been issued
        if (!pv_ready(g - 1) || !take_turn()) break;  // PV of the item's last tile
        ptx::tc_fence_after();
        issue_pv(g - 1, first_pv);
        ptx::tc_commit_pair(ctl.bar(BAR_O_FULL + i));
        pass_turn();
      }
      // Drain: every MMA this thread issued has finished before TMEM is released.
      ptx::tc_commit_pair(ctl.bar(BAR_DRAIN));
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(ctl.bar(BAR_DRAIN), 0)) {
        if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
          record_error(ctl.err, DFLASH_ERR_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue (warps 4..11, both CTAs)
    ptx::setmaxnreg_inc<kSoftmaxRegs>();
    const int half = (warp - 4) >> 2;  // query tile of the pair
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t s_col = tmem + lane_off + kColS + 128u * half;
    const uint32_t o_col = tmem + lane_off + kColO + 128u * half;
    const uint32_t p_full = ctl.bar(BAR_P_FULL + half);
    const uint32_t p_full_lead = ptx::mapa(p_full, 0u);
    const float c2 = p.scale_log2;
    uint32_t g = 0, n_full = 0;
    bool stop = false;
    for (int k = 0; !stop && k * G < a.n_items; ++k) {
      const int idx = item_of_round(k);
      if (idx >= a.n_items) continue;
      const Item it = decode_item<DENSE>(a, idx, rank);
      if (!it.ok) continue;
      // this half's scalars (selected, so that the item's arrays stay in registers)
      const bool h_has = half ? it.has[1] : it.has[0];
      const int h_r0 = half ? it.r0[1] : it.r0[0], h_r1 = half ? it.r1[1] : it.r1[0];
      const int h_amin = half ? it.amin[1] : it.amin[0], h_amax = half ? it.amax[1] : it.amax[0];
      const uint8_t* h_cls = half ? it.cls[1] : it.cls[0];
      const int i = h_r0 + row;
      const bool row_ok = h_has && i < h_r1;
      const int S = it.sg.S, Qn = it.sg.Q, K = S + Qn;
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
      for (int kt = next_tile<DENSE>(a, it, -1); kt < it.nkt; kt = next_tile<DENSE>(a, it, kt)) {
        any_tile = true;
        const int cls = half_class<DENSE>(a, it.sg, h_has, h_r0, h_r1, h_amin, h_amax, h_cls, kt);
        const int k0 = kt * kBN;
        int kind;
        if (!row_ok || cls == DFLASH_TILE_SKIP) kind = kPrepNone;
        else if (cls == DFLASH_TILE_FULL && k0 + kBN <= K) kind = kPrepFull;
        else kind = DENSE ? kPrepDense : kPrepAnchored;
        const PrepCtx pc{ctx_lim - k0, nlo - k0, nhi - k0, mrow ? mrow + k0 : nullptr, K - k0,
                         a.mask_vec != 0, c2};
        if (!ctl.wait_cluster(BAR_S_FULL + half, g & 1u)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        // The online softmax of attn_tc.cu: one TMEM read per 64-column half, a
        // running reference maximum that moves only when a half's maximum exceeds
        // it by more than 2^8, and P packed to bf16 pairs over the first 64
        // columns of S.
        const bool scaled = kind == kPrepDense;  // dense scores are already in base-2 units
        const float cm = scaled ? 1.f : c2;
        float2 lsum = make_float2(0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float x[64];
          ptx::tmem_ld32(s_col + 64u * hh, reinterpret_cast<uint32_t*>(x));
          ptx::tmem_ld32(s_col + 64u * hh + 32u, reinterpret_cast<uint32_t*>(x) + 32);
          ptx::tmem_wait_ld();
          mask64(x, kind, 64 * hh, pc);
          const float mh = max64(x) * cm;
          if (mh > m_used + 8.0f) {  // also when m is still -inf and this half sees a key
            if (m_used != -INFINITY) {
              const float alpha = ptx::ex2(m_used - mh);
#pragma unroll 1
              for (int cc = 0; cc < kDv; cc += 32) {
                uint32_t o[32];
                ptx::tmem_ld32(o_col + cc, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                ptx::tmem_st32(o_col + cc, o);
              }
              if (hh == 1) {  // P of columns 0-63, written with the old reference
                uint32_t pr[32];
                ptx::tmem_wait_st();
                ptx::tmem_ld32(s_col, pr);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  pr[e] = ptx::pack_bf16x2(__uint_as_float(pr[e] << 16) * alpha,
                                           __uint_as_float(pr[e] & 0xFFFF0000u) * alpha);
                ptx::tmem_st32(s_col, pr);
              }
              ptx::tmem_wait_st();
              l *= alpha;
              lsum.x *= alpha;
              lsum.y *= alpha;
            }
            m_used = mh;
          }
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
        }
        l += lsum.x + lsum.y;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        // One arrival per warp on the even CTA's barrier, once the warp's 32 rows of P are in TMEM.
        __syncwarp();
        if (lane == 0) {
          if (lead) ptx::mbar_arrive(p_full);
          else ptx::mbar_arrive_remote_relaxed(p_full_lead);  // P is complete in TMEM (tcgen05.wait::st)
        }
        ++g;
      }
      if (stop) break;
      // ---- epilogue: out = O / l (bf16, round to nearest even), lse = (m + log2 l) ln 2
      uint32_t ob[kDv / 2];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (any_tile) {
        if (!ctl.wait_cluster(BAR_O_FULL + half, n_full & 1u)) break;
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
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                              ((it.sg.q0 + i) * p.H + it.h) * (long long)kDv);
        if (a.out_v8) {
          // a row is 256 contiguous bytes: eight 32-byte stores (a sector each)
#pragma unroll
          for (int v = 0; v < kDv / 16; ++v) ptx::st_global_v8(dst + 2 * v, ob + 8 * v);
        } else {
#pragma unroll
          for (int v = 0; v < kDv / 8; ++v) dst[v] = make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]);
        }
        if (p.lse)
          p.lse[it.sg.lse0 + (long long)it.h * it.sg.lse_hs + i] =
              l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the even CTA's MMAs have drained; TMEM of both CTAs is free to release
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn_tc2(const AttnParams& p, int segments, int nqt, long long q_rows, long long kv_rows,
                            cudaStream_t stream) {
  Tc2Args a;
  a.p = p;
  a.segments = segments;
  a.nqt = nqt;
  a.nquad = (nqt + 3) / 4;
  a.n_items = a.nquad * segments * p.H;
  a.mask_vec = 0;
  if (p.mode == kDense) a.mask_vec = (((uintptr_t)p.mask & 15u) == 0) && ((p.S + p.Q) % 8 == 0);
  a.out_v8 = ((uintptr_t)p.out & 31u) == 0;
  if (a.n_items <= 0) return cudaSuccess;
  CUtensorMap mq, mkn, mkr, mv;
  if (!make_map_3d(&mq, p.q, q_rows, p.H, kDn + kDr, kBM) || !make_map_3d(&mkn, p.kn, kv_rows, p.H, kDn, kBN / 2) ||
      !make_map_2d(&mkr, p.kr, kv_rows, kDr, kBN / 2) || !make_map_3d(&mv, p.v, kv_rows, p.H, kDv, kBN))
    return cudaErrorInvalidValue;
  const int nsm = sm_count();
  if (nsm < 2) return cudaErrorInvalidDevice;
  // The setmaxnreg split assumes the kernel launches with exactly kLaunchRegs
  // registers per thread; any other count would make setmaxnreg.inc wait forever.
  auto kernel = p.mode == kDense ? attn_tc2_kernel<true> : attn_tc2_kernel<false>;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || fa.numRegs != kLaunchRegs)
    return cudaErrorInvalidConfiguration;
  const int clusters = a.n_items < nsm / 2 ? a.n_items : nsm / 2;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  kernel<<<2 * clusters, kThreads, kSmemBytes, stream>>>(a, mq, mkn, mkr, mv);
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
