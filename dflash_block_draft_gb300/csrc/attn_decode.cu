// attn_decode.cu -- split-context block attention for decode-shaped ragged
// batches (few draft rows per request, long context), sm_103a.
//
// Serving drafts one block per request over its cached context
// (max.pipelines.architectures.dflash_kimi_k25 page, DFlashKimiK25:
// forward_block over the draft KV cache, input_row_offsets,
// ctx_at_draft_cache_length).  A request has at most 16 query rows but up to
// tens of thousands of keys, so one (request, head) is far too little work for
// one SM and the pass is bound by the K/V bytes read from HBM.  The context is
// therefore cut into splits of kSplitTiles 128-key tiles; every
// (request, split, head) is a work unit that writes a normalised partial
// output and its log-sum-exp, and a combine kernel merges the splits:
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s O_s / sum_s w_s,
//   lse = M + log(sum_s w_s).
//
// The MMAs are swapped so that the 128 keys of a tile are the M dimension:
//   S^T [128 keys x 16 rows]  = K_tile . Q^T      (A = K from smem, B = Q from smem)
//   O^T [128 dv   x 16 rows] += V^T . P^T          (A = V, MN-major, B = P^T from smem)
// both accumulating in TMEM.  Softmax threads own one key (TMEM lane) each and
// keep, per query row, a reference maximum shared by all 128 threads: a tile
// changes it only when some score exceeds it by more than 2^8 (a warp OR-vote
// finds that), so most tiles need no cross-thread reduction.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2..5 softmax and epilogue.  Shared memory: the Q tile (3 panels
// of 16 rows), a ring of 10 panels holding two K/V tiles (the two V panels of
// a tile are adjacent), and P^T (2 panels).  Waits are bounded as in the
// prefill kernel.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBN = 128;            // keys per tile
constexpr int kQN = 16;             // query rows per request (MMA N)
// At most this many tiles per work unit (4096 keys): a request's context is cut
// into ceil(tiles / kSplitTiles) splits of equal size (within one tile).  Each
// unit pays a Q load, a pipeline fill and an epilogue, and longer units leave a
// longer tail: limits of 16, 24, 32, 48 and 64 tiles measured 76, 80, 82, 79 and
// 79 % of the HBM peak on the decode workload with full splits plus a remainder;
// equal splits added 1 % at 32.
constexpr int kSplitTiles = 32;
constexpr uint32_t kPanel = 128 * 128;      // K/V panel: 128 rows x 128 bytes
constexpr uint32_t kQPanel = kQN * 128;     // Q / P^T panel: 16 rows x 128 bytes
constexpr uint32_t kRing = 10;
constexpr uint32_t kPanelsPerTile = 5;      // k_nope x2, k_rope, v x2
constexpr uint32_t kOffRing = 0;
constexpr uint32_t kOffQ = kOffRing + kRing * kPanel;
constexpr uint32_t kOffP = kOffQ + 3 * kQPanel;
constexpr uint32_t kOffBar = kOffP + 4 * kQPanel;  // P^T double buffer, 2 panels each

enum {
  BAR_Q_FULL = 0,
  BAR_Q_EMPTY = 1,
  BAR_RING_FULL = 2,
  BAR_RING_EMPTY = BAR_RING_FULL + kRing,
  BAR_S_FULL = BAR_RING_EMPTY + kRing,  // 2: S^T double buffer
  BAR_P_FULL = BAR_S_FULL + 2,          // 2: P^T double buffer
  BAR_PV_DONE = BAR_P_FULL + 2,         // one phase per PV
  BAR_O_FULL = BAR_PV_DONE + 1,
  BAR_DRAIN = BAR_O_FULL + 1,
  kNumBars = BAR_DRAIN + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kOffRed = kOffAbort + 12;               // softmax scratch (floats)
constexpr uint32_t kRedFloats = 4 * kQN + 3 + 3 * kQN;     // per-warp maxima/sums, vote words, row key bounds
constexpr uint32_t kSmemBytes = kOffRed + 4 * kRedFloats + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

constexpr uint32_t kTmemCols = 64;
constexpr uint32_t kColS = 0, kColO = 32;  // S^T buffers at 0 and 16

constexpr int kThreads = 192;
using tc::Ctl;
using tc::kWaitBudgetNs;
constexpr uint32_t kSoftmaxBarrier = 1;  // named barrier of the 4 softmax warps

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(128, kQN, 0, 0);  // K and Q both K-major
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, kQN, 1, 0);  // V^T MN-major, P^T K-major

struct DecodeArgs {
  AttnParams p;
  const int* prefix;  // [R+1] work units (splits) per request, exclusive prefix
  float* part_o;      // [units][kQN][kDv]
  float* part_lse;    // [units][kQN]
  int max_slots;      // request-splits the workspace holds
};

struct Unit {
  int ok;
  int r, s, h;
  Seg sg;
  int kt0, kt1;  // tiles [kt0, kt1) of the request's key axis
  int amin, amax;
  long long slot;  // partial-output index
};

__device__ __forceinline__ Unit decode_unit(const DecodeArgs& a, int u) {
  Unit it;
  const AttnParams& p = a.p;
  it.h = u % p.H;
  const int w = u / p.H;
  int lo = 0, hi = p.R - 1;  // request r with prefix[r] <= w < prefix[r+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.prefix[mid] <= w) lo = mid;
    else hi = mid - 1;
  }
  it.r = lo;
  it.s = w - a.prefix[lo];
  it.slot = w;
  it.sg = resolve_segment(p, it.r);
  it.ok = it.sg.ok && it.sg.Q <= kQN && w < a.max_slots;
  if (!it.ok) return it;
  const int nkt = (it.sg.S + it.sg.Q + kBN - 1) / kBN;
  // ceil(nkt / kSplitTiles) splits of equal size (within one tile)
  const int nsplit = (nkt + kSplitTiles - 1) / kSplitTiles;
  it.kt0 = (int)((long long)it.s * nkt / nsplit);
  it.kt1 = (int)((long long)(it.s + 1) * nkt / nsplit);
  it.amin = it.sg.S;
  it.amax = 0;
  for (int j = 0; j <= (it.sg.Q - 1) / p.bs; ++j) {
    int an = p.anchors[it.sg.anc0 + j];
    an = an < 0 ? 0 : (an > it.sg.S ? it.sg.S : an);
    it.amin = min(it.amin, an);
    it.amax = max(it.amax, an);
  }
  return it;
}

__device__ __forceinline__ int unit_class(const DecodeArgs& a, const Unit& it, int kt) {
  return anchored_tile_class(it.sg.S, it.sg.Q, a.p.bs, 0, it.sg.Q, it.amin, it.amax, kt);
}

__device__ __forceinline__ int next_tile(const DecodeArgs& a, const Unit& it, int kt) {
  for (++kt; kt < it.kt1; ++kt)
    if (unit_class(a, it, kt) != DFLASH_TILE_SKIP) return kt;
  return it.kt1;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_kernel(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmKn, const __grid_constant__ CUtensorMap tmKr,
                       const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& p = a.p;
  const int n_units = a.prefix[p.R] * p.H;

  Ctl ctl;
  ctl.bar0 = sbase + kOffBar;
  ctl.abort = reinterpret_cast<volatile int*>(smem + kOffAbort);
  ctl.err = p.err;
  ctl.budget = p.wait_ns;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);
  float* red = reinterpret_cast<float*>(smem + kOffRed);  // [4][kQN] per-warp values
  unsigned* vote = reinterpret_cast<unsigned*>(red + 4 * kQN);  // [3] vote words, used in rotation
  // [3][kQN] per row: anchor (context keys below it are visible), first and
  // one-past-last key of the row's own noise block
  int* s_ctx = reinterpret_cast<int*>(red + 4 * kQN + 3);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ctl.bar(BAR_Q_FULL), 1);
    ptx::mbar_init(ctl.bar(BAR_Q_EMPTY), 1);
    for (uint32_t s = 0; s < kRing; ++s) {
      ptx::mbar_init(ctl.bar(BAR_RING_FULL + s), 1);
      ptx::mbar_init(ctl.bar(BAR_RING_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(ctl.bar(BAR_S_FULL + b), 1);
      ptx::mbar_init(ctl.bar(BAR_P_FULL + b), 128);
    }
    ptx::mbar_init(ctl.bar(BAR_PV_DONE), 1);
    ptx::mbar_init(ctl.bar(BAR_O_FULL), 1);
    ptx::mbar_init(ctl.bar(BAR_DRAIN), 1);
    *ctl.abort = 0;
    vote[0] = vote[1] = vote[2] = 0u;
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pc = 0, n = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit it = decode_unit(a, u);
        if (!it.ok) continue;
        if (n > 0 && !ctl.wait(BAR_Q_EMPTY, (n - 1) & 1u)) break;
        ptx::mbar_arrive_expect_tx(ctl.bar(BAR_Q_FULL), 3 * kQPanel);
        for (int pn = 0; pn < 3; ++pn)
          ptx::tma_load_3d(sbase + kOffQ + pn * kQPanel, &tmQ, ctl.bar(BAR_Q_FULL), 64 * pn, it.h,
                           (int)it.sg.q0);
        ++n;
        if ((int)blockIdx.x == p.stall_cta) break;  // timeout test: this unit's key tiles never arrive
        for (int kt = next_tile(a, it, it.kt0 - 1); kt < it.kt1 && !stop; kt = next_tile(a, it, kt)) {
          const int krow = (int)(it.sg.kv0 + (long long)kt * kBN);
          for (uint32_t pn = 0; pn < kPanelsPerTile; ++pn, ++pc) {
            const uint32_t s = pc % kRing;
            if (!ctl.wait(BAR_RING_EMPTY + s, ((pc / kRing) & 1u) ^ 1u)) {
              stop = true;
              break;
            }
            const uint32_t dst = ring + s * kPanel;
            const uint32_t fb = ctl.bar(BAR_RING_FULL + s);
            ptx::mbar_arrive_expect_tx(fb, kPanel);
            if (pn < 2) ptx::tma_load_3d(dst, &tmKn, fb, 64 * pn, it.h, krow);
            else if (pn == 2) ptx::tma_load_2d(dst, &tmKr, fb, 0, krow);
            else ptx::tma_load_3d(dst, &tmV, fb, 64 * (pn - 3), it.h, krow);
          }
        }
      }
      // Wind-down (also after a timeout): the loads still outstanding -- at most
      // the last kRing panels and the last Q tile -- land before the CTA exits.
      for (uint32_t i = pc > kRing ? pc - kRing : 0u; i < pc; ++i)
        ctl.wait_landed(BAR_RING_FULL + i % kRing, (i / kRing) & 1u);
      if (n > 0) ctl.wait_landed(BAR_Q_FULL, (n - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0, n = 0;
      const uint32_t sQ = sbase + kOffQ, sP = sbase + kOffP;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const Unit it = decode_unit(a, u);
        if (!it.ok) continue;
        if (!ctl.wait(BAR_Q_FULL, n & 1u)) break;
        ++n;
        // S^T of the next tile is computed while the softmax works on this one.
        auto issue_qk = [&](uint32_t gg) -> bool {
          const uint32_t kp = gg * kPanelsPerTile;
          for (uint32_t pn = 0; pn < 3; ++pn)
            if (!ctl.wait(BAR_RING_FULL + (kp + pn) % kRing, ((kp + pn) / kRing) & 1u)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < (kDn + kDr) / 16; ++ks) {
            const uint32_t pn = (uint32_t)(ks >> 2), sub = (uint32_t)(ks & 3) * 32u;
            const uint32_t kslot = (kp + pn) % kRing;
            ptx::mma_ss(tmem + kColS + 16u * (gg & 1u), ptx::smem_desc(ring + kslot * kPanel + sub, 16, 1024),
                        ptx::smem_desc(sQ + pn * kQPanel + sub, 16, 1024), kIdescQK, ks > 0);
          }
          ptx::tc_commit(ctl.bar(BAR_S_FULL + (gg & 1u)));
          for (uint32_t pn = 0; pn < 3; ++pn) ptx::tc_commit(ctl.bar(BAR_RING_EMPTY + (kp + pn) % kRing));
          return true;
        };
        int kt = next_tile(a, it, it.kt0 - 1);
        if (kt >= it.kt1) {  // nothing visible in this split
          ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));
          continue;
        }
        if (!issue_qk(g)) break;
        bool first = true;
        for (;;) {
          const int kn = next_tile(a, it, kt);
          if (kn < it.kt1) {
            if (!issue_qk(g + 1)) { stop = true; break; }
          } else {
            ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));
          }
          // O^T += V^T P^T for tile g
          const uint32_t kp = g * kPanelsPerTile;
          if (!ctl.wait(BAR_P_FULL + (g & 1u), (g >> 1) & 1u) ||
              !ctl.wait(BAR_RING_FULL + (kp + 3) % kRing, ((kp + 3) / kRing) & 1u) ||
              !ctl.wait(BAR_RING_FULL + (kp + 4) % kRing, ((kp + 4) / kRing) & 1u)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t v0 = ring + ((kp + 3) % kRing) * kPanel;  // the two V panels are adjacent
          const uint32_t sPg = sP + (g & 1u) * 2u * kQPanel;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            ptx::mma_ss(tmem + kColO, ptx::smem_desc(v0 + (uint32_t)ks * 2048u, kPanel, 1024),
                        ptx::smem_desc(sPg + (uint32_t)(ks >> 2) * kQPanel + (uint32_t)(ks & 3) * 32u, 16, 1024),
                        kIdescPV, !(first && ks == 0));
          }
          first = false;
          ptx::tc_commit(ctl.bar(BAR_PV_DONE));
          ptx::tc_commit(ctl.bar(BAR_RING_EMPTY + (kp + 3) % kRing));
          ptx::tc_commit(ctl.bar(BAR_RING_EMPTY + (kp + 4) % kRing));
          ++g;
          if (kn >= it.kt1) break;
          kt = kn;
        }
        if (stop) break;
        ptx::tc_commit(ctl.bar(BAR_O_FULL));
      }
      ptx::tc_commit(ctl.bar(BAR_DRAIN));
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(ctl.bar(BAR_DRAIN), 0)) {
        if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
          record_error(ctl.err, DFLASH_ERR_TIMEOUT);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 2..5)
    const int quad = warp & 3;
    const int wi = warp - 2;                 // softmax warp index 0..3
    const int t = quad * 32 + lane;          // TMEM lane: key within the tile (S^T), dv (O^T)
    const int st = threadIdx.x - 64;         // 0..127
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    uint32_t g = 0, n = 0, vslot = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const Unit it = decode_unit(a, u);
      if (!it.ok) continue;
      const int S = it.sg.S, Qn = it.sg.Q, K = S + Qn;
      if (st < kQN) {
        const int blk = st / p.bs;
        s_ctx[st] = st < Qn ? row_anchor(p, it.sg, st) : 0;
        s_ctx[kQN + st] = st < Qn ? S + blk * p.bs : 0;
        s_ctx[2 * kQN + st] = st < Qn ? S + min(blk * p.bs + p.bs, Qn) : 0;
      }
      ptx::named_barrier(kSoftmaxBarrier, 128);
      float m_ref[kQN], l_part[kQN];
#pragma unroll
      for (int q = 0; q < kQN; ++q) {
        m_ref[q] = -INFINITY;
        l_part[q] = 0.f;
      }
      bool first = true;
      for (int kt = next_tile(a, it, it.kt0 - 1); kt < it.kt1; kt = next_tile(a, it, kt), ++g) {
        const int key = kt * kBN + t;  // this thread's key, relative to the request
        const bool full = unit_class(a, it, kt) == DFLASH_TILE_FULL && kt * kBN + kBN <= K;
        // Which rows see this thread's key, as a bit mask worked out before the
        // scores arrive, without branches (rows past Qn hold empty ranges).
        uint32_t vmask = (1u << Qn) - 1u;
        if (!full) {
          vmask = 0u;
#pragma unroll
          for (int q = 0; q < kQN; ++q)
            vmask |= (uint32_t)((key < s_ctx[q]) | ((key >= s_ctx[kQN + q]) & (key < s_ctx[2 * kQN + q]))) << q;
        }
        if (!ctl.wait(BAR_S_FULL + (g & 1u), (g >> 1) & 1u)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        float x[kQN];
        ptx::tmem_ld16(tmem + lane_off + kColS + 16u * (g & 1u), reinterpret_cast<uint32_t*>(x));
        ptx::tmem_wait_ld();
        uint32_t flags = 0;
#pragma unroll
        for (int q = 0; q < kQN; ++q) {
          x[q] = (vmask >> q) & 1u ? x[q] * c2 : -INFINITY;
          if (x[q] > m_ref[q] + 8.0f) flags |= 1u << q;
        }
        // Does any of the 128 keys move some row's reference maximum?
        flags = __reduce_or_sync(0xffffffffu, flags);
        if (lane == 0 && flags) atomicOr(&vote[vslot], flags);
        ptx::named_barrier(kSoftmaxBarrier, 128);
        flags = vote[vslot];
        // The word two tiles ahead was last read before the previous barrier and is
        // next written after the following one: clear it now.
        if (st == 0) vote[vslot == 0 ? 2 : vslot - 1] = 0u;
        vslot = vslot == 2 ? 0 : vslot + 1;
        if (flags) {
          // exact tile maxima of the flagged rows
#pragma unroll
          for (int q = 0; q < kQN; ++q) {
            if (!((flags >> q) & 1u)) continue;
            float mx = x[q];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane == 0) red[wi * kQN + q] = mx;
          }
          ptx::named_barrier(kSoftmaxBarrier, 128);
          float alpha[kQN];
          bool rescale = false;
#pragma unroll
          for (int q = 0; q < kQN; ++q) {
            alpha[q] = 1.f;
            if (!((flags >> q) & 1u)) continue;
            const float mx = fmaxf(fmaxf(red[q], red[kQN + q]), fmaxf(red[2 * kQN + q], red[3 * kQN + q]));
            const float mn = fmaxf(m_ref[q], mx);
            alpha[q] = m_ref[q] == -INFINITY ? 0.f : ptx::ex2(m_ref[q] - mn);
            m_ref[q] = mn;
            l_part[q] *= alpha[q];
            rescale = true;
          }
          if (rescale && !first) {
            // O^T column q (this thread's dv lane) scaled to the new reference, once
            // PV of the previous tile has completed.
            if (!ctl.wait(BAR_PV_DONE, (g - 1) & 1u)) {
              stop = true;
              break;
            }
            ptx::tc_fence_after();
            uint32_t o[kQN];
            ptx::tmem_ld16(tmem + lane_off + kColO, o);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < kQN; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
            ptx::tmem_st16(tmem + lane_off + kColO, o);
            ptx::tmem_wait_st();
          }
          ptx::named_barrier(kSoftmaxBarrier, 128);  // red[] is free again
        }
        // p = exp2(x - m_ref); P^T[row q][key t] in the 128-byte-swizzled K-major layout
        uint8_t* pt = smem + kOffP + (g & 1u) * 2u * kQPanel + (t >> 6) * kQPanel;
        const int cb = (t & 63) * 2;  // byte offset of this key inside a 128-byte row
#pragma unroll
        for (int q = 0; q < kQN; ++q) {
          const float pq = m_ref[q] == -INFINITY ? 0.f : ptx::ex2(x[q] - m_ref[q]);
          l_part[q] += pq;
          const int chunk = (cb >> 4) ^ (q & 7);
          *reinterpret_cast<__nv_bfloat16*>(pt + q * 128 + chunk * 16 + (cb & 15)) = __float2bfloat16_rn(pq);
        }
        ptx::fence_proxy_async_smem();  // P^T written by threads, read by the tensor core
        ptx::tc_fence_before();
        ptx::mbar_arrive(ctl.bar(BAR_P_FULL + (g & 1u)));
        first = false;
      }
      if (stop) break;
      // ---- epilogue: partial O = O^T / l and lse for each row of this unit
      // l[q] = sum over the 128 key threads
#pragma unroll
      for (int q = 0; q < kQN; ++q) {
        float v = l_part[q];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red[wi * kQN + q] = v;
      }
      ptx::named_barrier(kSoftmaxBarrier, 128);
      float inv[kQN], lrow[kQN];
#pragma unroll
      for (int q = 0; q < kQN; ++q) {
        lrow[q] = red[q] + red[kQN + q] + red[2 * kQN + q] + red[3 * kQN + q];
        inv[q] = lrow[q] > 0.f ? 1.f / lrow[q] : 0.f;
      }
      float* po = a.part_o + it.slot * p.H * (long long)(kQN * kDv) + (long long)it.h * (kQN * kDv);
      if (!first) {
        if (!ctl.wait(BAR_O_FULL, n & 1u)) break;
        ++n;
        ptx::tc_fence_after();
        uint32_t o[kQN];
        ptx::tmem_ld16(tmem + lane_off + kColO, o);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kQN; ++q) po[q * kDv + t] = __uint_as_float(o[q]) * inv[q];
      } else {
#pragma unroll
        for (int q = 0; q < kQN; ++q) po[q * kDv + t] = 0.f;
      }
      if (st < kQN) {
        float mr = -INFINITY;
#pragma unroll
        for (int q = 0; q < kQN; ++q)
          if (q == st) mr = m_ref[q];
        float lr = 0.f;
#pragma unroll
        for (int q = 0; q < kQN; ++q)
          if (q == st) lr = lrow[q];
        a.part_lse[(it.slot * p.H + it.h) * kQN + st] = lr > 0.f ? (mr + log2f(lr)) * 0.6931471805599453f : -INFINITY;
      }
      ptx::named_barrier(kSoftmaxBarrier, 128);  // red[] and s_ctx[] reused by the next unit
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// Per-request work-unit counts and their exclusive prefix, one CTA.  Invalid
// offsets get zero units (recorded in the error word by the attention kernel's
// segment check; here they are simply skipped).
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) decode_plan_kernel(AttnParams p, int* prefix, int max_slots) {
  __shared__ int part[kPlanThreads];
  const int R = p.R;
  const int per = (R + kPlanThreads - 1) / kPlanThreads;
  const int r0 = threadIdx.x * per, r1 = min(R, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) {
    const Seg sg = resolve_segment(p, r);
    if (sg.ok && sg.Q <= kQN) {
      const int nkt = (sg.S + sg.Q + kBN - 1) / kBN;
      sum += (nkt + kSplitTiles - 1) / kSplitTiles;
    } else if (sg.ok) {
      record_error(p.err, DFLASH_ERR_INVALID);  // q_len beyond the declared max_q_len
    }
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {  // inclusive scan
    const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
  for (int r = r0; r < r1; ++r) {
    prefix[r] = run;
    const Seg sg = resolve_segment(p, r);
    if (sg.ok && sg.Q <= kQN) run += ((sg.S + sg.Q + kBN - 1) / kBN + kSplitTiles - 1) / kSplitTiles;
  }
  if (threadIdx.x == kPlanThreads - 1) {
    prefix[R] = part[kPlanThreads - 1];
    // overlapping offsets could ask for more splits than the workspace holds
    if (part[kPlanThreads - 1] > max_slots) record_error(p.err, DFLASH_ERR_INVALID);
  }
}

// Merge the split partials of every (query row, head): one CTA of kDv threads.
// One warp per (row, head); a lane owns 4 consecutive dv values (16-byte loads).
constexpr int kCombineWarps = 8;
__global__ void __launch_bounds__(32 * kCombineWarps) decode_combine_kernel(AttnParams p, const int* prefix,
                                                                             const float* part_o,
                                                                             const float* part_lse, int max_slots) {
  const long long wid = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)p.total_q * p.H) return;
  const int row = (int)(wid / p.H), h = (int)(wid % p.H);
  int lo = 0, hi = p.R - 1;  // request owning this row
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.q_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int q = row - p.q_off[r];
  const int u0 = prefix[r], u1 = min(prefix[r + 1], max_slots);
  if (u1 <= u0 || q < 0 || q >= kQN || q >= p.q_off[r + 1] - p.q_off[r]) return;  // skipped request
  float M = -INFINITY;
  for (int u = u0; u < u1; ++u) M = fmaxf(M, part_lse[((long long)u * p.H + h) * kQN + q]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int u = u0; u < u1; ++u) {
      const float ls = part_lse[((long long)u * p.H + h) * kQN + q];
      const float w = ls == -INFINITY ? 0.f : __expf(ls - M);
      wsum += w;
      const float4 o = reinterpret_cast<const float4*>(part_o + (((long long)u * p.H + h) * kQN + q) * kDv)[lane];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat162 v01 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv), v23 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&v01);
  pk.y = *reinterpret_cast<uint32_t*>(&v23);
  reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + ((long long)row * p.H + h) * kDv)[lane] = pk;
  if (p.lse && lane == 0) p.lse[(long long)h * p.total_q + row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

int decode_max_units(int R, int total_kv) {
  // sum_r ceil(tiles_r / kSplitTiles) <= total_kv / (kSplitTiles*kBN) + 2 R (tile rounding and split rounding)
  return total_kv / (kSplitTiles * kBN) + 2 * R + 1;
}

size_t decode_workspace_bytes(int R, int H, int total_kv) {
  const size_t units = (size_t)decode_max_units(R, total_kv) * H;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(sizeof(int) * (R + 1)) + up(units * kQN * kDv * sizeof(float)) + up(units * kQN * sizeof(float));
}

bool decode_supported(int dn, int dr, int dv, int max_q_len) {
  return dn == kDn && dr == kDr && dv == kDv && max_q_len <= kQN;
}

cudaError_t launch_attn_decode(const AttnParams& p, void* ws, cudaStream_t stream) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t units = (size_t)decode_max_units(p.R, p.total_kv) * p.H;
  uint8_t* base = static_cast<uint8_t*>(ws);
  DecodeArgs a;
  a.p = p;
  a.prefix = reinterpret_cast<int*>(base);
  a.part_o = reinterpret_cast<float*>(base + up(sizeof(int) * (p.R + 1)));
  a.part_lse = reinterpret_cast<float*>(base + up(sizeof(int) * (p.R + 1)) + up(units * kQN * kDv * sizeof(float)));
  a.max_slots = decode_max_units(p.R, p.total_kv);
  decode_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p, const_cast<int*>(a.prefix), a.max_slots);
  count_launch();
  CUtensorMap mq, mkn, mkr, mv;
  if (!make_map_3d(&mq, p.q, p.total_q, p.H, kDn + kDr, kQN) || !make_map_3d(&mkn, p.kn, p.total_kv, p.H, kDn, kBN) ||
      !make_map_2d(&mkr, p.kr, p.total_kv, kDr, kBN) || !make_map_3d(&mv, p.v, p.total_kv, p.H, kDv, kBN))
    return cudaErrorInvalidValue;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = (int)((size_t)nsm < units ? (size_t)nsm : units);
  attn_decode_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, mq, mkn, mkr, mv);
  count_launch();
  decode_combine_kernel<<<(unsigned)(((long long)p.total_q * p.H + kCombineWarps - 1) / kCombineWarps),
                          32 * kCombineWarps, 0, stream>>>(p, a.prefix, a.part_o, a.part_lse, a.max_slots);
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
