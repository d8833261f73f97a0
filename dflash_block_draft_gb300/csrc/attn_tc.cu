// attn_tc.cu -- tensor-core (tcgen05 + TMEM + TMA) DFlash block attention, sm_103a.
//
// Shapes: bf16 q/k/v with d_nope = 128, d_rope = 64 (head-shared rope key),
// d_v = 128 -- the Kimi K3 MLA head layout of the DFlash draft
// (nemo_automodel.components.speculative.dflash.draft_kimi_k3 page:
// KimiK3DFlashAttention, one K/V per query head; module docstring: the
// qk_rope slice is a head-shared extension of the key, no rotary).
//
// One work item = (segment, 128-row query tile, head).  Per item the kernel
// walks the 128-key tiles of [context | noise] that the schedule marks
// FULL or PARTIAL (anchored rule, or the dense mask's tile classes) and keeps an
// online softmax per row:
//   S  = Q_nope K_nope^T + Q_rope K_rope^T      tcgen05 SS MMAs into TMEM (fp32)
//   P  = exp2(S * scale * log2 e - m)           4 softmax warps, one row per thread
//   O += P V                                    tcgen05 TS MMA, P (bf16) read from TMEM
//   out = O / l,  lse = (m + log2 l) ln 2
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and
// issues MMAs, warps 2..5 run the softmax and the epilogue.  Shared memory holds
// the Q tile (48 KB) and a 2-stage ring of K tiles (nope + rope, 48 KB) and V
// tiles (32 KB), all in the 128-byte-swizzled K-major layout TMA writes.
// TMEM (512 columns): S double buffer [0,256), O [256,384), P double buffer [384,512).
// The grid is persistent (one CTA per SM); items are dealt in a snake order over
// a longest-first list (query tiles with the most context first).
// Every mbarrier wait is bounded; a wait that runs past its budget records
// DFLASH_ERR_TIMEOUT, raises a CTA abort flag and the CTA winds down.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dflash {
namespace {

constexpr int kDn = 128, kDr = 64, kDv = 128;
constexpr int kBM = 128, kBN = 128;
constexpr uint32_t kPanel = kBM * 128;        // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kQBytes = 3 * kPanel;      // nope 0-63, nope 64-127, rope
constexpr uint32_t kKBytes = 3 * kPanel;
constexpr uint32_t kVBytes = 2 * kPanel;      // v 0-63, v 64-127
constexpr int kStages = 2;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + kStages * kKBytes;
constexpr uint32_t kOffBar = kOffV + kStages * kVBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // + alignment slack

// barrier slots (8 bytes each)
enum {
  BAR_Q_FULL = 0,
  BAR_Q_EMPTY = 1,
  BAR_K_FULL = 2,   // 2 stages
  BAR_K_EMPTY = 4,  // 2
  BAR_V_FULL = 6,   // 2
  BAR_V_EMPTY = 8,  // 2 (also marks "PV of this tile done")
  BAR_S_FULL = 10,  // 2
  BAR_P_FULL = 12,  // 2
  BAR_O_FULL = 14,
  BAR_DRAIN = 15,
  kNumBars = 16
};
constexpr uint32_t kOffTmemSlot = kOffBar + 8 * kNumBars;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;

constexpr int kThreads = 192;
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s per wait

constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBM, kBN, 0, 0);  // Q, K both K-major
constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBM, kDv, 0, 1);  // P from TMEM, V MN-major

struct TcArgs {
  AttnParams p;
  int segments;
  int nqt;      // query tiles per segment (max over segments for ragged)
  int n_items;  // nqt * segments * H
  int mask_vec; // dense: mask rows are 16-byte aligned
};

struct Item {
  int ok;
  int z, t, h;
  Seg sg;
  int r0, r1;
  int amin, amax;
  int nkt;
  const uint8_t* cls;
};

__device__ __forceinline__ Item decode_item(const TcArgs& a, int idx) {
  Item it;
  const AttnParams& p = a.p;
  const int zh = a.segments * p.H;
  it.t = a.nqt - 1 - idx / zh;  // longest (latest) query tiles first
  const int rem = idx % zh;
  it.z = rem / p.H;
  it.h = rem % p.H;
  it.sg = resolve_segment(p, it.z);
  it.ok = it.sg.ok;
  if (!it.ok) return it;
  it.r0 = it.t * kBM;
  if (it.r0 >= it.sg.Q) {
    it.ok = 0;
    return it;
  }
  it.r1 = min(it.r0 + kBM, it.sg.Q);
  it.nkt = (it.sg.S + it.sg.Q + kBN - 1) / kBN;
  it.cls = nullptr;
  it.amin = it.sg.S;
  it.amax = 0;
  if (p.mode == kDense) {
    it.cls = p.classes + ((long long)it.z * p.nqt + it.t) * p.nkt;
  } else {
    for (int j = it.r0 / p.bs; j <= (it.r1 - 1) / p.bs; ++j) {
      int an = p.anchors[it.sg.anc0 + j];
      an = an < 0 ? 0 : (an > it.sg.S ? it.sg.S : an);
      it.amin = min(it.amin, an);
      it.amax = max(it.amax, an);
    }
  }
  return it;
}

__device__ __forceinline__ int tile_class(const TcArgs& a, const Item& it, int kt) {
  if (a.p.mode == kDense) return it.cls[kt];
  return anchored_tile_class(it.sg.S, it.sg.Q, a.p.bs, it.r0, it.r1, it.amin, it.amax, kt);
}

__device__ __forceinline__ int next_tile(const TcArgs& a, const Item& it, int kt) {
  for (++kt; kt < it.nkt; ++kt)
    if (tile_class(a, it, kt) != DFLASH_TILE_SKIP) return kt;
  return it.nkt;
}

// Item index of this CTA's round k (snake order), or -1 when past the end.
__device__ __forceinline__ int item_of_round(const TcArgs& a, int k) {
  const int G = gridDim.x;
  const int idx = k * G + ((k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return idx;
}

struct Ctl {
  uint32_t bar0;
  volatile int* abort;
  unsigned* err;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  // Bounded wait for the completion of the phase with parity `parity`.
  __device__ bool wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    if (ptx::mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
      if (ptx::mbar_try_wait(b, parity)) return true;
      if ((n & 15u) == 0) {
        if (*abort) return false;
        if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
          *abort = 1;
          record_error(err, DFLASH_ERR_TIMEOUT);
          return false;
        }
      }
    }
  }
};

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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmemSlot);

  if (threadIdx.x == 0) {
    ptx::mbar_init(ctl.bar(BAR_Q_FULL), 1);
    ptx::mbar_init(ctl.bar(BAR_Q_EMPTY), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ctl.bar(BAR_K_FULL + s), 1);
      ptx::mbar_init(ctl.bar(BAR_K_EMPTY + s), 1);
      ptx::mbar_init(ctl.bar(BAR_V_FULL + s), 1);
      ptx::mbar_init(ctl.bar(BAR_V_EMPTY + s), 1);
      ptx::mbar_init(ctl.bar(BAR_S_FULL + s), 1);
      ptx::mbar_init(ctl.bar(BAR_P_FULL + s), 128);
    }
    ptx::mbar_init(ctl.bar(BAR_O_FULL), 1);
    ptx::mbar_init(ctl.bar(BAR_DRAIN), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t g = 0, n_items = 0;
      for (int k = 0;; ++k) {
        const int idx = item_of_round(a, k);
        if (k * (int)gridDim.x >= a.n_items) break;
        if (idx >= a.n_items) continue;
        const Item it = decode_item(a, idx);
        if (!it.ok) continue;
        if (n_items > 0 && !ctl.wait(BAR_Q_EMPTY, (n_items - 1) & 1u)) break;
        const int qrow = (int)(it.sg.q0 + it.r0);
        ptx::mbar_arrive_expect_tx(ctl.bar(BAR_Q_FULL), kQBytes);
        for (int pn = 0; pn < 3; ++pn)
          ptx::tma_load_3d(sbase + kOffQ + pn * kPanel, &tmQ, ctl.bar(BAR_Q_FULL), 64 * pn, it.h, qrow);
        ++n_items;
        bool stop = false;
        for (int kt = next_tile(a, it, -1); kt < it.nkt; kt = next_tile(a, it, kt)) {
          const int s = g & 1;
          const uint32_t u = g >> 1;
          const int krow = (int)(it.sg.kv0 + (long long)kt * kBN);
          if (!ctl.wait(BAR_K_EMPTY + s, (u & 1u) ^ 1u)) { stop = true; break; }
          const uint32_t kdst = sbase + kOffK + s * kKBytes;
          ptx::mbar_arrive_expect_tx(ctl.bar(BAR_K_FULL + s), kKBytes);
          ptx::tma_load_3d(kdst, &tmKn, ctl.bar(BAR_K_FULL + s), 0, it.h, krow);
          ptx::tma_load_3d(kdst + kPanel, &tmKn, ctl.bar(BAR_K_FULL + s), 64, it.h, krow);
          ptx::tma_load_2d(kdst + 2 * kPanel, &tmKr, ctl.bar(BAR_K_FULL + s), 0, krow);
          if (!ctl.wait(BAR_V_EMPTY + s, (u & 1u) ^ 1u)) { stop = true; break; }
          const uint32_t vdst = sbase + kOffV + s * kVBytes;
          ptx::mbar_arrive_expect_tx(ctl.bar(BAR_V_FULL + s), kVBytes);
          ptx::tma_load_3d(vdst, &tmV, ctl.bar(BAR_V_FULL + s), 0, it.h, krow);
          ptx::tma_load_3d(vdst + kPanel, &tmV, ctl.bar(BAR_V_FULL + s), 64, it.h, krow);
          ++g;
        }
        if (stop) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0, n_items = 0;
      const uint32_t sQ = sbase + kOffQ;
      auto issue_qk = [&](uint32_t gg) -> bool {
        const int s = gg & 1;
        if (!ctl.wait(BAR_K_FULL + s, (gg >> 1) & 1u)) return false;
        ptx::tc_fence_after();
        const uint32_t sK = sbase + kOffK + s * kKBytes;
        const uint32_t d = tmem + kColS + (uint32_t)s * kBN;
#pragma unroll
        for (int ks = 0; ks < (kDn + kDr) / 16; ++ks) {
          const uint32_t off = (uint32_t)(ks >> 2) * kPanel + (uint32_t)(ks & 3) * 32u;
          ptx::mma_ss(d, ptx::smem_desc(sQ + off, 16, 1024), ptx::smem_desc(sK + off, 16, 1024), kIdescQK,
                      ks > 0);
        }
        ptx::tc_commit(ctl.bar(BAR_S_FULL + s));
        ptx::tc_commit(ctl.bar(BAR_K_EMPTY + s));
        return true;
      };
      bool stop = false;
      for (int k = 0; !stop; ++k) {
        const int idx = item_of_round(a, k);
        if (k * (int)gridDim.x >= a.n_items) break;
        if (idx >= a.n_items) continue;
        const Item it = decode_item(a, idx);
        if (!it.ok) continue;
        if (!ctl.wait(BAR_Q_FULL, n_items & 1u)) break;
        ++n_items;
        int kt = next_tile(a, it, -1);
        if (kt >= it.nkt) {  // nothing visible in this tile row: no MMA, release Q
          ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));
          continue;
        }
        if (!issue_qk(g)) break;
        for (int j = 0;; ++j) {
          const int kn = next_tile(a, it, kt);
          if (kn < it.nkt) {
            if (!issue_qk(g + 1)) { stop = true; break; }
          } else {
            ptx::tc_commit(ctl.bar(BAR_Q_EMPTY));
          }
          const int s = g & 1;
          const uint32_t par = (g >> 1) & 1u;
          if (!ctl.wait(BAR_P_FULL + s, par) || !ctl.wait(BAR_V_FULL + s, par)) { stop = true; break; }
          ptx::tc_fence_after();
          const uint32_t sV = sbase + kOffV + s * kVBytes;
          const uint32_t pcol = tmem + kColP + (uint32_t)s * 64u;
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            // P columns: 16 keys = 8 packed bf16x2 columns; V rows: 16 keys = 2 x 1024-byte groups.
            ptx::mma_ts(tmem + kColO, pcol + (uint32_t)ks * 8u, ptx::smem_desc(sV + (uint32_t)ks * 2048u, kPanel, 1024),
                        kIdescPV, (j > 0 || ks > 0));
          }
          ptx::tc_commit(ctl.bar(BAR_V_EMPTY + s));
          ++g;
          if (kn >= it.nkt) {
            ptx::tc_commit(ctl.bar(BAR_O_FULL));
            break;
          }
          kt = kn;
        }
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
  } else {
    // ------------------------------------------------------------ softmax + epilogue (warps 2..5)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;             // TMEM lane = query row within the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const float c2 = p.scale_log2;
    uint32_t g = 0, n_full = 0;
    bool stop = false;
    for (int k = 0; !stop; ++k) {
      const int idx = item_of_round(a, k);
      if (k * (int)gridDim.x >= a.n_items) break;
      if (idx >= a.n_items) continue;
      const Item it = decode_item(a, idx);
      if (!it.ok) continue;
      const int i = it.r0 + row;
      const bool row_ok = i < it.r1;
      const int S = it.sg.S, Qn = it.sg.Q, K = S + Qn;
      int ctx_lim = 0, nlo = 0, nhi = 0;
      const __nv_bfloat16* mrow = nullptr;
      if (p.mode == kDense) {
        mrow = static_cast<const __nv_bfloat16*>(p.mask) + ((long long)it.z * p.Q + (row_ok ? i : 0)) * (long long)K;
      } else if (row_ok) {
        ctx_lim = row_anchor(p, it.sg, i);
        const int blk = i / p.bs;
        nlo = S + blk * p.bs;
        nhi = S + min(blk * p.bs + p.bs, Qn);
      }
      float m_used = -INFINITY, l = 0.f;
      bool any_tile = false;
      for (int kt = next_tile(a, it, -1); kt < it.nkt; kt = next_tile(a, it, kt)) {
        any_tile = true;
        const int cls = tile_class(a, it, kt);
        const int s = g & 1;
        if (!ctl.wait(BAR_S_FULL + s, (g >> 1) & 1u)) { stop = true; break; }
        ptx::tc_fence_after();
        float x[kBN];
        {
          uint32_t* xr = reinterpret_cast<uint32_t*>(x);
          const uint32_t sa = tmem + lane_off + kColS + (uint32_t)s * kBN;
          ptx::tmem_ld32(sa, xr);
          ptx::tmem_ld32(sa + 32, xr + 32);
          ptx::tmem_ld32(sa + 64, xr + 64);
          ptx::tmem_ld32(sa + 96, xr + 96);
          ptx::tmem_wait_ld();
        }
        const int k0 = kt * kBN;
        float mt = -INFINITY;
        bool scaled = false;  // x already in base-2 units (dense partial tiles)
        // A FULL tile that runs past the segment's last key still needs the
        // per-key test: the columns past S+Q hold the next segment's keys.
        const bool full = cls == DFLASH_TILE_FULL && k0 + kBN <= K;
        if (!row_ok) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) x[c] = -INFINITY;
        } else if (full) {
#pragma unroll
          for (int c = 0; c < kBN; ++c) mt = fmaxf(mt, x[c]);
        } else if (p.mode != kDense) {
          // anchored: context keys k < ctx_lim, noise keys of the row's own block
          const int c_ctx = ctx_lim - k0, c_lo = nlo - k0, c_hi = nhi - k0;
#pragma unroll
          for (int c = 0; c < kBN; ++c) {
            const bool vis = c < c_ctx || (c >= c_lo && c < c_hi);
            x[c] = vis ? x[c] : -INFINITY;
            mt = fmaxf(mt, x[c]);
          }
        } else {
          scaled = true;
          const int kmax = K - k0;
          if (a.mask_vec && kmax >= kBN) {
            const uint4* mp = reinterpret_cast<const uint4*>(mrow + k0);
#pragma unroll
            for (int v8 = 0; v8 < kBN / 8; ++v8) {
              const uint4 w = __ldg(mp + v8);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  const int c = v8 * 8 + u * 2 + hh;
                  const float mk = __uint_as_float((hh ? (ws[u] & 0xFFFF0000u) : (ws[u] << 16)));
                  x[c] = mk == -INFINITY ? -INFINITY : fmaf(x[c], c2, fmaxf(mk * kLog2e, -3.0e38f));
                  mt = fmaxf(mt, x[c]);
                }
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < kBN; ++c) {
              const float mk = c < kmax ? __bfloat162float(mrow[k0 + c]) : -INFINITY;
              x[c] = mk == -INFINITY ? -INFINITY : fmaf(x[c], c2, fmaxf(mk * kLog2e, -3.0e38f));
              mt = fmaxf(mt, x[c]);
            }
          }
        }
        const float m_tile = scaled ? mt : mt * c2;  // base-2 units
        if (m_tile != -INFINITY) {
          if (m_used == -INFINITY) {
            m_used = m_tile;  // nothing accumulated for this row yet
          } else if (m_tile > m_used + 8.0f) {
            // Rescale O and l to the new maximum once PV of the previous tile is done.
            const float alpha = ptx::ex2(m_used - m_tile);
            const uint32_t gp = g - 1;
            if (!ctl.wait(BAR_V_EMPTY + (gp & 1), (gp >> 1) & 1u)) { stop = true; break; }
            ptx::tc_fence_after();
            const uint32_t oa = tmem + lane_off + kColO;
#pragma unroll
            for (int cc = 0; cc < kDv; cc += 32) {
              uint32_t o[32];
              ptx::tmem_ld32(oa + cc, o);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              ptx::tmem_st32(oa + cc, o);
            }
            ptx::tmem_wait_st();
            l *= alpha;
            m_used = m_tile;
          }
        }
        const float msub = m_used == -INFINITY ? 0.f : m_used;
        // p = exp2(x - m) packed to bf16 pairs (lower key in the low half), written to TMEM in two halves.
        const float mul = scaled ? 1.f : c2;
        float lsum = 0.f;
        const uint32_t pa = tmem + lane_off + kColP + (uint32_t)s * 64u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float p0 = ptx::ex2(fmaf(x[64 * half + c], mul, -msub));
            const float p1 = ptx::ex2(fmaf(x[64 * half + c + 1], mul, -msub));
            lsum += p0 + p1;
            pk[c / 2] = ptx::pack_bf16x2(p0, p1);
          }
          ptx::tmem_st32(pa + 32u * half, pk);
        }
        l += lsum;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(ctl.bar(BAR_P_FULL + s));
        ++g;
      }
      if (stop) break;
      // ---- epilogue: out = O / l (bf16, round to nearest even), lse = (m + log2 l) ln 2
      uint32_t ob[kDv / 2];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (any_tile) {
        if (!ctl.wait(BAR_O_FULL, n_full & 1u)) break;
        ++n_full;
        ptx::tc_fence_after();
        const uint32_t oa = tmem + lane_off + kColO;
#pragma unroll
        for (int cc = 0; cc < kDv; cc += 32) {
          uint32_t o[32];
          ptx::tmem_ld32(oa + cc, o);
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
#pragma unroll
        for (int v = 0; v < kDv / 8; ++v) dst[v] = make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]);
        if (p.lse)
          p.lse[it.sg.lse0 + (long long)it.h * it.sg.lse_hs + i] =
              l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
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
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// rows x heads x width (bf16), box = 64 x 1 x 128, 128-byte swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, long long rows, int heads, int width) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)width * 2 * heads};
  const cuuint32_t box[3] = {64, 1, 128};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, const void* base, long long rows, int width) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
  const cuuint32_t box[2] = {64, 128};
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

}  // namespace

bool tc_supported(int dn, int dr, int dv) { return dn == kDn && dr == kDr && dv == kDv; }

cudaError_t launch_attn_tc(const AttnParams& p, int segments, int nqt, long long q_rows, long long kv_rows,
                           cudaStream_t stream) {
  TcArgs a;
  a.p = p;
  a.segments = segments;
  a.nqt = nqt;
  a.n_items = nqt * segments * p.H;
  a.mask_vec = 0;
  if (p.mode == kDense) a.mask_vec = (((uintptr_t)p.mask & 15u) == 0) && ((p.S + p.Q) % 8 == 0);
  if (a.n_items <= 0) return cudaSuccess;
  CUtensorMap mq, mkn, mkr, mv;
  if (!make_map_3d(&mq, p.q, q_rows, p.H, kDn + kDr) || !make_map_3d(&mkn, p.kn, kv_rows, p.H, kDn) ||
      !make_map_2d(&mkr, p.kr, kv_rows, kDr) || !make_map_3d(&mv, p.v, kv_rows, p.H, kDv))
    return cudaErrorInvalidValue;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  const int grid = a.n_items < nsm ? a.n_items : nsm;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, mq, mkn, mkr, mv);
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
