// tc_common.cuh -- device helpers of the tensor-core attention kernel
// (attn_tc.cu): bounded mbarrier waits and the per-row score preparation of
// the softmax.  Internal header.
#pragma once

#include <math.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dflash {
namespace tc {

constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s per wait unless the caller sets a budget
constexpr uint32_t kSleepHintNs = 100000;           // re-check the budget every ~0.1 ms of sleep

struct Ctl {
  uint32_t bar0;
  volatile int* abort;
  unsigned* err;
  uint64_t budget = kWaitBudgetNs;
  __device__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
  __device__ void give_up() const {
    *abort = 1;
    record_error(err, DFLASH_ERR_TIMEOUT);
  }
  // Bounded wait for the completion of the phase with parity `parity`.
  __device__ bool wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    if (ptx::mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
      // sleep on the barrier (woken by the phase completing) rather than spin
      if (ptx::mbar_try_wait_sleep(b, parity, kSleepHintNs)) return true;
      if (*abort) return false;
      if (ptx::globaltimer() - t0 > budget) {
        give_up();
        return false;
      }
    }
  }
  // Wind-down wait for a TMA load this thread issued: bulk copies of valid
  // memory always land, so this ignores the abort flag; it is still bounded
  // (kWaitBudgetNs) and records DFLASH_ERR_TIMEOUT if it ever runs out.
  __device__ void wait_landed(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait_sleep(b, parity, kSleepHintNs)) {
      if (ptx::globaltimer() - t0 > kWaitBudgetNs) {
        record_error(err, DFLASH_ERR_TIMEOUT);
        return;
      }
    }
  }
};

// How a softmax thread prepares a tile's scores for its row.
enum { kPrepFull = 0, kPrepAnchored = 1, kPrepDense = 2, kPrepNone = 3 };

struct PrepCtx {
  int c_ctx, c_lo, c_hi;      // anchored: visible columns c < c_ctx or c_lo <= c < c_hi
  const __nv_bfloat16* mask;  // dense: mask row at the tile's first key
  int kmax;                   // dense: columns >= kmax lie past the segment
  bool mvec;                  // dense: 16-byte mask loads allowed
  float c2;                   // scale * log2(e)
};

__device__ __forceinline__ float max64(const float* x) {
  float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    a0 = ptx::max3(a0, x[c], x[c + 1]);
    a1 = ptx::max3(a1, x[c + 2], x[c + 3]);
    a2 = ptx::max3(a2, x[c + 4], x[c + 5]);
    a3 = ptx::max3(a3, x[c + 6], x[c + 7]);
  }
  return ptx::max3(fmaxf(a0, a1), a2, a3);
}

__device__ __forceinline__ float dense_term(float s, float mk, float c2) {
  // base-2 score with the additive mask; -inf stays -inf, huge finite values are
  // clamped so that their base-2 image stays finite
  return mk == -INFINITY ? -INFINITY : fmaf(s, c2, fmaxf(mk * kLog2e, -3.0e38f));
}

// Bits [lo, hi) of a 64-bit word, clipped to [0, 64).
__device__ __forceinline__ uint64_t range_bits(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 64);
  if (hi <= lo) return 0ull;
  const uint64_t below_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
  return below_hi & ~((1ull << lo) - 1ull);
}

// Applies the row's mask to the 64 scores of tile columns [c0, c0+64) in place:
// FULL leaves raw scores, anchored sets hidden keys to -inf (raw scores stay
// raw), dense turns scores into base-2 units plus the mask, NONE sets all -inf.
// DENSE selects the mask kind at compile time, so that each kernel carries only
// its own masking code (the softmax loop is instruction-cache bound).
template <bool DENSE>
__device__ __forceinline__ void mask64(float* x, int kind, int c0, const PrepCtx& pc) {
  if (kind == kPrepFull) return;
  if (kind == kPrepNone) {
#pragma unroll
    for (int c = 0; c < 64; ++c) x[c] = -INFINITY;
    return;
  }
  if (!DENSE) {
    // visible: c < c_ctx (context below the anchor) or c_lo <= c < c_hi (own block)
    const uint64_t vis = range_bits(0, pc.c_ctx - c0) | range_bits(pc.c_lo - c0, pc.c_hi - c0);
    const uint32_t lo = (uint32_t)vis, hi = (uint32_t)(vis >> 32);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      x[c] = (lo >> c) & 1u ? x[c] : -INFINITY;
      x[32 + c] = (hi >> c) & 1u ? x[32 + c] : -INFINITY;
    }
    return;
  }
  if (pc.mvec && pc.kmax >= c0 + 64) {
    const uint4* mp = reinterpret_cast<const uint4*>(pc.mask + c0);
#pragma unroll
    for (int v8 = 0; v8 < 8; ++v8) {
      const uint4 w = __ldg(mp + v8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = v8 * 8 + u * 2;
        x[c] = dense_term(x[c], __uint_as_float(ws[u] << 16), pc.c2);
        x[c + 1] = dense_term(x[c + 1], __uint_as_float(ws[u] & 0xFFFF0000u), pc.c2);
      }
    }
  } else {
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float mk = c0 + c < pc.kmax ? __bfloat162float(pc.mask[c0 + c]) : -INFINITY;
      x[c] = dense_term(x[c], mk, pc.c2);
    }
  }
}

}  // namespace tc
}  // namespace dflash
