// common.cuh -- shared device-side definitions of the DFlash block-attention
// library (sm_103a).  Internal; the public interface is include/dflash_attn.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash_attn.h"

namespace dflash {

enum Mode : int { kDense = DFLASH_MODE_DENSE, kAnchored = DFLASH_MODE_ANCHORED, kRagged = DFLASH_MODE_RAGGED };

constexpr int kTileM = DFLASH_TILE_M;
constexpr int kTileN = DFLASH_TILE_N;
constexpr float kLog2e = 1.4426950408889634f;

// Everything a kernel needs to locate one problem.  The batched entry points
// are B "segments" of identical shape; the ragged one has R segments whose
// bounds come from the offset arrays.
struct AttnParams {
  const void* q;
  const void* kn;
  const void* kr;
  const void* v;
  const void* mask;  // dense only: [B,1,Q,S+Q]
  void* out;
  float* lse;  // nullable
  int H, dn, dr, dv;
  float scale;       // softmax scale (natural units)
  float scale_log2;  // scale * log2(e), for kernels that keep scores in base-2 units
  int mode;
  // batched (dense / anchored)
  int B, S, Q, nb, bs;
  const int32_t* anchors;
  // ragged
  int R, total_q, total_kv;
  int max_q;  // the caller's bound on every request's q_len (kernels size their grids by it)
  const int32_t* q_off;
  const int32_t* kv_off;
  // dense tile classes [B, nqt, nkt] (uint8), produced by the mask scan
  const uint8_t* classes;
  int nqt, nkt;
  unsigned* err;  // device error word
  // Bounded waits: the budget of one mbarrier wait, and (tests of the timeout
  // path only; -1 otherwise) the CTA whose producer leaves its first work
  // item's key tiles unloaded so that its consumers' waits run out.
  unsigned long long wait_ns;
  int stall_cta;
  // Backward: how many tile flags a CTA may keep in shared memory (the kernels
  // cap it at their table's size; tests of the path past the table lower it).
  int flag_tiles;
};

// One segment (batch row or request), resolved on the device.
struct Seg {
  int ok;
  int S, Q;                 // context and query lengths
  long long q0, kv0;        // first query token, first key token
  long long anc0;           // anchors index of block 0
  long long lse0, lse_hs;   // lse index of (h=0, i=0) and per-head stride
  int b;                    // batch index (dense: mask and classes)
};

__device__ __forceinline__ void record_error(unsigned* err, unsigned code) {
  if (err) atomicCAS(err, 0u, code);
}

__device__ __forceinline__ Seg resolve_segment(const AttnParams& p, int z) {
  Seg s;
  s.ok = 1;
  s.b = z;
  if (p.mode == kRagged) {
    const int q0 = p.q_off[z], q1 = p.q_off[z + 1];
    const int k0 = p.kv_off[z], k1 = p.kv_off[z + 1];
    const int ql = q1 - q0, kl = k1 - k0;
    if (q0 < 0 || k0 < 0 || q1 > p.total_q || k1 > p.total_kv || ql < p.bs || ql % p.bs != 0 ||
        q0 % p.bs != 0 || kl < ql || ql > p.max_q) {
      s.ok = 0;
      record_error(p.err, DFLASH_ERR_INVALID);
      return s;
    }
    s.S = kl - ql;
    s.Q = ql;
    s.q0 = q0;
    s.kv0 = k0;
    s.anc0 = q0 / p.bs;
    s.lse0 = q0;
    s.lse_hs = p.total_q;
  } else {
    s.S = p.S;
    s.Q = p.Q;
    s.q0 = (long long)z * p.Q;
    s.kv0 = (long long)z * (p.S + p.Q);
    s.anc0 = (long long)z * p.nb;
    s.lse0 = (long long)z * p.H * p.Q;
    s.lse_hs = p.Q;
  }
  return s;
}

// Anchor of query row i (clamped to [0, S]; out-of-range values are recorded).
__device__ __forceinline__ int row_anchor(const AttnParams& p, const Seg& s, int i) {
  int a = p.anchors[s.anc0 + i / p.bs];
  if (a < 0 || a > s.S) {
    record_error(p.err, DFLASH_ERR_INVALID);
    a = a < 0 ? 0 : s.S;
  }
  return a;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace dflash
