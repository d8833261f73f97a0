// attn_bwd.cu -- backward pass of DFlash block attention on the CUDA cores
// (fp32 arithmetic, bf16 or fp32 tensors).
//
// The forward (KimiK3DFlashAttention.forward on the DFlash Kimi K3 draft page:
// softmax over [context | noise block] keys under the block mask) belongs to
// a draft that is trained, so its gradients are needed.  For L = sum dout . out,
// per head and query row i over the visible keys k, with P the softmax
// weights recomputed from the forward's log-sum-exp:
//   dP(i,k) = dout(i) . v(k)          D(i) = dout(i) . out(i)
//   dS(i,k) = P(i,k) (dP(i,k) - D(i))
//   dq(i)   = scale sum_k dS(i,k) [k_nope(k) | k_rope(k)]
//   dk(k)   = scale sum_i dS(i,k) q(i)     (the rope part summed over heads)
//   dv(k)   = sum_i P(i,k) dout(i)
// Kernels, in stream order:
//   bwd_prep     D per (row, head); zeroes the fp32 dk_rope accumulator; the
//                largest anchor of each query tile (anchored rule);
//   bwd_dq       one CTA per (query tile, head, batch row), looping over the
//                key tiles its rows see; dq stays in registers;
//   bwd_dkdv     one CTA per (key tile, head, batch row), looping over the
//                query tiles that see the key tile; dk_nope and dv stay in
//                registers, the rope part is added into the accumulator;
//   bwd_finish   the accumulator to dk_rope in the tensors' type.
// Tiles are BT x BT (64, or 32 when the head dims need more shared memory);
// 256 threads form a 16 x 16 grid: thread (ty, tx) owns rows ty + 16a and
// columns tx + 16c of every product it computes.
#include <math.h>
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dflash {

// Shared-memory bytes of one backward CTA with tile bt (both tile kernels use
// the same carve-up: two dqk-wide tiles, two dv-wide tiles, two bt x bt tiles
// and five per-row words).
size_t bwd_smem_bytes(int bt, int dqk, int dv) {
  return sizeof(float) * ((size_t)bt * (dqk + 1) * 2 + (size_t)bt * (dv + 1) * 2 + (size_t)bt * (bt + 1) * 2 +
                          (size_t)bt * 5);
}

namespace {

constexpr int kBwdThreads = 256;

struct BwdArgs {
  AttnParams p;      // forward problem: mode, sizes, q/k/v, anchors or mask+classes; out = forward output
  const float* lse;  // forward lse [B,H,Q] (natural log)
  const void* dout;  // [B,Q,H,dv]
  void* dq;          // [B,Q,H,dqk]
  void* dkn;         // [B,S+Q,H,dn]
  void* dkr;         // [B,S+Q,dr]
  void* dvo;         // [B,S+Q,H,dv]
  float* D;          // [B,H,Q]
  float* dkr_acc;    // [B,S+Q,dr]
  int* tile_amax;    // [B,nqt] (anchored): largest anchor of each query tile
  int* tile_amin;    // [B,nqt] (anchored): smallest anchor of each query tile
  int bt;            // tile edge
  int nqt, nkt;      // query / key tiles of bt
};

// Visibility of one query row under the anchored rule: context keys [0, ctx)
// and noise keys [nlo, nhi) (key indices within the batch row).  Rows past Q
// see nothing.
struct RowVis {
  int ctx, nlo, nhi;
};

__device__ __forceinline__ RowVis anchored_row(const AttnParams& p, int b, int i) {
  RowVis r{0, 0, 0};
  if (i >= p.Q) return r;
  int a = p.anchors[(long long)b * p.nb + i / p.bs];
  if (a < 0 || a > p.S) {
    record_error(p.err, DFLASH_ERR_INVALID);
    a = a < 0 ? 0 : p.S;
  }
  const int blk = i / p.bs;
  r.ctx = a;
  r.nlo = p.S + blk * p.bs;
  r.nhi = p.S + min(blk * p.bs + p.bs, p.Q);
  return r;
}

template <typename T>
__device__ __forceinline__ float ldf(const void* base, long long i) {
  return to_f32(static_cast<const T*>(base)[i]);
}

// Stages `rows` token rows starting at token tok0 + r0 of a [tokens, H, w]
// tensor (head h) into columns col0 .. col0+w-1 of a shared tile with row
// pitch `pitch`.  Rows at or past `limit` (relative to tok0) are zero.
template <typename T>
__device__ __forceinline__ void stage(float* dst, int pitch, int col0, const void* src, long long tok0, int r0,
                                      int limit, int H, int h, int w, int rows) {
  for (int e = threadIdx.x; e < rows * w; e += kBwdThreads) {
    const int r = e / w, d = e - r * w;
    float x = 0.f;
    if (r0 + r < limit) x = ldf<T>(src, ((tok0 + r0 + r) * H + h) * (long long)w + d);
    dst[r * pitch + col0 + d] = x;
  }
}

// Does any row of query tile [r0, r1) see any key of [k0, k1)?  Dense masks
// use the 128 x 128 tile classes of the mask scan (a BT tile lies inside one
// of them); the anchored rule uses the tile's largest anchor and its blocks.
__device__ __forceinline__ bool tile_needed(const BwdArgs& a, int b, int r0, int r1, int k0, int k1, int amax) {
  const AttnParams& p = a.p;
  if (p.mode == kDense)
    return p.classes[((long long)b * p.nqt + r0 / kTileM) * p.nkt + k0 / kTileN] != DFLASH_TILE_SKIP;
  if (k0 < p.S && k0 < amax) return true;
  const int u0 = p.S + (r0 / p.bs) * p.bs;
  const int u1 = p.S + min(((r1 - 1) / p.bs + 1) * p.bs, p.Q);
  return k0 < u1 && k1 > u0;
}

// P(i,k) and dS(i,k) of one (row, key) from the raw score dot product x and
// dP; vis_add: 0 for a visible anchored key or the dense mask value, -inf
// for an invisible key.
__device__ __forceinline__ void p_ds(float x, float dp, float add, float c2, float lse2, float Di, float& P,
                                     float& dS) {
  P = 0.f;
  dS = 0.f;
  if (add != -INFINITY) {
    P = exp2f(fmaf(x, c2, add * kLog2e) - lse2);
    dS = P * (dp - Di);
  }
}

// Additive term of (row i, key k): anchored 0 / -inf, dense the mask entry.
template <typename T>
__device__ __forceinline__ float mask_term(const AttnParams& p, int b, int i, int k, const int* rv, int r) {
  if (i >= p.Q || k >= p.S + p.Q) return -INFINITY;
  if (p.mode == kDense) return ldf<T>(p.mask, ((long long)b * p.Q + i) * (p.S + p.Q) + k);
  const bool vis = k < rv[3 * r] || (k >= rv[3 * r + 1] && k < rv[3 * r + 2]);
  return vis ? 0.f : -INFINITY;
}

// Loads lse (base 2), D and the anchored visibility of rows r0 .. r0+BT-1.
template <int BT>
__device__ __forceinline__ void stage_rows(const BwdArgs& a, int b, int h, int r0, float* lse2, float* Dr, int* rv) {
  const AttnParams& p = a.p;
  for (int r = threadIdx.x; r < BT; r += kBwdThreads) {
    const int i = r0 + r;
    const bool ok = i < p.Q;
    const long long li = ((long long)b * p.H + h) * p.Q + i;
    lse2[r] = ok ? a.lse[li] * kLog2e : 0.f;
    Dr[r] = ok ? a.D[li] : 0.f;
    RowVis v{0, 0, 0};
    if (p.mode == kAnchored) v = anchored_row(p, b, i);
    rv[3 * r] = v.ctx;
    rv[3 * r + 1] = v.nlo;
    rv[3 * r + 2] = v.nhi;
  }
}

// ---------------------------------------------------------------- prep
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) bwd_prep_kernel(const BwdArgs a) {
  const AttnParams& p = a.p;
  const long long nrows = (long long)p.B * p.Q * p.H;
  const int lane = threadIdx.x & 31;
  const long long warp0 = ((long long)blockIdx.x * kBwdThreads + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * kBwdThreads) >> 5;
  for (long long w = warp0; w < nrows; w += nwarps) {
    // w = (b*Q + i)*H + h: the row's dv values are contiguous in out and dout
    float s = 0.f;
    for (int d = lane; d < p.dv; d += 32) s += ldf<T>(p.out, w * p.dv + d) * ldf<T>(a.dout, w * p.dv + d);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const long long bi = w / p.H;
      const int h = (int)(w - bi * p.H);
      const long long b = bi / p.Q, i = bi - b * p.Q;
      a.D[(b * p.H + h) * p.Q + i] = s;
    }
  }
  const long long t0 = (long long)blockIdx.x * kBwdThreads + threadIdx.x;
  const long long nt = (long long)gridDim.x * kBwdThreads;
  const long long nacc = (long long)p.B * (p.S + p.Q) * p.dr;
  for (long long e = t0; e < nacc; e += nt) a.dkr_acc[e] = 0.f;
  if (p.mode == kAnchored) {
    for (long long e = t0; e < (long long)p.B * a.nqt; e += nt) {
      const int b = (int)(e / a.nqt), t = (int)(e - (long long)b * a.nqt);
      const int r0 = t * a.bt, r1 = min(r0 + a.bt, p.Q);
      int amax = 0, amin = p.S;
      for (int j = r0 / p.bs; j <= (r1 - 1) / p.bs; ++j) {
        const int an = min(max(p.anchors[(long long)b * p.nb + j], 0), p.S);
        amax = max(amax, an);
        amin = min(amin, an);
      }
      a.tile_amax[e] = amax;
      a.tile_amin[e] = amin;
    }
  }
}

// ---------------------------------------------------------------- dq
template <typename T, int BT>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const BwdArgs a) {
  constexpr int RT = BT / 16;
  constexpr int kMaxC = DFLASH_BWD_MAX_DQK / 16;
  extern __shared__ float smf[];
  const AttnParams& p = a.p;
  const int t = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int S = p.S, Q = p.Q, K = S + Q, dn = p.dn, dr = p.dr, dqk = dn + dr, dv = p.dv;
  const int LQ = dqk + 1, LV = dv + 1, LS = BT + 1;
  float* Qs = smf;
  float* dOs = Qs + BT * LQ;
  float* Ks = dOs + BT * LV;
  float* Vs = Ks + BT * LQ;
  float* dSs = Vs + BT * LV;
  float* lse2 = dSs + 2 * BT * LS;
  float* Dr = lse2 + BT;
  int* rv = reinterpret_cast<int*>(Dr + BT);  // [BT][3]
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int r0 = t * BT, r1 = min(r0 + BT, Q);
  const long long qtok = (long long)b * Q, ktok = (long long)b * K;
  const float c2 = p.scale_log2;

  stage<T>(Qs, LQ, 0, p.q, qtok, r0, Q, p.H, h, dqk, BT);
  stage<T>(dOs, LV, 0, a.dout, qtok, r0, Q, p.H, h, dv, BT);
  stage_rows<BT>(a, b, h, r0, lse2, Dr, rv);
  __syncthreads();
  int amax = 0;
  if (p.mode == kAnchored) amax = a.tile_amax[(long long)b * a.nqt + t];

  float acc[RT][kMaxC];
#pragma unroll
  for (int i = 0; i < RT; ++i)
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) acc[i][c] = 0.f;

  for (int kt = 0; kt < a.nkt; ++kt) {
    const int k0 = kt * BT, k1 = min(k0 + BT, K);
    if (!tile_needed(a, b, r0, r1, k0, k1, amax)) continue;
    __syncthreads();  // the previous tile's K, V and dS are no longer read
    stage<T>(Ks, LQ, 0, p.kn, ktok, k0, K, p.H, h, dn, BT);
    stage<T>(Ks, LQ, dn, p.kr, ktok, k0, K, 1, 0, dr, BT);
    stage<T>(Vs, LV, 0, p.v, ktok, k0, K, p.H, h, dv, BT);
    __syncthreads();
    // S and dP for rows ty + 16i, keys tx + 16j
    float s[RT][RT], dp[RT][RT];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < RT; ++j) s[i][j] = dp[i][j] = 0.f;
    for (int d = 0; d < dqk; ++d) {
      float qa[RT], kb[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) qa[i] = Qs[(ty + 16 * i) * LQ + d];
#pragma unroll
      for (int j = 0; j < RT; ++j) kb[j] = Ks[(tx + 16 * j) * LQ + d];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RT; ++j) s[i][j] = fmaf(qa[i], kb[j], s[i][j]);
    }
    for (int d = 0; d < dv; ++d) {
      float oa[RT], vb[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) oa[i] = dOs[(ty + 16 * i) * LV + d];
#pragma unroll
      for (int j = 0; j < RT; ++j) vb[j] = Vs[(tx + 16 * j) * LV + d];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RT; ++j) dp[i][j] = fmaf(oa[i], vb[j], dp[i][j]);
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int r = ty + 16 * i;
#pragma unroll
      for (int j = 0; j < RT; ++j) {
        const int c = tx + 16 * j;
        float P, dS;
        p_ds(s[i][j], dp[i][j], mask_term<T>(p, b, r0 + r, k0 + c, rv, r), c2, lse2[r], Dr[r], P, dS);
        dSs[r * LS + c] = dS;
      }
    }
    __syncthreads();
    // dq(rows ty + 16i, columns tx + 16c) += dS . K
    for (int kk = 0; kk < BT; ++kk) {
      float g[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) g[i] = dSs[(ty + 16 * i) * LS + kk];
#pragma unroll
      for (int c = 0; c < kMaxC; ++c) {
        const int d = tx + 16 * c;
        if (d < dqk) {
          const float kv = Ks[kk * LQ + d];
#pragma unroll
          for (int i = 0; i < RT; ++i) acc[i][c] = fmaf(g[i], kv, acc[i][c]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RT; ++i) {
    const int row = r0 + ty + 16 * i;
    if (row >= Q) continue;
    T* dst = static_cast<T*>(a.dq) + ((qtok + row) * p.H + h) * (long long)dqk;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int d = tx + 16 * c;
      if (d < dqk) dst[d] = from_f32<T>(acc[i][c] * p.scale);
    }
  }
}

// ---------------------------------------------------------------- dk, dv
template <typename T, int BT>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const BwdArgs a) {
  constexpr int RT = BT / 16;
  constexpr int kMaxC = DFLASH_BWD_MAX_DQK / 16;
  constexpr int kMaxV = DFLASH_BWD_MAX_DV / 16;
  extern __shared__ float smf[];
  const AttnParams& p = a.p;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int S = p.S, Q = p.Q, K = S + Q, dn = p.dn, dr = p.dr, dqk = dn + dr, dv = p.dv;
  const int LQ = dqk + 1, LV = dv + 1, LS = BT + 1;
  float* Qs = smf;
  float* dOs = Qs + BT * LQ;
  float* Ks = dOs + BT * LV;
  float* Vs = Ks + BT * LQ;
  float* Pt = Vs + BT * LV;   // P^T  [key][row]
  float* dSt = Pt + BT * LS;  // dS^T [key][row]
  float* lse2 = dSt + BT * LS;
  float* Dr = lse2 + BT;
  int* rv = reinterpret_cast<int*>(Dr + BT);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  const int k0 = kt * BT, k1 = min(k0 + BT, K);
  const long long qtok = (long long)b * Q, ktok = (long long)b * K;
  const float c2 = p.scale_log2;

  stage<T>(Ks, LQ, 0, p.kn, ktok, k0, K, p.H, h, dn, BT);
  stage<T>(Ks, LQ, dn, p.kr, ktok, k0, K, 1, 0, dr, BT);
  stage<T>(Vs, LV, 0, p.v, ktok, k0, K, p.H, h, dv, BT);

  float ak[RT][kMaxC], av[RT][kMaxV];
#pragma unroll
  for (int i = 0; i < RT; ++i) {
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) ak[i][c] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxV; ++c) av[i][c] = 0.f;
  }

  for (int t = 0; t < a.nqt; ++t) {
    const int r0 = t * BT, r1 = min(r0 + BT, Q);
    const int amax = p.mode == kAnchored ? a.tile_amax[(long long)b * a.nqt + t] : 0;
    if (!tile_needed(a, b, r0, r1, k0, k1, amax)) continue;
    __syncthreads();  // the previous tile's Q, dO, P^T and dS^T are no longer read
    stage<T>(Qs, LQ, 0, p.q, qtok, r0, Q, p.H, h, dqk, BT);
    stage<T>(dOs, LV, 0, a.dout, qtok, r0, Q, p.H, h, dv, BT);
    stage_rows<BT>(a, b, h, r0, lse2, Dr, rv);
    __syncthreads();
    // S^T and dP^T for keys ty + 16i, rows tx + 16j
    float s[RT][RT], dp[RT][RT];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < RT; ++j) s[i][j] = dp[i][j] = 0.f;
    for (int d = 0; d < dqk; ++d) {
      float ka[RT], qb[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) ka[i] = Ks[(ty + 16 * i) * LQ + d];
#pragma unroll
      for (int j = 0; j < RT; ++j) qb[j] = Qs[(tx + 16 * j) * LQ + d];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RT; ++j) s[i][j] = fmaf(ka[i], qb[j], s[i][j]);
    }
    for (int d = 0; d < dv; ++d) {
      float va[RT], ob[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) va[i] = Vs[(ty + 16 * i) * LV + d];
#pragma unroll
      for (int j = 0; j < RT; ++j) ob[j] = dOs[(tx + 16 * j) * LV + d];
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < RT; ++j) dp[i][j] = fmaf(va[i], ob[j], dp[i][j]);
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int kr = ty + 16 * i;
#pragma unroll
      for (int j = 0; j < RT; ++j) {
        const int r = tx + 16 * j;
        float P, dS;
        p_ds(s[i][j], dp[i][j], mask_term<T>(p, b, r0 + r, k0 + kr, rv, r), c2, lse2[r], Dr[r], P, dS);
        Pt[kr * LS + r] = P;
        dSt[kr * LS + r] = dS;
      }
    }
    __syncthreads();
    // dv(keys ty + 16i, columns tx + 16c) += P^T . dout; dk += dS^T . q
    for (int rr = 0; rr < BT; ++rr) {
      float pw[RT], gw[RT];
#pragma unroll
      for (int i = 0; i < RT; ++i) {
        pw[i] = Pt[(ty + 16 * i) * LS + rr];
        gw[i] = dSt[(ty + 16 * i) * LS + rr];
      }
#pragma unroll
      for (int c = 0; c < kMaxV; ++c) {
        const int d = tx + 16 * c;
        if (d < dv) {
          const float o = dOs[rr * LV + d];
#pragma unroll
          for (int i = 0; i < RT; ++i) av[i][c] = fmaf(pw[i], o, av[i][c]);
        }
      }
#pragma unroll
      for (int c = 0; c < kMaxC; ++c) {
        const int d = tx + 16 * c;
        if (d < dqk) {
          const float qv = Qs[rr * LQ + d];
#pragma unroll
          for (int i = 0; i < RT; ++i) ak[i][c] = fmaf(gw[i], qv, ak[i][c]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < RT; ++i) {
    const int key = k0 + ty + 16 * i;
    if (key >= K) continue;
    T* dvd = static_cast<T*>(a.dvo) + ((ktok + key) * p.H + h) * (long long)dv;
#pragma unroll
    for (int c = 0; c < kMaxV; ++c) {
      const int d = tx + 16 * c;
      if (d < dv) dvd[d] = from_f32<T>(av[i][c]);
    }
    T* dkd = static_cast<T*>(a.dkn) + ((ktok + key) * p.H + h) * (long long)dn;
    float* racc = a.dkr_acc + (ktok + key) * (long long)dr;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int d = tx + 16 * c;
      if (d < dn) dkd[d] = from_f32<T>(ak[i][c] * p.scale);
      else if (d < dqk) atomicAdd(racc + (d - dn), ak[i][c] * p.scale);
    }
  }
}

// ---------------------------------------------------------------- finish
template <typename T>
__global__ void __launch_bounds__(kBwdThreads) bwd_finish_kernel(const float* __restrict__ acc, T* __restrict__ dst,
                                                                 long long n) {
  for (long long e = (long long)blockIdx.x * kBwdThreads + threadIdx.x; e < n;
       e += (long long)gridDim.x * kBwdThreads)
    dst[e] = from_f32<T>(acc[e]);
}

template <typename T, int BT>
cudaError_t launch_tiles(const BwdArgs& a, size_t smem, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<T, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_dkdv_kernel<T, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const AttnParams& p = a.p;
  if (a.nqt > 0) {
    bwd_dq_kernel<T, BT><<<dim3(a.nqt, p.H, p.B), kBwdThreads, smem, stream>>>(a);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  bwd_dkdv_kernel<T, BT><<<dim3(a.nkt, p.H, p.B), kBwdThreads, smem, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// bf16 with the Kimi K3 MLA head dims runs on the tensor-core kernels of
// attn_bwd_tc.cu (DFLASH_FORCE_SIMT=1 keeps it on the CUDA cores, for tests).
bool use_bwd_tc(const AttnParams& p, bool bf16) {
  if (!bf16 || !bwd_tc_supported(p.dn, p.dr, p.dv)) return false;
  if ((long long)p.B * p.Q + 128 >= (1ll << 31) || (long long)p.B * (p.S + p.Q) + 128 >= (1ll << 31)) return false;
  if ((long long)p.H * p.B * (((long long)p.S + p.Q + 127) / 128) >= (1ll << 31)) return false;  // 1-D grid
  const char* v = getenv("DFLASH_FORCE_SIMT");
  return !(v && v[0] && v[0] != '0');
}

template <typename T>
cudaError_t launch_bwd_t(const BwdArgs& a0, bool tc, cudaStream_t stream) {
  BwdArgs a = a0;
  const AttnParams& p = a.p;
  const int dqk = p.dn + p.dr;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  const int bt = tc || bwd_smem_bytes(64, dqk, p.dv) <= (size_t)optin ? 64 : 32;
  const size_t smem = bwd_smem_bytes(bt, dqk, p.dv);
  if (!tc && smem > (size_t)optin) return cudaErrorInvalidConfiguration;
  a.bt = bt;
  a.nqt = (p.Q + bt - 1) / bt;
  a.nkt = (p.S + p.Q + bt - 1) / bt;
  const long long work = std::max<long long>((long long)p.B * p.Q * p.H * 32,
                                             std::max<long long>((long long)p.B * (p.S + p.Q) * p.dr,
                                                                 (long long)p.B * a.nqt));
  const int grid = (int)std::min<long long>((work + kBwdThreads - 1) / kBwdThreads, 152ll * 16);
  bwd_prep_kernel<T><<<std::max(grid, 1), kBwdThreads, 0, stream>>>(a);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (tc)
    e = launch_attn_bwd_tc(p, a.lse, a.dout, a.dq, a.dkn, a.dvo, a.D, a.dkr_acc, a.tile_amax, a.tile_amin,
                           stream);
  else
    e = bt == 64 ? launch_tiles<T, 64>(a, smem, stream) : launch_tiles<T, 32>(a, smem, stream);
  if (e != cudaSuccess) return e;
  const long long n = (long long)p.B * (p.S + p.Q) * p.dr;
  if (n > 0) {
    const int g = (int)std::min<long long>((n + kBwdThreads - 1) / kBwdThreads, 152ll * 8);
    bwd_finish_kernel<T><<<g, kBwdThreads, 0, stream>>>(a.dkr_acc, static_cast<T*>(a.dkr), n);
    count_launch();
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnParams& p, bool bf16, const float* lse, const void* dout, void* dq,
                            void* dkn, void* dkr, void* dv, float* D, float* dkr_acc, int* tile_amax,
                            cudaStream_t stream) {
  BwdArgs a;
  a.p = p;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dkn = dkn;
  a.dkr = dkr;
  a.dvo = dv;
  a.D = D;
  a.dkr_acc = dkr_acc;
  a.tile_amax = tile_amax;
  a.tile_amin = tile_amax + bwd_max_qtiles(p.B, p.Q);
  a.bt = 0;
  a.nqt = a.nkt = 0;
  return bf16 ? launch_bwd_t<__nv_bfloat16>(a, use_bwd_tc(p, true), stream) : launch_bwd_t<float>(a, false, stream);
}

// Largest query-tile count the backward's tile-maximum array must hold.
long long bwd_max_qtiles(int B, int Q) { return (long long)B * ((Q + 31) / 32); }

}  // namespace dflash
