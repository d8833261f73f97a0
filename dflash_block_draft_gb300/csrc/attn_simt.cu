// attn_simt.cu -- exact CUDA-core (FFMA) block attention for every entry point.
//
// This is the path for fp32 inputs (fp32 products and sums; no tf32) and for
// head dims the tensor-core kernel does not cover.  One CTA owns kRows query
// rows of one (segment, head); key/value chunks of kChunk keys are staged in
// shared memory as fp32 and shared by all rows, with an online (running-max)
// softmax.  Scores stay in natural units (scale * q.k + mask) so that a very
// large finite mask value cannot overflow; exponentials are taken as
// exp2((s - m) * log2 e).  Visibility follows the entry point: the dense additive
// mask (KimiK3DFlashAttention.forward of the DFlash Kimi K3 draft page), or the
// anchored block rule (context p < a_j plus the row's own block).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dflash {
namespace {

constexpr int kRows = 16;    // query rows per CTA
constexpr int kChunk = 32;   // keys per staged chunk
constexpr int kThreads = 128;
constexpr int kMaxJ = DFLASH_MAX_DV / 8;  // output columns per thread

template <typename T>
struct SimtKernel {
  // Shared memory layout (floats):
  //   qs [kRows][dqk+1] | ks [kChunk][dqk+1] | vs [kChunk][dv] | ps [kRows][kChunk+1]
  static __device__ void run(const AttnParams& p) {
    extern __shared__ float smem[];
    const int z = blockIdx.z, h = blockIdx.y;
    const Seg sg = resolve_segment(p, z);
    if (!sg.ok) return;
    const int r0 = blockIdx.x * kRows;
    if (r0 >= sg.Q) return;
    const int r1 = min(r0 + kRows, sg.Q);
    const int dqk = p.dn + p.dr, dv = p.dv, H = p.H;
    const int qstride = dqk + 1;
    float* qs = smem;
    float* ks = qs + kRows * qstride;
    float* vs = ks + kChunk * qstride;
    float* ps = vs + kChunk * dv;

    const int t = threadIdx.x;
    const int r = t >> 3;      // row owned by this thread (0..15)
    const int lane8 = t & 7;   // key / column slot
    const int i = r0 + r;      // query row within the segment
    const bool row_ok = i < r1;

    const T* q = static_cast<const T*>(p.q);
    const T* kn = static_cast<const T*>(p.kn);
    const T* kr = static_cast<const T*>(p.kr);
    const T* v = static_cast<const T*>(p.v);
    const T* mask = static_cast<const T*>(p.mask);

    // Stage the query rows (zeros past the segment's tail).
    for (int e = t; e < kRows * dqk; e += kThreads) {
      const int rr = e / dqk, d = e % dqk;
      float x = 0.f;
      if (r0 + rr < r1) x = to_f32(q[((sg.q0 + r0 + rr) * H + h) * (long long)dqk + d]);
      qs[rr * qstride + d] = x;
    }

    // Visibility data.
    const int K = sg.S + sg.Q;
    int a_row = 0, blk_lo = 0, blk_hi = 0, amax = 0;
    if (p.mode != kDense) {
      a_row = row_ok ? row_anchor(p, sg, i) : 0;
      amax = 0;
      for (int rr = r0; rr < r1; ++rr) amax = max(amax, row_anchor(p, sg, rr));
      blk_lo = r0 / p.bs;
      blk_hi = (r1 - 1) / p.bs;
    }
    const long long mask_row = ((long long)sg.b * p.Q + i) * (long long)K;

    float m = -INFINITY, l = 0.f;
    float o[kMaxJ];
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j) o[j] = 0.f;

    auto chunk = [&](int k0, int nk) {
      __syncthreads();  // previous chunk fully consumed
      for (int e = t; e < kChunk * dqk; e += kThreads) {
        const int kk = e / dqk, d = e % dqk;
        float x = 0.f;
        if (kk < nk) {
          const long long tok = sg.kv0 + k0 + kk;
          x = d < p.dn ? to_f32(kn[(tok * H + h) * (long long)p.dn + d])
                       : to_f32(kr[tok * (long long)p.dr + (d - p.dn)]);
        }
        ks[kk * qstride + d] = x;
      }
      for (int e = t; e < kChunk * dv; e += kThreads) {
        const int kk = e / dv, d = e % dv;
        float x = 0.f;
        if (kk < nk) x = to_f32(v[((sg.kv0 + k0 + kk) * H + h) * (long long)dv + d]);
        vs[kk * dv + d] = x;
      }
      __syncthreads();
      // Scores for keys lane8 + 8u of row r, in base-2 units.
      float s[kChunk / 8];
      float cmax = -INFINITY;
#pragma unroll
      for (int u = 0; u < kChunk / 8; ++u) {
        const int kk = lane8 + 8 * u;
        const int key = k0 + kk;
        bool vis = row_ok && kk < nk;
        float add = 0.f;
        if (vis) {
          if (p.mode == kDense) {
            add = to_f32(mask[mask_row + key]);
            vis = add != -INFINITY;
          } else {
            vis = key < sg.S ? key < a_row : ((key - sg.S) / p.bs == i / p.bs);
          }
        }
        float acc = 0.f;
        if (vis) {
          const float* qr = qs + r * qstride;
          const float* kr_ = ks + kk * qstride;
          for (int d = 0; d < dqk; ++d) acc = fmaf(qr[d], kr_[d], acc);
          s[u] = fmaf(acc, p.scale, add);
        } else {
          s[u] = -INFINITY;
        }
        cmax = fmaxf(cmax, s[u]);
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, off));
      const float m_new = fmaxf(m, cmax);
      float alpha = 1.f, psum = 0.f;
      if (m_new != -INFINITY) {
        alpha = exp2f((m - m_new) * kLog2e);  // m = -inf gives 0
#pragma unroll
        for (int u = 0; u < kChunk / 8; ++u) {
          const float pu = s[u] == -INFINITY ? 0.f : exp2f((s[u] - m_new) * kLog2e);
          s[u] = pu;
          psum += pu;
        }
      } else {
#pragma unroll
        for (int u = 0; u < kChunk / 8; ++u) s[u] = 0.f;
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l = l * alpha + psum;
      m = m_new;
#pragma unroll
      for (int u = 0; u < kChunk / 8; ++u) ps[r * (kChunk + 1) + lane8 + 8 * u] = s[u];
      __syncthreads();
#pragma unroll
      for (int j = 0; j < kMaxJ; ++j) {
        const int c = lane8 + 8 * j;
        if (c < dv) {
          float acc = o[j] * alpha;
          for (int kk = 0; kk < nk; ++kk) acc = fmaf(ps[r * (kChunk + 1) + kk], vs[kk * dv + c], acc);
          o[j] = acc;
        }
      }
    };

    auto key_range = [&](int k_begin, int k_end) {
      for (int k0 = k_begin; k0 < k_end; k0 += kChunk) chunk(k0, min(kChunk, k_end - k0));
    };

    if (p.mode == kDense) {
      const int qt = r0 / kTileM;
      const uint8_t* cls = p.classes ? p.classes + ((long long)sg.b * p.nqt + qt) * p.nkt : nullptr;
      const int nkt = (K + kTileN - 1) / kTileN;
      for (int kt = 0; kt < nkt; ++kt) {
        if (cls && cls[kt] == DFLASH_TILE_SKIP) continue;
        key_range(kt * kTileN, min(K, (kt + 1) * kTileN));
      }
    } else {
      // Context keys visible to some row, then the noise keys of the rows' blocks.
      key_range(0, min(amax, sg.S));
      key_range(sg.S + blk_lo * p.bs, sg.S + min((blk_hi + 1) * p.bs, sg.Q));
    }

    if (!row_ok) return;
    T* out = static_cast<T*>(p.out);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const long long ob = ((sg.q0 + i) * H + h) * (long long)dv;
#pragma unroll
    for (int j = 0; j < kMaxJ; ++j) {
      const int c = lane8 + 8 * j;
      if (c < dv) out[ob + c] = from_f32<T>(o[j] * inv);
    }
    if (p.lse && lane8 == 0) {
      p.lse[sg.lse0 + h * sg.lse_hs + i] = l > 0.f ? m + logf(l) : -INFINITY;
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnParams p) {
  SimtKernel<T>::run(p);
}

}  // namespace

size_t simt_smem_bytes(int dqk, int dv) {
  return sizeof(float) * ((size_t)kRows * (dqk + 1) + (size_t)kChunk * (dqk + 1) + (size_t)kChunk * dv +
                          (size_t)kRows * (kChunk + 1));
}

cudaError_t launch_attn_simt(const AttnParams& p, bool bf16, int segments, int max_q, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes(p.dn + p.dr, p.dv);
  const dim3 grid((max_q + kRows - 1) / kRows, p.H, segments);
  if (grid.x == 0 || segments == 0) return cudaSuccess;
  if (bf16) {
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attn_simt_kernel<__nv_bfloat16><<<grid, kThreads, smem, stream>>>(p);
    count_launch();
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attn_simt_kernel<float><<<grid, kThreads, smem, stream>>>(p);
    count_launch();
  }
  return cudaGetLastError();
}

}  // namespace dflash
