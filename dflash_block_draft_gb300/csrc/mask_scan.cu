// mask_scan.cu -- classify every 128x128 tile of a dense additive mask.
//
// The dense entry point receives the DFlash block mask as an additive tensor
// [B, 1, Q, S+Q] (KimiK3DFlashAttention.forward on the DFlash Kimi K3 draft
// page passes it unchanged to SDPA).  Reading it once up front lets the
// attention kernels skip all -inf tiles and skip mask reads on all-0 tiles.
// The scan is bound by HBM: each mask byte is read exactly once, with 16-byte
// loads when rows are 16-byte aligned.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dflash {
namespace {

constexpr int kScanThreads = 128;  // one CTA per tile: a 2048-tile mask fits in one wave

__device__ __forceinline__ void classify_bits(uint32_t bits, bool is_bf16, bool& zero, bool& neginf) {
  if (is_bf16) {
    zero = (bits & 0x7FFFu) == 0u;
    neginf = bits == 0xFF80u;
  } else {
    zero = (bits & 0x7FFFFFFFu) == 0u;
    neginf = bits == 0xFF800000u;
  }
}

// kVB: bytes per vector load (32 or 16; rows and base aligned to it).
template <bool kBf16, int kVB>
__global__ void __launch_bounds__(kScanThreads) mask_scan_kernel(const void* __restrict__ mask, int S, int Q,
                                                                 int nqt, int nkt, bool vec_ok,
                                                                 uint8_t* __restrict__ classes) {
  const int kt = blockIdx.x, qt = blockIdx.y, b = blockIdx.z;
  const int K = S + Q;
  const int r0 = qt * kTileM, c0 = kt * kTileN;
  const int c1 = min(c0 + kTileN, K);
  bool all_zero = true, all_ninf = true;
  if (vec_ok && c1 - c0 == kTileN) {
    // The tile's rows as kVB-byte chunks; consecutive threads take consecutive
    // chunks of a row, so a warp reads whole rows (coalesced), and every load
    // of a thread is independent of the others.
    constexpr int kVec = kBf16 ? kTileN * 2 / kVB : kTileN * 4 / kVB;  // chunks per row
#pragma unroll
    for (int t = 0; t < kVec; ++t) {
      const int c = t * kScanThreads + (int)threadIdx.x;
      const int row = r0 + c / kVec;
      if (row >= Q) continue;
      const char* p = static_cast<const char*>(mask) + (((size_t)b * Q + row) * (size_t)K + c0) * (kBf16 ? 2 : 4) +
                      kVB * (c % kVec);
      uint32_t ws[kVB / 4];
      if (kVB == 32) {
        ptx::ld_global_nc_v8(p, ws);
      } else {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        ws[0] = w.x;
        ws[1] = w.y;
        ws[2] = w.z;
        ws[3] = w.w;
      }
#pragma unroll
      for (int u = 0; u < kVB / 4; ++u) {
        bool z0, n0;
        if (kBf16) {
          bool z1, n1;
          classify_bits(ws[u] & 0xFFFFu, true, z0, n0);
          classify_bits(ws[u] >> 16, true, z1, n1);
          all_zero &= z0 && z1;
          all_ninf &= n0 && n1;
        } else {
          classify_bits(ws[u], false, z0, n0);
          all_zero &= z0;
          all_ninf &= n0;
        }
      }
    }
  } else {
    // ragged tile or unaligned rows: element by element, a row per thread
    const int row = r0 + (int)threadIdx.x;
    if (row < Q) {
      const size_t base = ((size_t)b * Q + row) * (size_t)K;
      for (int c = c0; c < c1; ++c) {
        uint32_t bits = kBf16 ? (uint32_t) static_cast<const uint16_t*>(mask)[base + c]
                              : static_cast<const uint32_t*>(mask)[base + c];
        bool z, n;
        classify_bits(bits, kBf16, z, n);
        all_zero &= z;
        all_ninf &= n;
      }
    }
  }
  const int zero = __syncthreads_and(all_zero);
  const int ninf = __syncthreads_and(all_ninf);
  if (threadIdx.x == 0) {
    uint8_t c = DFLASH_TILE_PARTIAL;
    if (zero) c = DFLASH_TILE_FULL;
    else if (ninf) c = DFLASH_TILE_SKIP;
    classes[((size_t)b * nqt + qt) * nkt + kt] = c;
  }
}

// The additive DFlash block mask of the anchored rule: row i of batch row b
// (block j = i / bs) is 0 on context keys p < a_j and on its own block's noise
// keys, -inf elsewhere.  One CTA per (row, batch row); 16-byte stores.
template <bool kBf16>
__global__ void __launch_bounds__(256) build_mask_kernel(const int32_t* __restrict__ anchors, int S, int Q, int nb,
                                                         int bs, void* __restrict__ mask, unsigned* err) {
  const int i = blockIdx.x, b = blockIdx.y;
  const int K = S + Q;
  int a = anchors[(size_t)b * nb + i / bs];
  if (a < 0 || a > S) {
    if (threadIdx.x == 0) record_error(err, DFLASH_ERR_INVALID);
    a = a < 0 ? 0 : S;
  }
  const int blk = i / bs;
  const int nlo = S + blk * bs, nhi = S + min(blk * bs + bs, Q);
  const size_t row = ((size_t)b * Q + i) * (size_t)K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const bool vis = k < a || (k >= nlo && k < nhi);
    if (kBf16) static_cast<uint16_t*>(mask)[row + k] = vis ? 0u : 0xFF80u;
    else static_cast<uint32_t*>(mask)[row + k] = vis ? 0u : 0xFF800000u;
  }
}

}  // namespace

cudaError_t launch_build_mask(const int32_t* anchors, bool bf16, int B, int S, int Q, int nb, int bs, void* mask,
                              unsigned* err, cudaStream_t stream) {
  if (B == 0 || Q == 0) return cudaSuccess;
  const dim3 grid(Q, B);
  if (bf16) build_mask_kernel<true><<<grid, 256, 0, stream>>>(anchors, S, Q, nb, bs, mask, err);
  else build_mask_kernel<false><<<grid, 256, 0, stream>>>(anchors, S, Q, nb, bs, mask, err);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mask_scan(const void* mask, bool bf16, int B, int S, int Q, uint8_t* classes,
                             cudaStream_t stream) {
  const int K = S + Q;
  const int nqt = (Q + kTileM - 1) / kTileM, nkt = (K + kTileN - 1) / kTileN;
  if (B == 0 || nqt == 0 || nkt == 0) return cudaSuccess;
  const size_t esz = bf16 ? 2 : 4;
  const bool vec32 = ((uintptr_t)mask % 32 == 0) && ((size_t)K * esz) % 32 == 0;
  const bool vec_ok = ((uintptr_t)mask % 16 == 0) && ((size_t)K * esz) % 16 == 0;
  const dim3 grid(nkt, nqt, B);
  if (bf16 && vec32)
    mask_scan_kernel<true, 32><<<grid, kScanThreads, 0, stream>>>(mask, S, Q, nqt, nkt, true, classes);
  else if (bf16)
    mask_scan_kernel<true, 16><<<grid, kScanThreads, 0, stream>>>(mask, S, Q, nqt, nkt, vec_ok, classes);
  else if (vec32)
    mask_scan_kernel<false, 32><<<grid, kScanThreads, 0, stream>>>(mask, S, Q, nqt, nkt, true, classes);
  else
    mask_scan_kernel<false, 16><<<grid, kScanThreads, 0, stream>>>(mask, S, Q, nqt, nkt, vec_ok, classes);
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
