// internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dflash_attn.h"

namespace dflash {

struct AttnParams;

// Tile class of key tile kt (keys [kt*TILE_N, min((kt+1)*TILE_N, S+Q))) for the
// query rows [r0, r1) of one segment under the anchored rule, given the
// minimum and maximum anchor of those rows (anchors clamped to [0, S]).
//   context part [k0, min(k1,S)):  all rows see it iff min(k1,S) <= amin,
//                                   no row sees it iff k0 >= amax;
//   noise part: a row sees only its own block, so the rows together see the
//   union of their blocks [blk(r0)*bs, min((blk(r1-1)+1)*bs, Q)), and every row
//   sees every noise key only when all rows share one block that covers it.
__host__ __device__ inline int anchored_tile_class(int S, int Q, int bs, int r0, int r1, int amin, int amax,
                                                   int kt) {
  const int K = S + Q;
  const int k0 = kt * DFLASH_TILE_N;
  const int k1 = k0 + DFLASH_TILE_N < K ? k0 + DFLASH_TILE_N : K;
  const int c1 = k1 < S ? k1 : S;
  bool ctx_all = true, ctx_none = true;
  if (k0 < c1) {
    ctx_all = c1 <= amin;
    ctx_none = k0 >= amax;
  }
  const int n0 = (k0 > S ? k0 : S) - S, n1 = k1 - S;
  bool nz_all = true, nz_none = true;
  if (n0 < n1) {
    const int b_lo = r0 / bs, b_hi = (r1 - 1) / bs;
    const int u0 = b_lo * bs;
    const int u1 = (b_hi + 1) * bs < Q ? (b_hi + 1) * bs : Q;
    nz_none = n1 <= u0 || n0 >= u1;
    nz_all = b_lo == b_hi && n0 >= u0 && n1 <= u1;
  }
  if (ctx_all && nz_all) return DFLASH_TILE_FULL;
  if (ctx_none && nz_none) return DFLASH_TILE_SKIP;
  return DFLASH_TILE_PARTIAL;
}

// Launch counter behind dflash_kernel_launches(); every launcher bumps it.
void count_launch();

size_t simt_smem_bytes(int dqk, int dv);
cudaError_t launch_attn_simt(const AttnParams& p, bool bf16, int segments, int max_q, cudaStream_t stream);
// TMA tensor maps over bf16 tensors, 128-byte swizzle, box {64, 1, box_rows} / {64, box_rows}.
bool make_map_3d(CUtensorMap* m, const void* base, long long rows, int heads, int width, int box_rows);
bool make_map_2d(CUtensorMap* m, const void* base, long long rows, int width, int box_rows);
// General 3-D bf16 map, 128-byte swizzle: dims innermost first, byte strides of
// dims 1 and 2, box extents (box[0] * 2 bytes = 128).
bool make_map_3d_box(CUtensorMap* m, const void* base, const unsigned long long dims[3],
                     const unsigned long long strides_bytes[2], const unsigned box[3]);
int sm_count();

bool tc_supported(int dn, int dr, int dv);
cudaError_t launch_attn_tc(const AttnParams& p, int segments, int nqt, long long q_rows, long long kv_rows,
                           cudaStream_t stream);
// Split-context decode path (ragged batches with at most 16 rows per request).
bool decode_supported(int dn, int dr, int dv, int max_q_len);
int decode_max_units(int R, int total_kv);
size_t decode_workspace_bytes(int R, int H, int total_kv);
cudaError_t launch_attn_decode(const AttnParams& p, void* ws, cudaStream_t stream);

// Backward pass (attn_bwd.cu): prep, dq, dk/dv and rope-finish kernels.
// Workspace: D [B,H,Q] fp32, dkr_acc [B,S+Q,d_rope] fp32, tile_amax
// [2 * bwd_max_qtiles(B,Q)] int32 (largest, then smallest anchor of each query
// tile); dense calls also need p.classes.
size_t bwd_smem_bytes(int bt, int dqk, int dv);
long long bwd_max_qtiles(int B, int Q);
cudaError_t launch_attn_bwd(const AttnParams& p, bool bf16, const float* lse, const void* dout, void* dq,
                            void* dkn, void* dkr, void* dv, float* D, float* dkr_acc, int* tile_amax,
                            cudaStream_t stream);

// Tensor-core backward (attn_bwd_tc.cu) for the Kimi K3 MLA head dims (bf16):
// dq and dk/dv kernels; D, the zeroed dk_rope accumulator and the 64-row tile
// maxima come from the prep kernel of attn_bwd.cu.
bool bwd_tc_supported(int dn, int dr, int dv);
cudaError_t launch_attn_bwd_tc(const AttnParams& p, const float* lse, const void* dout, void* dq, void* dkn,
                               void* dv, const float* D, float* dkr_acc, const int* tile_amax64,
                               const int* tile_amin64, cudaStream_t stream);

// Compressed-latent ragged attention (attn_latent.cu).  Expanded path: per-head
// k_nope / v written from the latents (any dims, fp32 or bf16).  Absorbed path
// (bf16 Kimi K3 MLA dims, kv_lora_rank 512, decode-shaped requests): q
// absorption GEMM, latent attention with split-context partials, combine, and
// the output projection GEMM, all in the workspace.
size_t latent_expand_bytes(int H, int dn, int dv, int total_kv, bool bf16);
cudaError_t launch_latent_expand(const void* c_kv, const void* w, bool bf16, int total_kv, int H, int dn, int dv,
                                 int rank, void* kn_out, void* v_out, cudaStream_t stream);
bool latent_absorbed_supported(int H, int dn, int dr, int dv, int rank, int max_q_len);
size_t latent_absorbed_bytes(int R, int H, int total_q, int total_kv);
cudaError_t launch_latent_absorbed(const AttnParams& p, const void* c_kv, const void* w, void* ws,
                                   cudaStream_t stream);

cudaError_t launch_build_mask(const int32_t* anchors, bool bf16, int B, int S, int Q, int nb, int bs, void* mask,
                              unsigned* err, cudaStream_t stream);
cudaError_t launch_mask_scan(const void* mask, bool bf16, int B, int S, int Q, uint8_t* classes,
                             cudaStream_t stream);

}  // namespace dflash
