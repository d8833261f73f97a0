// api.cu -- the C ABI: host validation, workspace layout and kernel dispatch.
//
// Every entry point validates on the host before it launches anything, then
// enqueues its kernels on the caller's stream and returns without
// synchronising.  No device memory is allocated here.
#include <limits.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dflash {

// Per-device error word for conditions only a kernel can see.
__device__ unsigned g_error_word;

namespace {
std::atomic<uint64_t> g_launches{0};
// Test fault injection (dflash_test_inject_stall): wait budget and stalled CTA.
std::atomic<unsigned long long> g_wait_ns{0};
std::atomic<int> g_stall_cta{-1};
// Test hook (dflash_test_limit_tile_flags): backward tile flags kept in shared memory.
std::atomic<int> g_flag_tiles{0};
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
}
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
std::atomic<unsigned*> g_err_ptr[kMaxDevices];

unsigned* error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return nullptr;
    p = static_cast<unsigned*>(addr);
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

bool env_flag(const char* name) {
  const char* v = getenv(name);
  return v && v[0] && strcmp(v, "0") != 0;
}

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t ctrl = 0;     // 256 B of counters for persistent kernels
  size_t classes = 0;  // dense tile classes
  size_t total = 0;
};

Layout layout_batched(int mode, int B, int S, int Q) {
  Layout L;
  L.ctrl = 0;
  size_t off = kAlign;
  if (mode == kDense) {
    const size_t nqt = (size_t)(Q + kTileM - 1) / kTileM, nkt = (size_t)(S + Q + kTileN - 1) / kTileN;
    L.classes = off;
    off += round_up((size_t)B * nqt * nkt);
  }
  L.total = off;
  return L;
}

// Backward workspace: [ctrl | classes (dense) | D | dk_rope accumulator | tile maxima].
struct BwdLayout {
  size_t classes = 0, D = 0, acc = 0, amax = 0, total = 0;
};

BwdLayout layout_backward(bool dense, int B, int H, int S, int Q, int dr) {
  BwdLayout L;
  size_t off = kAlign;
  if (dense) {
    const size_t nqt = (size_t)(Q + kTileM - 1) / kTileM, nkt = (size_t)(S + Q + kTileN - 1) / kTileN;
    L.classes = off;
    off += round_up((size_t)B * nqt * nkt);
  }
  L.D = off;
  off += round_up(sizeof(float) * (size_t)B * H * Q);
  L.acc = off;
  off += round_up(sizeof(float) * (size_t)B * (S + Q) * dr);
  L.amax = off;
  off += round_up(2 * sizeof(int) * (size_t)bwd_max_qtiles(B, Q));
  L.total = off;
  return L;
}

Layout layout_ragged(int R, int H, bool decode, int total_kv) {
  Layout L;
  L.total = kAlign + (decode ? round_up(decode_workspace_bytes(R, H, total_kv)) : 0);
  return L;
}

// Ragged batches whose requests have at most 16 rows take the split-context
// decode kernels (bf16, Kimi K3 MLA head dims).
bool use_decode(dflash_dtype_t dtype, int dn, int dr, int dv, int max_q_len) {
  return dtype == DFLASH_BF16 && decode_supported(dn, dr, dv, max_q_len) && !env_flag("DFLASH_FORCE_SIMT") &&
         !env_flag("DFLASH_NO_SPLIT");
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

dflash_status_t check_heads(int H, int dn, int dr, int dv) {
  if (H <= 0 || dn < 0 || dr < 0 || dv <= 0 || dn + dr <= 0) return DFLASH_ERR_SHAPE;
  if (dn + dr > DFLASH_MAX_DQK || dv > DFLASH_MAX_DV) return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

dflash_status_t check_dims(const dflash_dims_t* d) {
  if (!d) return DFLASH_ERR_INVALID;
  if (d->B < 0 || d->S < 0 || d->Q < 0) return DFLASH_ERR_SHAPE;
  if (isnan(d->scale) || isinf(d->scale)) return DFLASH_ERR_INVALID;
  const dflash_status_t st = check_heads(d->H, d->d_nope, d->d_rope, d->d_v);
  if (st != DFLASH_OK) return st;
  // Token and element counts must stay inside the kernels' index arithmetic.
  const long long K = (long long)d->S + d->Q;
  if (K >= (1ll << 31) - kTileN) return DFLASH_ERR_UNSUPPORTED;
  if ((long long)d->B * K * d->H * (d->d_nope + d->d_rope + d->d_v) >= (1ll << 62)) return DFLASH_ERR_UNSUPPORTED;
  if (d->B > 65535 || d->H > 65535) return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

dflash_status_t check_dtype(dflash_dtype_t t) {
  return (t == DFLASH_BF16 || t == DFLASH_FP32) ? DFLASH_OK : DFLASH_ERR_DTYPE;
}

dflash_status_t check_tensors(const void* q, const void* kn, const void* kr, const void* v, void* out,
                              const float* lse, int dr) {
  if (!q || !kn || !v || !out || (dr > 0 && !kr)) return DFLASH_ERR_INVALID;
  if (!aligned16(q) || !aligned16(kn) || (dr > 0 && !aligned16(kr)) || !aligned16(v) || !aligned16(out))
    return DFLASH_ERR_ALIGN;
  if (lse && ((uintptr_t)lse & 3u)) return DFLASH_ERR_ALIGN;
  return DFLASH_OK;
}

dflash_status_t check_workspace(const void* ws, size_t bytes, size_t need) {
  if (bytes < need) return DFLASH_ERR_WORKSPACE;
  if (need > 0 && (!ws || ((uintptr_t)ws % kAlign) != 0)) return DFLASH_ERR_WORKSPACE;
  return DFLASH_OK;
}

float resolve_scale(float scale, int dn, int dr) {
  return scale > 0.f ? scale : (float)(1.0 / sqrt((double)(dn + dr)));
}

AttnParams base_params(int H, int dn, int dr, int dv, float scale, const void* q, const void* kn,
                       const void* kr, const void* v, void* out, float* lse) {
  AttnParams p;
  memset(&p, 0, sizeof p);
  p.q = q;
  p.kn = kn;
  p.kr = kr;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.H = H;
  p.dn = dn;
  p.dr = dr;
  p.dv = dv;
  p.scale = resolve_scale(scale, dn, dr);
  p.scale_log2 = (float)((double)p.scale * 1.4426950408889634);
  p.err = error_word();
  const unsigned long long w = g_wait_ns.load(std::memory_order_relaxed);
  p.wait_ns = w ? w : kDefaultWaitNs;
  p.stall_cta = g_stall_cta.load(std::memory_order_relaxed);
  const int nf = g_flag_tiles.load(std::memory_order_relaxed);
  p.flag_tiles = nf > 0 ? nf : INT_MAX;
  return p;
}

dflash_status_t launched(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA; }

// The tensor-core kernel takes bf16 with the Kimi K3 MLA head dims and token
// counts that fit TMA's 32-bit coordinates; DFLASH_FORCE_SIMT=1 routes every
// call to the exact CUDA-core kernel instead (used to test both kernels).
bool use_tc(dflash_dtype_t dtype, int dn, int dr, int dv, long long q_rows, long long kv_rows) {
  if (dtype != DFLASH_BF16 || !tc_supported(dn, dr, dv)) return false;
  if (q_rows + kTileM >= (1ll << 31) || kv_rows + kTileN >= (1ll << 31)) return false;
  return !env_flag("DFLASH_FORCE_SIMT");
}

cudaError_t launch_tc(const AttnParams& p, int segments, int nqt, long long q_rows, long long kv_rows,
                      cudaStream_t stream) {
  return launch_attn_tc(p, segments, nqt, q_rows, kv_rows, stream);
}

dflash_status_t check_ragged(int R, int H, int d_nope, int d_rope, int d_v, float scale, dflash_dtype_t dtype,
                             int block_size, int total_q, int total_kv, int max_q_len) {
  dflash_status_t st;
  if ((st = check_dtype(dtype)) != DFLASH_OK) return st;
  if (R < 0 || total_q < 0 || total_kv < 0 || max_q_len < 0 || block_size <= 0) return DFLASH_ERR_SHAPE;
  if ((st = check_heads(H, d_nope, d_rope, d_v)) != DFLASH_OK) return st;
  if (isnan(scale) || isinf(scale)) return DFLASH_ERR_INVALID;
  if (R > 65535 || H > 65535) return DFLASH_ERR_UNSUPPORTED;
  return DFLASH_OK;
}

AttnParams ragged_params(int R, int H, int dn, int dr, int dv, float scale, const void* q, const void* kn,
                         const void* kr, const void* v, const int32_t* q_offsets, const int32_t* kv_offsets,
                         const int32_t* anchors, int bs, int total_q, int total_kv, int max_q_len, void* out,
                         float* lse) {
  AttnParams p = base_params(H, dn, dr, dv, scale, q, kn, kr, v, out, lse);
  p.mode = kRagged;
  p.R = R;
  p.total_q = total_q;
  p.total_kv = total_kv;
  p.max_q = max_q_len;
  p.q_off = q_offsets;
  p.kv_off = kv_offsets;
  p.anchors = anchors;
  p.bs = bs;
  return p;
}

// Kernel choice for a validated ragged call: the split-context decode kernels,
// the tensor-core kernel, or the exact CUDA-core kernel.
dflash_status_t ragged_dispatch(const AttnParams& p, dflash_dtype_t dtype, bool decode, void* decode_ws,
                                cudaStream_t stream) {
  if (decode && (long long)p.total_q + kTileM < (1ll << 31) && (long long)p.total_kv + kTileN < (1ll << 31))
    return launched(launch_attn_decode(p, decode_ws, stream));
  if (use_tc(dtype, p.dn, p.dr, p.dv, p.total_q, p.total_kv))
    return launched(launch_tc(p, p.R, (p.max_q + kTileM - 1) / kTileM, p.total_q, p.total_kv, stream));
  return launched(launch_attn_simt(p, dtype == DFLASH_BF16, p.R, p.max_q, stream));
}

// Workspace of the compressed-latent entry point: the absorbed tensor-core
// path's buffers, or the expanded keys and values plus the ragged kernels'
// workspace.  DFLASH_LATENT_EXPAND=1 (tests) forces the expanded path.
struct LatentLayout {
  bool absorbed = false, decode = false;
  size_t absorbed_ws = 0, kn = 0, v = 0, ragged_ws = 0, total = 0;
};

LatentLayout layout_latent(int R, int H, int dn, int dr, int dv, int rank, dflash_dtype_t dtype, int total_q,
                           int total_kv, int max_q_len) {
  LatentLayout L;
  L.absorbed = dtype == DFLASH_BF16 && latent_absorbed_supported(H, dn, dr, dv, rank, max_q_len) &&
               !env_flag("DFLASH_FORCE_SIMT") && !env_flag("DFLASH_LATENT_EXPAND") &&
               (long long)total_q + kTileM < (1ll << 31) && (long long)total_kv + kTileN < (1ll << 31);
  size_t off = kAlign;
  if (L.absorbed) {
    L.absorbed_ws = off;
    off += round_up(latent_absorbed_bytes(R, H, total_q, total_kv));
  } else {
    const bool bf16 = dtype == DFLASH_BF16;
    L.kn = off;
    off += round_up((size_t)total_kv * H * dn * (bf16 ? 2 : 4));
    L.v = off;
    off += round_up((size_t)total_kv * H * dv * (bf16 ? 2 : 4));
    L.decode = use_decode(dtype, dn, dr, dv, max_q_len);
    L.ragged_ws = off;
    off += L.decode ? round_up(decode_workspace_bytes(R, H, total_kv)) : 0;
  }
  L.total = off;
  return L;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" {

const char* dflash_status_string(dflash_status_t s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID: return "invalid argument";
    case DFLASH_ERR_SHAPE: return "inconsistent shapes";
    case DFLASH_ERR_DTYPE: return "unsupported dtype";
    case DFLASH_ERR_ALIGN: return "tensor not 16-byte aligned";
    case DFLASH_ERR_UNSUPPORTED: return "shape beyond kernel limits";
    case DFLASH_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

size_t dflash_attn_workspace_size(int mode, const dflash_dims_t* dims, dflash_dtype_t dtype, int R, int H,
                                  int d_nope, int d_rope, int d_v, int total_q, int total_kv,
                                  int max_q_len) {
  if (check_dtype(dtype) != DFLASH_OK) return 0;
  if (mode == kDense || mode == kAnchored) {
    if (check_dims(dims) != DFLASH_OK) return 0;
    return layout_batched(mode, dims->B, dims->S, dims->Q).total;
  }
  if (mode == DFLASH_MODE_DENSE_BACKWARD || mode == DFLASH_MODE_ANCHORED_BACKWARD) {
    if (check_dims(dims) != DFLASH_OK) return 0;
    return layout_backward(mode == DFLASH_MODE_DENSE_BACKWARD, dims->B, dims->H, dims->S, dims->Q, dims->d_rope)
        .total;
  }
  if (mode == kRagged) {
    if (R <= 0 || check_heads(H, d_nope, d_rope, d_v) != DFLASH_OK || total_q < 0 || total_kv < 0 ||
        max_q_len < 0)
      return 0;
    return layout_ragged(R, H, use_decode(dtype, d_nope, d_rope, d_v, max_q_len), total_kv).total;
  }
  return 0;
}

dflash_status_t dflash_build_schedule_host(int B, int S, int Q, const int32_t* anchors, int nb, int block_size,
                                           uint8_t* classes) {
  if (B < 0 || S < 0 || Q < 0 || nb < 0 || block_size <= 0) return DFLASH_ERR_SHAPE;
  if ((long long)nb * block_size != Q) return DFLASH_ERR_SHAPE;
  if ((B > 0 && Q > 0 && !anchors) || !classes) return DFLASH_ERR_INVALID;
  const int nqt = (Q + kTileM - 1) / kTileM, nkt = (S + Q + kTileN - 1) / kTileN;
  for (long long i = 0; i < (long long)B * nb; ++i)
    if (anchors[i] < 0 || anchors[i] > S) return DFLASH_ERR_INVALID;
  for (int b = 0; b < B; ++b)
    for (int qt = 0; qt < nqt; ++qt) {
      const int r0 = qt * kTileM, r1 = r0 + kTileM < Q ? r0 + kTileM : Q;
      int amin = S, amax = 0;
      for (int j = r0 / block_size; j <= (r1 - 1) / block_size; ++j) {
        const int a = anchors[(size_t)b * nb + j];
        amin = a < amin ? a : amin;
        amax = a > amax ? a : amax;
      }
      for (int kt = 0; kt < nkt; ++kt)
        classes[((size_t)b * nqt + qt) * nkt + kt] =
            (uint8_t)anchored_tile_class(S, Q, block_size, r0, r1, amin, amax, kt);
    }
  return DFLASH_OK;
}

dflash_status_t dflash_scan_mask(int B, int S, int Q, dflash_dtype_t dtype, const void* mask, uint8_t* classes,
                                 dflash_stream_t stream) {
  if (check_dtype(dtype) != DFLASH_OK) return DFLASH_ERR_DTYPE;
  if (B < 0 || S < 0 || Q < 0) return DFLASH_ERR_SHAPE;
  if (B == 0 || Q == 0) return DFLASH_OK;
  if (!mask || !classes) return DFLASH_ERR_INVALID;
  return launched(launch_mask_scan(mask, dtype == DFLASH_BF16, B, S, Q, classes, (cudaStream_t)stream));
}

dflash_status_t dflash_build_mask(int B, int S, int Q, const int32_t* anchors, int nb, int block_size,
                                  dflash_dtype_t dtype, void* mask, dflash_stream_t stream) {
  if (check_dtype(dtype) != DFLASH_OK) return DFLASH_ERR_DTYPE;
  if (B < 0 || S < 0 || Q < 0 || nb < 0 || block_size <= 0 || (long long)nb * block_size != Q)
    return DFLASH_ERR_SHAPE;
  if ((long long)S + Q >= (1ll << 31) || Q > (1 << 30) || B > 65535) return DFLASH_ERR_UNSUPPORTED;
  if (B == 0 || Q == 0) return DFLASH_OK;
  if (!anchors || !mask) return DFLASH_ERR_INVALID;
  return launched(launch_build_mask(anchors, dtype == DFLASH_BF16, B, S, Q, nb, block_size, mask, error_word(),
                                    (cudaStream_t)stream));
}

dflash_status_t dflash_attn_dense(const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                  const void* k_nope, const void* k_rope, const void* v, const void* mask,
                                  void* out, float* lse, void* workspace, size_t ws_bytes,
                                  dflash_stream_t stream) {
  dflash_status_t st;
  if ((st = check_dtype(dtype)) != DFLASH_OK) return st;
  if ((st = check_dims(dims)) != DFLASH_OK) return st;
  if (dims->B == 0 || dims->Q == 0) return DFLASH_OK;
  if ((st = check_tensors(q, k_nope, k_rope, v, out, lse, dims->d_rope)) != DFLASH_OK) return st;
  if (!mask) return DFLASH_ERR_INVALID;
  if (!aligned16(mask)) return DFLASH_ERR_ALIGN;
  const Layout L = layout_batched(kDense, dims->B, dims->S, dims->Q);
  if ((st = check_workspace(workspace, ws_bytes, L.total)) != DFLASH_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool bf16 = dtype == DFLASH_BF16;
  uint8_t* classes = static_cast<uint8_t*>(workspace) + L.classes;
  cudaError_t e = launch_mask_scan(mask, bf16, dims->B, dims->S, dims->Q, classes, s);
  if (e != cudaSuccess) return DFLASH_ERR_CUDA;
  AttnParams p = base_params(dims->H, dims->d_nope, dims->d_rope, dims->d_v, dims->scale, q, k_nope, k_rope, v,
                             out, lse);
  p.mode = kDense;
  p.mask = mask;
  p.B = dims->B;
  p.S = dims->S;
  p.Q = dims->Q;
  p.classes = classes;
  p.nqt = (dims->Q + kTileM - 1) / kTileM;
  p.nkt = (dims->S + dims->Q + kTileN - 1) / kTileN;
  const long long q_rows = (long long)dims->B * dims->Q, kv_rows = (long long)dims->B * (dims->S + dims->Q);
  if (use_tc(dtype, dims->d_nope, dims->d_rope, dims->d_v, q_rows, kv_rows))
    return launched(launch_tc(p, dims->B, p.nqt, q_rows, kv_rows, s));
  return launched(launch_attn_simt(p, bf16, dims->B, dims->Q, s));
}

dflash_status_t dflash_attn_anchored(const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                     const void* k_nope, const void* k_rope, const void* v,
                                     const int32_t* anchors, int nb, int block_size, void* out, float* lse,
                                     void* workspace, size_t ws_bytes, dflash_stream_t stream) {
  dflash_status_t st;
  if ((st = check_dtype(dtype)) != DFLASH_OK) return st;
  if ((st = check_dims(dims)) != DFLASH_OK) return st;
  if (block_size <= 0 || nb < 0 || (long long)nb * block_size != dims->Q) return DFLASH_ERR_SHAPE;
  if (dims->B == 0 || dims->Q == 0) return DFLASH_OK;
  if ((st = check_tensors(q, k_nope, k_rope, v, out, lse, dims->d_rope)) != DFLASH_OK) return st;
  if (!anchors) return DFLASH_ERR_INVALID;
  const Layout L = layout_batched(kAnchored, dims->B, dims->S, dims->Q);
  if ((st = check_workspace(workspace, ws_bytes, L.total)) != DFLASH_OK) return st;
  AttnParams p = base_params(dims->H, dims->d_nope, dims->d_rope, dims->d_v, dims->scale, q, k_nope, k_rope, v,
                             out, lse);
  p.mode = kAnchored;
  p.B = dims->B;
  p.S = dims->S;
  p.Q = dims->Q;
  p.nb = nb;
  p.bs = block_size;
  p.anchors = anchors;
  const long long q_rows = (long long)dims->B * dims->Q, kv_rows = (long long)dims->B * (dims->S + dims->Q);
  if (use_tc(dtype, dims->d_nope, dims->d_rope, dims->d_v, q_rows, kv_rows))
    return launched(launch_tc(p, dims->B, (dims->Q + kTileM - 1) / kTileM, q_rows, kv_rows,
                                   (cudaStream_t)stream));
  return launched(launch_attn_simt(p, dtype == DFLASH_BF16, dims->B, dims->Q, (cudaStream_t)stream));
}

dflash_status_t dflash_attn_ragged(int R, int H, int d_nope, int d_rope, int d_v, float scale,
                                   dflash_dtype_t dtype, const void* q, const void* k_nope, const void* k_rope,
                                   const void* v, const int32_t* q_offsets, const int32_t* kv_offsets,
                                   const int32_t* anchors, int block_size, int total_q, int total_kv,
                                   int max_q_len, void* out, float* lse, void* workspace, size_t ws_bytes,
                                   dflash_stream_t stream) {
  dflash_status_t st;
  if ((st = check_ragged(R, H, d_nope, d_rope, d_v, scale, dtype, block_size, total_q, total_kv, max_q_len)) !=
      DFLASH_OK)
    return st;
  if (R == 0 || total_q == 0) return DFLASH_OK;
  if ((st = check_tensors(q, k_nope, k_rope, v, out, lse, d_rope)) != DFLASH_OK) return st;
  if (!q_offsets || !kv_offsets || !anchors) return DFLASH_ERR_INVALID;
  if (max_q_len == 0) return DFLASH_ERR_SHAPE;
  const bool decode = use_decode(dtype, d_nope, d_rope, d_v, max_q_len);
  const Layout L = layout_ragged(R, H, decode, total_kv);
  if ((st = check_workspace(workspace, ws_bytes, L.total)) != DFLASH_OK) return st;
  AttnParams p = ragged_params(R, H, d_nope, d_rope, d_v, scale, q, k_nope, k_rope, v, q_offsets, kv_offsets, anchors,
                               block_size, total_q, total_kv, max_q_len, out, lse);
  return ragged_dispatch(p, dtype, decode, static_cast<uint8_t*>(workspace) + kAlign, (cudaStream_t)stream);
}

size_t dflash_attn_latent_workspace_size(int R, int H, int d_nope, int d_rope, int d_v, int kv_rank,
                                         dflash_dtype_t dtype, int total_q, int total_kv, int max_q_len) {
  if (check_dtype(dtype) != DFLASH_OK || R <= 0 || check_heads(H, d_nope, d_rope, d_v) != DFLASH_OK ||
      kv_rank <= 0 || kv_rank > DFLASH_MAX_KV_RANK || total_q < 0 || total_kv < 0 || max_q_len < 0)
    return 0;
  return layout_latent(R, H, d_nope, d_rope, d_v, kv_rank, dtype, total_q, total_kv, max_q_len).total;
}

dflash_status_t dflash_attn_latent_ragged(int R, int H, int d_nope, int d_rope, int d_v, int kv_rank, float scale,
                                          dflash_dtype_t dtype, const void* q, const void* c_kv, const void* k_rope,
                                          const void* w_kv_b, const int32_t* q_offsets, const int32_t* kv_offsets,
                                          const int32_t* anchors, int block_size, int total_q, int total_kv,
                                          int max_q_len, void* out, float* lse, void* workspace, size_t ws_bytes,
                                          dflash_stream_t stream) {
  dflash_status_t st;
  if ((st = check_ragged(R, H, d_nope, d_rope, d_v, scale, dtype, block_size, total_q, total_kv, max_q_len)) !=
      DFLASH_OK)
    return st;
  if (kv_rank <= 0) return DFLASH_ERR_SHAPE;
  if (kv_rank > DFLASH_MAX_KV_RANK) return DFLASH_ERR_UNSUPPORTED;
  if (R == 0 || total_q == 0) return DFLASH_OK;
  if (!q || !c_kv || !w_kv_b || !out || (d_rope > 0 && !k_rope)) return DFLASH_ERR_INVALID;
  if (!aligned16(q) || !aligned16(c_kv) || !aligned16(w_kv_b) || !aligned16(out) || (d_rope > 0 && !aligned16(k_rope)))
    return DFLASH_ERR_ALIGN;
  if (lse && ((uintptr_t)lse & 3u)) return DFLASH_ERR_ALIGN;
  if (!q_offsets || !kv_offsets || !anchors) return DFLASH_ERR_INVALID;
  if (max_q_len == 0) return DFLASH_ERR_SHAPE;
  const LatentLayout L = layout_latent(R, H, d_nope, d_rope, d_v, kv_rank, dtype, total_q, total_kv, max_q_len);
  if ((st = check_workspace(workspace, ws_bytes, L.total)) != DFLASH_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  cudaStream_t s = (cudaStream_t)stream;
  if (L.absorbed) {
    AttnParams p = ragged_params(R, H, d_nope, d_rope, d_v, scale, q, nullptr, k_rope, nullptr, q_offsets,
                                 kv_offsets, anchors, block_size, total_q, total_kv, max_q_len, out, lse);
    return launched(launch_latent_absorbed(p, c_kv, w_kv_b, w + L.absorbed_ws, s));
  }
  // Expanded: per-head keys and values in the workspace, then the ragged kernels.
  void* kn = w + L.kn;
  void* vv = w + L.v;
  cudaError_t e = launch_latent_expand(c_kv, w_kv_b, dtype == DFLASH_BF16, total_kv, H, d_nope, d_v, kv_rank, kn, vv, s);
  if (e != cudaSuccess) return DFLASH_ERR_CUDA;
  AttnParams p = ragged_params(R, H, d_nope, d_rope, d_v, scale, q, kn, k_rope, vv, q_offsets, kv_offsets, anchors,
                               block_size, total_q, total_kv, max_q_len, out, lse);
  return ragged_dispatch(p, dtype, L.decode, w + L.ragged_ws, s);
}

}  // extern "C"

namespace dflash {
namespace {

// Shared validation and launch of the two backward entry points.
dflash_status_t backward_common(bool dense, const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                const void* kn, const void* kr, const void* v, const int32_t* anchors, int nb,
                                int bs, const void* mask, const void* out, const float* lse, const void* dout,
                                void* dq, void* dkn, void* dkr, void* dv, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  dflash_status_t st;
  if ((st = check_dtype(dtype)) != DFLASH_OK) return st;
  if ((st = check_dims(dims)) != DFLASH_OK) return st;
  if (!dense && (bs <= 0 || nb < 0 || (long long)nb * bs != dims->Q)) return DFLASH_ERR_SHAPE;
  if (dims->d_nope + dims->d_rope > DFLASH_BWD_MAX_DQK || dims->d_v > DFLASH_BWD_MAX_DV)
    return DFLASH_ERR_UNSUPPORTED;
  if (dims->B == 0 || (long long)dims->S + dims->Q == 0) return DFLASH_OK;
  if (dims->Q == 0) {
    // No query row: every key gradient is 0 (q, out, lse, dout and dq are empty).
    if (!dkn || !dv || (dims->d_rope > 0 && !dkr)) return DFLASH_ERR_INVALID;
    if (!aligned16(dkn) || !aligned16(dv) || (dims->d_rope > 0 && !aligned16(dkr))) return DFLASH_ERR_ALIGN;
    const size_t esz = dtype == DFLASH_BF16 ? 2 : 4;
    const size_t keys = (size_t)dims->B * dims->S;
    cudaError_t e = cudaMemsetAsync(dkn, 0, keys * dims->H * dims->d_nope * esz, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, keys * dims->H * dims->d_v * esz, stream);
    if (e == cudaSuccess && dims->d_rope > 0) e = cudaMemsetAsync(dkr, 0, keys * dims->d_rope * esz, stream);
    return launched(e);
  }
  if ((st = check_tensors(q, kn, kr, v, const_cast<void*>(out), lse, dims->d_rope)) != DFLASH_OK) return st;
  if (!lse || !dout || !dq || !dkn || !dv || (dims->d_rope > 0 && !dkr)) return DFLASH_ERR_INVALID;
  if ((dense && !mask) || (!dense && !anchors)) return DFLASH_ERR_INVALID;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dkn) || !aligned16(dv) ||
      (dims->d_rope > 0 && !aligned16(dkr)) || (dense && !aligned16(mask)))
    return DFLASH_ERR_ALIGN;
  const BwdLayout L = layout_backward(dense, dims->B, dims->H, dims->S, dims->Q, dims->d_rope);
  if ((st = check_workspace(ws, ws_bytes, L.total)) != DFLASH_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  AttnParams p = base_params(dims->H, dims->d_nope, dims->d_rope, dims->d_v, dims->scale, q, kn, kr, v,
                             const_cast<void*>(out), nullptr);
  p.B = dims->B;
  p.S = dims->S;
  p.Q = dims->Q;
  const bool bf16 = dtype == DFLASH_BF16;
  if (dense) {
    p.mode = kDense;
    p.mask = mask;
    p.classes = w + L.classes;
    p.nqt = (dims->Q + kTileM - 1) / kTileM;
    p.nkt = (dims->S + dims->Q + kTileN - 1) / kTileN;
    if (dims->Q > 0 &&
        launch_mask_scan(mask, bf16, dims->B, dims->S, dims->Q, w + L.classes, stream) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  } else {
    p.mode = kAnchored;
    p.nb = nb;
    p.bs = bs;
    p.anchors = anchors;
  }
  return launched(launch_attn_bwd(p, bf16, lse, dout, dq, dkn, dkr, dv, reinterpret_cast<float*>(w + L.D),
                                  reinterpret_cast<float*>(w + L.acc), reinterpret_cast<int*>(w + L.amax),
                                  stream));
}

}  // namespace
}  // namespace dflash

extern "C" {

dflash_status_t dflash_attn_anchored_backward(const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                              const void* k_nope, const void* k_rope, const void* v,
                                              const int32_t* anchors, int nb, int block_size, const void* out,
                                              const float* lse, const void* dout, void* dq, void* dk_nope,
                                              void* dk_rope, void* dv, void* workspace, size_t ws_bytes,
                                              dflash_stream_t stream) {
  return backward_common(false, dims, dtype, q, k_nope, k_rope, v, anchors, nb, block_size, nullptr, out, lse,
                         dout, dq, dk_nope, dk_rope, dv, workspace, ws_bytes, (cudaStream_t)stream);
}

dflash_status_t dflash_attn_dense_backward(const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                           const void* k_nope, const void* k_rope, const void* v, const void* mask,
                                           const void* out, const float* lse, const void* dout, void* dq,
                                           void* dk_nope, void* dk_rope, void* dv, void* workspace,
                                           size_t ws_bytes, dflash_stream_t stream) {
  return backward_common(true, dims, dtype, q, k_nope, k_rope, v, nullptr, 0, 0, mask, out, lse, dout, dq,
                         dk_nope, dk_rope, dv, workspace, ws_bytes, (cudaStream_t)stream);
}

uint64_t dflash_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

void dflash_test_inject_stall(unsigned long long wait_budget_ns, int stall_cta) {
  g_wait_ns.store(wait_budget_ns, std::memory_order_relaxed);
  g_stall_cta.store(stall_cta < 0 ? -1 : stall_cta, std::memory_order_relaxed);
}

void dflash_test_limit_tile_flags(int n) { g_flag_tiles.store(n > 0 ? n : 0, std::memory_order_relaxed); }

dflash_status_t dflash_last_device_error(dflash_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DFLASH_ERR_CUDA;
  unsigned* p = error_word();
  if (!p) return DFLASH_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return DFLASH_ERR_CUDA;
  }
  return (dflash_status_t)v;
}

}  // extern "C"
