// attn_latent.cu -- ragged DFlash block attention over compressed KV latents
// (Kimi K3 MLA), sm_103a.
//
// The draft's attention is MLA: each token carries a KV latent c (kv_lora_rank
// values) and the head-shared rope key, and kv_b_proj expands the latent to
// one qk_nope + v slice per head (KimiK3DFlashAttention on the DFlash Kimi K3
// draft page; KimiK3DSparkAttention attributes kv_lora_rank and kv_b_proj on
// the DSpark Kimi K3 draft page; the Kimi K3 target page's MLA
// context-parallel attention moves exactly these kv_lora_rank + qk_rope values
// per token).  With the projection viewed per head as w[h, e, c] (rows e <
// d_nope the key part, the rest the value part):
//   k_nope[t,h] = W_UK[h] c[t],   v[t,h] = W_UV[h] c[t]
// and the attention is the ragged anchored one over those keys and values.
//
// Two ways to compute it:
//  * Expanded (any head dims, fp32 or bf16): a CUDA-core kernel writes k_nope
//    and v for every token and head into the workspace, and the ragged
//    kernels run on them.
//  * Absorbed (bf16, d_nope = d_v = 128, d_rope = 64, kv_lora_rank = 512, at
//    most 16 query rows per request -- the serving decode shape): the key
//    projection is folded into the query and the value projection applied
//    after the softmax, so the attention reads each token's 1152 bytes of
//    latent + rope key once per head group instead of 16.5 KB of expanded
//    per-head keys and values:
//      q_abs[i,h]   = [W_UK[h]^T q_nope[i,h] | q_rope[i,h]]      (head GEMM)
//      s(i,h,k)     = scale * q_abs[i,h] . [c[k] | k_rope[k]]
//      o_lat[i,h]   = sum_k softmax(s)_k c[k]                     (latent attention)
//      out[i,h]     = W_UV[h] o_lat[i,h]                          (head GEMM)
//    The latent attention shares every key between all heads, so one work
//    unit holds 64 query rows (4 heads x 16 draft tokens) against 128-key
//    tiles: S^T = K_tile Q^T (M = 128 keys, N = 64 rows, K = 576) and
//    O^T += C_tile^T P^T (M = 4 x 128 latent dims, N = 64, K = 128 keys),
//    accumulated in TMEM.  The context is split into units of kLSplit key
//    tiles whose normalised partials are merged by a log-sum-exp combine.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace dflash {
namespace {

// ============================================================================
// Expanded path: k_nope / v from the latents on CUDA cores.
// ============================================================================
constexpr int kExpTok = 32;       // tokens per CTA
constexpr int kExpThreads = 256;  // one thread per expanded row e (loops when d_nope + d_v > 256)

// CTA (token block, head): stages the tokens' latents in shared memory (fp32)
// and every thread accumulates rows e of w[h] against them, fp32 FMAs.
template <typename T>
__global__ void __launch_bounds__(kExpThreads) latent_expand_kernel(const T* __restrict__ c_kv,
                                                                    const T* __restrict__ w, int total_kv, int H,
                                                                    int dn, int dv, int rank, T* kn_out,
                                                                    T* v_out) {
  extern __shared__ float cs[];  // [kExpTok][rank]
  const int t0 = blockIdx.x * kExpTok, h = blockIdx.y;
  const int nt = min(kExpTok, total_kv - t0);
  for (int e = threadIdx.x; e < kExpTok * rank; e += blockDim.x) {
    const int t = e / rank, c = e % rank;
    cs[e] = t < nt ? to_f32(c_kv[(long long)(t0 + t) * rank + c]) : 0.f;
  }
  __syncthreads();
  const int E = dn + dv;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const T* wr = w + ((long long)h * E + e) * rank;
    float acc[kExpTok];
#pragma unroll
    for (int t = 0; t < kExpTok; ++t) acc[t] = 0.f;
    for (int c = 0; c < rank; ++c) {
      const float wv = to_f32(wr[c]);
#pragma unroll
      for (int t = 0; t < kExpTok; ++t) acc[t] = fmaf(wv, cs[t * rank + c], acc[t]);
    }
#pragma unroll
    for (int t = 0; t < kExpTok; ++t) {
      if (t >= nt) break;
      const long long tok = t0 + t;
      if (e < dn) kn_out[(tok * H + h) * dn + e] = from_f32<T>(acc[t]);
      else v_out[(tok * H + h) * dv + (e - dn)] = from_f32<T>(acc[t]);
    }
  }
}

// ============================================================================
// Head GEMM (tensor cores): for each head h and 128-row tile,
//   C[rows, n0 : n0+NT] = A_h[rows, 0:K] . B_h[n0 : n0+NT, 0:K]^T
// bf16 operands staged by TMA (128-byte swizzle), fp32 accumulator in TMEM,
// bf16 result.  A_h is a [rows, H, width] tensor at column a_col0; B_h is a
// slice of w[h] (w: [H, E, rank]).  Two uses:
//   absorb  (BMN = true):  A = q_nope, K = d_nope, B_h[n][k] = W_UK[h][k][n]
//                          (MN-major: n = latent index is contiguous);
//                          C -> q_abs[:, h, 0:rank], plus a copy of q_rope
//                          into q_abs[:, h, rank:rank+d_rope].
//   project (BMN = false): A = o_lat, K = rank, B_h[n][k] = W_UV[h][n][k]
//                          (K-major); C -> out[:, h, 0:d_v].
// One thread issues the loads (a ring of kGStages K chunks of 64) and the
// MMAs; the four warps then read one TMEM lane (row) each.
// ============================================================================
constexpr int kGThreads = 128;
constexpr uint32_t kGStages = 4;

template <int NT, bool BMN>
struct GemmCfg {
  static constexpr uint32_t kABytes = 128 * 128;           // 128 rows x 64 k
  static constexpr uint32_t kBBytes = NT * 128;            // NT x 64 k
  static constexpr uint32_t kStage = kABytes + kBBytes;
  static constexpr uint32_t kOffBar = kGStages * kStage;
  static constexpr uint32_t kSmem = kOffBar + 8 * (2 * kGStages + 2) + 16 + 1024;
  static constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, NT, 0, BMN ? 1 : 0);
};

struct GemmArgs {
  int rows, H, kchunks;   // rows of A, heads, K / 64
  int b_row0;             // first row e of w[h] in B (K-major: n rows; MN-major: k rows)
  int n0_per_tile;        // C columns per grid.z step (= NT)
  void* out;              // C base: [rows, H, out_width]
  int out_width, out_col0;
  const void* rope_src;   // absorb: q [rows, H, src_width]; copies src cols [src_col0, +rope) -> out cols [rope_dst, +rope)
  int src_width, src_col0, rope, rope_dst;
  unsigned* err;
  unsigned long long wait_ns;
};

template <int NT, bool BMN>
__global__ void __launch_bounds__(kGThreads, 1)
    head_gemm_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  using C = GemmCfg<NT, BMN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * 128, h = blockIdx.y, n0 = blockIdx.z * NT;
  enum { FULL = 0, EMPTY = kGStages, DONE = 2 * kGStages, DRAIN = 2 * kGStages + 1 };
  tc::Ctl ctl;
  ctl.bar0 = sbase + C::kOffBar;
  ctl.abort = reinterpret_cast<volatile int*>(smem + C::kOffBar + 8 * (2 * kGStages + 2));
  ctl.err = g.err;
  ctl.budget = g.wait_ns;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + 8 * (2 * kGStages + 2) + 8);
  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < kGStages; ++s) {
      ptx::mbar_init(ctl.bar(FULL + s), 1);
      ptx::mbar_init(ctl.bar(EMPTY + s), 1);
    }
    ptx::mbar_init(ctl.bar(DONE), 1);
    ptx::mbar_init(ctl.bar(DRAIN), 1);
    *ctl.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), NT);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // Loads run kGStages - 1 chunks ahead of the MMAs; every wait is bounded.
    auto load = [&](int c) -> bool {
      const uint32_t s = (uint32_t)c % kGStages;
      if (!ctl.wait(EMPTY + s, (((uint32_t)c / kGStages) & 1u) ^ 1u)) return false;
      const uint32_t a = sbase + s * C::kStage, b = a + C::kABytes;
      ptx::mbar_arrive_expect_tx(ctl.bar(FULL + s), C::kStage);
      ptx::tma_load_3d(a, &tmA, ctl.bar(FULL + s), 64 * c, h, row0);
      if (BMN) {
        // NT/64 panels of [64 k-rows x 64 n] (k = rows of w[h], n = latent index)
        for (int j = 0; j < NT / 64; ++j)
          ptx::tma_load_3d(b + j * 8192u, &tmB, ctl.bar(FULL + s), n0 + 64 * j, g.b_row0 + 64 * c, h);
      } else {
        // one panel of [NT n-rows x 64 k]
        ptx::tma_load_3d(b, &tmB, ctl.bar(FULL + s), 64 * c, g.b_row0 + n0, h);
      }
      return true;
    };
    bool ok = true;
    int issued = 0;
    for (; issued < g.kchunks && issued < (int)kGStages - 1 && ok; ++issued) ok = load(issued);
    for (int c = 0; c < g.kchunks && ok; ++c) {
      if (issued < g.kchunks) {
        ok = load(issued);
        ++issued;
        if (!ok) break;
      }
      const uint32_t s = (uint32_t)c % kGStages;
      if (!ctl.wait(FULL + s, ((uint32_t)c / kGStages) & 1u)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a = sbase + s * C::kStage, b = a + C::kABytes;
      const uint64_t da = ptx::smem_desc(a, 16, 1024);
      const uint64_t db = BMN ? ptx::smem_desc(b, 8192, 1024) : ptx::smem_desc(b, 16, 1024);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        // A and K-major B advance 32 bytes along the swizzled row; MN-major B
        // advances 16 k-rows (2048 bytes)
        const uint64_t bk = BMN ? db + ((uint32_t)(ks * 2048) >> 4) : db + ((uint32_t)(ks * 32) >> 4);
        ptx::mma_ss(tmem, da + ((uint32_t)(ks * 32) >> 4), bk, C::kIdesc, (c > 0 || ks > 0) ? 1u : 0u);
      }
      ptx::tc_commit(ctl.bar(EMPTY + s));
    }
    if (ok) ptx::tc_commit(ctl.bar(DONE));
    // Wind-down: the loads issued land and the MMAs issued complete before exit.
    for (int c = issued - (int)kGStages + 1; c < issued; ++c)
      if (c >= 0) ctl.wait_landed(FULL + (uint32_t)c % kGStages, ((uint32_t)c / kGStages) & 1u);
    ptx::tc_commit(ctl.bar(DRAIN));
    ctl.wait_landed(DRAIN, 0);
  }
  __syncwarp();
  // ---- epilogue: one row per thread
  const int row = row0 + warp * 32 + lane;
  if (__all_sync(0xffffffffu, ctl.wait(DONE, 0))) {
    ptx::tc_fence_after();
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(g.out) + ((long long)row * g.H + h) * g.out_width + g.out_col0 + n0;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int cc = 0; cc < NT; cc += 32) {
      uint32_t v[32];
      ptx::tmem_ld32(taddr + cc, v);
      ptx::tmem_wait_ld();
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = ptx::pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
      if (row < g.rows) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + cc);
#pragma unroll
        for (int e = 0; e < 4; ++e) d4[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
  }
  if (g.rope > 0 && blockIdx.z == 0 && row < g.rows) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(g.rope_src) +
                                                      ((long long)row * g.H + h) * g.src_width + g.src_col0);
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.out) +
                                          ((long long)row * g.H + h) * g.out_width + g.rope_dst);
    for (int e = 0; e < g.rope / 8; ++e) dst[e] = src[e];
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, NT);
  }
}

template <int NT, bool BMN>
cudaError_t launch_head_gemm(const GemmArgs& g, const CUtensorMap& mA, const CUtensorMap& mB, int ntiles,
                             cudaStream_t stream) {
  using C = GemmCfg<NT, BMN>;
  auto k = head_gemm_kernel<NT, BMN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
  if (e != cudaSuccess) return e;
  const dim3 grid((g.rows + 127) / 128, g.H, ntiles);
  k<<<grid, kGThreads, C::kSmem, stream>>>(g, mA, mB);
  count_launch();
  return cudaGetLastError();
}

// ============================================================================
// Latent attention (tensor cores).
// Unit = (request, split of kLSplit key tiles, group of kLHeads heads): 64
// query rows, row n = 4 * token + head-in-group (the TMA box order of q_abs).
// Warp roles (384 threads): warp 0 TMA producer; warp 1 TMEM owner and MMA
// issuer of QK over latent panels 0-3 and the rope panel and of PV for latent
// blocks 0, 1; warp 2 the MMA issuer of QK over latent panels 4-7 (its own S^T
// accumulator, which the softmax adds) and of PV for blocks 2, 3 -- two issuing
// threads interleave their N = 64 MMAs, and the S and PV barriers complete on
// both commits; warp 3 idle; warps 4..11 softmax and epilogue -- two warps per
// TMEM lane quarter (keys 32q..32q+31), each owning 32 of the 64 rows.  The
// control warpgroup gives registers back (setmaxnreg 104) so that the softmax
// warps get 200: 128*104 + 256*200 = 384*168, the launch budget.
// Shared memory: Q^T (9 panels of 64 rows x 64 dims), one key tile as 9 slots
// of 128 keys x 64 dims (8 latent panels, then the rope panel), and one 8 KB
// P^T panel (64 rows x 64 keys, bf16, K-major).  PV runs in two key halves
// through that panel: the softmax warps of keys 0-63 write it, PV of those
// keys goes out for all four latent blocks, then the warps of keys 64-127
// overwrite it and the second half goes out.  The rope slot is therefore free
// as soon as QK of a tile completes, and the next tile's rope panel loads
// while this tile's softmax and PV run; each latent slot is refilled as soon
// as the second-half PV reading it completes.
// TMEM: S^T [0,64) and [320,384) (128 keys x 64 rows, the two halves of the QK
// contraction), O^T blocks [64 + 64m, +64), m < 4 (128 latent dims x 64 rows each).
// ============================================================================
constexpr int kLRank = 512, kLDr = 64;
constexpr int kLPanels = (kLRank + kLDr) / 64;  // 9
constexpr int kLBN = 128;                       // keys per tile
constexpr int kLHeads = 4, kLTok = 16, kLRows = kLHeads * kLTok;
// At most this many key tiles per unit (3072 keys): a request's context is cut
// into ceil(tiles / kLSplit) splits of equal size (within one tile).  Each unit
// pays a Q load, a pipeline fill and an epilogue, and longer units leave a longer
// tail.  On the latent decode workload, full splits plus a remainder measured
// 1.88, 1.80, 1.83, 1.95, 1.90 and 2.09 ms for 24, 28, 32, 40, 48 and 64 tiles;
// equal splits 1.78, 1.75, 1.73, 1.75 and 1.74 ms for 16, 20, 24, 28 and 32.
constexpr int kLSplit = 24;
constexpr uint32_t kLQPanel = kLRows * 128;     // 8 KB
constexpr uint32_t kLKPanel = kLBN * 128;       // 16 KB
constexpr uint32_t kLOffQ = 0;
constexpr uint32_t kLOffK = kLPanels * kLQPanel;
constexpr uint32_t kLOffP = kLOffK + kLPanels * kLKPanel;
constexpr uint32_t kLOffBar = kLOffP + kLQPanel;
enum {
  LB_Q_FULL = 0,
  LB_Q_EMPTY = 1,
  LB_SLOT_FULL = 2,
  LB_SLOT_EMPTY = LB_SLOT_FULL + kLPanels,
  LB_S_FULL = LB_SLOT_EMPTY + kLPanels,
  LB_P_LO = LB_S_FULL + 1,     // 128 arrivals: P^T of keys 0-63 written
  LB_P_FREE = LB_P_LO + 1,     // first-half PV issued and complete: the P^T panel may be overwritten
  LB_P_HI = LB_P_FREE + 1,     // 128 arrivals: P^T of keys 64-127 written
  LB_PV_DONE = LB_P_HI + 1,    // one phase per tile
  LB_O_FULL = LB_PV_DONE + 1,
  LB_DRAIN = LB_O_FULL + 1,
  LB_DRAIN2 = LB_DRAIN + 1,    // the second PV issuer's drain
  kLBars = LB_DRAIN2 + 1
};
constexpr uint32_t kLOffSlot = kLOffBar + 8 * kLBars;
constexpr uint32_t kLOffAbort = kLOffSlot + 4;
constexpr uint32_t kLOffRed = kLOffAbort + 12;
constexpr uint32_t kLRedWords = 4 * kLRows + 9 + 3 * kLTok;  // maxima/sums [4][64], vote [3][3], token bounds [3][16]
constexpr uint32_t kLSmem = kLOffRed + 4 * kLRedWords + 1024;
static_assert(kLSmem <= 232448, "shared memory budget");
constexpr uint32_t kLTmemCols = 512;
constexpr uint32_t kLColS = 0, kLColO = 64, kLColS2 = 320;  // S^T: latent panels 0-3 + rope, and 4-7
constexpr int kLQkSplit = 4;  // QK: warp 1 takes latent panels 0-3 and the rope panel, warp 2 panels 4-7
constexpr int kLThreads = 384;
constexpr int kLLaunchRegs = 168;  // 65536 / 384, rounded down to a multiple of 8
constexpr uint32_t kLCtlRegs = 104, kLSoftRegs = 200;
static_assert(128 * kLCtlRegs + 256 * kLSoftRegs == kLThreads * kLLaunchRegs, "register split");
constexpr uint32_t kLSoftBar = 1;
constexpr uint32_t kLIdQK = ptx::idesc_bf16_f32(128, kLRows, 0, 0);  // K tile and Q^T, both K-major
constexpr uint32_t kLIdPV = ptx::idesc_bf16_f32(128, kLRows, 1, 0);  // V^T MN-major, P^T K-major

struct LatentArgs {
  AttnParams p;       // ragged segments (q_off, kv_off, anchors, bs, total_q/kv, max_q), scale, errors, waits
  const int* prefix;  // [R+1] splits per request, exclusive prefix
  float* part_o;      // [units][kLRows][kLRank], unit = (request-split) * groups + group
  float* part_lse;    // [units][kLRows] natural log
  int groups;         // H / kLHeads
  int max_slots;      // request-splits the workspace holds
};

struct LUnit {
  int ok;
  int gidx;
  Seg sg;
  int kt0, kt1;
  int amin, amax;
  long long unit;
};

__device__ __forceinline__ LUnit latent_unit(const LatentArgs& a, int u) {
  LUnit it;
  const AttnParams& p = a.p;
  it.gidx = u % a.groups;
  const int w = u / a.groups;
  int lo = 0, hi = p.R - 1;  // request r with prefix[r] <= w < prefix[r+1]
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.prefix[mid] <= w) lo = mid;
    else hi = mid - 1;
  }
  it.unit = u;
  it.sg = resolve_segment(p, lo);
  it.ok = it.sg.ok && it.sg.Q <= kLTok && w < a.max_slots;
  if (!it.ok) return it;
  const int nkt = (it.sg.S + it.sg.Q + kLBN - 1) / kLBN;
  // ceil(nkt / kLSplit) splits of equal size (within one tile)
  const int nsplit = (nkt + kLSplit - 1) / kLSplit, s = w - a.prefix[lo];
  it.kt0 = (int)((long long)s * nkt / nsplit);
  it.kt1 = (int)((long long)(s + 1) * nkt / nsplit);
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

__device__ __forceinline__ int lunit_class(const LatentArgs& a, const LUnit& it, int kt) {
  return anchored_tile_class(it.sg.S, it.sg.Q, a.p.bs, 0, it.sg.Q, it.amin, it.amax, kt);
}

__device__ __forceinline__ int lnext_tile(const LatentArgs& a, const LUnit& it, int kt) {
  for (++kt; kt < it.kt1; ++kt)
    if (lunit_class(a, it, kt) != DFLASH_TILE_SKIP) return kt;
  return it.kt1;
}

// Load order of a key tile's panels: the rope slot first, then latent 0..7.
__device__ __forceinline__ int lslot_of(int i) { return i == 0 ? kLPanels - 1 : i - 1; }

__global__ void __launch_bounds__(kLThreads, 1)
    latent_attn_kernel(const __grid_constant__ LatentArgs a, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmR) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnParams& p = a.p;
  const int n_units = a.prefix[p.R] * a.groups;

  tc::Ctl ctl;
  ctl.bar0 = sbase + kLOffBar;
  ctl.abort = reinterpret_cast<volatile int*>(smem + kLOffAbort);
  ctl.err = p.err;
  ctl.budget = p.wait_ns;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kLOffSlot);
  float* red = reinterpret_cast<float*>(smem + kLOffRed);                // [4][64]
  unsigned* vote = reinterpret_cast<unsigned*>(red + 4 * kLRows);        // [3][3]
  int* s_ctx = reinterpret_cast<int*>(vote + 9);                         // [3][16]: anchor, block lo, hi

  if (threadIdx.x == 0) {
    ptx::mbar_init(ctl.bar(LB_Q_FULL), 1);
    ptx::mbar_init(ctl.bar(LB_Q_EMPTY), 2);  // both QK issuers
    for (int s = 0; s < kLPanels; ++s) {
      ptx::mbar_init(ctl.bar(LB_SLOT_FULL + s), 1);
      ptx::mbar_init(ctl.bar(LB_SLOT_EMPTY + s), 1);
    }
    ptx::mbar_init(ctl.bar(LB_S_FULL), 2);
    ptx::mbar_init(ctl.bar(LB_P_LO), 128);
    ptx::mbar_init(ctl.bar(LB_P_FREE), 2);  // both PV issuers
    ptx::mbar_init(ctl.bar(LB_P_HI), 128);
    ptx::mbar_init(ctl.bar(LB_PV_DONE), 2);
    ptx::mbar_init(ctl.bar(LB_O_FULL), 2);
    ptx::mbar_init(ctl.bar(LB_DRAIN), 1);
    ptx::mbar_init(ctl.bar(LB_DRAIN2), 1);
    *ctl.abort = 0;
    for (int i = 0; i < 9; ++i) vote[i] = 0u;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmC);
    ptx::prefetch_tmap(&tmR);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kLTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ = sbase + kLOffQ, sK = sbase + kLOffK;
  if (warp < 4) ptx::setmaxnreg_dec<kLCtlRegs>();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pc = 0, n = 0;  // panels issued, units issued
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const LUnit it = latent_unit(a, u);
        if (!it.ok) continue;
        if (n > 0 && !ctl.wait(LB_Q_EMPTY, (n - 1) & 1u)) break;
        ptx::mbar_arrive_expect_tx(ctl.bar(LB_Q_FULL), kLPanels * kLQPanel);
        for (int pn = 0; pn < kLPanels; ++pn)
          ptx::tma_load_3d(sQ + pn * kLQPanel, &tmQ, ctl.bar(LB_Q_FULL), 64 * pn, kLHeads * it.gidx, (int)it.sg.q0);
        ++n;
        if ((int)blockIdx.x == p.stall_cta) break;  // timeout test: this unit's key tiles never arrive
        for (int kt = lnext_tile(a, it, it.kt0 - 1); kt < it.kt1 && !stop; kt = lnext_tile(a, it, kt)) {
          const int krow = (int)(it.sg.kv0 + (long long)kt * kLBN);
          // the rope panel first: its slot is freed by QK, the latent slots only by PV
          for (int ip = 0; ip < kLPanels; ++ip) {
            const int pn = lslot_of(ip);
            const uint32_t tile = pc / kLPanels;
            if (!ctl.wait(LB_SLOT_EMPTY + pn, (tile & 1u) ^ 1u)) {
              stop = true;
              break;
            }
            const uint32_t fb = ctl.bar(LB_SLOT_FULL + pn);
            ptx::mbar_arrive_expect_tx(fb, kLKPanel);
            if (pn < kLPanels - 1) ptx::tma_load_2d(sK + pn * kLKPanel, &tmC, fb, 64 * pn, krow);
            else ptx::tma_load_2d(sK + pn * kLKPanel, &tmR, fb, 0, krow);
            ++pc;
          }
        }
      }
      // Wind-down: the outstanding loads (the last kLPanels panels, the last Q)
      // land before the CTA exits.
      for (uint32_t i = pc > (uint32_t)kLPanels ? pc - kLPanels : 0u; i < pc; ++i)
        ctl.wait_landed(LB_SLOT_FULL + lslot_of((int)(i % kLPanels)), (i / kLPanels) & 1u);
      if (n > 0) ctl.wait_landed(LB_Q_FULL, (n - 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (QK of panels 0-3 + rope, PV of blocks 0, 1)
    if (lane == 0) {
      uint32_t g = 0, n = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const LUnit it = latent_unit(a, u);
        if (!it.ok) continue;
        if (!ctl.wait(LB_Q_FULL, n & 1u)) break;
        ++n;
        int kt = lnext_tile(a, it, it.kt0 - 1);
        if (kt >= it.kt1) {  // nothing visible in this split
          ptx::tc_commit(ctl.bar(LB_Q_EMPTY));
          continue;
        }
        bool first = true;
        for (;;) {
          const int kn = lnext_tile(a, it, kt);
          // S^T = K_tile Q^T.  S^T is free: the softmax read S^T of the previous
          // tile before its P^T arrival, which PV of that tile waited for.
          for (int ip = 0; ip <= kLQkSplit && !stop; ++ip) {
            const int pn = ip < kLQkSplit ? ip : kLPanels - 1;  // latent 0..3, then rope
            if (!ctl.wait(LB_SLOT_FULL + pn, g & 1u)) {
              stop = true;
              break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              ptx::mma_ss(tmem + kLColS, ptx::smem_desc(sK + pn * kLKPanel + ks * 32, 16, 1024),
                          ptx::smem_desc(sQ + pn * kLQPanel + ks * 32, 16, 1024), kLIdQK, (ip | ks) != 0);
          }
          if (stop) break;
          ptx::tc_commit(ctl.bar(LB_S_FULL));
          ptx::tc_commit(ctl.bar(LB_SLOT_EMPTY + kLPanels - 1));  // the rope slot: read by QK only
          if (kn >= it.kt1) ptx::tc_commit(ctl.bar(LB_Q_EMPTY));  // every QK of this unit issued
          // O^T += V^T P^T in two key halves through the one P^T panel; a latent
          // block's two slots are released as soon as its second half completes.
          const uint32_t sP = sbase + kLOffP;
          if (!ctl.wait(LB_P_LO, g & 1u)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int m = 0; m < 2; ++m) {  // latent blocks 0, 1 (warp 2 issues 2, 3)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              ptx::mma_ss(tmem + kLColO + 64u * m, ptx::smem_desc(sK + 2 * m * kLKPanel + ks * 2048, kLKPanel, 1024),
                          ptx::smem_desc(sP + ks * 32, 16, 1024), kLIdPV, !(first && ks == 0));
          }
          ptx::tc_commit(ctl.bar(LB_P_FREE));
          if (!ctl.wait(LB_P_HI, g & 1u)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int ks = 4; ks < 8; ++ks)
              ptx::mma_ss(tmem + kLColO + 64u * m, ptx::smem_desc(sK + 2 * m * kLKPanel + ks * 2048, kLKPanel, 1024),
                          ptx::smem_desc(sP + (ks - 4) * 32, 16, 1024), kLIdPV, 1u);
            ptx::tc_commit(ctl.bar(LB_SLOT_EMPTY + 2 * m));
            ptx::tc_commit(ctl.bar(LB_SLOT_EMPTY + 2 * m + 1));
          }
          ptx::tc_commit(ctl.bar(LB_PV_DONE));
          first = false;
          ++g;
          if (kn >= it.kt1) break;
          kt = kn;
        }
        if (stop) break;
        ptx::tc_commit(ctl.bar(LB_O_FULL));
      }
      ptx::tc_commit(ctl.bar(LB_DRAIN));
      ctl.wait_landed(LB_DRAIN, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ second MMA issuer
    // QK of latent panels 4-7 and O^T of latent blocks 2 and 3, so that the two
    // streams of N = 64 MMAs interleave; it follows the units and tiles of warp 1.
    if (lane == 0) {
      uint32_t g = 0, n = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const LUnit it = latent_unit(a, u);
        if (!it.ok) continue;
        if (!ctl.wait(LB_Q_FULL, n & 1u)) break;
        ++n;
        int kt = lnext_tile(a, it, it.kt0 - 1);
        if (kt >= it.kt1) {
          ptx::tc_commit(ctl.bar(LB_Q_EMPTY));
          continue;
        }
        bool first = true;
        const uint32_t sP = sbase + kLOffP;
        for (;;) {
          const int kn = lnext_tile(a, it, kt);
          // S^T of latent panels 4..7 into its own accumulator (the softmax adds the two)
          for (int pn = kLQkSplit; pn < kLPanels - 1 && !stop; ++pn) {
            if (!ctl.wait(LB_SLOT_FULL + pn, g & 1u)) {
              stop = true;
              break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              ptx::mma_ss(tmem + kLColS2, ptx::smem_desc(sK + pn * kLKPanel + ks * 32, 16, 1024),
                          ptx::smem_desc(sQ + pn * kLQPanel + ks * 32, 16, 1024), kLIdQK,
                          (pn != kLQkSplit || ks != 0) ? 1u : 0u);
          }
          if (stop) break;
          ptx::tc_commit(ctl.bar(LB_S_FULL));
          if (kn >= it.kt1) ptx::tc_commit(ctl.bar(LB_Q_EMPTY));
          if (!ctl.wait(LB_P_LO, g & 1u)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int m = 2; m < 4; ++m) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              ptx::mma_ss(tmem + kLColO + 64u * m, ptx::smem_desc(sK + 2 * m * kLKPanel + ks * 2048, kLKPanel, 1024),
                          ptx::smem_desc(sP + ks * 32, 16, 1024), kLIdPV, !(first && ks == 0));
          }
          ptx::tc_commit(ctl.bar(LB_P_FREE));
          if (!ctl.wait(LB_P_HI, g & 1u)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int m = 2; m < 4; ++m) {
#pragma unroll
            for (int ks = 4; ks < 8; ++ks)
              ptx::mma_ss(tmem + kLColO + 64u * m, ptx::smem_desc(sK + 2 * m * kLKPanel + ks * 2048, kLKPanel, 1024),
                          ptx::smem_desc(sP + (ks - 4) * 32, 16, 1024), kLIdPV, 1u);
            ptx::tc_commit(ctl.bar(LB_SLOT_EMPTY + 2 * m));
            ptx::tc_commit(ctl.bar(LB_SLOT_EMPTY + 2 * m + 1));
          }
          ptx::tc_commit(ctl.bar(LB_PV_DONE));
          first = false;
          ++g;
          if (kn >= it.kt1) break;
          kt = kn;
        }
        if (stop) break;
        ptx::tc_commit(ctl.bar(LB_O_FULL));
      }
      ptx::tc_commit(ctl.bar(LB_DRAIN2));
      ctl.wait_landed(LB_DRAIN2, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue (warps 4..11)
    ptx::setmaxnreg_inc<kLSoftRegs>();
    const int q = warp & 3;              // TMEM lane quarter: keys 32q .. 32q+31
    const int hf = (warp - 4) >> 2;      // rows 32hf .. 32hf+31
    const int st = threadIdx.x - 128;    // 0..255
    const int kin = q * 32 + lane;       // key within the tile
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const float c2 = p.scale_log2;
    uint32_t g = 0, n = 0, vslot = 0;
    bool stop = false;
    for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
      const LUnit it = latent_unit(a, u);
      if (!it.ok) continue;
      const int S = it.sg.S, Qn = it.sg.Q, K = S + Qn;
      if (st < kLTok) {
        // per draft token: its anchor, and its own block's noise keys [lo, hi)
        const int blk = st / p.bs;
        s_ctx[st] = st < Qn ? row_anchor(p, it.sg, st) : 0;
        s_ctx[kLTok + st] = S + blk * p.bs;
        s_ctx[2 * kLTok + st] = S + min(blk * p.bs + p.bs, Qn);
      }
      ptx::named_barrier(kLSoftBar, 256);
      // This thread's 32 rows are the 4 heads of draft tokens 8hf .. 8hf+7: the
      // visibility of its key is decided once per token and spread over the 4 rows.
      uint32_t rows_valid = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (8 * hf + u < Qn) rows_valid |= 0xFu << (4 * u);
      float m_ref[32], l_part[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        m_ref[c] = -INFINITY;
        l_part[c] = 0.f;
      }
      bool first = true;
      for (int kt = lnext_tile(a, it, it.kt0 - 1); kt < it.kt1; kt = lnext_tile(a, it, kt), ++g) {
        const int key = kt * kLBN + kin;  // this thread's key, relative to the request
        const bool full = lunit_class(a, it, kt) == DFLASH_TILE_FULL && kt * kLBN + kLBN <= K;
        // The wait result is made warp-uniform (TMEM loads are warp-collective)
        // and then group-uniform through the vote words (named barriers follow).
        // which of the half's 32 rows see this thread's key, worked out before the
        // scores arrive and without branches (four rows per draft token)
        uint32_t vmask = rows_valid;
        if (!full) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int t = 8 * hf + u;
            const uint32_t v = (uint32_t)((key < s_ctx[t]) | ((key >= s_ctx[kLTok + t]) & (key < s_ctx[2 * kLTok + t])));
            vmask &= ~((v ^ 1u) * (0xFu << (4 * u)));
          }
        }
        const bool ok = __all_sync(0xffffffffu, ctl.wait(LB_S_FULL, g & 1u));
        float x[32];
        uint32_t flags = 0;
        if (ok) {
          ptx::tc_fence_after();
          float x2[32];
          ptx::tmem_ld32(tmem + lane_off + kLColS + 32u * hf, reinterpret_cast<uint32_t*>(x));
          ptx::tmem_ld32(tmem + lane_off + kLColS2 + 32u * hf, reinterpret_cast<uint32_t*>(x2));
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) x[c] += x2[c];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            x[c] = (vmask >> c) & 1u ? x[c] * c2 : -INFINITY;
            if (x[c] > m_ref[c] + 8.0f) flags |= 1u << c;
          }
        }
        flags = __reduce_or_sync(0xffffffffu, flags);
        if (lane == 0) {
          if (flags) atomicOr(&vote[vslot * 3 + hf], flags);
          if (!ok) atomicOr(&vote[vslot * 3 + 2], 1u);
        }
        ptx::named_barrier(kLSoftBar, 256);
        const uint32_t f0 = vote[vslot * 3], f1 = vote[vslot * 3 + 1], fab = vote[vslot * 3 + 2];
        // The words two tiles ahead were last read before the previous barrier and
        // are next written after the following one: clear them now.
        if (st == 0) {
          const uint32_t v2 = vslot == 0 ? 2u : vslot - 1u;
          vote[v2 * 3] = vote[v2 * 3 + 1] = vote[v2 * 3 + 2] = 0u;
        }
        vslot = vslot == 2 ? 0 : vslot + 1;
        if (fab) {
          stop = true;
          break;
        }
        flags = hf ? f1 : f0;
        if (f0 | f1) {
          // exact tile maxima of the flagged rows (over the 128 keys: 4 warps of this half)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (!((flags >> c) & 1u)) continue;
            float mx = x[c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane == 0) red[q * kLRows + 32 * hf + c] = mx;
          }
          ptx::named_barrier(kLSoftBar, 256);
          float alpha[32];
          bool rescale = false;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            alpha[c] = 1.f;
            if (!((flags >> c) & 1u)) continue;
            const int r = 32 * hf + c;
            const float mx = fmaxf(fmaxf(red[r], red[kLRows + r]), fmaxf(red[2 * kLRows + r], red[3 * kLRows + r]));
            const float mn = fmaxf(m_ref[c], mx);
            alpha[c] = m_ref[c] == -INFINITY ? 0.f : ptx::ex2(m_ref[c] - mn);
            m_ref[c] = mn;
            l_part[c] *= alpha[c];
            rescale = true;
          }
          // rescale is uniform over this half's warps (their flags are the same word)
          if (rescale && !first) {
            // O^T columns of this half's rows scaled to the new references, once PV
            // of the previous tile has completed.
            if (__all_sync(0xffffffffu, ctl.wait(LB_PV_DONE, (g - 1) & 1u))) {
              ptx::tc_fence_after();
#pragma unroll 1
              for (int m = 0; m < 4; ++m) {
                uint32_t o[32];
                const uint32_t ta = tmem + lane_off + kLColO + 64u * m + 32u * hf;
                ptx::tmem_ld32(ta, o);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha[c]);
                ptx::tmem_st32(ta, o);
              }
              ptx::tmem_wait_st();
            }
          }
          ptx::named_barrier(kLSoftBar, 256);  // red[] is free again
        }
        // p = exp2(x - m_ref), as bf16; then P^T[row][key] into the P^T panel
        // (128-byte-swizzled K-major): keys 0-63 first, keys 64-127 once PV of
        // the first half has completed.
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = m_ref[c] == -INFINITY ? 0.f : ptx::ex2(x[c] - m_ref[c]);
          const float p1 = m_ref[c + 1] == -INFINITY ? 0.f : ptx::ex2(x[c + 1] - m_ref[c + 1]);
          l_part[c] += p0;
          l_part[c + 1] += p1;
          pk[c / 2] = ptx::pack_bf16x2(p0, p1);
        }
        const bool hi_keys = kin >= 64;  // warp-uniform: quarters 2 and 3
        if (hi_keys) ctl.wait(LB_P_FREE, g & 1u);
        uint8_t* pt = smem + kLOffP;
        const int cb = (kin & 63) * 2;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int r = 32 * hf + c;
          *reinterpret_cast<uint16_t*>(pt + r * 128 + ((((cb >> 4) ^ (r & 7))) << 4) + (cb & 15)) =
              (uint16_t)(pk[c / 2] >> (16 * (c & 1)));
        }
        ptx::fence_proxy_async_smem();  // P^T written by threads, read by the tensor core
        ptx::tc_fence_before();
        ptx::mbar_arrive(ctl.bar(hi_keys ? LB_P_HI : LB_P_LO));
        first = false;
      }
      if (stop) break;
      // ---- epilogue: partial O = O^T / l and lse for each row of this unit
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float v = l_part[c];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0) red[q * kLRows + 32 * hf + c] = v;
      }
      ptx::named_barrier(kLSoftBar, 256);
      float inv[32], lrow[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int r = 32 * hf + c;
        lrow[c] = red[r] + red[kLRows + r] + red[2 * kLRows + r] + red[3 * kLRows + r];
        inv[c] = lrow[c] > 0.f ? 1.f / lrow[c] : 0.f;
      }
      float* po = a.part_o + it.unit * (long long)(kLRows * kLRank);
      const bool have_o = !first && __all_sync(0xffffffffu, ctl.wait(LB_O_FULL, n & 1u));
      if (!first) ++n;
      if (have_o) {
        ptx::tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
          uint32_t o[32];
          ptx::tmem_ld32(tmem + lane_off + kLColO + 64u * m + 32u * hf, o);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            po[(32 * hf + c) * kLRank + 128 * m + kin] = __uint_as_float(o[c]) * inv[c];
        }
      } else {
#pragma unroll 1
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int c = 0; c < 32; ++c) po[(32 * hf + c) * kLRank + 128 * m + kin] = 0.f;
      }
      if (q == 0) {
        float mr = -INFINITY, lr = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (c == lane) {
            mr = m_ref[c];
            lr = lrow[c];
          }
        a.part_lse[it.unit * kLRows + 32 * hf + lane] =
            lr > 0.f && have_o ? (mr + log2f(lr)) * 0.6931471805599453f : -INFINITY;
      }
      ptx::named_barrier(kLSoftBar, 256);  // red[] and s_ctx[] reused by the next unit
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kLTmemCols);
  }
}

// Splits per request and their exclusive prefix (one CTA).
constexpr int kLPlanThreads = 1024;

__global__ void __launch_bounds__(kLPlanThreads) latent_plan_kernel(AttnParams p, int* prefix, int max_slots) {
  __shared__ int part[kLPlanThreads];
  const int R = p.R;
  const int per = (R + kLPlanThreads - 1) / kLPlanThreads;
  const int r0 = threadIdx.x * per, r1 = min(R, r0 + per);
  auto splits = [&](int r) -> int {
    const Seg sg = resolve_segment(p, r);
    if (!sg.ok) return 0;
    if (sg.Q > kLTok) {
      record_error(p.err, DFLASH_ERR_INVALID);
      return 0;
    }
    const int nkt = (sg.S + sg.Q + kLBN - 1) / kLBN;
    return (nkt + kLSplit - 1) / kLSplit;
  };
  int sum = 0;
  for (int r = r0; r < r1; ++r) sum += splits(r);
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int off = 1; off < kLPlanThreads; off <<= 1) {
    const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
  for (int r = r0; r < r1; ++r) {
    prefix[r] = run;
    run += splits(r);
  }
  if (threadIdx.x == kLPlanThreads - 1) {
    prefix[R] = part[kLPlanThreads - 1];
    if (part[kLPlanThreads - 1] > max_slots) record_error(p.err, DFLASH_ERR_INVALID);
  }
}

// Merge the splits of every (query row, head) into o_lat (bf16) and lse; one
// CTA of 128 threads (4 latent dims each) per (row, head).
__global__ void __launch_bounds__(128) latent_combine_kernel(AttnParams p, const int* prefix, const float* part_o,
                                                             const float* part_lse, int groups, int max_slots,
                                                             __nv_bfloat16* o_lat) {
  const int row = blockIdx.x, h = blockIdx.y;
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.q_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  const int r = lo;
  const int t = row - p.q_off[r];
  const int u0 = prefix[r], u1 = min(prefix[r + 1], max_slots);
  if (u1 <= u0 || t < 0 || t >= kLTok || t >= p.q_off[r + 1] - p.q_off[r]) {
    // a skipped request (invalid offsets, recorded by the plan kernel): its rows
    // project to 0, with lse -inf
    __nv_bfloat16* dst = o_lat + ((long long)row * p.H + h) * kLRank + 4 * threadIdx.x;
    *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
    if (p.lse && threadIdx.x == 0) p.lse[(long long)h * p.total_q + row] = -INFINITY;
    return;
  }
  const int gidx = h / kLHeads, nrow = t * kLHeads + (h % kLHeads);
  float M = -INFINITY;
  for (int w = u0; w < u1; ++w) M = fmaxf(M, part_lse[((long long)w * groups + gidx) * kLRows + nrow]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f}, wsum = 0.f;
  if (M != -INFINITY) {
    for (int w = u0; w < u1; ++w) {
      const long long unit = (long long)w * groups + gidx;
      const float ls = part_lse[unit * kLRows + nrow];
      const float wt = ls == -INFINITY ? 0.f : __expf(ls - M);
      wsum += wt;
      const float4 o = *reinterpret_cast<const float4*>(part_o + (unit * kLRows + nrow) * kLRank + 4 * threadIdx.x);
      acc[0] = fmaf(wt, o.x, acc[0]);
      acc[1] = fmaf(wt, o.y, acc[1]);
      acc[2] = fmaf(wt, o.z, acc[2]);
      acc[3] = fmaf(wt, o.w, acc[3]);
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = o_lat + ((long long)row * p.H + h) * kLRank + 4 * threadIdx.x;
  const uint32_t lo2 = ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv), hi2 = ptx::pack_bf16x2(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(dst) = make_uint2(lo2, hi2);
  if (p.lse && threadIdx.x == 0) p.lse[(long long)h * p.total_q + row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

}  // namespace

bool latent_absorbed_supported(int H, int dn, int dr, int dv, int rank, int max_q_len) {
  return dn == 128 && dr == kLDr && dv == 128 && rank == kLRank && max_q_len <= kLTok && H % kLHeads == 0;
}

static int latent_max_slots(int R, int total_kv) {
  // sum_r ceil(tiles_r / kLSplit) <= total_kv / (kLSplit * kLBN) + 2 R (tile and split rounding)
  return total_kv / (kLSplit * kLBN) + 2 * R + 1;
}

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
struct LatentLayout {
  size_t prefix, q_abs, o_lat, part_o, part_lse, total;
};
LatentLayout latent_layout(int R, int H, int total_q, int total_kv) {
  LatentLayout L;
  const size_t units = (size_t)latent_max_slots(R, total_kv) * (H / kLHeads);
  L.prefix = 0;
  L.q_abs = L.prefix + up256(sizeof(int) * (R + 1));
  L.o_lat = L.q_abs + up256((size_t)total_q * H * (kLRank + kLDr) * 2);
  L.part_o = L.o_lat + up256((size_t)total_q * H * kLRank * 2);
  L.part_lse = L.part_o + up256(units * kLRows * kLRank * sizeof(float));
  L.total = L.part_lse + up256(units * kLRows * sizeof(float));
  return L;
}
}  // namespace

size_t latent_absorbed_bytes(int R, int H, int total_q, int total_kv) {
  return latent_layout(R, H, total_q, total_kv).total;
}

cudaError_t launch_latent_absorbed(const AttnParams& p, const void* c_kv, const void* w, void* ws,
                                   cudaStream_t stream) {
  const LatentLayout L = latent_layout(p.R, p.H, p.total_q, p.total_kv);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int* prefix = reinterpret_cast<int*>(base + L.prefix);
  __nv_bfloat16* q_abs = reinterpret_cast<__nv_bfloat16*>(base + L.q_abs);
  __nv_bfloat16* o_lat = reinterpret_cast<__nv_bfloat16*>(base + L.o_lat);
  const int E = p.dn + p.dv, dqk = p.dn + p.dr, dabs = kLRank + kLDr;
  const unsigned long long H = (unsigned long long)p.H;

  // 1. q_abs = [W_UK^T q_nope | q_rope]
  CUtensorMap mq, mwk;
  {
    const unsigned long long dq[3] = {(unsigned long long)dqk, H, (unsigned long long)p.total_q};
    const unsigned long long sq[2] = {(unsigned long long)dqk * 2, (unsigned long long)dqk * 2 * H};
    const unsigned bq[3] = {64, 1, 128};
    const unsigned long long dw[3] = {(unsigned long long)kLRank, (unsigned long long)E, H};
    const unsigned long long sw[2] = {(unsigned long long)kLRank * 2, (unsigned long long)kLRank * 2 * E};
    const unsigned bw[3] = {64, 64, 1};
    if (!make_map_3d_box(&mq, p.q, dq, sq, bq) || !make_map_3d_box(&mwk, w, dw, sw, bw)) return cudaErrorInvalidValue;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.rows = p.total_q;
    g.H = p.H;
    g.kchunks = p.dn / 64;
    g.b_row0 = 0;
    g.out = q_abs;
    g.out_width = dabs;
    g.out_col0 = 0;
    g.rope_src = p.q;
    g.src_width = dqk;
    g.src_col0 = p.dn;
    g.rope = p.dr;
    g.rope_dst = kLRank;
    g.err = p.err;
    g.wait_ns = p.wait_ns;
    cudaError_t e = launch_head_gemm<256, true>(g, mq, mwk, kLRank / 256, stream);
    if (e != cudaSuccess) return e;
  }
  // 2. splits per request
  const int max_slots = latent_max_slots(p.R, p.total_kv);
  latent_plan_kernel<<<1, kLPlanThreads, 0, stream>>>(p, prefix, max_slots);
  count_launch();
  if (cudaGetLastError() != cudaSuccess) return cudaErrorLaunchFailure;
  // 3. latent attention
  {
    CUtensorMap mqa, mc, mr;
    const unsigned long long dqa[3] = {(unsigned long long)dabs, H, (unsigned long long)p.total_q};
    const unsigned long long sqa[2] = {(unsigned long long)dabs * 2, (unsigned long long)dabs * 2 * H};
    const unsigned bqa[3] = {64, (unsigned)kLHeads, (unsigned)kLTok};
    if (!make_map_3d_box(&mqa, q_abs, dqa, sqa, bqa) || !make_map_2d(&mc, c_kv, p.total_kv, kLRank, kLBN) ||
        !make_map_2d(&mr, p.kr, p.total_kv, kLDr, kLBN))
      return cudaErrorInvalidValue;
    LatentArgs a;
    a.p = p;
    a.prefix = prefix;
    a.part_o = reinterpret_cast<float*>(base + L.part_o);
    a.part_lse = reinterpret_cast<float*>(base + L.part_lse);
    a.groups = p.H / kLHeads;
    a.max_slots = max_slots;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    // The setmaxnreg split assumes the kernel launches with exactly kLLaunchRegs
    // registers per thread; any other count would make setmaxnreg.inc wait forever.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, latent_attn_kernel) != cudaSuccess || fa.numRegs != kLLaunchRegs)
      return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(latent_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLSmem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)max_slots * a.groups;
    const int grid = (int)(units < nsm ? units : nsm);
    latent_attn_kernel<<<grid, kLThreads, kLSmem, stream>>>(a, mqa, mc, mr);
    count_launch();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // 4. merge the splits: o_lat and lse
    latent_combine_kernel<<<dim3(p.total_q, p.H), 128, 0, stream>>>(p, prefix, a.part_o, a.part_lse, a.groups,
                                                                    max_slots, o_lat);
    count_launch();
  }
  // 5. out = W_UV o_lat
  {
    CUtensorMap mo, mwv;
    const unsigned long long d_o[3] = {(unsigned long long)kLRank, H, (unsigned long long)p.total_q};
    const unsigned long long s_o[2] = {(unsigned long long)kLRank * 2, (unsigned long long)kLRank * 2 * H};
    const unsigned b_o[3] = {64, 1, 128};
    const unsigned long long dw[3] = {(unsigned long long)kLRank, (unsigned long long)E, H};
    const unsigned long long sw[2] = {(unsigned long long)kLRank * 2, (unsigned long long)kLRank * 2 * E};
    const unsigned bw[3] = {64, 128, 1};
    if (!make_map_3d_box(&mo, o_lat, d_o, s_o, b_o) || !make_map_3d_box(&mwv, w, dw, sw, bw))
      return cudaErrorInvalidValue;
    GemmArgs g;
    memset(&g, 0, sizeof g);
    g.rows = p.total_q;
    g.H = p.H;
    g.kchunks = kLRank / 64;
    g.b_row0 = p.dn;
    g.out = p.out;
    g.out_width = p.dv;
    g.out_col0 = 0;
    g.err = p.err;
    g.wait_ns = p.wait_ns;
    cudaError_t e = launch_head_gemm<128, false>(g, mo, mwv, 1, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

size_t latent_expand_bytes(int H, int dn, int dv, int total_kv, bool bf16) {
  return (size_t)total_kv * H * (dn + dv) * (bf16 ? 2 : 4);
}

cudaError_t launch_latent_expand(const void* c_kv, const void* w, bool bf16, int total_kv, int H, int dn, int dv,
                                 int rank, void* kn_out, void* v_out, cudaStream_t stream) {
  if (total_kv <= 0) return cudaSuccess;
  const size_t smem = sizeof(float) * kExpTok * rank;
  const dim3 grid((total_kv + kExpTok - 1) / kExpTok, H);
  if (bf16) {
    auto k = latent_expand_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kExpThreads, smem, stream>>>(static_cast<const __nv_bfloat16*>(c_kv),
                                           static_cast<const __nv_bfloat16*>(w), total_kv, H, dn, dv, rank,
                                           static_cast<__nv_bfloat16*>(kn_out), static_cast<__nv_bfloat16*>(v_out));
  } else {
    auto k = latent_expand_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, kExpThreads, smem, stream>>>(static_cast<const float*>(c_kv), static_cast<const float*>(w), total_kv,
                                           H, dn, dv, rank, static_cast<float*>(kn_out), static_cast<float*>(v_out));
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace dflash
