/*
 * dflash_attn.h -- C ABI of the GB300 (sm_103a) DFlash draft block-attention
 * library.
 *
 * The operation.  A DFlash draft predicts a whole block of block_size tokens
 * in one non-causal forward whose keys and values are
 * [projected target-hidden context (S tokens) | noise block (Q tokens)]
 * (nemo_automodel.components.speculative.dflash.draft_kimi_k3 page, module
 * docstring).  Queries are the Q noise (draft) tokens: per
 * KimiK3DFlashAttention.forward the query axis has blocks x block_size rows
 * and the key axis the sequence plus those rows.  The backbone is Kimi K3
 * MLA: one K/V per query head with no GQA repeat (KimiK3DFlashAttention), and
 * NoPE: the rope part of the key is one vector per token, shared by all
 * heads, with no rotary embedding (module docstring).  Per head h, query row
 * i and key k:
 *
 *   s(i,k) = ( q_nope(i,h) . k_nope(k,h) + q_rope(i,h) . k_rope(k) ) * scale
 *            [+ mask(i,k) on the dense entry point]
 *   out(i,h) = sum_k softmax_k(s(i,.)) v(k,h)
 *
 * with scale = (d_nope + d_rope)^-0.5 by default
 * (nemo_automodel.components.speculative.dspark.draft_kimi_k3 page,
 * KimiK3DSparkAttention: q_head_dim = qk_nope_head_dim + qk_rope_head_dim,
 * scaling = q_head_dim ** -0.5).
 *
 * Layouts (row-major, contiguous, element type = dtype):
 *   q      [B, Q, H, d_nope + d_rope]   the nope part first, then the rope part
 *   k_nope [B, S+Q, H, d_nope]          keys 0..S-1 context, S..S+Q-1 noise
 *   k_rope [B, S+Q, d_rope]             one per token, shared by every head
 *   v      [B, S+Q, H, d_v]
 *   out    [B, Q, H, d_v]               written in dtype (bf16: round to nearest even)
 *   lse    [B, H, Q] fp32, optional     natural-log log-sum-exp of the scaled scores
 *   mask   [B, 1, Q, S+Q] (dense only)  additive, element type = dtype
 *
 * Ownership and execution.  Every pointer argument of the compute calls is a
 * device pointer owned by the caller; the library allocates no device memory
 * and uses only the caller's workspace.  Calls are asynchronous on the given
 * stream and never synchronise the host.  Errors are status codes; nothing is
 * thrown across the ABI.  Host-side validation happens before any launch, and
 * a call that returns an error launches nothing.  Conditions only the device
 * can see (an anchor outside [0, S], a wait that ran past its time limit) are
 * recorded in a per-device error word read by dflash_last_device_error().
 *
 * Rows that see no key (dense masks whose row is entirely -inf) produce
 * out = 0 and lse = -inf.  Mask entries must be finite or -inf.
 */
#ifndef DFLASH_ATTN_H_
#define DFLASH_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* dflash_stream_t;

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID = 1,     /* null pointer, negative size, bad anchor/offset on the device */
  DFLASH_ERR_SHAPE = 2,       /* inconsistent shapes (nb*block_size != Q, ...) */
  DFLASH_ERR_DTYPE = 3,       /* unknown dtype */
  DFLASH_ERR_ALIGN = 4,       /* a tensor base pointer is not 16-byte aligned */
  DFLASH_ERR_UNSUPPORTED = 5, /* head dims beyond the kernels' limits */
  DFLASH_ERR_WORKSPACE = 6,   /* workspace null, misaligned (256 B) or too small */
  DFLASH_ERR_CUDA = 7,        /* a CUDA runtime call or launch failed */
  DFLASH_ERR_TIMEOUT = 8      /* a bounded device wait gave up (kernel returned early) */
} dflash_status_t;

typedef enum { DFLASH_BF16 = 0, DFLASH_FP32 = 1 } dflash_dtype_t;

typedef struct {
  int B;      /* batch rows */
  int H;      /* heads (one K/V per query head) */
  int S;      /* context tokens */
  int Q;      /* noise (query) tokens = nb * block_size */
  int d_nope; /* qk_nope_head_dim */
  int d_rope; /* qk_rope_head_dim (head-shared key slice) */
  int d_v;    /* v_head_dim */
  float scale; /* <= 0 selects (d_nope + d_rope)^-0.5 */
} dflash_dims_t;

/* Tile grid of the schedule: DFLASH_TILE_M query rows x DFLASH_TILE_N keys,
 * anchored at query row 0 and key 0 of each batch row. */
#define DFLASH_TILE_M 128
#define DFLASH_TILE_N 128
enum { DFLASH_TILE_SKIP = 0, DFLASH_TILE_PARTIAL = 1, DFLASH_TILE_FULL = 2 };

/* Kernel limits.  bf16 with (d_nope, d_rope, d_v) = (128, 64, 128) runs on the
 * tensor-core (tcgen05) kernels; every other supported shape, and all fp32,
 * runs on the exact CUDA-core kernel. */
#define DFLASH_MAX_DQK 512 /* d_nope + d_rope */
#define DFLASH_MAX_DV 256

/*
 * Dense additive-mask entry point (KimiK3DFlashAttention.forward: the
 * additive mask [batch, 1, blocks*block_size, sequence + blocks*block_size]
 * is used unchanged).  A key is visible to a row iff its mask entry is not
 * -inf; the entry is added to the scaled score.  The mask is first scanned
 * on the device into per-tile classes (all 0 / all -inf / mixed) so that
 * all--inf tiles are skipped and all-0 tiles need no mask reads.
 *   workspace: >= dflash_attn_workspace_size(DFLASH_MODE_DENSE, ...) bytes,
 *              256-byte aligned, device memory; contents need no initialisation.
 */
DFLASH_API dflash_status_t dflash_attn_dense(const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q,
                                  const void* k_nope, const void* k_rope, const void* v,
                                  const void* mask, void* out, float* lse, void* workspace,
                                  size_t ws_bytes, dflash_stream_t stream);

/*
 * Anchored entry point.  anchors [B, nb] int32 on the device; Q = nb *
 * block_size.  Query row i of batch row b belongs to block j = i / block_size
 * and sees exactly the context keys p < anchors[b, j] and the block_size noise
 * keys S + j*block_size + t of its own block (the DFlash block contract of the
 * draft_kimi_k3 page: one block = [anchor, MASK, ...] predicted in one
 * non-causal forward).  Anchors must lie in [0, S]; sortedness and
 * distinctness are not required.  An anchor outside [0, S] is clamped and
 * recorded as DFLASH_ERR_INVALID in the device error word.
 */
DFLASH_API dflash_status_t dflash_attn_anchored(const dflash_dims_t* dims, dflash_dtype_t dtype,
                                     const void* q, const void* k_nope, const void* k_rope,
                                     const void* v, const int32_t* anchors, int nb,
                                     int block_size, void* out, float* lse, void* workspace,
                                     size_t ws_bytes, dflash_stream_t stream);

/*
 * Ragged (serving) entry point: R requests packed along the token axis by row
 * offsets (max.pipelines.architectures.dflash_kimi_k25 page, DFlashKimiK25:
 * input_row_offsets; ctx_at_draft_cache_length = True; supports_zero_draft_rows
 * = False).  Request r owns query rows [q_offsets[r], q_offsets[r+1]) and key
 * rows [kv_offsets[r], kv_offsets[r+1]); its keys are its context followed by
 * its q_len noise tokens, so S_r = kv_len - q_len.  q_len must be a positive
 * multiple of block_size and q_offsets[r] a multiple of block_size; anchors
 * are indexed by global block q_offsets[r]/block_size + local block, and obey
 * the anchored rule inside the request.
 *   q [total_q, H, d_nope+d_rope], k_nope [total_kv, H, d_nope],
 *   k_rope [total_kv, d_rope], v [total_kv, H, d_v], out [total_q, H, d_v],
 *   lse [H, total_q] fp32 (optional), offsets int32 [R+1] on the device.
 *   total_q, total_kv: extents of the packed tensors (q_offsets[R],
 *   kv_offsets[R]); max_q_len: an upper bound on every request's q_len.
 * Offsets that break these rules, and a request whose q_len exceeds
 * max_q_len, are recorded as DFLASH_ERR_INVALID in the device error word and
 * the offending request is skipped (its out and lse rows are not written).
 * Decode-shaped batches (small q_len, long context) are split along the
 * context and merged with a log-sum-exp combine kernel.
 */
DFLASH_API dflash_status_t dflash_attn_ragged(int R, int H, int d_nope, int d_rope, int d_v, float scale,
                                   dflash_dtype_t dtype, const void* q, const void* k_nope,
                                   const void* k_rope, const void* v, const int32_t* q_offsets,
                                   const int32_t* kv_offsets, const int32_t* anchors,
                                   int block_size, int total_q, int total_kv, int max_q_len,
                                   void* out, float* lse, void* workspace, size_t ws_bytes,
                                   dflash_stream_t stream);

/*
 * Ragged entry point over compressed KV latents (Kimi K3 MLA).  Each token
 * carries its KV latent c (kv_rank values, after the latent norm) and the
 * head-shared rope key; kv_b_proj expands the latent to one k_nope + v slice
 * per head (nemo_automodel.components.speculative.dflash.draft_kimi_k3 page,
 * KimiK3DFlashAttention: kv_b_proj produces num_attention_heads slices of
 * qk_nope_head_dim + v_head_dim; ...dspark.draft_kimi_k3 page,
 * KimiK3DSparkAttention: kv_lora_rank, kv_b_proj; nemo_automodel.components.
 * models.kimi_k3.model page: the compressed latent is kv_lora_rank +
 * qk_rope_head_dim values per token).  With w_kv_b viewed as [H, d_nope + d_v,
 * kv_rank] (per head: the d_nope key rows, then the d_v value rows):
 *   k_nope[t,h,e] = sum_c w_kv_b[h,e,c] c_kv[t,c],
 *   v[t,h,e]      = sum_c w_kv_b[h,d_nope+e,c] c_kv[t,c],
 * and the result is dflash_attn_ragged over those keys and values (same
 * offsets, anchors, block rule, scale, out and lse).
 *   q [total_q, H, d_nope+d_rope], c_kv [total_kv, kv_rank],
 *   k_rope [total_kv, d_rope], w_kv_b [H, d_nope+d_v, kv_rank] (the
 *   projection weight, row-major), out [total_q, H, d_v], lse [H, total_q].
 * bf16 with (d_nope, d_rope, d_v, kv_rank) = (128, 64, 128, 512), H a multiple
 * of 4 and max_q_len <= 16 (the serving decode shape) runs absorbed on the
 * tensor cores: W_UK is folded into q, the attention runs over the latents
 * (every head reads each token's latent once), and W_UV is applied after the
 * softmax; q_abs and o_lat are rounded to bf16 on the way.  Every other shape
 * (and fp32) expands the keys and values into the workspace and runs the
 * ragged kernels on them.  A request skipped for invalid offsets or q_len >
 * max_q_len is recorded as DFLASH_ERR_INVALID; its rows are written as 0
 * (lse -inf) on the absorbed path and left unwritten on the expanded path.
 *   workspace: >= dflash_attn_latent_workspace_size(...) bytes, 256-byte
 *   aligned; needs no initialisation.
 */
#define DFLASH_MAX_KV_RANK 1024
DFLASH_API size_t dflash_attn_latent_workspace_size(int R, int H, int d_nope, int d_rope, int d_v, int kv_rank,
                                                    dflash_dtype_t dtype, int total_q, int total_kv, int max_q_len);
DFLASH_API dflash_status_t dflash_attn_latent_ragged(int R, int H, int d_nope, int d_rope, int d_v, int kv_rank,
                                                     float scale, dflash_dtype_t dtype, const void* q,
                                                     const void* c_kv, const void* k_rope, const void* w_kv_b,
                                                     const int32_t* q_offsets, const int32_t* kv_offsets,
                                                     const int32_t* anchors, int block_size, int total_q,
                                                     int total_kv, int max_q_len, void* out, float* lse,
                                                     void* workspace, size_t ws_bytes, dflash_stream_t stream);

/*
 * Dense entry point that allocates nothing and takes no workspace.  (No
 * counterpart on the pages: this is a convenience of this library.)
 *
 * For callers that cannot provide device scratch memory -- runtimes that plan
 * all device memory once at start-up and forbid allocations while serving,
 * or plugin interfaces whose fixed signature has no workspace argument.  The
 * dense path's only scratch, one class byte per 128x128 mask tile, lives in a
 * fixed device array inside the library (DFLASH_NOALLOC_MAX_TILES + 256 bytes,
 * held on every GPU that loads the library until the process exits).
 * Arguments and results are those of dflash_attn_dense.
 *   - Returns DFLASH_ERR_WORKSPACE when B * ceil(Q/128) * ceil((S+Q)/128)
 *     exceeds DFLASH_NOALLOC_MAX_TILES; nothing is launched then.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents (each call rewrites every byte it reads).  Calls that overlap
 *     on the GPU (different streams, or different host threads on one device)
 *     race on it and must be serialised by the caller.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define DFLASH_NOALLOC_MAX_TILES (1 << 20)
DFLASH_API dflash_status_t dflash_attn_dense_noalloc(const dflash_dims_t* dims, dflash_dtype_t dtype,
                                                     const void* q, const void* k_nope, const void* k_rope,
                                                     const void* v, const void* mask, void* out, float* lse,
                                                     dflash_stream_t stream);

enum {
  DFLASH_MODE_DENSE = 0,
  DFLASH_MODE_ANCHORED = 1,
  DFLASH_MODE_RAGGED = 2,
  DFLASH_MODE_DENSE_BACKWARD = 3,
  DFLASH_MODE_ANCHORED_BACKWARD = 4
};

/*
 * Backward pass of the anchored and dense entry points: gradients of the
 * scalar L = sum over (b, i, h, d) of dout * out.  The DFlash draft is a
 * trained module (nemo_automodel.components.speculative.dflash.draft_kimi_k3
 * page, module docstring), so the attention's gradients are needed.  Per head
 * and query row i over its visible keys k, with P the softmax weights
 * recomputed from the forward's lse:
 *   dP(i,k) = dout(i) . v(k),  D(i) = dout(i) . out(i),  dS = P (dP - D)
 *   dq(i)      = scale * sum_k dS(i,k) [k_nope(k) | k_rope(k)]
 *   dk_nope(k) = scale * sum_i dS(i,k) q_nope(i)
 *   dk_rope(k) = scale * sum_h sum_i dS(i,k) q_rope(i)   (one rope key per token
 *                serves every head, so its gradient is the sum over heads)
 *   dv(k)      = sum_i P(i,k) dout(i)
 * The mask (dense) is a constant input and gets no gradient.
 *   q, k_nope, k_rope, v, anchors/mask: the forward's inputs (same layouts).
 *   out [B,Q,H,d_v] and lse [B,H,Q] fp32: the forward's outputs for these
 *     inputs (lse is required here).
 *   dout [B,Q,H,d_v]: gradient of L with respect to out.
 *   dq [B,Q,H,d_nope+d_rope], dk_nope [B,S+Q,H,d_nope], dk_rope [B,S+Q,d_rope],
 *   dv [B,S+Q,H,d_v]: written in dtype; every element is written (keys no row
 *     sees get 0).  With Q = 0 only the key gradients are written (all 0) and
 *     the query-side pointers may be null.
 *   workspace: >= dflash_attn_workspace_size(DFLASH_MODE_*_BACKWARD, ...)
 *     bytes, 256-byte aligned, device memory; needs no initialisation.
 * Limits: d_nope + d_rope <= DFLASH_BWD_MAX_DQK and d_v <= DFLASH_BWD_MAX_DV
 * (else DFLASH_ERR_UNSUPPORTED).  Device pointers, 16-byte aligned; the call
 * is asynchronous on `stream` and allocates no device memory.  On the
 * tensor-core path (bf16, head dims 128/64/128) the dq kernel runs on a second
 * stream that the library creates once per host thread and device; it is
 * forked from `stream` (an event) and joined back into it before the call
 * returns, so work queued on `stream` afterwards sees every gradient.  Errors
 * as for the forward entry points.
 */
#define DFLASH_BWD_MAX_DQK 256
#define DFLASH_BWD_MAX_DV 128
DFLASH_API dflash_status_t dflash_attn_anchored_backward(
    const dflash_dims_t* dims, dflash_dtype_t dtype, const void* q, const void* k_nope, const void* k_rope,
    const void* v, const int32_t* anchors, int nb, int block_size, const void* out, const float* lse,
    const void* dout, void* dq, void* dk_nope, void* dk_rope, void* dv, void* workspace, size_t ws_bytes,
    dflash_stream_t stream);
DFLASH_API dflash_status_t dflash_attn_dense_backward(const dflash_dims_t* dims, dflash_dtype_t dtype,
                                                      const void* q, const void* k_nope, const void* k_rope,
                                                      const void* v, const void* mask, const void* out,
                                                      const float* lse, const void* dout, void* dq,
                                                      void* dk_nope, void* dk_rope, void* dv, void* workspace,
                                                      size_t ws_bytes, dflash_stream_t stream);

/*
 * Workspace bytes a call needs.  For DENSE/ANCHORED (and their _BACKWARD
 * modes) pass dims (dims->B, S, Q,
 * H, head dims) and ignore the ragged arguments; for RAGGED pass dims = NULL
 * and R, H, head dims via the ragged arguments.  Returns 0 on invalid input.
 */
DFLASH_API size_t dflash_attn_workspace_size(int mode, const dflash_dims_t* dims, dflash_dtype_t dtype,
                                  int R, int H, int d_nope, int d_rope, int d_v, int total_q,
                                  int total_kv, int max_q_len);

/*
 * Host builder of the anchored tile schedule (exported for tests).  anchors
 * [B, nb] int32 in HOST memory.  classes (host, uint8) receives
 * [B, ceil(Q/DFLASH_TILE_M), ceil((S+Q)/DFLASH_TILE_N)] tile classes
 * (DFLASH_TILE_*), computed from each tile's minimum and maximum anchor with
 * the same formula the kernels use.
 */
DFLASH_API dflash_status_t dflash_build_schedule_host(int B, int S, int Q, const int32_t* anchors, int nb,
                                           int block_size, uint8_t* classes);

/*
 * Device scan of a dense mask into tile classes (exported for tests): mask
 * [B,1,Q,S+Q] of dtype on the device, classes [B, ceil(Q/TILE_M),
 * ceil((S+Q)/TILE_N)] uint8 on the device.  An all-0 tile is FULL, an
 * all--inf tile SKIP, anything else PARTIAL.
 */
DFLASH_API dflash_status_t dflash_scan_mask(int B, int S, int Q, dflash_dtype_t dtype, const void* mask,
                                 uint8_t* classes, dflash_stream_t stream);

/*
 * Number of kernels this library has launched in the calling process since it
 * was loaded (all devices, all streams).  Diagnostic counter for benchmarks.
 */
DFLASH_API uint64_t dflash_kernel_launches(void);

/*
 * Builds the additive DFlash block mask of the anchored rule on the device:
 * mask [B, 1, Q, S+Q] of dtype gets 0 where row i (block j = i/block_size) may
 * attend -- context keys p < anchors[b, j] and the block_size noise keys of
 * block j -- and -inf everywhere else.  This is the dense mask the trainer
 * hands the draft (nemo_automodel.components.speculative.dflash.draft_kimi_k3
 * page, module docstring: the block structure is supplied entirely by the
 * attention mask; KimiK3DFlashAttention.forward: its shape).  anchors [B, nb]
 * int32 on the device; anchors outside [0, S] are clamped and recorded as
 * DFLASH_ERR_INVALID in the device error word.  Asynchronous on `stream`.
 */
DFLASH_API dflash_status_t dflash_build_mask(int B, int S, int Q, const int32_t* anchors, int nb, int block_size,
                                             dflash_dtype_t dtype, void* mask, dflash_stream_t stream);

/*
 * Test export: fault injection for the bounded-wait path.  Every mbarrier wait
 * of the tensor-core kernels (forward, split-context decode, latent decode and
 * backward) gives up after a budget -- 2 s unless set here -- records
 * DFLASH_ERR_TIMEOUT in the device error word, and the CTA winds down: its
 * issued TMA loads land, its issued MMAs complete, its TMEM is freed, and it
 * returns; the context stays usable.  This call sets, process-wide and for
 * every later call until it is called again:
 *   wait_budget_ns  budget of one wait (0 restores the 2 s default);
 *   stall_cta       the CTA (of each of those kernels) whose TMA producer
 *                   leaves its first work item's key tiles (the backward's
 *                   dk/dv kernel: query tiles) unloaded, so that the waits on
 *                   them run out (-1: none).  Other CTAs compute normally; the
 *                   stalled CTA's results are left unwritten or incomplete.
 * Not for production use; not synchronised with calls in flight.
 */
DFLASH_API void dflash_test_inject_stall(unsigned long long wait_budget_ns, int stall_cta);

/*
 * Test export: the backward kernels work out, once per CTA, which tiles of the
 * axis they loop over (dq: key tiles; dk/dv: query tiles) they need, and keep
 * these flags in a shared-memory table of 16384 entries; tiles past the table
 * are worked out when they come up.  This call caps the table at n entries
 * (n <= 0 restores the full table), process-wide for every later call, so that
 * tests reach the path past the table at small sizes.  Results do not depend
 * on n.  Not for production use; not synchronised with calls in flight.
 */
DFLASH_API void dflash_test_limit_tile_flags(int n);

/* Human-readable name of a status code (static storage). */
DFLASH_API const char* dflash_status_string(dflash_status_t status);

/*
 * Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns DFLASH_OK when no kernel recorded an error since the last
 * read, DFLASH_ERR_CUDA when the synchronisation itself failed.
 */
DFLASH_API dflash_status_t dflash_last_device_error(dflash_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_ATTN_H_ */
