/*
 * oracle.c -- plain fp64 CPU oracle for DFlash draft block attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file; only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or constant with
 * the CUDA library.
 *
 * What it computes (the plain definition; no tiling, no online softmax):
 *
 *   For every query row i of batch row b and head h, over the key axis
 *   [target-hidden context (S tokens) | noise block (Q tokens)]:
 *     s_k   = scale * ( q_nope . k_nope[k,h] + q_rope . k_rope[k] ) (+ mask[i,k])
 *     out   = sum_k softmax(s)_k * v[k,h]     over the visible keys k
 *     lse   = m + log(sum_k exp(s_k - m))     (natural log), m = max_k s_k
 *   A row with no visible key gives out = 0, lse = -inf.
 *
 * Sources (nemo_automodel.components.speculative.dflash.draft_kimi_k3 page):
 *   - module docstring: keys/values are [target-hidden context | noise block],
 *     one non-causal forward per block; the rope part of the key is one vector
 *     per token shared by all heads, without rotary embedding (NoPE);
 *   - KimiK3DFlashAttention: one K/V per query head (no GQA repeat);
 *   - KimiK3DFlashAttention.forward: additive mask of shape
 *     [batch, 1, blocks*block_size, sequence + blocks*block_size], passed to
 *     SDPA unchanged.
 * nemo_automodel.components.speculative.dspark.draft_kimi_k3 page,
 *   KimiK3DSparkAttention attributes: q_head_dim = qk_nope + qk_rope and
 *   scaling = q_head_dim ** -0.5.
 * Anchored visibility (the block mask the trainer builds, whose source is not
 * on the pages): a query in block j sees context positions p < a_j and the
 * block_size noise tokens of its own block j, nothing else.
 * Ragged layout (max.pipelines.architectures.dflash_kimi_k25 page,
 * DFlashKimiK25: ctx_at_draft_cache_length, input_row_offsets,
 * supports_zero_draft_rows = False): request r's keys are its context followed
 * by its q_len draft tokens, contiguous.
 *
 * Element types: 0 = bf16 (raw 16-bit patterns), 1 = fp32, 2 = fp64.  Every
 * input is widened to double exactly before use.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BF16 0
#define ORC_F32 1
#define ORC_F64 2

/* Tile classes of the brute-force schedule scan. */
#define ORC_TILE_SKIP 0
#define ORC_TILE_PARTIAL 1
#define ORC_TILE_FULL 2

static double ld(const void* p, int dt, size_t i) {
  if (dt == ORC_BF16) {
    /* bf16 is the top half of an IEEE binary32: widening is a 16-bit shift. */
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  if (dt == ORC_F32) return (double)((const float*)p)[i];
  return ((const double*)p)[i];
}

typedef struct {
  int H, dn, dr, dv, dt;
  double scale;
  const void *q, *kn, *kr, *v;
} io_t;

/* Raw dot product q[qrow,h,:] . [k_nope[krow,h,:] | k_rope[krow,:]]. */
static double qk_dot(const io_t* io, size_t qrow, size_t krow, int h) {
  const int dqk = io->dn + io->dr;
  const size_t qb = (qrow * io->H + h) * (size_t)dqk;
  const size_t kb = (krow * io->H + h) * (size_t)io->dn;
  const size_t rb = krow * (size_t)io->dr;
  double acc = 0.0;
  for (int d = 0; d < io->dn; ++d) acc += ld(io->q, io->dt, qb + d) * ld(io->kn, io->dt, kb + d);
  for (int d = 0; d < io->dr; ++d) acc += ld(io->q, io->dt, qb + io->dn + d) * ld(io->kr, io->dt, rb + d);
  return acc;
}

/*
 * Softmax-weighted sum over an explicit list of keys with their scores.
 * keys[] are absolute token rows of k/v; s[] the final scores.  out gets dv
 * values, *lse the natural-log log-sum-exp.  n == 0 gives out = 0, lse = -inf.
 */
static void softmax_sum(const io_t* io, int h, int n, const size_t* keys, const double* s,
                        double* out, double* lse) {
  for (int d = 0; d < io->dv; ++d) out[d] = 0.0;
  if (n == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = s[0];
  for (int t = 1; t < n; ++t)
    if (s[t] > m) m = s[t];
  double l = 0.0;
  for (int t = 0; t < n; ++t) {
    const double w = exp(s[t] - m);
    l += w;
    const size_t vb = (keys[t] * io->H + h) * (size_t)io->dv;
    for (int d = 0; d < io->dv; ++d) out[d] += w * ld(io->v, io->dt, vb + d);
  }
  for (int d = 0; d < io->dv; ++d) out[d] /= l;
  *lse = m + log(l);
}

/*
 * Visible key set of one row under the anchored rule, as relative key indices
 * into [0, S+Q).  Returns the count.  Context keys p < min(a, S); noise keys of
 * the row's own block, clipped to the row's Q.
 */
static int anchored_keys(int S, int Q, int bs, int a, int i, int* rel) {
  int n = 0;
  const int lim = a < S ? a : S;
  for (int p = 0; p < lim; ++p) rel[n++] = p;
  const int blk = i / bs;
  for (int t = 0; t < bs; ++t) {
    const int r = blk * bs + t;
    if (r < Q) rel[n++] = S + r;
  }
  return n;
}

static int nthreads_or_default(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) return nthreads;
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Dense additive mask [B,1,Q,S+Q]: visible iff mask != -inf, score += mask.  */
/* ------------------------------------------------------------------------ */
int oracle_dense(int B, int H, int S, int Q, int dn, int dr, int dv, double scale, int dt,
                 const void* q, const void* kn, const void* kr, const void* v,
                 const void* mask, int mask_dt, const int64_t* rows, int64_t nrows,
                 double* out, double* lse, int nthreads) {
  if (B < 0 || H <= 0 || S < 0 || Q < 0 || dn < 0 || dr < 0 || dv <= 0) return 1;
  const io_t io = {H, dn, dr, dv, dt, scale, q, kn, kr, v};
  const int K = S + Q;
  const int64_t total = rows ? nrows : (int64_t)B * Q;
  int bad = 0;
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
  {
    size_t* keys = (size_t*)malloc(sizeof(size_t) * (K > 0 ? K : 1));
    double* s = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < total * H; ++w) {
      const int64_t ri = w / H;
      const int h = (int)(w % H);
      const int64_t grow = rows ? rows[ri] : ri;
      if (grow < 0 || grow >= (int64_t)B * Q) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int b = (int)(grow / Q), i = (int)(grow % Q);
      int n = 0;
      for (int k = 0; k < K; ++k) {
        const double mk = ld(mask, mask_dt, ((size_t)b * Q + i) * (size_t)K + k);
        if (mk == -INFINITY) continue;
        keys[n] = (size_t)b * K + k;
        s[n] = scale * qk_dot(&io, (size_t)grow, keys[n], h) + mk;
        ++n;
      }
      softmax_sum(&io, h, n, keys, s, out + ((size_t)ri * H + h) * dv, lse + (size_t)ri * H + h);
    }
    free(keys);
    free(s);
  }
  return bad ? 2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Anchored: a query in block j sees context p < a_j and its own block.       */
/* ------------------------------------------------------------------------ */
int oracle_anchored(int B, int H, int S, int Q, int dn, int dr, int dv, double scale, int dt,
                    const void* q, const void* kn, const void* kr, const void* v,
                    const int32_t* anchors, int nb, int bs, const int64_t* rows, int64_t nrows,
                    double* out, double* lse, int nthreads) {
  if (B < 0 || H <= 0 || S < 0 || Q < 0 || bs <= 0 || nb * bs != Q || dv <= 0) return 1;
  const io_t io = {H, dn, dr, dv, dt, scale, q, kn, kr, v};
  const int K = S + Q;
  const int64_t total = rows ? nrows : (int64_t)B * Q;
  int bad = 0;
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
  {
    int* rel = (int*)malloc(sizeof(int) * (K > 0 ? K : 1));
    size_t* keys = (size_t*)malloc(sizeof(size_t) * (K > 0 ? K : 1));
    double* s = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < total * H; ++w) {
      const int64_t ri = w / H;
      const int h = (int)(w % H);
      const int64_t grow = rows ? rows[ri] : ri;
      if (grow < 0 || grow >= (int64_t)B * Q) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int b = (int)(grow / Q), i = (int)(grow % Q);
      const int a = anchors[(size_t)b * nb + i / bs];
      const int n = anchored_keys(S, Q, bs, a, i, rel);
      for (int t = 0; t < n; ++t) {
        keys[t] = (size_t)b * K + rel[t];
        s[t] = scale * qk_dot(&io, (size_t)grow, keys[t], h);
      }
      softmax_sum(&io, h, n, keys, s, out + ((size_t)ri * H + h) * dv, lse + (size_t)ri * H + h);
    }
    free(rel);
    free(keys);
    free(s);
  }
  return bad ? 2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Ragged: R requests packed by row offsets; anchored rule per request.        */
/* q rows [q_off[r], q_off[r+1]); key rows [kv_off[r], kv_off[r+1]) laid out   */
/* as [context (kv_len - q_len) | noise (q_len)].  anchors are indexed by the  */
/* global block number q_off[r]/bs + local block.                              */
/* ------------------------------------------------------------------------ */
static int find_request(const int32_t* q_off, int R, int64_t row) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (q_off[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

int oracle_ragged(int R, int H, int dn, int dr, int dv, double scale, int dt,
                  const void* q, const void* kn, const void* kr, const void* v,
                  const int32_t* q_off, const int32_t* kv_off, const int32_t* anchors, int bs,
                  const int64_t* rows, int64_t nrows, double* out, double* lse, int nthreads) {
  if (R <= 0 || H <= 0 || bs <= 0 || dv <= 0) return 1;
  const io_t io = {H, dn, dr, dv, dt, scale, q, kn, kr, v};
  int maxk = 1;
  for (int r = 0; r < R; ++r) {
    const int ql = q_off[r + 1] - q_off[r], kl = kv_off[r + 1] - kv_off[r];
    if (ql < bs || ql % bs || q_off[r] % bs || kl < ql) return 1;
    if (kl > maxk) maxk = kl;
  }
  const int64_t total = rows ? nrows : (int64_t)q_off[R];
  int bad = 0;
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
  {
    int* rel = (int*)malloc(sizeof(int) * maxk);
    size_t* keys = (size_t*)malloc(sizeof(size_t) * maxk);
    double* s = (double*)malloc(sizeof(double) * maxk);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < total * H; ++w) {
      const int64_t ri = w / H;
      const int h = (int)(w % H);
      const int64_t grow = rows ? rows[ri] : ri;
      if (grow < 0 || grow >= (int64_t)q_off[R]) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int r = find_request(q_off, R, grow);
      const int Qr = q_off[r + 1] - q_off[r];
      const int Sr = (kv_off[r + 1] - kv_off[r]) - Qr;
      const int i = (int)(grow - q_off[r]);
      const int a = anchors[q_off[r] / bs + i / bs];
      const int n = anchored_keys(Sr, Qr, bs, a, i, rel);
      for (int t = 0; t < n; ++t) {
        keys[t] = (size_t)kv_off[r] + rel[t];
        s[t] = scale * qk_dot(&io, (size_t)grow, keys[t], h);
      }
      softmax_sum(&io, h, n, keys, s, out + ((size_t)ri * H + h) * dv, lse + (size_t)ri * H + h);
    }
    free(rel);
    free(keys);
    free(s);
  }
  return bad ? 2 : 0;
}

/* ------------------------------------------------------------------------ */
/* Split-context + log-sum-exp merge, anchored rule.                          */
/* The key axis [0, S+Q) is cut into spans of `split` keys; each span gives a  */
/* normalised partial O_s and lse_s over its visible keys (O_s = 0, lse_s =    */
/* -inf when none), and the row result is                                      */
/*   M = max_s lse_s,  w_s = exp(lse_s - M),                                   */
/*   out = sum_s w_s O_s / sum_s w_s,  lse = M + log(sum_s w_s).               */
/* This is the merge rule the split-context decode path uses; the oracle       */
/* carries it so the rule itself is checked against the unsplit definition.    */
/* ------------------------------------------------------------------------ */
int oracle_anchored_split(int B, int H, int S, int Q, int dn, int dr, int dv, double scale, int dt,
                          const void* q, const void* kn, const void* kr, const void* v,
                          const int32_t* anchors, int nb, int bs, int split,
                          double* out, double* lse, int nthreads) {
  if (B < 0 || H <= 0 || bs <= 0 || nb * bs != Q || split <= 0 || dv <= 0) return 1;
  const io_t io = {H, dn, dr, dv, dt, scale, q, kn, kr, v};
  const int K = S + Q;
  const int nsplit = (K + split - 1) / split;
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
  {
    int* rel = (int*)malloc(sizeof(int) * (K > 0 ? K : 1));
    size_t* keys = (size_t*)malloc(sizeof(size_t) * (K > 0 ? K : 1));
    double* s = (double*)malloc(sizeof(double) * (K > 0 ? K : 1));
    double* Os = (double*)malloc(sizeof(double) * (size_t)(nsplit > 0 ? nsplit : 1) * dv);
    double* Ls = (double*)malloc(sizeof(double) * (nsplit > 0 ? nsplit : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < (int64_t)B * Q * H; ++w) {
      const int64_t grow = w / H;
      const int h = (int)(w % H);
      const int b = (int)(grow / Q), i = (int)(grow % Q);
      const int a = anchors[(size_t)b * nb + i / bs];
      const int n = anchored_keys(S, Q, bs, a, i, rel);
      for (int sp = 0; sp < nsplit; ++sp) {
        int m = 0;
        for (int t = 0; t < n; ++t) {
          if (rel[t] / split != sp) continue;
          keys[m] = (size_t)b * K + rel[t];
          s[m] = scale * qk_dot(&io, (size_t)grow, keys[m], h);
          ++m;
        }
        softmax_sum(&io, h, m, keys, s, Os + (size_t)sp * dv, Ls + sp);
      }
      double M = -INFINITY;
      for (int sp = 0; sp < nsplit; ++sp)
        if (Ls[sp] > M) M = Ls[sp];
      double* o = out + ((size_t)grow * H + h) * dv;
      for (int d = 0; d < dv; ++d) o[d] = 0.0;
      if (M == -INFINITY) {
        lse[(size_t)grow * H + h] = -INFINITY;
        continue;
      }
      double wsum = 0.0;
      for (int sp = 0; sp < nsplit; ++sp) {
        const double ws = exp(Ls[sp] - M);
        wsum += ws;
        for (int d = 0; d < dv; ++d) o[d] += ws * Os[(size_t)sp * dv + d];
      }
      for (int d = 0; d < dv; ++d) o[d] /= wsum;
      lse[(size_t)grow * H + h] = M + log(wsum);
    }
    free(rel);
    free(keys);
    free(s);
    free(Os);
    free(Ls);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward pass: gradients of the scalar L = sum_{b,i,h} dout(i,h) . out(i,h) */
/* with respect to q, k_nope, k_rope and v.  Differentiating the forward       */
/* definition row by row (softmax Jacobian dP/ds = diag(P) - P P^T), for each  */
/* batch row b, head h and query row i over its visible keys k:               */
/*   P_k  = softmax_k(s)                                                      */
/*   dP_k = dout(i,h) . v(k,h)                                                */
/*   D    = sum_k P_k dP_k                  (equals dout(i,h) . out(i,h))      */
/*   dS_k = P_k (dP_k - D)                  (dL/ds_k)                          */
/*   dq(i,h)      = scale * sum_k dS_k [k_nope(k,h) | k_rope(k)]               */
/*   dk_nope(k,h) += scale * dS_k q_nope(i,h)                                  */
/*   dk_rope(k)   += scale * dS_k q_rope(i,h)     summed over heads, since one */
/*                                                k_rope serves every head     */
/*   dv(k,h)      += P_k dout(i,h)                                             */
/* Visibility is the anchored rule (anchors != NULL) or the dense mask's       */
/* non--inf entries (mask != NULL); the mask is a constant input and gets no   */
/* gradient.  A row that sees no key contributes nothing.                     */
/* pairs: optional subset of (b*H + h) to evaluate (NULL: all); outputs of     */
/* other pairs stay 0 and dk_rope sums only the listed heads.                  */
/* Outputs (fp64, zeroed here): dq [B,Q,H,dn+dr], dkn [B,S+Q,H,dn],            */
/* dkr [B,S+Q,dr], dvo [B,S+Q,H,dv].                                           */
/* ------------------------------------------------------------------------ */
int oracle_backward(int B, int H, int S, int Q, int dn, int dr, int dv, double scale, int dt,
                    const void* q, const void* kn, const void* kr, const void* v, const void* dout,
                    const int32_t* anchors, int nb, int bs, const void* mask, int mask_dt,
                    const int64_t* pairs, int64_t npairs, double* dq, double* dkn, double* dkr,
                    double* dvo, int nthreads) {
  if (B < 0 || H <= 0 || S < 0 || Q < 0 || dn < 0 || dr < 0 || dv <= 0) return 1;
  if (!mask && (!anchors || bs <= 0 || nb * bs != Q)) return 1;
  const io_t io = {H, dn, dr, dv, dt, scale, q, kn, kr, v};
  const int K = S + Q, dqk = dn + dr;
  memset(dq, 0, sizeof(double) * (size_t)B * Q * H * dqk);
  memset(dkn, 0, sizeof(double) * (size_t)B * K * H * dn);
  memset(dkr, 0, sizeof(double) * (size_t)B * K * dr);
  memset(dvo, 0, sizeof(double) * (size_t)B * K * H * dv);
  const int64_t total = pairs ? npairs : (int64_t)B * H;
  int bad = 0;
#pragma omp parallel num_threads(nthreads_or_default(nthreads))
  {
    const int Kc = K > 0 ? K : 1;
    int* rel = (int*)malloc(sizeof(int) * Kc);
    int* kk = (int*)malloc(sizeof(int) * Kc);
    double* s = (double*)malloc(sizeof(double) * Kc);
    double* dS = (double*)malloc(sizeof(double) * Kc);
    double* dkr_part = (double*)malloc(sizeof(double) * (size_t)Kc * (dr > 0 ? dr : 1));
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < total; ++w) {
      const int64_t pr = pairs ? pairs[w] : w;
      if (pr < 0 || pr >= (int64_t)B * H) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int b = (int)(pr / H), h = (int)(pr % H);
      memset(dkr_part, 0, sizeof(double) * (size_t)K * dr);
      for (int i = 0; i < Q; ++i) {
        const size_t grow = (size_t)b * Q + i;
        int n = 0;
        if (mask) {
          for (int k = 0; k < K; ++k) {
            const double mk = ld(mask, mask_dt, grow * (size_t)K + k);
            if (mk == -INFINITY) continue;
            kk[n] = k;
            s[n] = scale * qk_dot(&io, grow, (size_t)b * K + k, h) + mk;
            ++n;
          }
        } else {
          n = anchored_keys(S, Q, bs, anchors[(size_t)b * nb + i / bs], i, rel);
          for (int t = 0; t < n; ++t) {
            kk[t] = rel[t];
            s[t] = scale * qk_dot(&io, grow, (size_t)b * K + rel[t], h);
          }
        }
        if (n == 0) continue;
        double m = s[0];
        for (int t = 1; t < n; ++t)
          if (s[t] > m) m = s[t];
        double l = 0.0;
        for (int t = 0; t < n; ++t) l += exp(s[t] - m);
        /* P_k (kept in s) and dP_k (kept in dS), then D */
        const size_t ob = (grow * H + h) * (size_t)dv;
        double D = 0.0;
        for (int t = 0; t < n; ++t) {
          s[t] = exp(s[t] - m) / l;
          const size_t vb = (((size_t)b * K + kk[t]) * H + h) * (size_t)dv;
          double dp = 0.0;
          for (int d = 0; d < dv; ++d) dp += ld(dout, dt, ob + d) * ld(v, dt, vb + d);
          dS[t] = dp;
          D += s[t] * dp;
        }
        const size_t qb = (grow * H + h) * (size_t)dqk;
        for (int t = 0; t < n; ++t) {
          const double g = s[t] * (dS[t] - D);
          const size_t key = (size_t)b * K + kk[t];
          const size_t knb = (key * H + h) * (size_t)dn, krb = key * (size_t)dr;
          for (int d = 0; d < dn; ++d) {
            dq[qb + d] += scale * g * ld(kn, dt, knb + d);
            dkn[knb + d] += scale * g * ld(q, dt, qb + d);
          }
          for (int d = 0; d < dr; ++d) {
            dq[qb + dn + d] += scale * g * ld(kr, dt, krb + d);
            dkr_part[(size_t)kk[t] * dr + d] += scale * g * ld(q, dt, qb + dn + d);
          }
          const size_t vb = (key * H + h) * (size_t)dv;
          for (int d = 0; d < dv; ++d) dvo[vb + d] += s[t] * ld(dout, dt, ob + d);
        }
      }
#pragma omp critical(oracle_dkr)
      {
        double* dst = dkr + (size_t)b * K * dr;
        for (size_t e = 0; e < (size_t)K * dr; ++e) dst[e] += dkr_part[e];
      }
    }
    free(rel);
    free(kk);
    free(s);
    free(dS);
    free(dkr_part);
  }
  return bad ? 2 : 0;
}

/* ------------------------------------------------------------------------ */
/* The additive block mask the anchored rule stands for: 0 where visible,      */
/* -inf elsewhere, laid out [B, 1, Q, S+Q] in fp32.                            */
/* ------------------------------------------------------------------------ */
int oracle_build_mask(int B, int S, int Q, const int32_t* anchors, int nb, int bs, float* mask) {
  if (B < 0 || S < 0 || bs <= 0 || nb * bs != Q) return 1;
  const int K = S + Q;
  for (int b = 0; b < B; ++b)
    for (int i = 0; i < Q; ++i) {
      float* row = mask + ((size_t)b * Q + i) * (size_t)K;
      for (int k = 0; k < K; ++k) row[k] = -INFINITY;
      const int a = anchors[(size_t)b * nb + i / bs];
      for (int p = 0; p < S && p < a; ++p) row[p] = 0.0f;
      const int blk = i / bs;
      for (int t = 0; t < bs; ++t)
        if (blk * bs + t < Q) row[S + blk * bs + t] = 0.0f;
    }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Brute-force tile classes: scan every (row, key) of every tile.              */
/* Tiles are tile_m query rows by tile_n keys on the grid anchored at row 0    */
/* and key 0, clipped to [0,Q) x [0,S+Q).                                      */
/*   anchored (mask == NULL): FULL if every pair is visible, SKIP if none.     */
/*   dense: FULL if every entry is exactly 0, SKIP if every entry is -inf,     */
/*   PARTIAL otherwise (any other finite value forces PARTIAL).                */
/* classes: uint8 [B, ceil(Q/tile_m), ceil((S+Q)/tile_n)].                     */
/* ------------------------------------------------------------------------ */
int oracle_tile_classes(int B, int S, int Q, int tile_m, int tile_n, const int32_t* anchors, int nb,
                        int bs, const void* mask, int mask_dt, uint8_t* classes) {
  if (B < 0 || tile_m <= 0 || tile_n <= 0) return 1;
  if (!mask && (bs <= 0 || nb * bs != Q)) return 1;
  const int K = S + Q;
  const int nqt = (Q + tile_m - 1) / tile_m, nkt = (K + tile_n - 1) / tile_n;
  int* rel = (int*)malloc(sizeof(int) * (K > 0 ? K : 1));
  char* vis = (char*)malloc(K > 0 ? K : 1);
  for (int b = 0; b < B; ++b)
    for (int tq = 0; tq < nqt; ++tq)
      for (int tk = 0; tk < nkt; ++tk) {
        int any = 0, all = 1, allzero = 1;
        for (int i = tq * tile_m; i < (tq + 1) * tile_m && i < Q; ++i) {
          if (!mask) {
            memset(vis, 0, K > 0 ? K : 1);
            const int n = anchored_keys(S, Q, bs, anchors[(size_t)b * nb + i / bs], i, rel);
            for (int t = 0; t < n; ++t) vis[rel[t]] = 1;
          }
          for (int k = tk * tile_n; k < (tk + 1) * tile_n && k < K; ++k) {
            int vk;
            if (mask) {
              const double mk = ld(mask, mask_dt, ((size_t)b * Q + i) * (size_t)K + k);
              vk = mk != -INFINITY;
              if (mk != 0.0) allzero = 0;
            } else {
              vk = vis[k];
              if (!vk) allzero = 0;
            }
            if (vk) any = 1;
            else all = 0;
          }
        }
        uint8_t c;
        if (!any) c = ORC_TILE_SKIP;
        else if (all && allzero) c = ORC_TILE_FULL;
        else c = ORC_TILE_PARTIAL;
        classes[((size_t)b * nqt + tq) * nkt + tk] = c;
      }
  free(rel);
  free(vis);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Compressed-latent MLA: the per-head keys and values a token's latent        */
/* expands to.  The attention's kv_b_proj maps each token's KV latent c        */
/* (kv_lora_rank values, after kv_a_layernorm) to one qk_nope + v slice per     */
/* head (KimiK3DSparkAttention attributes on the DSpark Kimi K3 draft page;    */
/* KimiK3DFlashAttention on the DFlash Kimi K3 draft page: kv_b_proj produces  */
/* num_attention_heads slices of qk_nope_head_dim + v_head_dim).  With that    */
/* projection's weight viewed per head as w[h, e, c] (e < dn: the key part,     */
/* e >= dn: the value part; c < rank):                                         */
/*   k_nope[t,h,e] = sum_c w[h, e, c]      c_kv[t, c]    (e < dn)              */
/*   v[t,h,e]      = sum_c w[h, dn + e, c] c_kv[t, c]    (e < dv)              */
/* The rope part of the key stays the head-shared k_rope[t] (the latent holds  */
/* kv_lora_rank + qk_rope_head_dim values per token: Kimi K3 target page, MLA  */
/* context-parallel attention).  Attention over the expanded keys and values  */
/* is then the ragged definition above.  Tokens [t0, t1) are expanded into     */
/* fp64 k_nope_out [t1-t0, H, dn] and v_out [t1-t0, H, dv].                    */
/* ------------------------------------------------------------------------ */
int oracle_latent_expand(int H, int dn, int dv, int rank, int dt, const void* c_kv, const void* w,
                         int64_t t0, int64_t t1, double* k_nope_out, double* v_out, int nthreads) {
  if (H <= 0 || dn < 0 || dv <= 0 || rank <= 0 || t1 < t0) return 1;
  const int E = dn + dv;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads_or_default(nthreads))
  for (int64_t t = t0; t < t1; ++t) {
    for (int h = 0; h < H; ++h)
      for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int c = 0; c < rank; ++c)
          acc += ld(w, dt, ((size_t)h * E + e) * (size_t)rank + c) * ld(c_kv, dt, (size_t)t * rank + c);
        if (e < dn) k_nope_out[((size_t)(t - t0) * H + h) * dn + e] = acc;
        else v_out[((size_t)(t - t0) * H + h) * dv + (e - dn)] = acc;
      }
  }
  return 0;
}

/* Number of OpenMP threads a parallel region gets by default. */
int oracle_max_threads(void) { return nthreads_or_default(0); }
