/*
 * mla_oracle.c -- plain fp64 CPU oracle for the Kimi K2 MLA causal-attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the CUDA
 * library is checked against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  The product path never calls it and
 * shares no code, header or constant with it.
 *
 * What it computes, step by step, in the order of the attention excerpt on the page
 * "Kimi K2 · Similarities" (section "Contextual evidence from Query-key similarity",
 * the MLA forward of modeling_deepseek.py):
 *
 *   1. query row   Q = [q_nope | q_pe]                       (query concat)
 *   2. key row     K = [k_nope | k_pe]   with k_pe the single rotary key of the
 *                  sequence, broadcast to every head        (key concat; "the key's
 *                  rotated part being the shared rotary key")
 *   3. score       s_j = (Q . K_j) * softmax_scale          (matmul, then scale)
 *   4. mask        s_j += M[i, j]                           (additive 4D mask)
 *   5. weights     w_j = exp(s_j - max) / sum exp(s - max)  (softmax over keys)
 *   6. output      o   = sum_j w_j V_j                      (weights times values)
 *
 * The cast of the weights to bf16 and dropout (p = attention_dropout = 0.0 in the
 * config.json excerpt on "Kimi K2 · Logits") are not applied in the exact mode: the
 * oracle is the exact value of the method, in fp64.
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *   - The mask (built by _prepare_4d_causal_attention_mask on "Kimi K2 · Causal mask",
 *     section "Construct causal mask"; its body is not shown) is 0 where key j is
 *     visible to query i and the most negative finite bf16 value elsewhere.  Key j is
 *     visible to query i iff j <= i + past_len (positions are numbered from the cached
 *     length) and j < kv_len[b] (right padding).  A key masked for both reasons gets
 *     the same single minimum, not twice it.
 *   - Tk = past_len + Tq: the cache update puts the cached prefix first and the new
 *     rows last.
 *   - softmax_scale is an argument; it is used as the float it arrives as, widened to
 *     double.
 *
 * Mode 1 ("eager") is a diagnostic: it rounds to bf16 where the eager PyTorch code on
 * the page produces a bf16 tensor (matmul output, scaled scores, masked scores, the
 * weights after the fp32 softmax, the output) and keeps everything else in fp64.  It
 * shows how far the eager bf16 sequence sits from the exact value; it is not a gate.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread (no fast-math).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_NOPE 128 /* qk_nope_head_dim, config.json excerpt */
#define D_ROPE 64  /* qk_rope_head_dim */
#define D_V 128    /* v_head_dim */

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE fp32. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16 value (ties to even), returned as double.
 * Used only by the eager-emulation diagnostic.  Goes through fp32 first, as the eager
 * code computes in fp32 before it stores bf16; values are finite here. */
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u) return (double)f; /* inf / nan untouched */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  u &= 0xffff0000u;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* finfo(bfloat16).min = -(2 - 2^-7) * 2^127, the value the 4D mask holds where a key
 * is hidden (the mask is built in the dtype of inputs_embeds, torch_dtype bfloat16). */
static const double MASK_MIN_BF16 = -3.3895313892515355e38;

typedef struct {
  const uint16_t *q_nope, *q_pe, *k_nope, *k_pe, *v;
  const int32_t* kv_len;
  const uint8_t* key_mask; /* [B][Tk], 0 = key hidden; NULL = no 2D padding mask */
  const uint16_t* c_kv;    /* latent rows [B][Tk][512]; NULL = per-head k_nope / v given */
  const uint16_t* w_kvb;   /* kv_b_proj weight [H*256][512] (latent mode) */
  int64_t B, H, Tq, Tk, past_len;
  double scale;
  const int64_t* rows;
  int64_t n_rows;
  int mode;
  const double* rope_inv_freq; /* NULL: inputs already rotated; else 32 frequencies */
  double rope_mscale;
  double* out;
  double* wsum;
  int64_t next; /* shared work counter, guarded by lock */
  pthread_mutex_t lock;
  int err;
} job_t;

/* Rotary embedding of the 64 rotary columns at position pos (rotate-half form):
 *   y[d]      = x[d]      cos(pos f_d) - x[d + 32] sin(pos f_d)
 *   y[d + 32] = x[d + 32] cos(pos f_d) + x[d]      sin(pos f_d),   d < 32,
 * with cos and sin multiplied by the YaRN mscale ratio. */
static void rotate64(double* y, const double* x, double pos, const double* f, double msc) {
  for (int d = 0; d < 32; ++d) {
    const double a = pos * f[d];
    const double c = cos(a) * msc, sn = sin(a) * msc;
    y[d] = x[d] * c - x[d + 32] * sn;
    y[d + 32] = x[d + 32] * c + x[d] * sn;
  }
}

#define D_LAT 512 /* kv_lora_rank */

/* One output row from the latent cache, in the pages' (non-absorbed) form: kv_b_proj maps
 * the latent row c_j of key j to 64 x (128 + 128) features; head h takes features
 * [256h, 256h + 128) as its no-rope key and [256h + 128, 256h + 256) as its value.  Then
 * the same concat, scores, mask and softmax as one_row.  s is scratch of Tk doubles;
 * kv is scratch of 256 doubles. */
static int one_row_latent(const job_t* J, int64_t flat, double* s, double* o) {
  const int64_t i = flat % J->Tq;
  const int64_t bh = flat / J->Tq;
  const int64_t b = bh / J->H;
  const int64_t h = bh % J->H;
  if (b >= J->B) return 1;
  const int64_t kvl = J->kv_len ? (int64_t)J->kv_len[b] : J->Tk;
  if (kvl < 1 || kvl > J->Tk) return 2;
  double q[D_NOPE + D_ROPE];
  for (int d = 0; d < D_NOPE; ++d) q[d] = bf16_to_double(J->q_nope[(bh * J->Tq + i) * D_NOPE + d]);
  for (int d = 0; d < D_ROPE; ++d) q[D_NOPE + d] = bf16_to_double(J->q_pe[(bh * J->Tq + i) * D_ROPE + d]);
  const uint16_t* wk = J->w_kvb + (h * 256) * D_LAT;        /* rows of the no-rope key */
  const uint16_t* wv = J->w_kvb + (h * 256 + 128) * D_LAT;  /* rows of the value */
  for (int64_t j = 0; j < J->Tk; ++j) {
    const uint16_t* c = J->c_kv + (b * J->Tk + j) * D_LAT;
    double acc = 0.0;
    for (int e = 0; e < D_NOPE; ++e) {
      double kn = 0.0; /* k_nope[b, h, j, e] = sum_d W[256h + e, d] c[d] */
      for (int d = 0; d < D_LAT; ++d) kn += bf16_to_double(wk[e * D_LAT + d]) * bf16_to_double(c[d]);
      acc += q[e] * kn;
    }
    const uint16_t* kr = J->k_pe + (b * J->Tk + j) * D_ROPE;
    for (int d = 0; d < D_ROPE; ++d) acc += q[D_NOPE + d] * bf16_to_double(kr[d]); /* shared rotary key */
    double sj = acc * J->scale;
    const int visible = (j <= i + J->past_len) && (j < kvl);
    sj += visible ? 0.0 : MASK_MIN_BF16;
    s[j] = sj;
  }
  double m = s[0];
  for (int64_t j = 1; j < J->Tk; ++j)
    if (s[j] > m) m = s[j];
  double denom = 0.0;
  for (int64_t j = 0; j < J->Tk; ++j) {
    s[j] = exp(s[j] - m);
    denom += s[j];
  }
  for (int e = 0; e < D_V; ++e) o[e] = 0.0;
  for (int64_t j = 0; j < J->Tk; ++j) {
    const double w = s[j] / denom;
    if (w == 0.0) continue;
    const uint16_t* c = J->c_kv + (b * J->Tk + j) * D_LAT;
    for (int e = 0; e < D_V; ++e) {
      double v = 0.0; /* v[b, h, j, e] = sum_d W[256h + 128 + e, d] c[d] */
      for (int d = 0; d < D_LAT; ++d) v += bf16_to_double(wv[e * D_LAT + d]) * bf16_to_double(c[d]);
      o[e] += w * v;
    }
  }
  return 0;
}

/* One output row o[b, h, i, :].  s is scratch of Tk doubles. */
static int one_row(const job_t* J, int64_t flat, double* s, double* o, double* wsum_out) {
  if (J->c_kv) return one_row_latent(J, flat, s, o);
  const int64_t i = flat % J->Tq;
  const int64_t bh = flat / J->Tq;
  const int64_t b = bh / J->H;
  if (b >= J->B) return 1;
  const int64_t kvl = J->kv_len ? (int64_t)J->kv_len[b] : J->Tk;
  if (kvl < 1 || kvl > J->Tk) return 2;
  const int eager = (J->mode == 1);

  /* Step 1: query row Q = [q_nope | q_pe] (192 values). */
  double q[D_NOPE + D_ROPE];
  const uint16_t* qn = J->q_nope + (bh * J->Tq + i) * D_NOPE;
  const uint16_t* qr = J->q_pe + (bh * J->Tq + i) * D_ROPE;
  for (int d = 0; d < D_NOPE; ++d) q[d] = bf16_to_double(qn[d]);
  for (int d = 0; d < D_ROPE; ++d) q[D_NOPE + d] = bf16_to_double(qr[d]);
  if (J->rope_inv_freq) {
    /* The query's rotary part arrives unrotated; query i sits at position past_len + i. */
    double raw[D_ROPE];
    for (int d = 0; d < D_ROPE; ++d) raw[d] = q[D_NOPE + d];
    rotate64(q + D_NOPE, raw, (double)(J->past_len + i), J->rope_inv_freq, J->rope_mscale);
  }

  /* The scale is a Python float multiplied into a bf16 tensor: eager computes the product
   * with the scale as an fp32 value, which is what J->scale holds in both modes. */
  const double scale_used = J->scale;
  for (int64_t j = 0; j < J->Tk; ++j) {
    /* Step 2: key row K_j = [k_nope[b,h,j] | k_pe[b,j]]; the rotary part has no head index. */
    const uint16_t* kn = J->k_nope + (bh * J->Tk + j) * D_NOPE;
    const uint16_t* kr = J->k_pe + (b * J->Tk + j) * D_ROPE;
    /* Step 3: dot product over all 192 columns, then the scale. */
    double acc = 0.0;
    for (int d = 0; d < D_NOPE; ++d) acc += q[d] * bf16_to_double(kn[d]);
    if (J->rope_inv_freq && j >= J->past_len) {
      /* A new key's rotary part arrives unrotated and is rotated at its position j; the
       * cached rows (j < past_len) were stored rotated. */
      double raw[D_ROPE], rot[D_ROPE];
      for (int d = 0; d < D_ROPE; ++d) raw[d] = bf16_to_double(kr[d]);
      rotate64(rot, raw, (double)j, J->rope_inv_freq, J->rope_mscale);
      for (int d = 0; d < D_ROPE; ++d) acc += q[D_NOPE + d] * rot[d];
    } else {
      for (int d = 0; d < D_ROPE; ++d) acc += q[D_NOPE + d] * bf16_to_double(kr[d]);
    }
    if (eager) acc = round_bf16(acc);
    double sj = acc * scale_used;
    if (eager) sj = round_bf16(sj);
    /* Step 4: additive mask.  A key hidden by the causal mask, by the right padding or by
     * the 2D padding mask gets the one minimum (the masks are merged, not summed). */
    const int visible = (j <= i + J->past_len) && (j < kvl) &&
                        (!J->key_mask || J->key_mask[b * J->Tk + j] != 0);
    sj += visible ? 0.0 : MASK_MIN_BF16;
    if (eager) sj = round_bf16(sj);
    s[j] = sj;
  }

  /* Step 5: softmax over the key axis (max-subtracted, then normalised). */
  double m = s[0];
  for (int64_t j = 1; j < J->Tk; ++j)
    if (s[j] > m) m = s[j];
  double denom = 0.0;
  for (int64_t j = 0; j < J->Tk; ++j) {
    s[j] = exp(s[j] - m);
    denom += s[j];
  }
  double wsum = 0.0;
  for (int64_t j = 0; j < J->Tk; ++j) {
    s[j] = s[j] / denom;
    if (eager) s[j] = round_bf16(s[j]);
    wsum += s[j];
  }

  /* Step 6: weighted sum of value rows. */
  for (int d = 0; d < D_V; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < J->Tk; ++j) {
    const double w = s[j];
    if (w == 0.0) continue; /* adds exactly zero; skipping does not change the sum */
    const uint16_t* vr = J->v + (bh * J->Tk + j) * D_V;
    for (int d = 0; d < D_V; ++d) o[d] += w * bf16_to_double(vr[d]);
  }
  if (eager)
    for (int d = 0; d < D_V; ++d) o[d] = round_bf16(o[d]);
  if (wsum_out) *wsum_out = wsum;
  return 0;
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)(J->Tk > 0 ? J->Tk : 1));
  if (!s) {
    pthread_mutex_lock(&J->lock);
    J->err = 3;
    pthread_mutex_unlock(&J->lock);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int64_t r0 = J->next;
    J->next += 16;
    pthread_mutex_unlock(&J->lock);
    if (r0 >= J->n_rows) break;
    int64_t r1 = r0 + 16 < J->n_rows ? r0 + 16 : J->n_rows;
    for (int64_t r = r0; r < r1; ++r) {
      const int64_t flat = J->rows ? J->rows[r] : r;
      int e = one_row(J, flat, s, J->out + r * D_V, J->wsum ? J->wsum + r : NULL);
      if (e) {
        pthread_mutex_lock(&J->lock);
        J->err = e;
        pthread_mutex_unlock(&J->lock);
      }
    }
  }
  free(s);
  return NULL;
}

/*
 * Compute output rows of the attention core.
 *   q_nope [B,H,Tq,128], q_pe [B,H,Tq,64], k_nope [B,H,Tk,128], k_pe [B,Tk,64],
 *   v [B,H,Tk,128]: bf16 bit patterns, row-major, contiguous.
 *   kv_len [B] (int32, may be NULL meaning Tk for every sequence).
 *   rows: n_rows flat row indices ((b*H + h)*Tq + i); NULL means all B*H*Tq rows.
 *   out [n_rows,128] and wsum [n_rows] (may be NULL): written as double.
 * Returns 0, or a nonzero code for bad arguments (shape, kv_len out of [1,Tk], alloc).
 */
static int rows_impl(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                     const uint16_t* k_pe, const uint16_t* v, const int32_t* kv_len, int64_t B,
                     int64_t H, int64_t Tq, int64_t Tk, int64_t past_len, float softmax_scale,
                     const int64_t* rows, int64_t n_rows, int mode, int nthreads, double* out,
                     double* wsum, const double* rope_inv_freq, double rope_mscale,
                     const uint8_t* key_mask) {
  if (B < 1 || H < 1 || Tq < 1 || Tk < 1 || past_len < 0 || Tk != past_len + Tq) return 10;
  if (!q_nope || !q_pe || !k_nope || !k_pe || !v || !out) return 11;
  if (mode != 0 && mode != 1) return 12;
  if (rows) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= B * H * Tq) return 13;
  } else {
    n_rows = B * H * Tq;
  }
  job_t J;
  memset(&J, 0, sizeof J);
  J.q_nope = q_nope; J.q_pe = q_pe; J.k_nope = k_nope; J.k_pe = k_pe; J.v = v;
  J.kv_len = kv_len;
  J.key_mask = key_mask;
  J.B = B; J.H = H; J.Tq = Tq; J.Tk = Tk; J.past_len = past_len;
  J.scale = (double)softmax_scale;
  J.rows = rows; J.n_rows = n_rows; J.mode = mode; J.out = out; J.wsum = wsum;
  J.rope_inv_freq = rope_inv_freq;
  J.rope_mscale = rope_mscale;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, worker, &J) == 0) ++started;
  if (started == 0) worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.err;
}

int mla_oracle_rows(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                    const uint16_t* k_pe, const uint16_t* v, const int32_t* kv_len, int64_t B,
                    int64_t H, int64_t Tq, int64_t Tk, int64_t past_len, float softmax_scale,
                    const int64_t* rows, int64_t n_rows, int mode, int nthreads, double* out,
                    double* wsum) {
  return rows_impl(q_nope, q_pe, k_nope, k_pe, v, kv_len, B, H, Tq, Tk, past_len, softmax_scale,
                   rows, n_rows, mode, nthreads, out, wsum, NULL, 1.0, NULL);
}

/*
 * The same rows with a 2D padding mask on the keys (the attention_mask argument of the
 * model, "Kimi K2 · Causal mask", §Construct causal mask: expanded to 4D and merged with the
 * causal mask before the scores): key_mask [B][Tk] bytes, 0 = hidden.  A hidden key gets
 * the same additive minimum as a causally hidden one.  A row whose keys are all hidden then
 * has every score equal to that minimum (the score is absorbed: |s| is far below the
 * spacing of doubles near 3.4e38), so its weights are uniform over all Tk keys, as in the
 * eager computation.
 */
int mla_oracle_rows_mask(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                         const uint16_t* k_pe, const uint16_t* v, const int32_t* kv_len,
                         const uint8_t* key_mask, int64_t B, int64_t H, int64_t Tq, int64_t Tk,
                         int64_t past_len, float softmax_scale, const int64_t* rows,
                         int64_t n_rows, int mode, int nthreads, double* out, double* wsum) {
  if (!key_mask) return 15;
  return rows_impl(q_nope, q_pe, k_nope, k_pe, v, kv_len, B, H, Tq, Tk, past_len, softmax_scale,
                   rows, n_rows, mode, nthreads, out, wsum, NULL, 1.0, key_mask);
}

/*
 * The same rows with the rotary step of the attention excerpt applied first
 * ("q_pe, k_pe = apply_rotary_pos_emb(q_pe, k_pe, cos, sin, position_ids)"): q_pe holds
 * unrotated query rows (query i at position past_len + i); k_pe rows j >= past_len hold
 * unrotated new keys (rotated at position j); rows j < past_len are cached, already rotated.
 * inv_freq: the 32 rotary frequencies; mscale: factor on cos and sin.
 */
int mla_oracle_rows_rope(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                         const uint16_t* k_pe, const uint16_t* v, const int32_t* kv_len,
                         int64_t B, int64_t H, int64_t Tq, int64_t Tk, int64_t past_len,
                         float softmax_scale, const int64_t* rows, int64_t n_rows, int nthreads,
                         double* out, const double* inv_freq, double mscale) {
  if (!inv_freq) return 14;
  return rows_impl(q_nope, q_pe, k_nope, k_pe, v, kv_len, B, H, Tq, Tk, past_len, softmax_scale,
                   rows, n_rows, 0, nthreads, out, NULL, inv_freq, mscale, NULL);
}

/*
 * Output rows of attention over the latent cache: c_kv [B][Tk][512] (the input of
 * kv_b_proj), k_pe [B][Tk][64] (the shared rotary key), w_kvb [H*256][512] (the kv_b_proj
 * weight, "Kimi K2 · Similarities", §Scale scores: kv_lora_rank -> num_heads x
 * (qk_nope_head_dim + v_head_dim)), q_nope [B][H][Tq][128], q_pe [B][H][Tq][64].  Computed
 * in the non-absorbed form (per-head keys and values materialised from the latent), so it
 * checks the absorbed kernels without sharing their algebra.
 */
int mla_oracle_latent_rows(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* c_kv,
                           const uint16_t* k_pe, const uint16_t* w_kvb, const int32_t* kv_len,
                           int64_t B, int64_t H, int64_t Tq, int64_t Tk, int64_t past_len,
                           float softmax_scale, const int64_t* rows, int64_t n_rows, int nthreads,
                           double* out) {
  if (!c_kv || !w_kvb || !q_nope || !q_pe || !k_pe || !out) return 11;
  if (B < 1 || H < 1 || Tq < 1 || Tk < 1 || past_len < 0 || Tk != past_len + Tq) return 10;
  if (rows) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= B * H * Tq) return 13;
  } else {
    n_rows = B * H * Tq;
  }
  job_t J;
  memset(&J, 0, sizeof J);
  J.q_nope = q_nope; J.q_pe = q_pe; J.k_pe = k_pe; J.c_kv = c_kv; J.w_kvb = w_kvb;
  J.kv_len = kv_len;
  J.B = B; J.H = H; J.Tq = Tq; J.Tk = Tk; J.past_len = past_len;
  J.scale = (double)softmax_scale;
  J.rows = rows; J.n_rows = n_rows; J.out = out;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, worker, &J) == 0) ++started;
  if (started == 0) worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.err;
}

/*
 * YaRN rotary frequencies for a 64-column rotary part (Peng et al., "YaRN: Efficient
 * Context Window Extension of Large Language Models", 2023), as configured by the
 * rope_scaling block of the config.json excerpt on "Kimi K2 · Logits":
 *   extrapolated f_d = theta^(-2d/64), interpolated f_d / factor;
 *   the dimension at which a wavelength makes n rotations over the original context L is
 *     dim(n) = 64 ln(L / (2 pi n)) / (2 ln theta);
 *   low = floor(dim(beta_fast)), high = ceil(dim(beta_slow)), clamped to [0, 31];
 *   ramp_d = clamp((d - low) / (high - low), 0, 1)  (high == low: high + 0.001);
 *   f_d = interpolated * ramp_d + extrapolated * (1 - ramp_d).
 * Returns through mscale_ratio the factor on cos and sin,
 *   m(factor, mscale) / m(factor, mscale_all_dim),  m(s, k) = 0.1 k ln s + 1 (s > 1), else 1.
 */
void mla_oracle_yarn(double theta, double factor, double orig_max_pos, double beta_fast,
                     double beta_slow, double mscale, double mscale_all_dim, double* inv_freq,
                     double* mscale_ratio) {
  const double pi = 3.14159265358979323846;
  double low = floor(64.0 * log(orig_max_pos / (2.0 * pi * beta_fast)) / (2.0 * log(theta)));
  double high = ceil(64.0 * log(orig_max_pos / (2.0 * pi * beta_slow)) / (2.0 * log(theta)));
  if (low < 0.0) low = 0.0;
  if (high > 31.0) high = 31.0;
  if (high == low) high += 0.001;
  for (int d = 0; d < 32; ++d) {
    const double extra = pow(theta, -2.0 * d / 64.0);
    const double inter = extra / factor;
    double ramp = ((double)d - low) / (high - low);
    if (ramp < 0.0) ramp = 0.0;
    if (ramp > 1.0) ramp = 1.0;
    inv_freq[d] = inter * ramp + extra * (1.0 - ramp);
  }
  const double m1 = factor > 1.0 ? 0.1 * mscale * log(factor) + 1.0 : 1.0;
  const double m2 = factor > 1.0 ? 0.1 * mscale_all_dim * log(factor) + 1.0 : 1.0;
  *mscale_ratio = m1 / m2;
}

/*
 * The rotary step alone: row r of x ([n][64] bf16 bits) rotated at position pos[r] into
 * out ([n][64] doubles), with the frequencies and mscale ratio of mla_oracle_yarn.  Used to
 * check rotated rows that a cache holds.
 */
int mla_oracle_rotate(const uint16_t* x, const int64_t* pos, int64_t n, const double* inv_freq,
                      double mscale, double* out) {
  if (!x || !pos || !inv_freq || !out || n < 0) return 1;
  for (int64_t r = 0; r < n; ++r) {
    double raw[D_ROPE];
    for (int d = 0; d < D_ROPE; ++d) raw[d] = bf16_to_double(x[r * D_ROPE + d]);
    rotate64(out + r * D_ROPE, raw, (double)pos[r], inv_freq, mscale);
  }
  return 0;
}

/* Exposed for the test that pins the diagnostic rounding against torch's own cast. */
double mla_oracle_round_bf16(double x) { return round_bf16(x); }

/*
 * Output projection of the attention output.  The MLA init excerpt on "Kimi K2 ·
 * Similarities" (section "Scale scores") defines o_proj as a linear map from
 * num_heads x v_head_dim to hidden_size, with bias = attention_bias (false in the
 * config.json excerpt on "Kimi K2 · Logits"): y = W x, W [N][K] as nn.Linear stores it.
 * Its input row for (b, i) is the heads' outputs concatenated in head order, feature
 * k = h * 128 + d of attn [B][H][T][128] (the reshape before o_proj is not shown on the
 * pages; this is the plain reading).  Sums in fp64 over exact bf16 products.
 * rows: flat indices b * T + i, or NULL for all B * T rows; out [n_rows][N].
 */
typedef struct {
  const uint16_t* attn;
  const uint16_t* w;
  int64_t B, H, T, N, K;
  const int64_t* rows;
  int64_t n_rows;
  double* out;
  int64_t next;
  int err;
  pthread_mutex_t lock;
} oproj_job_t;

static void* oproj_worker(void* arg) {
  oproj_job_t* J = (oproj_job_t*)arg;
  double* x = (double*)malloc((size_t)J->K * sizeof(double));
  if (!x) { /* reported: a row another worker does not pick up stays unwritten */
    pthread_mutex_lock(&J->lock);
    J->err = 3;
    pthread_mutex_unlock(&J->lock);
    return NULL;
  }
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int64_t r = J->next++;
    pthread_mutex_unlock(&J->lock);
    if (r >= J->n_rows) break;
    const int64_t flat = J->rows ? J->rows[r] : r;
    const int64_t b = flat / J->T, i = flat % J->T;
    for (int64_t h = 0; h < J->H; ++h) { /* concatenated head outputs */
      const uint16_t* src = J->attn + ((b * J->H + h) * J->T + i) * D_V;
      for (int64_t d = 0; d < D_V; ++d) x[h * D_V + d] = bf16_to_double(src[d]);
    }
    double* y = J->out + r * J->N;
    for (int64_t n = 0; n < J->N; ++n) {
      const uint16_t* wr = J->w + n * J->K; /* row n of the weight */
      double acc = 0.0;
      for (int64_t k = 0; k < J->K; ++k) acc += bf16_to_double(wr[k]) * x[k];
      y[n] = acc;
    }
  }
  free(x);
  return NULL;
}

int mla_oracle_oproj_rows(const uint16_t* attn, const uint16_t* w, int64_t B, int64_t H,
                          int64_t T, int64_t N, const int64_t* rows, int64_t n_rows,
                          int nthreads, double* out) {
  if (!attn || !w || !out) return 11;
  if (B < 1 || H < 1 || T < 1 || N < 1) return 10;
  if (rows) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= B * T) return 13;
  } else {
    n_rows = B * T;
  }
  oproj_job_t J;
  memset(&J, 0, sizeof J);
  J.attn = attn; J.w = w;
  J.B = B; J.H = H; J.T = T; J.N = N; J.K = H * D_V;
  J.rows = rows; J.n_rows = n_rows; J.out = out;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, oproj_worker, &J) == 0) ++started;
  if (started == 0) oproj_worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.lock);
  return J.err;
}
