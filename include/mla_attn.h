/*
 * mla_attn.h -- C ABI of the GB300 (sm_103a) MLA causal-attention library.
 *
 * The operation is the causal-attention core of Kimi K2's Multi-head Latent Attention,
 * as quoted on the page "Kimi K2 · Similarities" (section "Contextual evidence from
 * Query-key similarity", the MLA forward of modeling_deepseek.py) and on the page
 * "Weighted sum of values" (tensor card: weights [B,64,T,T] times values [B,64,T,128]
 * give [B,64,T,128]).  Per sequence b, head h and query i:
 *
 *   Q   = [q_nope[b,h,i,0:128] | q_pe[b,h,i,0:64]]           (query concat)
 *   K_j = [k_nope[b,h,j,0:128] | k_pe_shared[b,j,0:64]]      (key concat; one rotary
 *                                                             key row shared by all heads)
 *   s_j = softmax_scale * (Q . K_j)                          (scores, then scale)
 *   key j is visible iff j <= i + past_len and j < kv_len[b] (4D causal mask offset by
 *                                                             the cached length, plus
 *                                                             right padding)
 *   w   = softmax over visible j of s_j, in fp32             (hidden keys get weight 0)
 *   out[b,h,i,:] = sum_j bf16(w_j) * v[b,h,j,:]              (weights cast to bf16, then
 *                                                             the weighted sum of values)
 *
 * Dropout (attention_dropout = 0.0 in the config.json excerpt on "Kimi K2 · Logits") is
 * the identity and is not applied.  The cache layout follows the cache update in the
 * same excerpt: the Tk = past_len + Tq key/value rows hold the cached prefix first and
 * the Tq new rows last, and query i sits at position past_len + i (positions are
 * numbered from the cached length, page "Kimi K2 · Causal mask", section "Construct
 * causal mask").
 *
 * Head widths are fixed by the config.json excerpt: qk_nope_head_dim 128,
 * qk_rope_head_dim 64, v_head_dim 128.  The head count H is a runtime argument (64 in
 * Kimi K2).
 *
 * Data types and layout.  bf16 tensors are passed as uint16_t bit patterns; every tensor
 * is row-major and contiguous in the shape given, in DEVICE memory of the current CUDA
 * device:
 *   q_nope      [B, H, Tq, 128]      q_pe        [B, H, Tq, 64]
 *   k_nope      [B, H, Tk, 128]      k_pe_shared [B, Tk, 64]
 *   v           [B, H, Tk, 128]      out         [B, H, Tq, 128]
 *   kv_len      [B] int32, or NULL meaning kv_len[b] = Tk for every b
 * Every pointer must be 16-byte aligned (bulk/tensor copies move 16-byte units).
 *
 * Ownership.  The caller owns every buffer: inputs, out, kv_len and the workspace.  The
 * library never allocates or frees device memory on the call path.  Inputs are only
 * read; out is fully overwritten.  Work is enqueued asynchronously on cuda_stream (a
 * cudaStream_t, NULL for the legacy default stream); the call returns before it runs.
 *
 * Errors.  Host-side checks run before anything is enqueued and are returned directly
 * (nothing is launched when a check fails).  Problems only the device can see
 * (kv_len[b] outside [1, Tk]; a bounded wait that gave up) are recorded in a status word
 * inside the workspace; mla_attn_get_status reads it.  Such a call still completes: an
 * out-of-range kv_len is clamped to [1, Tk] for memory safety and the output for that
 * sequence is not meaningful.
 */
#ifndef MLA_ATTN_H_
#define MLA_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_NULL = 1,      /* a required pointer is NULL */
  MLA_ERR_SHAPE = 2,     /* B, H, Tq < 1, past_len < 0, Tk != past_len + Tq, or too large:
                            the score-shape check of the attention excerpt (scores must be
                            [B, H, Tq, Tk]) */
  MLA_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned */
  MLA_ERR_WORKSPACE = 4, /* workspace NULL or smaller than mla_attn_workspace_bytes() */
  MLA_ERR_DEVICE = 5,    /* the current device is not an sm_103 (GB300-class) GPU */
  MLA_ERR_CUDA = 6,      /* a CUDA runtime call or kernel launch failed */
  MLA_ERR_KVLEN = 7,     /* (device) some kv_len[b] outside [1, Tk] */
  MLA_ERR_TIMEOUT = 8,   /* (device) a bounded wait inside a kernel gave up */
  MLA_ERR_ARG = 9        /* an option value is out of range */
} mla_status;

/*
 * Bytes of device workspace mla_attn_fwd needs for these sizes (a status word plus the
 * split-KV partial results of the decode path).  The workspace must be zero-filled once
 * before its first use (cudaMemset); afterwards the library keeps the status word
 * consistent itself.  Returns 0 for invalid sizes.
 */
MLA_API size_t mla_attn_workspace_bytes(int B, int H, int Tq, int Tk);

/*
 * The attention core described at the top of this file.  past_len is the cached length
 * (Tk must equal past_len + Tq); softmax_scale (finite, > 0, else MLA_ERR_ARG) multiplies
 * the raw scores (192^-0.5 for Kimi K2 before any YaRN adjustment, which the caller folds
 * in).  Tq == 1 takes the
 * split-KV decode path; Tq > 1 the tensor-core prefill path.  Returns MLA_OK once the
 * work is enqueued, or a host-side error code.
 */
MLA_API mla_status mla_attn_fwd(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                        const uint16_t* k_pe_shared, const uint16_t* v, const int32_t* kv_len,
                        int B, int H, int Tq, int Tk, int past_len, float softmax_scale,
                        uint16_t* out, void* workspace, size_t workspace_bytes,
                        void* cuda_stream);

/* Path selection for mla_attn_fwd_ex. */
typedef enum { MLA_PATH_AUTO = 0, MLA_PATH_PREFILL = 1, MLA_PATH_DECODE = 2 } mla_path;

/*
 * Options for mla_attn_fwd_ex.  Zero-initialised options mean "choose automatically",
 * which is what mla_attn_fwd does.
 *   path:         force the prefill (any Tq >= 1) or decode (Tq == 1 only) path.
 *   decode_chunk: keys per split of the decode path (a multiple of 64, at most 65536);
 *                 0 lets the scheduler pick it from B, H and Tk.
 */
typedef struct {
  int path;
  int decode_chunk;
  int reserved[6];
} mla_attn_options;

/* mla_attn_fwd with explicit options (same arguments and semantics otherwise). */
MLA_API mla_status mla_attn_fwd_ex(const uint16_t* q_nope, const uint16_t* q_pe,
                           const uint16_t* k_nope, const uint16_t* k_pe_shared,
                           const uint16_t* v, const int32_t* kv_len, int B, int H, int Tq,
                           int Tk, int past_len, float softmax_scale, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* cuda_stream,
                           const mla_attn_options* options);

/*
 * Cache append + attention.  The cache update of the attention excerpt on "Kimi K2 ·
 * Similarities" (past_key_value.update: the new key/value rows follow the cached prefix)
 * fused with the core described at the top of this file:
 *
 *   k_nope_cache[b,h,past_len+t,:] = k_nope_new[b,h,t,:]    (t < Tq)
 *   k_pe_cache  [b,  past_len+t,:] = k_pe_new  [b,  t,:]
 *   v_cache     [b,h,past_len+t,:] = v_new     [b,h,t,:]
 *   out = attention over rows [0, Tk) of the caches, Tk = past_len + Tq
 *
 * Caches: k_nope_cache / v_cache [B, H, T_cap, 128], k_pe_cache [B, T_cap, 64], device,
 * T_cap >= past_len + Tq rows per (b, h) (per b for k_pe); rows outside [past_len, Tk) are
 * not written.  New rows: k_nope_new / v_new [B, H, Tq, 128], k_pe_new [B, Tq, 64].  The
 * other arguments are those of mla_attn_fwd (kv_len, when given, still hides keys >=
 * kv_len[b]; the new rows are written at past_len regardless).  With Tq == 1 the append
 * is fused into the decode kernel (the stage holding the new row reads it from the new
 * buffers; one CTA per head group writes it to the cache).  With Tq > 1, past_len a
 * multiple of 128 and kv_len NULL it is fused into the prefill kernel: key tiles past the
 * cached prefix are read from the new buffers, and the work unit holding each such tile on
 * its causal diagonal writes it into the caches (every new row is then read by its owner).
 * Other prefills run a copy kernel that appends the rows before the attention kernel.  The
 * output is the same either way.  Errors as for mla_attn_fwd; MLA_ERR_SHAPE also when
 * past_len + Tq > T_cap.
 */
MLA_API mla_status mla_attn_append_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                                       const uint16_t* k_nope_new, const uint16_t* k_pe_new,
                                       const uint16_t* v_new, uint16_t* k_nope_cache,
                                       uint16_t* k_pe_cache, uint16_t* v_cache,
                                       const int32_t* kv_len, int B, int H, int Tq, int T_cap,
                                       int past_len, float softmax_scale, uint16_t* out,
                                       void* workspace, size_t workspace_bytes,
                                       void* cuda_stream);

/*
 * Attention with a 2D padding mask on the keys.  The model's attention_mask ("Kimi K2 ·
 * Causal mask", section "Construct causal mask") is expanded to 4D and merged with the
 * causal mask, so a hidden key gets the same additive minimum as a causally hidden one:
 *
 *   key j is visible to query i of sequence b iff j <= i + past_len, j < kv_len[b] and
 *   key_mask[b * Tk + j] != 0
 *
 * key_mask: [B, Tk] bytes in device memory (any alignment), nonzero = attend.  Left
 * padding (a run of zeros first) and arbitrary holes are both expressible.  A query row
 * that sees no visible key at all has every score equal to the minimum, so its weights
 * are uniform over all Tk keys: its output is the mean of the Tk value rows (the eager
 * result; such rows are usually padding queries).  The other arguments are those of
 * mla_attn_fwd; the workspace must hold mla_attn_masked_workspace_bytes(B, H, Tq, Tk)
 * bytes (for Tq > 1 it also holds the mask packed to bits).  MLA_ERR_NULL without key_mask.
 */
MLA_API size_t mla_attn_masked_workspace_bytes(int B, int H, int Tq, int Tk);
MLA_API mla_status mla_attn_masked_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                                       const uint16_t* k_nope, const uint16_t* k_pe_shared,
                                       const uint16_t* v, const int32_t* kv_len,
                                       const uint8_t* key_mask, int B, int H, int Tq, int Tk,
                                       int past_len, float softmax_scale, uint16_t* out,
                                       void* workspace, size_t workspace_bytes,
                                       void* cuda_stream);

/*
 * Decode over the latent cache.  The MLA init excerpt on "Kimi K2 · Similarities" (section
 * "Scale scores") has kv_a_proj_with_mqa produce a 512-wide latent row plus the shared
 * 64-wide rotary key per token, and kv_b_proj map the latent to 64 heads x (128 no-rope
 * key + 128 value).  A cache of latent rows holds 1152 bytes per token instead of the
 * 32,896 of per-head keys and values.  This call computes, for Tq = 1 (query at the last
 * position, causality vacuous) and every head h,
 *
 *   k_nope[b,h,j] = W[256h : 256h+128] . c_kv[b,j]      (no-rope key of key j)
 *   v[b,h,j]      = W[256h+128 : 256h+256] . c_kv[b,j]  (value of key j)
 *   out[b,h]      = the attention core of mla_attn_fwd on [q_nope | q_pe] and
 *                   [k_nope | k_pe], keys j < kv_len[b]
 *
 * without materialising k_nope or v: the no-rope key rows of W are folded into the query
 * (q_lat = W_K^T q_nope), the value rows applied once to the weighted latent sum.  Reading
 * of the weight layout: per head, the first 128 of its 256 kv_b_proj output rows are the
 * no-rope key, the next 128 the value.
 *
 *   q_nope [B, H, 128], q_pe [B, H, 64]           (bf16, device)
 *   c_kv   [B, Tk, 512], k_pe [B, Tk, 64]         (bf16, device: the latent cache)
 *   w_kvb  [H * 256, 512]                         (bf16, device: the kv_b_proj weight)
 *   kv_len [B] int32 or NULL, out [B, H, 128]
 * H must be at most 64.  Workspace: mla_latent_workspace_bytes(B, H, Tk), zeroed once.
 * Errors as for mla_attn_fwd.
 */
MLA_API size_t mla_latent_workspace_bytes(int B, int H, int Tk);
MLA_API mla_status mla_latent_decode_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                                         const uint16_t* c_kv, const uint16_t* k_pe,
                                         const uint16_t* w_kvb, const int32_t* kv_len, int B,
                                         int H, int Tk, float softmax_scale, uint16_t* out,
                                         void* workspace, size_t workspace_bytes,
                                         void* cuda_stream);

/*
 * Output projection (o_proj) of the attention output.  The MLA init excerpt on "Kimi K2 ·
 * Similarities" (section "Scale scores") ends the attention block with
 * o_proj = nn.Linear(num_heads * v_head_dim, hidden_size, bias = attention_bias); the
 * config.json excerpt on "Kimi K2 · Logits" has hidden_size 7168 and attention_bias false.
 * Reading of its input (the forward's reshape is not shown): the row for (b, i) is the
 * heads' outputs concatenated in head order, feature k = 128 h + d of attn, which is read in
 * place in the layout mla_attn_fwd writes.
 *
 *   attn [B, H, T, 128]   bf16, device
 *   w_o  [N, H * 128]     bf16, device (nn.Linear's weight: out_features x in_features)
 *   y    [B, T, N]        bf16, device, fully overwritten:
 *   y[b, i, n] = sum over h, d of w_o[n, 128 h + d] * attn[b, h, i, d]  (fp32 accumulation)
 * N must be a multiple of 32 and every pointer 16-byte aligned.  Workspace:
 * mla_oproj_workspace_bytes() (the status word), zeroed once.  Errors: MLA_ERR_NULL,
 * MLA_ERR_SHAPE (a size < 1, N not a multiple of 32, a tensor too large), MLA_ERR_ALIGN,
 * MLA_ERR_WORKSPACE, MLA_ERR_DEVICE, MLA_ERR_CUDA; a bounded wait that gives up sets
 * MLA_ERR_TIMEOUT in the status word (mla_attn_get_status).
 */
MLA_API size_t mla_oproj_workspace_bytes(void);
MLA_API mla_status mla_oproj_fwd(const uint16_t* attn, const uint16_t* w_o, int B, int H, int T,
                                 int N, uint16_t* y, void* workspace, size_t workspace_bytes,
                                 void* cuda_stream);

/*
 * Rotary embedding.  The attention excerpt on "Kimi K2 · Similarities" rotates the query's
 * and the new keys' rotary parts before the cache update (rotary_emb gives cos and sin for
 * the positions, apply_rotary_pos_emb rotates q_pe and k_pe), and the rope_scaling block of
 * the config.json excerpt on "Kimi K2 · Logits" selects YaRN scaling (Peng et al., "YaRN:
 * Efficient Context Window Extension of Large Language Models", 2023).  The pages give the
 * calls and the configuration, not the function bodies; the library takes the published
 * YaRN method:
 *   extrapolated f_d = theta^(-2d/64), interpolated f_d / factor   (d = 0..31)
 *   dim(n) = 64 ln(L / (2 pi n)) / (2 ln theta)   (L = original_max_position)
 *   low = floor(dim(beta_fast)), high = ceil(dim(beta_slow)), clamped to [0, 31]
 *   ramp_d = clamp((d - low) / (high - low), 0, 1)   (high == low: high + 0.001)
 *   f_d = interpolated * ramp_d + extrapolated * (1 - ramp_d)
 *   mscale ratio = m(factor, mscale) / m(factor, mscale_all_dim),
 *                  m(s, k) = 0.1 k ln s + 1 for s > 1, else 1
 * and the rotate-half rotation of the 64 rotary columns of a row at position p:
 *   y[d]    = x[d]    * c - x[d+32] * s
 *   y[d+32] = x[d+32] * c + x[d]    * s,     c = cos(p f_d) * ratio, s = sin(p f_d) * ratio
 * Kimi K2's values: theta 50000, factor 32, original_max_position 4096, beta_fast 1,
 * beta_slow 1, mscale 1, mscale_all_dim 1.
 */
typedef struct {
  double rope_theta;            /* > 1 */
  double factor;                /* >= 1 */
  double original_max_position; /* > 0 */
  double beta_fast;             /* >= beta_slow */
  double beta_slow;             /* > 0 */
  double mscale;
  double mscale_all_dim;
} mla_rope_config;

/*
 * Host only: the 32 frequencies f_d and the mscale ratio of a configuration (written
 * through the non-NULL pointers).  MLA_ERR_NULL without cfg; MLA_ERR_ARG for values out of
 * the ranges above or not finite.
 */
MLA_API mla_status mla_rope_frequencies(const mla_rope_config* cfg, double* inv_freq,
                                        double* mscale_ratio);

/*
 * Fills table (device, float, [max_pos][64], 16-byte aligned) with cos(p f_d) * ratio in
 * columns 0..31 and sin(p f_d) * ratio in columns 32..63 for positions p < max_pos; the
 * angles are formed and evaluated in double, then rounded to float.  Build it once per
 * configuration and pass it to mla_attn_rope_append_fwd.  Enqueued on cuda_stream.
 */
MLA_API mla_status mla_rope_table(const mla_rope_config* cfg, int max_pos, float* table,
                                  void* cuda_stream);

/* Bytes of workspace mla_attn_rope_append_fwd needs (0 for invalid sizes). */
MLA_API size_t mla_attn_rope_workspace_bytes(int B, int H, int Tq, int Tk);

/*
 * Rotary step + cache append + attention.  As mla_attn_append_fwd, except that q_pe_raw
 * and k_pe_new_raw arrive unrotated: query t and new key t are rotated at position
 * past_len + t with the table from mla_rope_table (table_rows >= past_len + Tq rows, else
 * MLA_ERR_SHAPE); the rotated new keys are what the k_pe cache receives (cached rows are
 * stored rotated and are not rotated again); the rotated queries are kept in the
 * workspace (at least mla_attn_rope_workspace_bytes(B, H, Tq, past_len + Tq) bytes, zeroed
 * once like mla_attn_fwd's).  Rotated values are rounded to bf16, the type of the cache.
 * With Tq == 1 the decode kernel itself rotates the query and the new rotary key (one
 * launch besides the split merge) and appends the new rows.  With Tq > 1 a rotation kernel
 * runs first: for a prefill that fuses the append (past_len a multiple of 128, kv_len
 * NULL; see mla_attn_append_fwd) it only rotates the queries and the new rotary keys into
 * the workspace and the prefill kernel appends all three new rows; otherwise it also writes
 * the rotated keys and the no-rope key and value rows into the caches before the prefill
 * kernel runs.  All host checks run before anything is enqueued.
 */
MLA_API mla_status mla_attn_rope_append_fwd(const uint16_t* q_nope, const uint16_t* q_pe_raw,
                                            const uint16_t* k_nope_new,
                                            const uint16_t* k_pe_new_raw, const uint16_t* v_new,
                                            uint16_t* k_nope_cache, uint16_t* k_pe_cache,
                                            uint16_t* v_cache, const int32_t* kv_len, int B,
                                            int H, int Tq, int T_cap, int past_len,
                                            float softmax_scale, const float* rope_table,
                                            int table_rows, uint16_t* out, void* workspace,
                                            size_t workspace_bytes, void* cuda_stream);

/*
 * Synchronises cuda_stream, reads the device status word in the workspace, clears it,
 * and returns it (MLA_OK if no kernel recorded a problem since the last read).
 */
MLA_API mla_status mla_attn_get_status(void* workspace, void* cuda_stream);

/* Static, human-readable name of a status code. */
MLA_API const char* mla_status_string(mla_status status);

/*
 * The decode scheduler's choice for these sizes: keys per split and number of splits
 * (written through the non-NULL pointers).  Pure host arithmetic; returns MLA_ERR_SHAPE
 * for invalid sizes.
 */
MLA_API mla_status mla_attn_decode_plan(int B, int H, int Tk, int* chunk, int* splits);

/*
 * Decode (Tq == 1, past_len = Tk - 1) without a caller-provided workspace.  The pages
 * have no counterpart to this call: it exists for callers that cannot allocate device
 * memory for the library (a server whose KV-cache pool owns all free HBM, a plugin inside
 * a framework whose allocator owns the device, a loop that cannot afford cudaMalloc's
 * implicit synchronisation).  The split-KV partials live in a 32 MiB array inside the
 * library image, which every GPU that loads the library holds until the process exits.
 *
 * Arguments and result are those of mla_attn_fwd with Tq = 1 and the same split plan, so
 * the output matches mla_attn_fwd's.  device_status (device int, may be NULL) receives
 * device-detected errors (MLA_ERR_KVLEN, MLA_ERR_TIMEOUT) the way the workspace status
 * word does; the caller zeroes and reads it.  Pass it: with device_status NULL those
 * errors go unreported, and after a bounded wait gives up (a split that never wrote its
 * partial) the merge may read partials a previous call left in the array, so the output
 * is undefined without any sign of it.  Returns MLA_ERR_WORKSPACE when the plan for these
 * sizes needs more than the 32 MiB array (B * H * splits partials of 520 bytes each).
 *
 * The call allocates nothing.  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and keeps it for the rest of
 * the process; make that first call before any stream capture.  The kept address belongs
 * to the device's context of that time: after cudaDeviceReset on that device it is stale,
 * so do not call this function on a device that has been reset since its first call.  All
 * calls share the array: calls that overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller.
 */
MLA_API mla_status mla_attn_decode_noalloc(const uint16_t* q_nope, const uint16_t* q_pe,
                                           const uint16_t* k_nope, const uint16_t* k_pe_shared,
                                           const uint16_t* v, const int32_t* kv_len, int B,
                                           int H, int Tk, float softmax_scale, uint16_t* out,
                                           int* device_status, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_ATTN_H_ */
