// kernels.h -- internal launch interface between the C-ABI host code and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mla_attn.h"

namespace mla {

// Decode (Tq == 1): split-KV partial pass, then a combine pass when there are several
// splits.  Partials live in the caller's workspace: part_ml [B*H*splits][2] = (max, sum)
// in the log2 domain, part_acc [B*H*splits][128] = unnormalised weighted value sums.
struct DecodeArgs {
  const uint16_t* q_nope;
  const uint16_t* q_pe;
  const uint16_t* k_nope;
  const uint16_t* k_pe;
  const uint16_t* v;
  const int32_t* kv_len;  // may be null
  uint16_t* out;
  float* part_ml;
  float* part_acc;
  int* status;
  int B, H, Tk;
  int chunk;   // keys per split
  int splits;  // ceil(Tk / chunk)
  float scale_log2;  // softmax_scale * log2(e)
  int kv_rows;       // rows per (b, h) of k_nope / v and per b of k_pe (>= Tk)
  // Optional fused cache append (all null otherwise): key row Tk-1 is taken from new_*
  // ([B,H,1,128], [B,1,64], [B,H,1,128]) instead of the cache, and written into the cache
  // at row Tk-1 through cache_* (the same buffers as k_nope / k_pe / v).
  const uint16_t* new_k_nope;
  const uint16_t* new_k_pe;
  const uint16_t* new_v;
  uint16_t* cache_k_nope;
  uint16_t* cache_k_pe;
  uint16_t* cache_v;
  // Optional 2D padding mask [B][Tk] (0 = key hidden); null otherwise.
  const uint8_t* key_mask;
  // Optional rotary step (with the fused append only): q_pe and new_k_pe arrive unrotated
  // and are rotated at position Tk - 1 with this row of the cos/sin table (64 floats: cos of
  // the 32 angles, then sin); null otherwise.
  const float* rope_cs;
};

// Decode kernel configuration (shared with the scheduler).
constexpr int kDecHeadsPerCta = 4;   // heads sharing one rotary-key tile
constexpr int kDecTokensPerStage = 16;
constexpr int kDecMinChunk = 64;
constexpr int kDecMaxChunk = 65536;

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// The decode scheduler's choice for given sizes on a GPU with `sms` SMs.
struct DecodePlan {
  int chunk;
  int splits;
};
DecodePlan plan_decode(int B, int H, int Tk, int sms, int forced_chunk);

// Prefill (Tq >= 1): fused tensor-core kernel.
struct PrefillArgs {
  const uint16_t* q_nope;
  const uint16_t* q_pe;
  const uint16_t* k_nope;
  const uint16_t* k_pe;
  const uint16_t* v;
  const int32_t* kv_len;  // may be null
  uint16_t* out;
  int* status;
  int B, H, Tq, Tk, past_len;
  float scale_log2;
  int kv_rows;  // rows per (b, h) of k_nope / v and per b of k_pe (>= Tk)
  // Optional 2D padding mask packed by launch_key_bits: [B][ceil(Tk/128)][4] words, bit e
  // of word c of key tile t = visibility of key 128 t + 32 c + e.  Null: no mask.
  const uint32_t* key_bits;
  // Optional fused cache append (all null otherwise; needs past_len a multiple of 128 and
  // no kv_len): key tiles from past_len / 128 on are read from the new rows
  // ([B,H,Tq,128], [B,Tq,64], [B,H,Tq,128]) instead of k_nope / k_pe / v, and the unit that
  // holds each such tile on its diagonal writes it into the caches (the same buffers as
  // k_nope / k_pe / v, kv_rows rows per (b, h) or b) at rows [past_len, past_len + Tq).
  const uint16_t* new_k_nope;
  const uint16_t* new_k_pe;
  const uint16_t* new_v;
};

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Cache append for Tq > 1: new rows [B,H,Tq,128] / [B,Tq,64] / [B,H,Tq,128] are copied to
// rows [past_len, past_len + Tq) of caches with kv_rows rows per (b, h) (per b for k_pe).
struct AppendArgs {
  const uint16_t* new_k_nope;
  const uint16_t* new_k_pe;
  const uint16_t* new_v;
  uint16_t* cache_k_nope;
  uint16_t* cache_k_pe;
  uint16_t* cache_v;
  int B, H, Tq, past_len, kv_rows;
};
cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream);

// YaRN frequencies and mscale ratio of a configuration (host arithmetic, double).
void yarn_frequencies(const mla_rope_config& cfg, double* inv_freq, double* mscale);

// cos / sin table [max_pos][64] (cos in columns 0..31, sin in 32..63, times the ratio).
cudaError_t launch_rope_table(float* cos_sin, int max_pos, const mla_rope_config& cfg,
                              cudaStream_t stream);

// Rotary pre-pass: query t and new rotary key t are rotated at position past_len + t.
// Rotated queries go to q_pe_rot [B,H,Tq,64]; rotated keys (b, t) to
// k_pe_dst + ((b * k_pe_rows) + k_pe_row0 + t) * 64.  When new_k_nope is non-null the
// no-rope key and value rows are also appended to the caches at rows past_len + t.
struct RopeAppendArgs {
  const uint16_t* q_pe_raw;
  uint16_t* q_pe_rot;
  const uint16_t* k_pe_raw;
  uint16_t* k_pe_dst;
  int k_pe_rows, k_pe_row0;
  const uint16_t* new_k_nope;
  const uint16_t* new_v;
  uint16_t* cache_k_nope;
  uint16_t* cache_v;
  const float* cos_sin;
  int B, H, Tq, past_len, kv_rows;
};
cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream);

// Packing of the 2D padding mask for the prefill kernel.
struct KeyBitsArgs {
  const uint8_t* key_mask;  // [B][Tk]
  uint32_t* bits;           // [B][n_kt][4]
  int B, Tk, n_kt;
};
cudaError_t launch_key_bits(const KeyBitsArgs& a, cudaStream_t stream);

// Rows that see no visible key under the 2D padding mask: out = mean of all Tk value rows.
struct FixupArgs {
  const uint8_t* key_mask;  // [B][Tk]
  const int32_t* kv_len;    // may be null
  const uint16_t* v;        // [B][H][kv_rows][128]
  uint16_t* out;            // [B][H][Tq][128]
  int B, H, Tq, Tk, past_len, kv_rows;
  int heads_per_cta;        // set by the launcher
};
cudaError_t launch_masked_rows_fixup(const FixupArgs& a, cudaStream_t stream);

// bf16 tensor viewed as {inner, rows, planes} (planes plane_rows rows apart) as a tensor
// map with 128-byte swizzled {64, box_rows, 1} boxes; rows past `rows` read as zeros.
bool encode_bf16_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t planes, uint64_t plane_rows, uint32_t box_rows);

// bf16 tensor map of any rank (<= 5) with 128-byte swizzled boxes; dims innermost first,
// strides_bytes for dims 1.. (rank - 1 entries); elements past dims read as zeros.
bool encode_bf16_tiled(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box);

// Output projection (o_proj) of the attention output: y [B,T,N] = W [N,H*128] applied to
// each (b, i) row of attn [B,H,T,128] with the heads concatenated in head order.
struct OprojArgs {
  const uint16_t* attn;
  const uint16_t* w;
  uint16_t* y;
  int* status;
  int B, H, T, N;
};
cudaError_t launch_oproj(const OprojArgs& a, cudaStream_t stream);

// Decode over the latent cache (absorbed kv_b_proj).  Shapes: q_nope [B,H,128], q_pe
// [B,H,64], c_kv [B,kv_rows,512], k_pe [B,kv_rows,64], w_kvb [H*256,512]; out [B,H,128].
// Workspace pieces (device): q_lat bf16 [B,H,512], seq_tile0 int32 [B+1] (the split kernel's
// partition), part_ml f32 [(grid+B)*H][2], part_acc f32 [(grid+B)*H][512] (partial c + b of
// CTA c and sequence b, then head).
struct LatentArgs {
  const uint16_t* q_nope;
  const uint16_t* q_pe;
  const uint16_t* c_kv;
  const uint16_t* k_pe;
  const uint16_t* w_kvb;
  const int32_t* kv_len;
  uint16_t* out;
  uint16_t* q_lat;
  int32_t* seq_tile0;
  float* part_ml;
  float* part_acc;
  int* status;
  int B, H, Tk, kv_rows, grid;
  float scale_log2;
};
constexpr int kLatTile = 128;  // keys per tile of the latent kernel
cudaError_t launch_latent(const LatentArgs& a, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace mla
