// host.cu -- the C ABI of libmla_attn.so: argument checks, workspace layout, the decode
// split scheduler, kernel launches and the device status word.
//
// The checks mirror the guards of the attention excerpt on "Kimi K2 · Similarities":
// the scores must have shape [B, H, Tq, Tk] with Tk the cached length plus the new
// rows, and a mask must be present (here it is implied by past_len and kv_len, so it is
// always present).  Failing checks return an error code; nothing is launched.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "kernels.h"
#include "mla_attn.h"

namespace mla {
namespace {

constexpr size_t kStatusBytes = 256;  // status word + padding at the start of the workspace
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxElems = int64_t(1) << 40;

// 0 = unknown, 1 = sm_103, 2 = other.  Per device, filled on first use.
std::atomic<int> g_dev_kind[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status check_device(int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  int kind = g_dev_kind[dev].load(std::memory_order_acquire);
  if (kind == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
    kind = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_sms[dev].store(sms, std::memory_order_relaxed);
    g_dev_kind[dev].store(kind, std::memory_order_release);
  }
  if (kind != 1) return MLA_ERR_DEVICE;
  if (sms_out) *sms_out = g_dev_sms[dev].load(std::memory_order_relaxed);
  return MLA_OK;
}

mla_status check_shape(int B, int H, int Tq, int Tk, int past_len) {
  if (B < 1 || H < 1 || Tq < 1 || past_len < 0) return MLA_ERR_SHAPE;
  if ((int64_t)past_len + Tq != (int64_t)Tk) return MLA_ERR_SHAPE;
  if ((int64_t)B * H * Tk * 128 > kMaxElems) return MLA_ERR_SHAPE;
  if (B > 65535) return MLA_ERR_SHAPE;  // grid z of the decode launch
  return MLA_OK;
}

// Partials: (max, sum) pairs, then the 128-float accumulators starting on a 256-byte
// boundary (the kernels access them with 16-byte vector loads and stores).
size_t decode_ml_bytes(int B, int H, int splits) {
  const size_t raw = (size_t)B * H * splits * 2 * sizeof(float);
  return (raw + 255) & ~(size_t)255;
}

size_t decode_workspace(int B, int H, int splits) {
  if (splits <= 1) return kStatusBytes;
  return kStatusBytes + decode_ml_bytes(B, H, splits) +
         (size_t)B * H * splits * 128 * sizeof(float);
}

// Packed 2D padding mask for the prefill kernel: [B][ceil(Tk/128)][4] words.
size_t key_bits_bytes(int B, int Tk) {
  return ((size_t)B * ((Tk + 127) / 128) * 16 + 255) & ~(size_t)255;
}

// Latent-cache decode: one CTA per SM (its shared memory allows no more), each taking an
// equal share of all sequences' 128-key tiles (the kernel partitions them from kv_len on the
// device), capped at the tiles there can be.  Each CTA writes one 64 heads x 512 fp32
// partial per sequence it touches: at most grid + B partials.
struct LatentPlan {
  int grid;
};
LatentPlan plan_latent(int B, int Tk, int sms) {
  const int64_t tiles = (int64_t)B * ((Tk + kLatTile - 1) / kLatTile);
  LatentPlan pl;
  pl.grid = (int)std::min<int64_t>(tiles, sms);
  return pl;
}
size_t r256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t latent_q_bytes(int B, int H) { return r256((size_t)B * H * 512 * 2); }
size_t latent_tile0_bytes(int B) { return r256((size_t)(B + 1) * 4); }
size_t latent_ml_bytes(int B, int H, int grid) { return r256((size_t)(grid + B) * H * 8); }
size_t latent_acc_bytes(int B, int H, int grid) {
  return r256((size_t)(grid + B) * H * 512 * 4);
}
size_t latent_workspace(int B, int H, int grid) {
  return kStatusBytes + latent_q_bytes(B, H) + latent_tile0_bytes(B) +
         latent_ml_bytes(B, H, grid) + latent_acc_bytes(B, H, grid);
}

// Rotary workspace: rotated queries [B,H,Tq,64] then rotated new rotary keys [B,Tq,64],
// each on a 256-byte boundary, after the attention call's own workspace.
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
size_t q_rot_bytes(int B, int H, int Tq) { return round256((size_t)B * H * Tq * 64 * 2); }
size_t rope_bytes(int B, int H, int Tq) {
  return q_rot_bytes(B, H, Tq) + round256((size_t)B * Tq * 64 * 2);
}

bool rope_config_ok(const mla_rope_config& c) {
  const double v[7] = {c.rope_theta, c.factor, c.original_max_position, c.beta_fast,
                       c.beta_slow, c.mscale, c.mscale_all_dim};
  for (double x : v)
    if (!std::isfinite(x)) return false;
  if (!(c.rope_theta > 1.0 && c.factor >= 1.0 && c.original_max_position > 0.0 &&
        c.beta_slow > 0.0 && c.beta_fast >= c.beta_slow))
    return false;
  // the ratio's denominator 0.1 mscale_all_dim ln(factor) + 1 must not vanish
  return c.factor == 1.0 || 0.1 * c.mscale_all_dim * std::log(c.factor) + 1.0 != 0.0;
}

}  // namespace

// Keys per split for the decode path (the kernel runs 2 CTAs per SM).  When there are at
// least as many (sequence, head group) units as SMs, take the largest power-of-two multiple
// of 64 keys (at most 1024) that still leaves two full waves of one CTA per SM.  Fewer
// units split the keys so that the whole grid is about one wave of 2 CTAs per SM.
DecodePlan plan_decode(int B, int H, int Tk, int sms, int forced_chunk) {
  const int64_t groups = (int64_t)B * ((H + kDecHeadsPerCta - 1) / kDecHeadsPerCta);
  DecodePlan pl;
  const bool few = groups < (int64_t)sms;
  if (forced_chunk > 0) {
    pl.chunk = forced_chunk;
  } else if (!few) {
    int c = kDecMinChunk;
    while (c < 1024) {
      const int64_t next = groups * ((Tk + 2 * c - 1) / (2 * c));
      if (next < 2 * (int64_t)sms) break;
      c *= 2;
    }
    pl.chunk = c;
  } else {
    const int64_t want = std::max<int64_t>(1, (2 * (int64_t)sms) / groups);
    int64_t c = (Tk + want - 1) / want;
    c = std::max<int64_t>(32, (c + 31) / 32 * 32);
    pl.chunk = (int)std::min<int64_t>(c, kDecMaxChunk);
  }
  pl.splits = (Tk + pl.chunk - 1) / pl.chunk;
  return pl;
}

int device_sm_count() {
  int sms = 0;
  return check_device(&sms) == MLA_OK ? sms : 0;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_NULL: return "MLA_ERR_NULL: a required pointer is NULL";
    case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE: invalid sizes (need B,H,Tq>=1, past_len>=0, Tk==past_len+Tq)";
    case MLA_ERR_ALIGN: return "MLA_ERR_ALIGN: a pointer is not 16-byte aligned";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_DEVICE: return "MLA_ERR_DEVICE: current device is not sm_103";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA runtime or launch failure";
    case MLA_ERR_KVLEN: return "MLA_ERR_KVLEN: kv_len[b] outside [1, Tk]";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded wait in a kernel gave up";
    case MLA_ERR_ARG: return "MLA_ERR_ARG: option out of range";
  }
  return "unknown mla_status";
}

mla_status mla_attn_decode_plan(int B, int H, int Tk, int* chunk, int* splits) {
  if (B < 1 || H < 1 || Tk < 1) return MLA_ERR_SHAPE;
  int sms = 0;
  if (check_device(&sms) != MLA_OK || sms <= 0) sms = 152;  // GB300 SM count when no device
  const DecodePlan pl = plan_decode(B, H, Tk, sms, 0);
  if (chunk) *chunk = pl.chunk;
  if (splits) *splits = pl.splits;
  return MLA_OK;
}

size_t mla_attn_workspace_bytes(int B, int H, int Tq, int Tk) {
  if (B < 1 || H < 1 || Tq < 1 || Tk < Tq) return 0;
  if (Tq != 1) return kStatusBytes;
  int c = 0, s = 0;
  mla_attn_decode_plan(B, H, Tk, &c, &s);
  return decode_workspace(B, H, s);
}

}  // extern "C"

namespace mla {
namespace {

mla_status launch_fixup(const uint8_t* key_mask, const int32_t* kv_len, const uint16_t* v,
                        uint16_t* out, int B, int H, int Tq, int Tk, int past_len, int kv_rows,
                        cudaStream_t stream) {
  FixupArgs f;
  f.key_mask = key_mask; f.kv_len = kv_len; f.v = v; f.out = out;
  f.B = B; f.H = H; f.Tq = Tq; f.Tk = Tk; f.past_len = past_len; f.kv_rows = kv_rows;
  return launch_masked_rows_fixup(f, stream) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

bool prefill_can_fuse_append(int past_len, const int32_t* kv_len, const uint8_t* key_mask) {
  return past_len % 128 == 0 && kv_len == nullptr && key_mask == nullptr;
}

struct AppendPtrs {
  const uint16_t* new_k_nope;
  const uint16_t* new_k_pe;
  const uint16_t* new_v;
  uint16_t* cache_k_nope;
  uint16_t* cache_k_pe;
  uint16_t* cache_v;
  // Decode only: q_pe and new_k_pe arrive unrotated and the decode kernel rotates them with
  // this cos/sin table row (position Tk - 1); null: already rotated.
  const float* rope_cs;
};

// Argument checks and launch shared by the attention entry points.  kv_rows is the row
// stride of the key/value buffers (>= Tk); app (decode only) fuses the cache append;
// check_only runs every check and returns without launching; key_mask (may be null) is the
// 2D padding mask [B][Tk] on keys.
mla_status attention_impl(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                          const uint16_t* k_pe_shared, const uint16_t* v, const int32_t* kv_len,
                          int B, int H, int Tq, int Tk, int past_len, float softmax_scale,
                          uint16_t* out, void* workspace, size_t workspace_bytes,
                          void* cuda_stream, const mla_attn_options* options, int kv_rows,
                          const AppendPtrs* app, bool check_only = false,
                          const uint8_t* key_mask = nullptr) {
  if (!q_nope || !q_pe || !k_nope || !k_pe_shared || !v || !out) return MLA_ERR_NULL;
  if (!workspace) return MLA_ERR_WORKSPACE;
  mla_status st = check_shape(B, H, Tq, Tk, past_len);
  if (st != MLA_OK) return st;
  if (kv_rows < Tk || (int64_t)B * H * kv_rows * 128 > kMaxElems) return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(k_nope) || !aligned16(k_pe_shared) ||
      !aligned16(v) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0)
    return MLA_ERR_ALIGN;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.0f)) return MLA_ERR_ARG;
  int path = options ? options->path : MLA_PATH_AUTO;
  if (path < MLA_PATH_AUTO || path > MLA_PATH_DECODE) return MLA_ERR_ARG;
  if (path == MLA_PATH_AUTO) path = (Tq == 1) ? MLA_PATH_DECODE : MLA_PATH_PREFILL;
  if (path == MLA_PATH_DECODE && Tq != 1) return MLA_ERR_ARG;
  // The prefill kernel fuses the append only for a prefix of whole 128-key tiles and
  // sequences without kv_len (every new row is then read by the unit that writes it).
  if (app && path != MLA_PATH_DECODE && !prefill_can_fuse_append(past_len, kv_len, key_mask))
    return MLA_ERR_ARG;
  int sms = 0;
  st = check_device(&sms);
  if (st != MLA_OK) return st;

  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  int* status = static_cast<int*>(workspace);
  const float scale_log2 = softmax_scale * 1.4426950408889634f;

  if (path == MLA_PATH_DECODE) {
    const int forced = options ? options->decode_chunk : 0;
    if (forced != 0 &&
        (forced < kDecMinChunk || forced > kDecMaxChunk || forced % kDecMinChunk != 0))
      return MLA_ERR_ARG;
    const DecodePlan pl = plan_decode(B, H, Tk, sms, forced);
    const int chunk = pl.chunk, splits = pl.splits;
    if (splits > 65535) return MLA_ERR_ARG;
    if (workspace_bytes < decode_workspace(B, H, splits)) return MLA_ERR_WORKSPACE;
    if (check_only) return MLA_OK;
    DecodeArgs a{};
    a.q_nope = q_nope; a.q_pe = q_pe; a.k_nope = k_nope; a.k_pe = k_pe_shared; a.v = v;
    a.kv_len = kv_len; a.out = out; a.status = status;
    uint8_t* part = static_cast<uint8_t*>(workspace) + kStatusBytes;
    a.part_ml = reinterpret_cast<float*>(part);
    a.part_acc = reinterpret_cast<float*>(part + decode_ml_bytes(B, H, splits));
    a.B = B; a.H = H; a.Tk = Tk; a.chunk = chunk; a.splits = splits;
    a.scale_log2 = scale_log2;
    a.kv_rows = kv_rows;
    if (app) {
      a.new_k_nope = app->new_k_nope; a.new_k_pe = app->new_k_pe; a.new_v = app->new_v;
      a.cache_k_nope = app->cache_k_nope; a.cache_k_pe = app->cache_k_pe;
      a.cache_v = app->cache_v;
      a.rope_cs = app->rope_cs;
    }
    a.key_mask = key_mask;
    if (launch_decode(a, stream) != cudaSuccess) return MLA_ERR_CUDA;
    return key_mask ? launch_fixup(key_mask, kv_len, v, out, B, H, Tq, Tk, past_len, kv_rows,
                                   stream)
                    : MLA_OK;
  }

  const size_t need = kStatusBytes + (key_mask ? key_bits_bytes(B, Tk) : 0);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (check_only) return MLA_OK;
  uint32_t* key_bits = nullptr;
  if (key_mask) {
    KeyBitsArgs kb;
    kb.key_mask = key_mask;
    kb.bits = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + kStatusBytes);
    kb.B = B; kb.Tk = Tk; kb.n_kt = (Tk + 127) / 128;
    if (launch_key_bits(kb, stream) != cudaSuccess) return MLA_ERR_CUDA;
    key_bits = kb.bits;
  }
  PrefillArgs a{};
  a.q_nope = q_nope; a.q_pe = q_pe; a.k_nope = k_nope; a.k_pe = k_pe_shared; a.v = v;
  a.kv_len = kv_len; a.out = out; a.status = status;
  a.B = B; a.H = H; a.Tq = Tq; a.Tk = Tk; a.past_len = past_len;
  a.scale_log2 = scale_log2;
  a.kv_rows = kv_rows;
  a.key_bits = key_bits;
  if (app) {
    a.new_k_nope = app->new_k_nope;
    a.new_k_pe = app->new_k_pe;
    a.new_v = app->new_v;
  }
  if (launch_prefill(a, stream) != cudaSuccess) return MLA_ERR_CUDA;
  return key_mask ? launch_fixup(key_mask, kv_len, v, out, B, H, Tq, Tk, past_len, kv_rows,
                                 stream)
                  : MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" {

mla_status mla_attn_fwd_ex(const uint16_t* q_nope, const uint16_t* q_pe,
                           const uint16_t* k_nope, const uint16_t* k_pe_shared,
                           const uint16_t* v, const int32_t* kv_len, int B, int H, int Tq,
                           int Tk, int past_len, float softmax_scale, uint16_t* out,
                           void* workspace, size_t workspace_bytes, void* cuda_stream,
                           const mla_attn_options* options) {
  return attention_impl(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, B, H, Tq, Tk, past_len,
                        softmax_scale, out, workspace, workspace_bytes, cuda_stream, options, Tk,
                        nullptr);
}

mla_status mla_attn_append_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                               const uint16_t* k_nope_new, const uint16_t* k_pe_new,
                               const uint16_t* v_new, uint16_t* k_nope_cache,
                               uint16_t* k_pe_cache, uint16_t* v_cache, const int32_t* kv_len,
                               int B, int H, int Tq, int T_cap, int past_len,
                               float softmax_scale, uint16_t* out, void* workspace,
                               size_t workspace_bytes, void* cuda_stream) {
  if (!k_nope_new || !k_pe_new || !v_new || !k_nope_cache || !k_pe_cache || !v_cache)
    return MLA_ERR_NULL;
  if (B < 1 || H < 1 || Tq < 1 || past_len < 0 || (int64_t)past_len + Tq > (int64_t)T_cap)
    return MLA_ERR_SHAPE;
  if (!aligned16(k_nope_new) || !aligned16(k_pe_new) || !aligned16(v_new))
    return MLA_ERR_ALIGN;
  const int Tk = past_len + Tq;
  if (Tq == 1) {
    // Decode: the append is fused into the attention kernel.
    AppendPtrs app = {k_nope_new, k_pe_new, v_new, k_nope_cache, k_pe_cache, v_cache, nullptr};
    return attention_impl(q_nope, q_pe, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H, Tq, Tk,
                          past_len, softmax_scale, out, workspace, workspace_bytes, cuda_stream,
                          nullptr, T_cap, &app);
  }
  if (prefill_can_fuse_append(past_len, kv_len, nullptr)) {
    // Prefill on a prefix of whole key tiles: the attention kernel reads the new rows where
    // they are and writes them into the caches itself.
    AppendPtrs app = {k_nope_new, k_pe_new, v_new, k_nope_cache, k_pe_cache, v_cache, nullptr};
    return attention_impl(q_nope, q_pe, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H, Tq, Tk,
                          past_len, softmax_scale, out, workspace, workspace_bytes, cuda_stream,
                          nullptr, T_cap, &app);
  }
  // Other prefills: the checks run first (nothing is enqueued on failure), then the copy
  // kernel appends the new rows, then attention reads the cache.
  mla_status st = attention_impl(q_nope, q_pe, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H,
                                 Tq, Tk, past_len, softmax_scale, out, workspace,
                                 workspace_bytes, cuda_stream, nullptr, T_cap, nullptr, true);
  if (st != MLA_OK) return st;
  AppendArgs ap;
  ap.new_k_nope = k_nope_new; ap.new_k_pe = k_pe_new; ap.new_v = v_new;
  ap.cache_k_nope = k_nope_cache; ap.cache_k_pe = k_pe_cache; ap.cache_v = v_cache;
  ap.B = B; ap.H = H; ap.Tq = Tq; ap.past_len = past_len; ap.kv_rows = T_cap;
  if (launch_kv_append(ap, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return attention_impl(q_nope, q_pe, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H, Tq, Tk,
                        past_len, softmax_scale, out, workspace, workspace_bytes, cuda_stream,
                        nullptr, T_cap, nullptr);
}

mla_status mla_rope_frequencies(const mla_rope_config* cfg, double* inv_freq,
                                double* mscale_ratio) {
  if (!cfg) return MLA_ERR_NULL;
  if (!rope_config_ok(*cfg)) return MLA_ERR_ARG;
  double f[32], m = 1.0;
  yarn_frequencies(*cfg, f, &m);
  if (inv_freq) std::memcpy(inv_freq, f, sizeof(f));
  if (mscale_ratio) *mscale_ratio = m;
  return MLA_OK;
}

mla_status mla_rope_table(const mla_rope_config* cfg, int max_pos, float* table,
                          void* cuda_stream) {
  if (!cfg || !table) return MLA_ERR_NULL;
  if (max_pos < 1) return MLA_ERR_SHAPE;
  if (!aligned16(table)) return MLA_ERR_ALIGN;
  if (!rope_config_ok(*cfg)) return MLA_ERR_ARG;
  const mla_status st = check_device(nullptr);
  if (st != MLA_OK) return st;
  return launch_rope_table(table, max_pos, *cfg, static_cast<cudaStream_t>(cuda_stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

size_t mla_attn_rope_workspace_bytes(int B, int H, int Tq, int Tk) {
  const size_t base = mla_attn_workspace_bytes(B, H, Tq, Tk);
  if (base == 0) return 0;
  return round256(base) + rope_bytes(B, H, Tq);
}

mla_status mla_attn_rope_append_fwd(const uint16_t* q_nope, const uint16_t* q_pe_raw,
                                    const uint16_t* k_nope_new, const uint16_t* k_pe_new_raw,
                                    const uint16_t* v_new, uint16_t* k_nope_cache,
                                    uint16_t* k_pe_cache, uint16_t* v_cache,
                                    const int32_t* kv_len, int B, int H, int Tq, int T_cap,
                                    int past_len, float softmax_scale, const float* rope_table,
                                    int table_rows, uint16_t* out, void* workspace,
                                    size_t workspace_bytes, void* cuda_stream) {
  if (!q_pe_raw || !k_nope_new || !k_pe_new_raw || !v_new || !k_nope_cache || !k_pe_cache ||
      !v_cache || !rope_table)
    return MLA_ERR_NULL;
  if (B < 1 || H < 1 || Tq < 1 || past_len < 0 || (int64_t)past_len + Tq > (int64_t)T_cap)
    return MLA_ERR_SHAPE;
  const int Tk = past_len + Tq;
  if (table_rows < Tk) return MLA_ERR_SHAPE;
  if (!aligned16(q_pe_raw) || !aligned16(k_nope_new) || !aligned16(k_pe_new_raw) ||
      !aligned16(v_new) || !aligned16(rope_table))
    return MLA_ERR_ALIGN;
  if (!workspace) return MLA_ERR_WORKSPACE;
  const size_t base = mla_attn_workspace_bytes(B, H, Tq, Tk);
  if (base == 0) return MLA_ERR_SHAPE;
  if (workspace_bytes < round256(base) + rope_bytes(B, H, Tq)) return MLA_ERR_WORKSPACE;
  uint8_t* rot = static_cast<uint8_t*>(workspace) + round256(base);
  uint16_t* q_pe_rot = reinterpret_cast<uint16_t*>(rot);
  uint16_t* k_pe_rot = reinterpret_cast<uint16_t*>(rot + q_rot_bytes(B, H, Tq));

  if (Tq == 1) {
    // Decode: one kernel rotates the query's and the new key's rotary parts (row past_len of
    // the table), appends the new rows and attends.
    AppendPtrs dec = {k_nope_new, k_pe_new_raw, v_new, k_nope_cache, k_pe_cache, v_cache,
                      rope_table + (size_t)past_len * 64};
    return attention_impl(q_nope, q_pe_raw, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H, Tq,
                          Tk, past_len, softmax_scale, out, workspace, workspace_bytes,
                          cuda_stream, nullptr, T_cap, &dec);
  }
  // Prefill: every check of the attention call runs before anything is enqueued.  On a
  // prefix of whole key tiles without kv_len the append happens inside the attention
  // kernel (from the rotated keys in the workspace); other prefills copy first.
  AppendPtrs app = {k_nope_new, k_pe_rot, v_new, k_nope_cache, k_pe_cache, v_cache, nullptr};
  const bool fuse = prefill_can_fuse_append(past_len, kv_len, nullptr);
  const AppendPtrs* fused = fuse ? &app : nullptr;
  mla_status st = attention_impl(q_nope, q_pe_rot, k_nope_cache, k_pe_cache, v_cache, kv_len, B,
                                 H, Tq, Tk, past_len, softmax_scale, out, workspace,
                                 workspace_bytes, cuda_stream, nullptr, T_cap, fused, true);
  if (st != MLA_OK) return st;

  RopeAppendArgs r{};
  r.q_pe_raw = q_pe_raw; r.q_pe_rot = q_pe_rot; r.k_pe_raw = k_pe_new_raw;
  r.cos_sin = rope_table;
  r.B = B; r.H = H; r.Tq = Tq; r.past_len = past_len; r.kv_rows = T_cap;
  if (fuse) {
    // Rotate into the workspace; the attention kernel appends all three new rows.
    r.k_pe_dst = k_pe_rot; r.k_pe_rows = Tq; r.k_pe_row0 = 0;
  } else {
    r.k_pe_dst = k_pe_cache; r.k_pe_rows = T_cap; r.k_pe_row0 = past_len;
    r.new_k_nope = k_nope_new; r.new_v = v_new;
    r.cache_k_nope = k_nope_cache; r.cache_v = v_cache;
  }
  if (launch_rope_append(r, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return attention_impl(q_nope, q_pe_rot, k_nope_cache, k_pe_cache, v_cache, kv_len, B, H, Tq,
                        Tk, past_len, softmax_scale, out, workspace, workspace_bytes,
                        cuda_stream, nullptr, T_cap, fused);
}

size_t mla_attn_masked_workspace_bytes(int B, int H, int Tq, int Tk) {
  const size_t base = mla_attn_workspace_bytes(B, H, Tq, Tk);
  if (base == 0) return 0;
  return Tq == 1 ? base : kStatusBytes + key_bits_bytes(B, Tk);
}

mla_status mla_attn_masked_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                               const uint16_t* k_nope, const uint16_t* k_pe_shared,
                               const uint16_t* v, const int32_t* kv_len,
                               const uint8_t* key_mask, int B, int H, int Tq, int Tk,
                               int past_len, float softmax_scale, uint16_t* out,
                               void* workspace, size_t workspace_bytes, void* cuda_stream) {
  if (!key_mask) return MLA_ERR_NULL;
  return attention_impl(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, B, H, Tq, Tk, past_len,
                        softmax_scale, out, workspace, workspace_bytes, cuda_stream, nullptr, Tk,
                        nullptr, false, key_mask);
}

size_t mla_latent_workspace_bytes(int B, int H, int Tk) {
  if (B < 1 || H < 1 || H > 64 || Tk < 1) return 0;
  int sms = 0;
  if (check_device(&sms) != MLA_OK || sms <= 0) sms = 152;
  return latent_workspace(B, H, plan_latent(B, Tk, sms).grid);
}

mla_status mla_latent_decode_fwd(const uint16_t* q_nope, const uint16_t* q_pe,
                                 const uint16_t* c_kv, const uint16_t* k_pe,
                                 const uint16_t* w_kvb, const int32_t* kv_len, int B, int H,
                                 int Tk, float softmax_scale, uint16_t* out, void* workspace,
                                 size_t workspace_bytes, void* cuda_stream) {
  if (!q_nope || !q_pe || !c_kv || !k_pe || !w_kvb || !out) return MLA_ERR_NULL;
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (B < 1 || H < 1 || H > 64 || Tk < 1 || B > 65535) return MLA_ERR_SHAPE;
  if ((int64_t)B * Tk * 512 > kMaxElems) return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(c_kv) || !aligned16(k_pe) ||
      !aligned16(w_kvb) || !aligned16(out) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0)
    return MLA_ERR_ALIGN;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.0f)) return MLA_ERR_ARG;
  int sms = 0;
  mla_status st = check_device(&sms);
  if (st != MLA_OK) return st;
  const LatentPlan pl = plan_latent(B, Tk, sms);
  if (workspace_bytes < latent_workspace(B, H, pl.grid)) return MLA_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  LatentArgs a{};
  a.q_nope = q_nope; a.q_pe = q_pe; a.c_kv = c_kv; a.k_pe = k_pe; a.w_kvb = w_kvb;
  a.kv_len = kv_len; a.out = out;
  a.status = reinterpret_cast<int*>(w);
  uint8_t* cur = w + kStatusBytes;
  a.q_lat = reinterpret_cast<uint16_t*>(cur);
  cur += latent_q_bytes(B, H);
  a.seq_tile0 = reinterpret_cast<int32_t*>(cur);
  cur += latent_tile0_bytes(B);
  a.part_ml = reinterpret_cast<float*>(cur);
  cur += latent_ml_bytes(B, H, pl.grid);
  a.part_acc = reinterpret_cast<float*>(cur);
  a.B = B; a.H = H; a.Tk = Tk; a.kv_rows = Tk; a.grid = pl.grid;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_latent(a, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? MLA_OK
                                                                                  : MLA_ERR_CUDA;
}

size_t mla_oproj_workspace_bytes(void) { return kStatusBytes; }

mla_status mla_oproj_fwd(const uint16_t* attn, const uint16_t* w_o, int B, int H, int T, int N,
                         uint16_t* y, void* workspace, size_t workspace_bytes,
                         void* cuda_stream) {
  if (!attn || !w_o || !y) return MLA_ERR_NULL;
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (B < 1 || H < 1 || T < 1 || N < 1 || N % 32 != 0) return MLA_ERR_SHAPE;
  if ((int64_t)B * H * T * 128 > kMaxElems || (int64_t)N * H * 128 > kMaxElems ||
      (int64_t)B * T * N > kMaxElems || (int64_t)H * 128 * 2 > (int64_t(1) << 30))
    return MLA_ERR_SHAPE;
  if (!aligned16(attn) || !aligned16(w_o) || !aligned16(y) || !aligned16(workspace))
    return MLA_ERR_ALIGN;
  if (workspace_bytes < kStatusBytes) return MLA_ERR_WORKSPACE;
  int sms = 0;
  mla_status st = check_device(&sms);
  if (st != MLA_OK) return st;
  OprojArgs a{};
  a.attn = attn; a.w = w_o; a.y = y;
  a.status = static_cast<int*>(workspace);
  a.B = B; a.H = H; a.T = T; a.N = N;
  return launch_oproj(a, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? MLA_OK
                                                                                : MLA_ERR_CUDA;
}

mla_status mla_attn_fwd(const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* k_nope,
                        const uint16_t* k_pe_shared, const uint16_t* v, const int32_t* kv_len,
                        int B, int H, int Tq, int Tk, int past_len, float softmax_scale,
                        uint16_t* out, void* workspace, size_t workspace_bytes,
                        void* cuda_stream) {
  return mla_attn_fwd_ex(q_nope, q_pe, k_nope, k_pe_shared, v, kv_len, B, H, Tq, Tk, past_len,
                         softmax_scale, out, workspace, workspace_bytes, cuda_stream, nullptr);
}

mla_status mla_attn_get_status(void* workspace, void* cuda_stream) {
  if (!workspace) return MLA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (host < 0 || host > MLA_ERR_ARG) return MLA_ERR_CUDA;
  return static_cast<mla_status>(host);
}

}  // extern "C"
