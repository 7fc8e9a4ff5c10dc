// rope.cu -- YaRN rotary embedding for the attention core's rotary parts, fused with the
// cache append.
//
// The attention excerpt on "Kimi K2 · Similarities" rotates the query and key rotary parts
// before the cache update (rotary_emb gives cos and sin for the positions,
// apply_rotary_pos_emb rotates q_pe and k_pe), positions counted from the cached length;
// the rope_scaling block of the config.json excerpt ("Kimi K2 · Logits") selects YaRN.
// The frequencies follow the published YaRN method (Peng et al. 2023); the rotation is the
// rotate-half form on the 64 rotary columns:
//   y[d] = x[d] cos - x[d+32] sin,   y[d+32] = x[d+32] cos + x[d] sin,   d < 32.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace mla {
namespace {

struct TableArgs {
  float* cos_sin;  // [max_pos][64]: cos of the 32 angles, then sin, times the mscale ratio
  int max_pos;
  double inv_freq[32];
  double mscale;
};

__global__ void __launch_bounds__(256) rope_table_kernel(const TableArgs a) {
  const size_t n = (size_t)a.max_pos * 32;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t pos = i >> 5;
    const int d = (int)(i & 31);
    double s, c;
    sincos((double)pos * a.inv_freq[d], &s, &c);  // double: angles reach 10^5 radians
    a.cos_sin[pos * 64 + d] = (float)(c * a.mscale);
    a.cos_sin[pos * 64 + 32 + d] = (float)(s * a.mscale);
  }
}

// Rotates one 64-column bf16 row; 8 threads per row, thread k handles columns
// [4k, 4k+4) and [32 + 4k, 32 + 4k + 4).
__device__ __forceinline__ void rotate_row(const uint16_t* src, uint16_t* dst,
                                           const float* cs, int k) {
  const uint2 lo = *reinterpret_cast<const uint2*>(src + 4 * k);
  const uint2 hi = *reinterpret_cast<const uint2*>(src + 32 + 4 * k);
  const float4 c = *reinterpret_cast<const float4*>(cs + 4 * k);
  const float4 s = *reinterpret_cast<const float4*>(cs + 32 + 4 * k);
  const float x1[4] = {bf16lo_to_f32(lo.x), bf16hi_to_f32(lo.x), bf16lo_to_f32(lo.y),
                       bf16hi_to_f32(lo.y)};
  const float x2[4] = {bf16lo_to_f32(hi.x), bf16hi_to_f32(hi.x), bf16lo_to_f32(hi.y),
                       bf16hi_to_f32(hi.y)};
  const float cc[4] = {c.x, c.y, c.z, c.w}, ss[4] = {s.x, s.y, s.z, s.w};
  float y1[4], y2[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    y1[e] = fmaf(x1[e], cc[e], -x2[e] * ss[e]);
    y2[e] = fmaf(x2[e], cc[e], x1[e] * ss[e]);
  }
  uint2 o1, o2;
  o1.x = pack_bf16x2(y1[0], y1[1]);
  o1.y = pack_bf16x2(y1[2], y1[3]);
  o2.x = pack_bf16x2(y2[0], y2[1]);
  o2.y = pack_bf16x2(y2[2], y2[3]);
  *reinterpret_cast<uint2*>(dst + 4 * k) = o1;
  *reinterpret_cast<uint2*>(dst + 32 + 4 * k) = o2;
}

// One pass over the new rows: rotated query rotary parts into q_pe_rot, rotated new key
// rotary parts into k_pe_dst, and (when requested) the new no-rope key and value rows into
// the caches.  Eight threads per 64-column rotary row, one thread per 16 bytes of copy.
__global__ void __launch_bounds__(256) rope_append_kernel(const RopeAppendArgs a) {
  const size_t q_rows = (size_t)a.B * a.H * a.Tq;
  const size_t k_rows = (size_t)a.B * a.Tq;
  const size_t chunks = a.new_k_nope ? (size_t)a.B * a.H * a.Tq * 16 : 0;  // per tensor
  const size_t n = (q_rows + k_rows) * 8 + 2 * chunks;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < q_rows * 8) {
      const size_t row = i >> 3;  // (b*H + h)*Tq + t
      const int t = (int)(row % a.Tq);
      rotate_row(a.q_pe_raw + row * 64, a.q_pe_rot + row * 64,
                 a.cos_sin + (size_t)(a.past_len + t) * 64, (int)(i & 7));
    } else if (i < (q_rows + k_rows) * 8) {
      const size_t row = (i - q_rows * 8) >> 3;  // b*Tq + t
      const size_t b = row / a.Tq;
      const int t = (int)(row % a.Tq);
      rotate_row(a.k_pe_raw + row * 64,
                 a.k_pe_dst + (b * a.k_pe_rows + a.k_pe_row0 + t) * 64,
                 a.cos_sin + (size_t)(a.past_len + t) * 64, (int)(i & 7));
    } else {
      size_t k = i - (q_rows + k_rows) * 8;
      const bool is_v = k >= chunks;
      if (is_v) k -= chunks;
      const size_t row = k >> 4, c = k & 15;  // row = (b*H + h)*Tq + t
      const size_t bh = row / a.Tq, t = row % a.Tq;
      const uint4* src =
          reinterpret_cast<const uint4*>((is_v ? a.new_v : a.new_k_nope) + row * 128);
      uint4* dst = reinterpret_cast<uint4*>((is_v ? a.cache_v : a.cache_k_nope) +
                                            (bh * a.kv_rows + a.past_len + t) * 128);
      dst[c] = src[c];
    }
  }
}

unsigned grid_for(size_t n) {
  const int sms = device_sm_count();
  const size_t blocks = std::min<size_t>((n + 255) / 256, (size_t)(sms > 0 ? sms : 152) * 8);
  return (unsigned)std::max<size_t>(blocks, 1);
}

}  // namespace

// YaRN frequencies (extrapolated theta^(-2d/64), interpolated / factor, linear ramp between
// the dimensions whose wavelengths make beta_fast and beta_slow rotations over the original
// context) and the ratio of attention factors 0.1 k ln(factor) + 1, k = mscale over
// k = mscale_all_dim.
void yarn_frequencies(const mla_rope_config& c, double* inv_freq, double* mscale) {
  const double two_pi = 6.283185307179586;
  auto dim_for = [&](double rotations) {
    return 64.0 * std::log(c.original_max_position / (two_pi * rotations)) /
           (2.0 * std::log(c.rope_theta));
  };
  const double lo = std::max(std::floor(dim_for(c.beta_fast)), 0.0);
  double hi = std::min(std::ceil(dim_for(c.beta_slow)), 31.0);
  if (hi == lo) hi += 0.001;
  for (int d = 0; d < 32; ++d) {
    const double plain = std::pow(c.rope_theta, -2.0 * d / 64.0);
    const double w = std::min(std::max((d - lo) / (hi - lo), 0.0), 1.0);  // 1: interpolate
    inv_freq[d] = plain / c.factor * w + plain * (1.0 - w);
  }
  auto attn = [&](double k) { return c.factor > 1.0 ? 0.1 * k * std::log(c.factor) + 1.0 : 1.0; };
  *mscale = attn(c.mscale) / attn(c.mscale_all_dim);
}

cudaError_t launch_rope_table(float* cos_sin, int max_pos, const mla_rope_config& cfg,
                              cudaStream_t stream) {
  TableArgs a;
  a.cos_sin = cos_sin;
  a.max_pos = max_pos;
  yarn_frequencies(cfg, a.inv_freq, &a.mscale);
  rope_table_kernel<<<grid_for((size_t)max_pos * 32), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream) {
  const size_t n = ((size_t)a.B * a.H * a.Tq + (size_t)a.B * a.Tq) * 8 +
                   (a.new_k_nope ? (size_t)a.B * a.H * a.Tq * 32 : 0);
  rope_append_kernel<<<grid_for(n), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
