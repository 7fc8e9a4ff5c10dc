// mask.cu -- the 2D padding mask on keys: packing for the prefill kernel, and the rows that
// no key is visible to.
//
// The model's 2D attention_mask ("Kimi K2 · Causal mask", §Construct causal mask) is
// expanded to 4D and merged with the causal mask, so a hidden key receives the same
// additive minimum as a causally hidden one.  A query row that sees no visible key at all
// then has every score equal to that minimum, and its softmax weights are uniform over
// all Tk keys: its output is the plain mean of the Tk value rows.  The attention kernels
// skip hidden keys; masked_rows_fixup_kernel writes those uniform rows afterwards.
#include <algorithm>
#include <climits>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace mla {
namespace {

// Bit e of word c of key tile kt of sequence b is key kt*128 + 32c + e's visibility.
// Keys at or past Tk read as visible (the causal limit already hides them).
__global__ void __launch_bounds__(256) key_bits_kernel(const KeyBitsArgs a) {
  const size_t n = (size_t)a.B * a.n_kt * 4;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t b = i / ((size_t)a.n_kt * 4);
    const int k0 = (int)(i % ((size_t)a.n_kt * 4)) * 32;  // first key of this word
    const uint8_t* row = a.key_mask + b * a.Tk;
    uint32_t w = 0;
#pragma unroll 8
    for (int e = 0; e < 32; ++e) {
      const int j = k0 + e;
      const bool vis = j >= a.Tk || row[j] != 0;
      w |= (uint32_t)vis << e;
    }
    a.bits[i] = w;
  }
}

// One CTA of 256 threads per (16-column group cg, group of heads, sequence b).  Query row
// i of sequence b sees no visible key when i + past_len is below the first key that is
// visible (key_mask set and j < kv_len[b]).  Those rows get the mean of all Tk value rows.
// Columns are split eight ways so that the whole read of V (every row of every head that
// needs the mean) is spread over many SMs: each thread sums 8 columns of every 128th row.
__global__ void __launch_bounds__(256) masked_rows_fixup_kernel(const FixupArgs a) {
  __shared__ int s_first;
  __shared__ float s_part[8][16];
  __shared__ float s_mean[16];
  const int cg = blockIdx.x;  // columns [16 cg, 16 cg + 16)
  const int h0 = blockIdx.y * a.heads_per_cta;
  const int b = blockIdx.z;
  if (threadIdx.x == 0) s_first = INT_MAX;
  __syncthreads();
  int kvl = a.kv_len ? a.kv_len[b] : a.Tk;
  kvl = min(max(kvl, 1), a.Tk);
  const uint8_t* mrow = a.key_mask + (size_t)b * a.Tk;
  for (int j = threadIdx.x; j < kvl; j += blockDim.x) {
    if (mrow[j] != 0) {
      atomicMin(&s_first, j);  // this thread's first hit is its smallest index
      break;
    }
  }
  __syncthreads();
  const int first = s_first;
  const int n_rows =
      first == INT_MAX ? a.Tq : min(a.Tq, max(0, first - a.past_len));
  if (n_rows == 0) return;  // uniform across the CTA

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int ch = threadIdx.x & 1;   // columns 16 cg + 8 ch .. + 8
  const int r0 = threadIdx.x >> 1;  // rows r0, r0 + 128, ...
  const int col = cg * 16 + ch * 8;
  const float inv_tk = 1.0f / (float)a.Tk;
  const int h1 = min(h0 + a.heads_per_cta, a.H);
  for (int h = h0; h < h1; ++h) {
    const size_t bh = (size_t)b * a.H + h;
    const uint16_t* vb = a.v + bh * a.kv_rows * 128 + col;
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add = [&](const uint4 w) {
      s[0] += bf16lo_to_f32(w.x);
      s[1] += bf16hi_to_f32(w.x);
      s[2] += bf16lo_to_f32(w.y);
      s[3] += bf16hi_to_f32(w.y);
      s[4] += bf16lo_to_f32(w.z);
      s[5] += bf16hi_to_f32(w.z);
      s[6] += bf16lo_to_f32(w.w);
      s[7] += bf16hi_to_f32(w.w);
    };
    // Eight independent 16-byte loads in flight per thread (the read of V is latency-bound:
    // bytes in flight per SM set its rate), then the sums.
    int j = r0;
    for (; j + 7 * 128 < a.Tk; j += 8 * 128) {
      uint4 w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        w[k] = __ldcs(reinterpret_cast<const uint4*>(vb + (size_t)(j + k * 128) * 128));
#pragma unroll
      for (int k = 0; k < 8; ++k) add(w[k]);
    }
    for (; j < a.Tk; j += 128) add(__ldcs(reinterpret_cast<const uint4*>(vb + (size_t)j * 128)));
    // Lanes of one column half differ in bits 1..4.
#pragma unroll
    for (int k = 0; k < 8; ++k) {
#pragma unroll
      for (int x = 2; x < 32; x <<= 1) s[k] += __shfl_xor_sync(0xffffffffu, s[k], x);
    }
    if (lane < 2) {
#pragma unroll
      for (int k = 0; k < 8; ++k) s_part[warp][lane * 8 + k] = s[k];
    }
    __syncthreads();
    if (threadIdx.x < 16) {
      float t = 0.f;
#pragma unroll
      for (int g = 0; g < 8; ++g) t += s_part[g][threadIdx.x];
      s_mean[threadIdx.x] = t * inv_tk;
    }
    __syncthreads();
    // Rows i < n_rows, two threads per row (8 columns each).
    uint4 word;
    word.x = pack_bf16x2(s_mean[ch * 8 + 0], s_mean[ch * 8 + 1]);
    word.y = pack_bf16x2(s_mean[ch * 8 + 2], s_mean[ch * 8 + 3]);
    word.z = pack_bf16x2(s_mean[ch * 8 + 4], s_mean[ch * 8 + 5]);
    word.w = pack_bf16x2(s_mean[ch * 8 + 6], s_mean[ch * 8 + 7]);
    for (int i = r0; i < n_rows; i += 128)
      *reinterpret_cast<uint4*>(a.out + (bh * a.Tq + i) * 128 + col) = word;
    __syncthreads();  // s_part and s_mean are reused by the next head
  }
}

unsigned grid_for(size_t n) {
  const int sms = device_sm_count();
  const size_t blocks = (n + 255) / 256;
  const size_t cap = (size_t)(sms > 0 ? sms : 152) * 8;
  return (unsigned)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

}  // namespace

cudaError_t launch_key_bits(const KeyBitsArgs& a, cudaStream_t stream) {
  key_bits_kernel<<<grid_for((size_t)a.B * a.n_kt * 4), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_masked_rows_fixup(const FixupArgs& in, cudaStream_t stream) {
  // Heads per CTA: one, unless 8 * B * H CTAs would be more than eight per SM.
  FixupArgs a = in;
  const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
  const long long ctas = 8LL * a.B * a.H;
  a.heads_per_cta = (int)std::min<long long>(a.H, std::max<long long>(1, ctas / (8LL * sms)));
  dim3 grid(8, (a.H + a.heads_per_cta - 1) / a.heads_per_cta, a.B);
  masked_rows_fixup_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
