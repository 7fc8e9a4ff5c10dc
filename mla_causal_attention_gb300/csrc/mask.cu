// mask.cu -- the 2D padding mask on keys: packing for the prefill kernel, and the rows that
// no key is visible to.
//
// The model's 2D attention_mask ("Kimi K2 · Causal mask", §Construct causal mask) is
// expanded to 4D and merged with the causal mask, so a hidden key receives the same
// additive minimum as a causally hidden one.  A query row that sees no visible key at all
// then has every score equal to that minimum, and its softmax weights are uniform over
// all Tk keys: its output is the plain mean of the Tk value rows.  The attention kernels
// skip hidden keys; masked_rows_fixup_kernel writes those uniform rows afterwards.
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

// One CTA of 256 threads per (sequence b, group of 8 heads).  Query row i of sequence b
// sees no visible key when i + past_len is below the first key that is visible (key_mask
// set and j < kv_len[b]).  Those rows get the mean of all Tk value rows.
__global__ void __launch_bounds__(256) masked_rows_fixup_kernel(const FixupArgs a) {
  __shared__ int s_first;
  __shared__ float s_part[8][128];
  const int b = blockIdx.y;
  const int h0 = blockIdx.x * 8;
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
  const int grp = threadIdx.x >> 5;  // 8 row groups
  const float inv_tk = 1.0f / (float)a.Tk;
  for (int h = h0; h < min(h0 + 8, a.H); ++h) {
    const size_t bh = (size_t)b * a.H + h;
    const uint16_t* vb = a.v + bh * a.kv_rows * 128;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;  // columns 4 lane .. 4 lane + 3
    for (int j = grp; j < a.Tk; j += 8) {
      const uint2 w = *reinterpret_cast<const uint2*>(vb + (size_t)j * 128 + lane * 4);
      s0 += bf16lo_to_f32(w.x);
      s1 += bf16hi_to_f32(w.x);
      s2 += bf16lo_to_f32(w.y);
      s3 += bf16hi_to_f32(w.y);
    }
    s_part[grp][lane * 4 + 0] = s0;
    s_part[grp][lane * 4 + 1] = s1;
    s_part[grp][lane * 4 + 2] = s2;
    s_part[grp][lane * 4 + 3] = s3;
    __syncthreads();
    if (threadIdx.x < 128) {
      float t = 0.f;
#pragma unroll
      for (int g = 0; g < 8; ++g) t += s_part[g][threadIdx.x];
      s_part[0][threadIdx.x] = t * inv_tk;
    }
    __syncthreads();
    // Rows i < n_rows, 64 threads per row (2 columns each).
    const int c = (threadIdx.x & 63) * 2;
    const uint32_t word = pack_bf16x2(s_part[0][c], s_part[0][c + 1]);
    for (int i = threadIdx.x >> 6; i < n_rows; i += 4)
      *reinterpret_cast<uint32_t*>(a.out + (bh * a.Tq + i) * 128 + c) = word;
    __syncthreads();  // s_part is reused by the next head
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

cudaError_t launch_masked_rows_fixup(const FixupArgs& a, cudaStream_t stream) {
  dim3 grid((a.H + 7) / 8, a.B);
  masked_rows_fixup_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
