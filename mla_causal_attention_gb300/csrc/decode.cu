// decode.cu -- split-KV decode kernel (Tq == 1) and its combine pass, sm_103a.
//
// Per sequence b and head h the single query attends to keys j < kv_len[b]:
//   s_j = softmax_scale * ([q_nope | q_pe] . [k_nope[b,h,j] | k_pe_shared[b,j]])
//   out = sum_j softmax(s)_j v[b,h,j]
// (the attention excerpt on "Kimi K2 · Similarities"; with Tq = 1 and Tk = past_len + 1
// the causal limit admits every cached key, so only kv_len, and the optional 2D padding
// mask on keys, hide keys).
//
// Work split: one CTA per (group of 4 heads, key chunk, sequence).  One producer thread
// streams each 16-key stage with 1-D bulk copies into a 3-deep shared-memory ring: the
// shared rotary-key rows once per stage, then the no-rope key and value rows of the four
// heads.  Two consumer warps per head split the stage's keys: 8 lanes per key form the
// 192-wide dot product (conflict-free 128-bit shared loads, 3 shuffles), the warp keeps a running
// (max, sum) in the log2 domain, and every lane accumulates 4 output columns.  The CTA
// writes either the final bf16 row (single split) or a (max, sum, acc[128]) partial that
// the combine kernel merges:  m = max m_s,  l = sum 2^(m_s - m) l_s,
// out = sum 2^(m_s - m) acc_s / l.
#include <atomic>
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace mla {
namespace {

template <int G, int T, int NST, int WPH>
struct DecCfg {
  static constexpr int kConsumerWarps = G * WPH;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kTokPerWarp = T / WPH;
  static constexpr int kPasses = kTokPerWarp / 4;
  static constexpr uint32_t kKpeBytes = T * 128;
  static constexpr uint32_t kKnBytes = T * 256;
  static constexpr uint32_t kVBytes = T * 256;
  static constexpr uint32_t kStageBytes = kKpeBytes + G * (kKnBytes + kVBytes);
  static constexpr uint32_t kMergeBytes = kConsumerWarps * 132 * 4;
  static constexpr uint32_t kBarBytes = 128;
  static constexpr uint32_t kSmemBytes = NST * kStageBytes + kMergeBytes + kBarBytes;
  static_assert(T % (4 * WPH) == 0, "stage keys must split into 4-key passes per warp");
  static_assert(kStageBytes % 128 == 0, "stage alignment");
};

__device__ __forceinline__ float dot8(const uint4 k, const float* q) {
  float s = 0.f;
  s = fmaf(q[0], bf16lo_to_f32(k.x), s);
  s = fmaf(q[1], bf16hi_to_f32(k.x), s);
  s = fmaf(q[2], bf16lo_to_f32(k.y), s);
  s = fmaf(q[3], bf16hi_to_f32(k.y), s);
  s = fmaf(q[4], bf16lo_to_f32(k.z), s);
  s = fmaf(q[5], bf16hi_to_f32(k.z), s);
  s = fmaf(q[6], bf16lo_to_f32(k.w), s);
  s = fmaf(q[7], bf16hi_to_f32(k.w), s);
  return s;
}

__device__ __forceinline__ void load8(const uint16_t* src, float scale, float* dst) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  dst[0] = bf16lo_to_f32(w.x) * scale;
  dst[1] = bf16hi_to_f32(w.x) * scale;
  dst[2] = bf16lo_to_f32(w.y) * scale;
  dst[3] = bf16hi_to_f32(w.y) * scale;
  dst[4] = bf16lo_to_f32(w.z) * scale;
  dst[5] = bf16hi_to_f32(w.z) * scale;
  dst[6] = bf16lo_to_f32(w.w) * scale;
  dst[7] = bf16hi_to_f32(w.w) * scale;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait used only to drain the producer's own copies before exit; ignores the
// abort flag (copies in flight must land before the CTA's shared memory goes away).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// KM: the 2D padding mask on keys is applied (p.key_mask); a separate instantiation so the
// unmasked kernel carries none of its per-key work.
// ROPE: q_pe and the new key row arrive unrotated (p.rope_cs); a separate instantiation so
// the other kernels carry none of its registers or per-pass work.
template <int G, int T, int NST, int WPH, int MINB, bool KM, bool ROPE>
__global__ void __launch_bounds__(DecCfg<G, T, NST, WPH>::kThreads, MINB)
    decode_splitkv_kernel(const DecodeArgs p) {
  using C = DecCfg<G, T, NST, WPH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* merge = reinterpret_cast<float*>(smem + NST * C::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NST * C::kStageBytes + C::kMergeBytes);
  uint64_t* empty = full + NST;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NST);
  uint64_t* rot_done = empty + NST + 1;  // the new key row rotated (ROPE only, one phase)

  const int hg = blockIdx.x;
  const int split = blockIdx.y;
  const int b = blockIdx.z;
  const int h0 = hg * G;
  const int ng = min(G, p.H - h0);

  int kvl = p.kv_len ? p.kv_len[b] : p.Tk;
  if (kvl < 1 || kvl > p.Tk) {
    if (threadIdx.x == 0 && hg == 0 && split == 0) set_status(p.status, MLA_ERR_KVLEN);
    kvl = min(max(kvl, 1), p.Tk);
  }
  // Let the combine grid (launched with programmatic stream serialisation) get scheduled
  // now; it waits for this grid's completion itself before reading any partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j0 = split * p.chunk;
  if (j0 >= kvl) return;  // uniform across the CTA: this split holds no visible key
  const int j1 = min(j0 + p.chunk, kvl);
  const int n_tiles = (j1 - j0 + T - 1) / T;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::kConsumerWarps);
    }
    if (ROPE) mbar_init(rot_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == C::kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint64_t pol_kpe = l2_policy_evict_last();  // re-read by the other head groups
      int issued = 0;
      for (int it = 0; it < n_tiles; ++it) {
        const int slot = it % NST;
        if (it >= NST) {
          if (!mbar_wait(&empty[slot], ((it / NST) - 1) & 1, p.status, abort_flag)) break;
        }
        const int jt = j0 + it * T;
        const int nt = min(T, j1 - jt);
        uint8_t* st = stages + slot * C::kStageBytes;
        mbar_arrive_expect_tx(&full[slot], (uint32_t)nt * (128u + (uint32_t)ng * 512u));
        // With a fused append, the stage holding key row Tk-1 takes that row from the new
        // token's buffers; the cache supplies the rows before it.
        const bool subst = p.new_k_nope != nullptr && jt + nt == p.Tk;
        const int nc = subst ? nt - 1 : nt;  // rows read from the cache
        if (nc > 0)
          bulk_g2s(st, p.k_pe + ((size_t)b * p.kv_rows + jt) * 64, nc * 128, &full[slot], pol_kpe);
        if (subst) bulk_g2s(st + nc * 128, p.new_k_pe + (size_t)b * 64, 128, &full[slot], pol);
        for (int g = 0; g < ng; ++g) {
          const size_t bh = (size_t)b * p.H + h0 + g;
          uint8_t* kn_dst = st + C::kKpeBytes + g * C::kKnBytes;
          uint8_t* v_dst = st + C::kKpeBytes + G * C::kKnBytes + g * C::kVBytes;
          if (nc > 0) {
            bulk_g2s(kn_dst, p.k_nope + (bh * p.kv_rows + jt) * 128, nc * 256, &full[slot], pol);
            bulk_g2s(v_dst, p.v + (bh * p.kv_rows + jt) * 128, nc * 256, &full[slot], pol);
          }
          if (subst) {
            bulk_g2s(kn_dst + nc * 256, p.new_k_nope + bh * 128, 256, &full[slot], pol);
            bulk_g2s(v_dst + nc * 256, p.new_v + bh * 128, 256, &full[slot], pol);
          }
        }
        ++issued;
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int it = max(0, issued - NST); it < issued; ++it)
        drain_wait(&full[it % NST], (it / NST) & 1);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int g = warp / WPH;
  const int wh = warp % WPH;
  const bool head_ok = g < ng;
  const int l8 = lane & 7;
  const int tk = lane >> 3;
  const size_t bh = (size_t)b * p.H + h0 + (head_ok ? g : 0);

  // This lane's slice of the query, pre-multiplied by softmax_scale * log2(e): no-rope
  // columns [8*l8, 8*l8+8) and [64+8*l8, 64+8*l8+8), rotary columns [8*l8, 8*l8+8).  With
  // this split the 8 lanes of a key read each 128-byte half-row of shared memory once,
  // so the 4 keys of a pass hit every bank exactly once per 16-byte load.
  float qn[16], qr[8];
  // With the rotary step: the cos / sin of this lane's eight rotary columns at position
  // Tk - 1 (the query's, and the new key's), columns 8 (l8 & 3) .. + 8 of either half.
  // Loaded where they are used (L2-resident), so they are not live across the key loop.
  constexpr bool rope = ROPE;
  auto rope_cs = [&](float (&c)[8], float (&sn)[8], int slice) {
    const float4* cs = reinterpret_cast<const float4*>(p.rope_cs + 8 * slice);
    const float4* ss = reinterpret_cast<const float4*>(p.rope_cs + 32 + 8 * slice);
    const float4 c0 = cs[0], c1 = cs[1], s0 = ss[0], s1 = ss[1];
    c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
    c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
    sn[4] = s1.x; sn[5] = s1.y; sn[6] = s1.z; sn[7] = s1.w;
  };
  {
    const uint16_t* qsrc = p.q_nope + bh * 128 + l8 * 8;
    load8(qsrc, p.scale_log2, qn);
    load8(qsrc + 64, p.scale_log2, qn + 8);
    if (rope) {
      // The rotary pair of column d is d + 32: lanes l8 and l8 ^ 4 of a key group.
      const uint4 own = *reinterpret_cast<const uint4*>(p.q_pe + bh * 64 + l8 * 8);
      const uint4 other = make_uint4(__shfl_xor_sync(0xffffffffu, own.x, 4),
                                     __shfl_xor_sync(0xffffffffu, own.y, 4),
                                     __shfl_xor_sync(0xffffffffu, own.z, 4),
                                     __shfl_xor_sync(0xffffffffu, own.w, 4));
      float rc[8], rs[8];
      rope_cs(rc, rs, l8 & 3);
      const uint4 rot = rope_rotate8(own, other, rc, rs, l8 >= 4);
      const uint32_t w[4] = {rot.x, rot.y, rot.z, rot.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        qr[2 * k] = bf16lo_to_f32(w[k]) * p.scale_log2;
        qr[2 * k + 1] = bf16hi_to_f32(w[k]) * p.scale_log2;
      }
    } else {
      load8(p.q_pe + bh * 64 + l8 * 8, p.scale_log2, qr);
    }
  }

  // Fused cache append: split 0 of each head group writes the new key/value rows into the
  // cache (row Tk-1); no CTA of this call reads that cache row.
  if (p.new_k_nope != nullptr && split == 0 && head_ok && wh == 0 && lane < 16) {
    const size_t row = bh * p.kv_rows + (p.Tk - 1);
    reinterpret_cast<uint4*>(p.cache_k_nope + row * 128)[lane] =
        reinterpret_cast<const uint4*>(p.new_k_nope + bh * 128)[lane];
    reinterpret_cast<uint4*>(p.cache_v + row * 128)[lane] =
        reinterpret_cast<const uint4*>(p.new_v + bh * 128)[lane];
    if (hg == 0 && g == 0 && lane < 8) {
      uint4 kp = reinterpret_cast<const uint4*>(p.new_k_pe + (size_t)b * 64)[lane];
      if (rope) {  // lanes 0..7 hold the row's eight column slices; pairs are lane ^ 4
        const uint4 other = make_uint4(__shfl_xor_sync(0xffu, kp.x, 4),
                                       __shfl_xor_sync(0xffu, kp.y, 4),
                                       __shfl_xor_sync(0xffu, kp.z, 4),
                                       __shfl_xor_sync(0xffu, kp.w, 4));
        float rc[8], rs[8];
        rope_cs(rc, rs, lane & 3);
        kp = rope_rotate8(kp, other, rc, rs, lane >= 4);
      }
      reinterpret_cast<uint4*>(p.cache_k_pe + ((size_t)b * p.kv_rows + p.Tk - 1) * 64)[lane] = kp;
    }
  }

  float m_run = -1e30f;  // finite sentinel: 2^(m_run - m_new) stays defined
  float l_run = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  // 2D padding mask: the mask bytes of this lane's keys, loaded one stage ahead so that
  // their latency never adds to a stage that has already landed.
  uint8_t mnext[C::kPasses];
  auto load_mask = [&](int it_m) {
#pragma unroll
    for (int ps = 0; ps < C::kPasses; ++ps) {
      const int jm = j0 + it_m * T + wh * C::kTokPerWarp + ps * 4 + tk;
      mnext[ps] = (KM && it_m < n_tiles && jm < j1) ? p.key_mask[(size_t)b * p.Tk + jm] : 1;
    }
  };
  if (KM) load_mask(0);

  for (int it = 0; it < n_tiles; ++it) {
    const int slot = it % NST;
    const int jt = j0 + it * T;
    const int nt = min(T, j1 - jt);
    // With the rotary step, this stage's new-token row (key Tk - 1, taken from the new
    // buffers) arrives unrotated: the lanes of that key rotate their slices in registers.
    const bool rot_stage = rope && p.new_k_nope != nullptr && jt + nt == p.Tk;
    bool hidden[C::kPasses];
#pragma unroll
    for (int ps = 0; ps < C::kPasses; ++ps) hidden[ps] = KM && mnext[ps] == 0;
    if (KM) load_mask(it + 1);
    if (!mbar_wait(&full[slot], (it / NST) & 1, p.status, abort_flag)) break;
    if (rot_stage) {
      // The stage's last row is the new key's rotary part, unrotated: lanes 0..7 of the first
      // consumer warp rotate it in place (pairs are lane ^ 4) and signal an mbarrier that
      // the other consumer warps wait on (bounded, like every wait).  One such stage per CTA.
      if (warp == 0) {
        if (lane < 8) {
          uint4* row = reinterpret_cast<uint4*>(stages + slot * C::kStageBytes + (nt - 1) * 128);
          const uint4 own = row[lane];
          const uint4 other = make_uint4(__shfl_xor_sync(0xffu, own.x, 4),
                                         __shfl_xor_sync(0xffu, own.y, 4),
                                         __shfl_xor_sync(0xffu, own.z, 4),
                                         __shfl_xor_sync(0xffu, own.w, 4));
          float rc[8], rs[8];
          rope_cs(rc, rs, lane & 3);
          row[lane] = rope_rotate8(own, other, rc, rs, lane >= 4);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rot_done);
      } else if (!mbar_wait(rot_done, 0, p.status, abort_flag)) {
        break;
      }
    }
    if (head_ok) {
      const uint8_t* st = stages + slot * C::kStageBytes;
      const uint8_t* kpe_s = st;
      const uint8_t* kn_s = st + C::kKpeBytes + g * C::kKnBytes;
      const uint8_t* v_s = st + C::kKpeBytes + G * C::kKnBytes + g * C::kVBytes;

      float sc[C::kPasses];
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        const int t = wh * C::kTokPerWarp + ps * 4 + tk;
        const uint8_t* krow = kn_s + t * 256 + l8 * 16;
        const uint4 a0 = *reinterpret_cast<const uint4*>(krow);
        const uint4 a1 = *reinterpret_cast<const uint4*>(krow + 128);
        const uint4 c0 = *reinterpret_cast<const uint4*>(kpe_s + t * 128 + l8 * 16);
        float d = dot8(a0, qn) + dot8(a1, qn + 8) + dot8(c0, qr);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        sc[ps] = (t < nt && !hidden[ps]) ? d : -INFINITY;
      }
      float mx = sc[0];
#pragma unroll
      for (int ps = 1; ps < C::kPasses; ++ps) mx = fmaxf(mx, sc[ps]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2_approx(m_run - m_new);
      float pr[C::kPasses];
      float ps_sum = 0.f;
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        pr[ps] = ex2_approx(sc[ps] - m_new);
        ps_sum += pr[ps];
      }
      ps_sum += __shfl_xor_sync(0xffffffffu, ps_sum, 8);
      ps_sum += __shfl_xor_sync(0xffffffffu, ps_sum, 16);
      l_run = l_run * alpha + ps_sum;
      m_run = m_new;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] *= alpha;
      // Value mix: lane owns columns [4*lane, 4*lane + 4).
#pragma unroll
      for (int tt = 0; tt < C::kTokPerWarp; ++tt) {
        const int t = wh * C::kTokPerWarp + tt;
        const float pt = __shfl_sync(0xffffffffu, pr[tt / 4], (tt % 4) * 8);
        if (t < nt) {
          const uint2 vv = *reinterpret_cast<const uint2*>(v_s + t * 256 + lane * 8);
          acc[0] = fmaf(pt, bf16lo_to_f32(vv.x), acc[0]);
          acc[1] = fmaf(pt, bf16hi_to_f32(vv.x), acc[1]);
          acc[2] = fmaf(pt, bf16lo_to_f32(vv.y), acc[2]);
          acc[3] = fmaf(pt, bf16hi_to_f32(vv.y), acc[3]);
        }
      }
    }
    __syncwarp();
#ifdef MLA_TEST_DROP_SLOT_RELEASE
    // Test build only: the first consumer warp of CTA (0, 0, 0) withholds its release of the
    // first stage's slot.  The producer's bounded wait for that slot then gives up, which
    // exercises the timeout report and the CTA's unwinding (copies drained, no partial
    // written).  The arrival carries no transaction bytes.
    const bool withhold = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && warp == 0 &&
                          it == 0;
#else
    constexpr bool withhold = false;
#endif
    if (lane == 0 && !withhold) mbar_arrive(&empty[slot]);
  }

  // Merge the WPH warps of each head through shared memory.
  float* mw = merge + warp * 132;
  if (lane == 0) {
    mw[0] = m_run;
    mw[1] = l_run;
  }
  *reinterpret_cast<float4*>(mw + 4 + lane * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  named_bar_sync(1, C::kConsumerWarps * 32);
  if (wh != 0 || !head_ok || *abort_flag) return;

  float m = -1e30f;
#pragma unroll
  for (int w = 0; w < WPH; ++w) m = fmaxf(m, merge[(warp + w) * 132]);
  float l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < WPH; ++w) {
    const float* src = merge + (warp + w) * 132;
    const float f = ex2_approx(src[0] - m);
    l += f * src[1];
    const float4 a = *reinterpret_cast<const float4*>(src + 4 + lane * 4);
    o[0] += f * a.x;
    o[1] += f * a.y;
    o[2] += f * a.z;
    o[3] += f * a.w;
  }
  if (p.splits == 1) {
    // l = 0 only when the 2D padding mask hides every key; that row is rewritten later.
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint2 w;
    w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(p.out + bh * 128 + lane * 4) = w;
  } else {
    const size_t pi = bh * p.splits + split;
    if (lane == 0) *reinterpret_cast<float2*>(p.part_ml + pi * 2) = make_float2(m, l);
    *reinterpret_cast<float4*>(p.part_acc + pi * 128 + lane * 4) =
        make_float4(o[0], o[1], o[2], o[3]);
  }
}

// One warp per (b, h): merge the partials of the splits that hold visible keys.
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs p) {
  // Launched as a programmatic dependent of the split kernel: wait until that grid has
  // completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= p.B * p.H) return;
  const int b = w / p.H;
  int kvl = p.kv_len ? p.kv_len[b] : p.Tk;
  kvl = min(max(kvl, 1), p.Tk);
  const int n = (kvl + p.chunk - 1) / p.chunk;
  const size_t base = (size_t)w * p.splits;
  // (max, sum) of up to 32 splits per pass, one split per lane, loaded in parallel; then
  // the 128-column accumulators in batches of 8 independent loads per lane, so a merge
  // costs a few memory round trips instead of one per split.
  float m = -1e30f;
  for (int s = lane; s < n; s += 32) m = fmaxf(m, p.part_ml[(base + s) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n; s0 += 32) {
    float f = 0.f;  // this lane's split weight 2^(m_s - m)
    if (s0 + lane < n) {
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (base + s0 + lane) * 2);
      f = ex2_approx(ml.x - m);
      l += f * ml.y;
    }
    const int cnt = min(32, n - s0);
    for (int s1 = 0; s1 < cnt; s1 += 8) {
      float4 a[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (s1 + k < cnt)
          a[k] = *reinterpret_cast<const float4*>(p.part_acc + (base + s0 + s1 + k) * 128 +
                                                  lane * 4);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float fk = __shfl_sync(0xffffffffu, f, s1 + k);
        if (s1 + k < cnt) {
          acc.x += fk * a[k].x;
          acc.y += fk * a[k].y;
          acc.z += fk * a[k].z;
          acc.w += fk * a[k].w;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;  // see the single-split case
  uint2 o;
  o.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  o.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.out + (size_t)w * 128 + lane * 4) = o;
}

template <int T, int MINB, bool KM, bool ROPE>
cudaError_t launch_split(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int G = kDecHeadsPerCta, NST = 3, WPH = 2;
  using C = DecCfg<G, T, NST, WPH>;
  auto kern = decode_splitkv_kernel<G, T, NST, WPH, MINB, KM, ROPE>;
  static std::atomic<uint64_t> attr_done{0};  // bit per device: smem attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  dim3 grid((a.H + G - 1) / G, a.splits, a.B);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  // 16-key stages, 2 CTAs per SM (204 KB of stages in flight per SM).  For every problem
  // size measured this beats 32-key stages at 1 CTA per SM, which hold the same bytes in
  // flight: two independent rings per SM hide each other's waits (ragged 64-sequence batch
  // 2.6% faster, 32 x 32768 keys 3.2%, 16 x 2048 keys 12%).
  cudaError_t e;
  if (a.key_mask && a.rope_cs) return cudaErrorInvalidValue;  // no such entry point
  if (a.key_mask)
    e = launch_split<kDecTokensPerStage, 2, true, false>(a, stream);
  else if (a.rope_cs)
    e = launch_split<kDecTokensPerStage, 2, false, true>(a, stream);
  else
    e = launch_split<kDecTokensPerStage, 2, false, false>(a, stream);
  if (e != cudaSuccess || a.splits == 1) return e;
  // The combine pass is a programmatic dependent launch: its launch latency overlaps
  // the tail of the split kernel.
  const int warps = a.B * a.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((warps + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, a);
}

}  // namespace mla
