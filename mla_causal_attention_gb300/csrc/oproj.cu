// oproj.cu -- the output projection (o_proj) after the attention core, on sm_103a tensor
// cores.
//
// The MLA init excerpt on "Kimi K2 · Similarities" (section "Scale scores") ends the attention
// block with o_proj, a linear map from num_heads x v_head_dim = 64 x 128 to hidden_size (7168
// and no bias in the config.json excerpt on "Kimi K2 · Logits").  Its input row for (b, i) is
// the heads' outputs concatenated in head order, so
//   y[b, i, n] = sum_{h, d} W[n, 128 h + d] attn[b, h, i, d]
// a GEMM with M = B * T rows, K = 128 H, N outputs.  It reads the attention output where the
// attention core left it ([B, H, T, 128]) through a 4-D tensor map: a 64-column slice of K is
// half of one head, and a 128-row box is 128 positions of one sequence (T > 1) or 128
// sequences (T = 1, decode).
//
// Persistent: one CTA per SM walks 128-row x BN-column output tiles (BN = 256; with few row
// tiles, as in decode, 48 or 64 so that about one CTA per SM streams its share of the
// weight), with two TMEM accumulators so one tile's epilogue overlaps the next tile's K
// loop.  256 threads:
//   warps 0, 2, 3  TMA producers (the A slice; the two halves of the weight slice);
//   warp 1         allocates the TMEM accumulator, issues M128 x BN x K16 MMAs (A and B
//                  both K-major from 128-byte swizzled shared memory);
//   warps 4-7      epilogue: TMEM -> registers -> bf16 -> global, one row per thread.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kOpBM = 128;      // rows per tile (TMEM lanes)
constexpr int kOpBK = 64;       // K per stage: one 128-byte swizzled row of bf16
constexpr int kOpASub = kOpBM * kOpBK * 2;  // 16 KB

template <int BN>
struct OpCfg {
  static constexpr int kBBytes = BN * kOpBK * 2;               // weight slice
  static constexpr int kStage = kOpASub + kBBytes;
  static constexpr int kStages = BN == 256 ? 4 : (BN == 48 ? 10 : 8);  // fill shared memory
  static constexpr int kTmemCols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
  static_assert(2 * kTmemCols <= 512, "two accumulators in TMEM");
  static_assert(kStage % 1024 == 0 && BN % 16 == 0, "stage alignment, MMA N");
  static constexpr int kBarOff = kStages * kStage;
  static constexpr int kSmem = kBarOff + 256 + 1024;
  static constexpr int kBoxN = BN > 128 ? 128 : BN;            // rows per weight box
  static constexpr int kWProd = BN / kBoxN;                    // weight producers
  static_assert(kSmem <= 232448, "shared memory per block");
};

struct OprojParams {
  CUtensorMap tm_a;  // attn {128, T, H, B}
  CUtensorMap tm_w;  // w {K, N}
  uint16_t* y;
  int* status;
  int B, H, T, N, K;
  int m_tiles_per_b;  // T > 1: row tiles per sequence; T == 1: 0
  int m_tiles, n_tiles;
};

struct OpBars {  // <= 256 bytes
  uint64_t full[10];
  uint64_t empty[10];
  uint64_t acc_full[2];   // accumulator buffer a holds a finished tile
  uint64_t acc_empty[2];  // accumulator buffer a read out (4 warp arrivals)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Output tile t: row tile t % m_tiles (rows (b, i0 .. i0 + 127) for T > 1, sequences
// b .. b + 127 for T == 1), column tile t / m_tiles.  Row tiles run fastest, so the CTAs
// resident at once share one weight column block in L2.
struct OpTile {
  int b, i0, n0;
};
__device__ __forceinline__ OpTile op_tile(const OprojParams& p, int t, int bn) {
  OpTile w;
  const int mt = t % p.m_tiles;
  w.n0 = (t / p.m_tiles) * bn;
  if (p.m_tiles_per_b > 0) {
    w.b = mt / p.m_tiles_per_b;
    w.i0 = (mt % p.m_tiles_per_b) * kOpBM;
  } else {
    w.b = mt * kOpBM;
    w.i0 = 0;
  }
  return w;
}

// 2-D and 4-D tiled copies global -> shared with an L2 cache policy (createpolicy) for the
// copied lines; the innermost coordinate times the element size must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d_policy(void* smem_dst, const void* tmap,
                                                   uint64_t* bar, int c0, int c1,
                                                   uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_policy(void* smem_dst, const void* tmap,
                                                   uint64_t* bar, int c0, int c1, int c2,
                                                   int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

static_assert(sizeof(OpBars) <= 256, "barrier block");

template <int BN>
__global__ void __launch_bounds__(256, 1) oproj_kernel(const __grid_constant__ OprojParams p) {
  using C = OpCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  OpBars* bars = reinterpret_cast<OpBars*>(smem + C::kBarOff);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KB = p.K / kOpBK;
  const int n_tiles = p.m_tiles * p.n_tiles;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1 + C::kWProd);  // the A producer and the weight producers
      mbar_init(&bars->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars->acc_full[a], 1);
      mbar_init(&bars->acc_empty[a], 4);  // the 4 epilogue warps
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 2 * C::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = bars->tmem_base;

  if ((warp == 0 || warp == 2 || warp == 3) && lane == 0) {
    // ================= TMA producers =================
    // warp 0: the A slice (16 KB); warps 2 and 3: weight rows n0 .. n0 + 127 and
    // n0 + 128 .. n0 + 255 (BN = 256; warp 2 alone for narrower tiles).  The k-block ring
    // runs on across the CTA's tiles.
    const int role = warp == 0 ? 0 : warp - 1;  // 0 = A, 1.. = weight box
    if (role <= C::kWProd) {
      prefetch_tmap(role == 0 ? (const void*)&p.tm_a : (const void*)&p.tm_w);
      // The input is re-read by every column tile: keep it in L2.  Each weight byte is read
      // once: let it go first.
      const uint64_t pol = role == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
      uint32_t g = 0;  // k-blocks posted over the run
      bool ok = true;
      for (int t = blockIdx.x; t < n_tiles && ok; t += G) {
        const OpTile w = op_tile(p, t, BN);
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int s = g % C::kStages;
          if (g >= (uint32_t)C::kStages &&
              !mbar_wait(&bars->empty[s], ((g / C::kStages) - 1) & 1, p.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* stage = smem + s * C::kStage;
          if (role == 0) {
            mbar_arrive_expect_tx(&bars->full[s], kOpASub);
            const int h = kb >> 1, d0 = (kb & 1) * kOpBK;
            tma_load_4d_policy(stage, &p.tm_a, &bars->full[s], d0, w.i0, h, w.b, pol);
          } else {
            mbar_arrive_expect_tx(&bars->full[s], C::kBoxN * kOpBK * 2);
            const int r = (role - 1) * C::kBoxN;
            tma_load_2d_policy(stage + kOpASub + r * kOpBK * 2, &p.tm_w, &bars->full[s],
                               kb * kOpBK, w.n0 + r, pol);
          }
        }
      }
      // Loads in flight must land before the CTA's shared memory is released.
      for (uint32_t k = g > (uint32_t)C::kStages ? g - C::kStages : 0; k < g; ++k) {
        const uint32_t a = smem_u32(&bars->full[k % C::kStages]);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(a, (k / C::kStages) & 1))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    // Tile j of this CTA accumulates in TMEM buffer j & 1, once the epilogue has read the
    // tile two back out of it.
    constexpr uint32_t kIdesc = tc::idesc_bf16_f32(kOpBM, BN, false);
    const uint64_t dhi = tc::smem_desc_sw128(0, 16, 1024);
    const uint32_t base_lo = smem_u32(smem) >> 4;
    bool ok = true;
    uint32_t g = 0;
    int j = 0;
    for (int t = blockIdx.x; t < n_tiles && ok; t += G, ++j) {
      const int ab = j & 1;
      if (j >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_empty[ab], ((j >> 1) - 1) & 1,
                                               p.status, abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t acc = tbase + ab * C::kTmemCols;
      for (int kb = 0; kb < KB; ++kb, ++g) {
        const int s = g % C::kStages;
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&bars->full[s], (g / C::kStages) & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t a_lo = base_lo + (s * C::kStage >> 4);
        const uint32_t b_lo = a_lo + (kOpASub >> 4);
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kOpBK / 16; ++kk) {
            const uint32_t koff = kk * (32 >> 4);
            tc::mma_ss(acc, dhi | (uint64_t)(a_lo + koff), dhi | (uint64_t)(b_lo + koff),
                       kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
#ifdef MLA_TEST_DROP_STAGE_RELEASE
          // Test build only: CTA 0 skips the release of its first stage.  The producers'
          // bounded waits for that stage then give up, which exercises the timeout report
          // and the unwinding (the MMAs in flight are still covered by the final commit
          // that precedes the release of tensor memory).
          const bool withhold = blockIdx.x == 0 && g == 0;
#else
          constexpr bool withhold = false;
#endif
          if (!withhold) tc::commit(&bars->empty[s]);
          if (kb == KB - 1) tc::commit(&bars->acc_full[ab]);
        }
        __syncwarp();
      }
    }
    // No MMA may still run when TMEM is released (also after a failed wait).
    if (tc::elect_one()) tc::commit(&bars->mma_done);
    __syncwarp();
    const uint32_t a = smem_u32(&bars->mma_done);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(a, 0))
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  } else if (warp >= 4) {
    // ================= epilogue =================
    const int q = warp & 3;
    const int r = q * 32 + lane;  // tile row = TMEM lane
    int j = 0;
    for (int t = blockIdx.x; t < n_tiles; t += G, ++j) {
      const int ab = j & 1;
      const bool got = __all_sync(
          0xffffffffu, mbar_wait(&bars->acc_full[ab], (j >> 1) & 1, p.status, abort_flag));
      if (!got) break;
      tc::fence_after_sync();
      const OpTile w = op_tile(p, t, BN);
      bool row_ok;
      size_t row;
      if (p.m_tiles_per_b > 0) {
        row_ok = w.i0 + r < p.T;
        row = (size_t)w.b * p.T + w.i0 + r;
      } else {
        row_ok = w.b + r < p.B;
        row = (size_t)(w.b + r);
      }
      uint16_t* dst = p.y + row * p.N + w.n0;
      const uint32_t t_row = tbase + ab * C::kTmemCols + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        tc::tmem_ld16(t_row + c * 16, v);
        tc::tmem_wait_ld();
        if (row_ok && w.n0 + c * 16 < p.N) {
          uint4* o = reinterpret_cast<uint4*>(dst + c * 16);
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint4 x;
            x.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]), __uint_as_float(v[8 * u + 1]));
            x.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]), __uint_as_float(v[8 * u + 3]));
            x.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]), __uint_as_float(v[8 * u + 5]));
            x.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]), __uint_as_float(v[8 * u + 7]));
            o[u] = x;
          }
        }
      }
      // This warp's rows of the accumulator are read: the MMA warp may reuse the buffer.
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty[ab]);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, 2 * C::kTmemCols);
  }
}

// Tensor maps cached by pointers and sizes (encoding costs microseconds of host time).
struct OpKey {
  const void* a;
  const void* w;
  int B, H, T, N, bn;
  bool operator==(const OpKey& o) const {
    return a == o.a && w == o.w && B == o.B && H == o.H && T == o.T && N == o.N && bn == o.bn;
  }
};
struct OpEntry {
  OpKey key;
  CUtensorMap a, w;
  bool valid;
};
std::mutex g_op_mu;
OpEntry g_op[8];
int g_op_next = 0;

bool oproj_maps(const OprojArgs& a, int bn, OprojParams* p) {
  const OpKey key{a.attn, a.w, a.B, a.H, a.T, a.N, bn};
  std::lock_guard<std::mutex> lk(g_op_mu);
  for (const OpEntry& e : g_op) {
    if (e.valid && e.key == key) {
      p->tm_a = e.a;
      p->tm_w = e.w;
      return true;
    }
  }
  const uint64_t dims_a[4] = {128, (uint64_t)a.T, (uint64_t)a.H, (uint64_t)a.B};
  const uint64_t str_a[3] = {256, (uint64_t)a.T * 256, (uint64_t)a.H * a.T * 256};
  const uint32_t box_a[4] = {64, a.T > 1 ? 128u : 1u, 1, a.T > 1 ? 1u : 128u};
  const uint64_t K = (uint64_t)a.H * 128;
  const uint64_t dims_w[2] = {K, (uint64_t)a.N};
  const uint64_t str_w[1] = {K * 2};
  const uint32_t box_w[2] = {64, (uint32_t)std::min(bn, 128)};
  if (!encode_bf16_tiled(&p->tm_a, a.attn, 4, dims_a, str_a, box_a) ||
      !encode_bf16_tiled(&p->tm_w, a.w, 2, dims_w, str_w, box_w))
    return false;
  OpEntry& e = g_op[g_op_next];
  g_op_next = (g_op_next + 1) % 8;
  e.key = key;
  e.a = p->tm_a;
  e.w = p->tm_w;
  e.valid = true;
  return true;
}

template <int BN>
cudaError_t launch_bn(const OprojArgs& a, int m_tiles, cudaStream_t stream) {
  using C = OpCfg<BN>;
  OprojParams p;
  if (!oproj_maps(a, BN, &p)) return cudaErrorInvalidValue;
  p.y = a.y;
  p.status = a.status;
  p.B = a.B;
  p.H = a.H;
  p.T = a.T;
  p.N = a.N;
  p.K = a.H * 128;
  p.m_tiles_per_b = a.T > 1 ? (a.T + kOpBM - 1) / kOpBM : 0;
  p.m_tiles = m_tiles;
  p.n_tiles = (a.N + BN - 1) / BN;
  static std::atomic<uint64_t> attr_done{0};  // bit per device: smem attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load() & bit)) {
    e = cudaFuncSetAttribute(oproj_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit);
  }
  // Persistent: one CTA per SM (at most one per tile), each walking tiles c, c + G, ...
  const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
  const int64_t tiles = (int64_t)m_tiles * p.n_tiles;
  if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
  oproj_kernel<BN><<<(unsigned)std::min<int64_t>(tiles, sms), 256, C::kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_oproj(const OprojArgs& a, cudaStream_t stream) {
  const int64_t m_tiles = a.T > 1 ? (int64_t)a.B * ((a.T + kOpBM - 1) / kOpBM)
                                  : ((int64_t)a.B + kOpBM - 1) / kOpBM;
  if (m_tiles > 0x7fffffff) return cudaErrorInvalidValue;
  // Few row tiles (decode): narrow column tiles so that about one CTA per SM streams its
  // share of the weight (48 columns: 150 tiles of a 7168-wide weight on 152 SMs).
  const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
  if (m_tiles * ((a.N + 255) / 256) < sms) {
    if (m_tiles * ((a.N + 47) / 48) <= sms) return launch_bn<48>(a, (int)m_tiles, stream);
    return launch_bn<64>(a, (int)m_tiles, stream);
  }
  return launch_bn<256>(a, (int)m_tiles, stream);
}

}  // namespace mla
