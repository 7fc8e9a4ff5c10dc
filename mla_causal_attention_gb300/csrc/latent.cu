// latent.cu -- decode over MLA's latent cache with the key/value up-projection absorbed,
// on sm_103a tensor cores.
//
// The MLA init excerpt on "Kimi K2 · Similarities" (§Scale scores) gives the joint key/value
// down-projection (kv_a_proj_with_mqa: a 512-wide latent plus the shared 64-wide rotary key)
// and the up-projection kv_b_proj: 512 -> 64 heads x (128 no-rope key + 128 value).  The
// cache can therefore hold the latent row c_j (and the rotary key) instead of 64 heads'
// keys and values, 1152 bytes per token instead of 32,896.  With W_K[h], W_V[h] the
// 128 x 512 blocks of kv_b_proj for head h:
//   q_nope . k_nope_j = q_nope . (W_K c_j) = (W_K^T q_nope) . c_j = q_lat . c_j
//   sum_j p_j v_j     = sum_j p_j W_V c_j  = W_V (sum_j p_j c_j)   = W_V o_lat
// so the attention runs over the latent rows for all 64 heads at once (one shared "key"
// [c_j | k_pe_j] of 576 columns, one shared "value" c_j of 512), between two small per-head
// projections.
//
// Kernels:
//   latent_absorb_kernel      q_lat[b,h] = W_K[h]^T q_nope[b,h]              (bf16 out)
//   latent_splitkv_kernel     one CTA per SM over an equal share of all sequences' 128-key
//                             tiles: scores for the 64 heads, online softmax per head,
//                             one o_lat partial per sequence it touches
//   latent_combine_up_kernel  merges the partials of (sequence, head) into o_lat, then
//                             out[b,h] = W_V[h] o_lat[b,h]                   (bf16 out)
// Each kernel after the first is a programmatic dependent launch of the one before.
//
// The split kernel runs both MMAs transposed, with keys (and latent columns) on the
// 128 TMEM lanes and the 64 heads as the N dimension:
//   S^T[128 keys, 64 heads]   = K_tile[128, 576] . Q^T        A = K tile (K-major), B = Q
//   O^T[512, 64 heads]       += C_tile^T[512, 128] . P       4 M-blocks of 128 latent
//                                                             columns; A = the tile's
//                                                             latent rows read MN-major,
//                                                             B = P [keys, heads] from
//                                                             shared memory (MN-major)
//   L[128, 64 heads]         += 1[128, 128] . P              the row sums, A = ones in TMEM
// so O^T takes 4 x 64 TMEM columns (a head-major O would need all 512), and the softmax
// needs no sum reduction: every row of L holds the running sum of each head's (bf16)
// weights, rescaled with O^T.  The tile's eight 64-column latent sub-tiles stay in eight
// fixed slots from the score pass through the value pass (latent sub-tile s of every tile
// lives in slot s); its rotary-key sub-tile is loaded into the P buffer, which is free
// during the score pass.  Each value block releases its two slots, so the next tile's first
// sub-tiles load while the current value mixes still run.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace mla {
namespace {

constexpr int kLD = 512;          // latent width (kv_lora_rank)
constexpr int kLSubK = 16384;     // 128 keys x 64 columns, bf16, 128-byte swizzled
constexpr int kLSubQ = 8192;      // 64 heads x 64 columns
constexpr int kLSlots = 8;        // latent sub-tile s of every key tile lives in slot s
constexpr int kLThreads = 384;    // warps 0, 2 producers, warp 1 MMA, warps 4-11 softmax
constexpr int kLOffQ = 0;                             // 9 sub-tiles: q_lat 0-511, q_pe
constexpr int kLOffRing = kLOffQ + 9 * kLSubQ;        // 73728
constexpr int kLOffP = kLOffRing + kLSlots * kLSubK;  // 204800: the tile's rotary keys
                                                      // (16 KB), then P [128 keys x 64]
constexpr int kLOffRed = kLOffP + kLSubK;             // 221184: softmax scratch
constexpr int kLOffBar = kLOffRed + 4096;             // 225280
constexpr int kLSmem = kLOffBar + 256 + 1024;         // + barriers + alignment slack
static_assert(kLSmem <= 232448, "shared memory per block");
constexpr float kLRescale = 8.0f;  // log2 units, as in the prefill kernel
// TMEM columns: S^T [0, 64), O^T blocks [64, 320), L [320, 384), the ones operand [384, 416).
constexpr uint32_t kLColO = 64, kLColL = 320, kLColOnes = 384;

struct LatentParams {
  CUtensorMap tm_q;   // q_lat {512, H, B}, boxes {64, 64, 1}
  CUtensorMap tm_qr;  // q_pe  {64, H, B},  boxes {64, 64, 1}
  CUtensorMap tm_c;   // c_kv  {512, Tk, B}, boxes {64, 128, 1}
  CUtensorMap tm_kr;  // k_pe  {64, Tk, B},  boxes {64, 128, 1}
  const int32_t* kv_len;
  int32_t* seq_tile0;  // [B + 1]: first tile of each sequence in the partition, then T
  float* part_ml;
  float* part_acc;
  int* status;
  int B, H, Tk;
  float scale_log2;
};

struct LBars {
  uint64_t full[kLSlots];   // slot s holds the current tile's latent sub-tile s
  uint64_t empty[kLSlots];  // slot s released by the value block that read it
  uint64_t pe_full;         // the tile's rotary keys are in the P buffer
  uint64_t pe_free;         // the previous tile's value mixes are done with P
  uint64_t q_full;
  uint64_t q_empty;         // the segment's last score MMA has read Q
  uint64_t s_full;          // S^T of the tile in TMEM
  uint64_t p_ready;         // P in shared memory, O^T and L rescaled (8 warp arrivals)
  uint64_t o_done;          // the segment's last value mix done
  uint64_t o_free;          // O^T and L of the segment read out (8 warp arrivals)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(LBars) <= 256, "barrier block");

__device__ __forceinline__ void ldrain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Barrier over the 8 softmax warps (named barrier 1) that ANDs a predicate across them.
__device__ __forceinline__ bool softmax_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " bar.red.and.pred po, 1, 256, pi;\n selp.u32 %0, 1, 0, po;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Maximum of v over the 32 lanes of the warp (every lane gets it).
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The work partition.  Sequence b holds n_b = ceil(kv_len[b] / 128) key tiles; laid end to
// end they form T tiles, and CTA c of G = min(gridDim.x, T) takes tiles [c T / G,
// (c + 1) T / G), so every CTA gets T / G >= 1 tiles to within one (CTAs past G exit).  A CTA's range crosses sequence boundaries: it walks the
// segments (one per sequence it touches) in order, and writes one partial per segment, at
// index c + b (unique: the (c, b) pairs covered form a staircase, monotone in both).
__device__ __forceinline__ int latent_tiles(const LatentParams& p, int b) {
  const int kv = p.kv_len ? min(max(p.kv_len[b], 1), p.Tk) : p.Tk;
  return (kv + kLatTile - 1) / kLatTile;
}
__device__ __forceinline__ int latent_kv(const LatentParams& p, int b) {
  return p.kv_len ? min(max(p.kv_len[b], 1), p.Tk) : p.Tk;
}

// One segment of a CTA's range: sequence b, its keys [j0, j1), nt tiles.
struct LSeg {
  int b, j0, j1, nt;
};
// Walks the segments of [t0, t1): start at sequence b0 whose first tile is P0.
struct LSegWalk {
  int b, P, t0, t1;
  __device__ __forceinline__ bool next(const LatentParams& p, LSeg& s) {
    if (P >= t1 || b >= p.B) return false;
    const int n = latent_tiles(p, b);
    const int lo = max(t0, P), hi = min(t1, P + n);
    s.b = b;
    s.j0 = (lo - P) * kLatTile;
    s.j1 = min(latent_kv(p, b), (hi - P) * kLatTile);
    s.nt = hi - lo;
    P += n;
    ++b;
    return true;
  }
};

__global__ void __launch_bounds__(kLThreads, 1)
    latent_splitkv_kernel(const __grid_constant__ LatentParams p) {
  grid_dep_launch();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sQ = smem + kLOffQ;
  uint8_t* sRing = smem + kLOffRing;
  uint8_t* sP = smem + kLOffP;
  LBars* bars = reinterpret_cast<LBars*>(smem + kLOffBar);
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;

  // ---- the partition: per-sequence tile counts, a block-wide scan, this CTA's range ----
  int* scan = reinterpret_cast<int*>(smem + kLOffRed);  // [12] warp totals, [16..17] result
  int T;  // tiles of all sequences
  {
    const int per = (p.B + kLThreads - 1) / kLThreads;
    const int bs = min(p.B, (int)threadIdx.x * per), be = min(p.B, bs + per);
    int mine = 0;
    bool bad = false;
    for (int bb = bs; bb < be; ++bb) {
      if (p.kv_len && (p.kv_len[bb] < 1 || p.kv_len[bb] > p.Tk)) bad = true;
      mine += latent_tiles(p, bb);
    }
    if (bad && c == 0) set_status(p.status, MLA_ERR_KVLEN);
    int incl = mine;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kLThreads / 32; ++w) {
      const int v = scan[w];
      if (w < warp) before += v;
      total += v;
    }
    const int excl = before + incl - mine;  // first tile of sequence bs
    const int G = min((int)gridDim.x, total);
    const int t0 = (int)((int64_t)c * total / G);
    if (excl <= t0 && t0 < excl + mine) {  // this thread's sequences hold tile t0
      int P = excl;
      for (int bb = bs; bb < be; ++bb) {
        const int n = latent_tiles(p, bb);
        if (P + n > t0) {
          scan[16] = bb;
          scan[17] = P;
          break;
        }
        P += n;
      }
    }
    if (c == 0) {  // the prefix array, for the combine
      int P = excl;
      for (int bb = bs; bb < be; ++bb) {
        p.seq_tile0[bb] = P;
        P += latent_tiles(p, bb);
      }
      if (threadIdx.x == 0) p.seq_tile0[p.B] = total;
    }
    T = total;
    __syncthreads();
  }
  const int G = min((int)gridDim.x, T);
  if (c >= G) return;  // uniform: no tiles for this CTA
  const int t0 = (int)((int64_t)c * T / G), t1 = (int)((int64_t)(c + 1) * T / G);
  const int b_first = scan[16], P_first = scan[17];
  __syncthreads();  // the scan scratch is reused by the softmax warps

  if (threadIdx.x == 0) {
    for (int i = 0; i < kLSlots; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->pe_full, 1);
    mbar_init(&bars->pe_free, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_ready, 8);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_free, 8);
    mbar_init(&bars->mma_done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = bars->tmem_base;
  LSegWalk walk{b_first, P_first, t0, t1};
  LSeg sg;

  if (warp == 0 || warp == 2) {
    // Two producer threads: one thread's TMA issue rate is well below what the SM takes in,
    // and a tile's loads are issued in one burst once its slots free up.  Producer pi owns
    // the latent slots s = pi (mod 2); producer 0 also loads Q, producer 1 the rotary keys.
    const int pi = warp >> 1;
    if (lane == 0) {
      // ================= TMA producers =================
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_qr);
      prefetch_tmap(&p.tm_c);
      prefetch_tmap(&p.tm_kr);
      bool ok = true;
      uint32_t g = 0;  // key tiles issued over the run
      int nseg = 0;    // segments whose Q was issued
      // Q of sequence bq, once the previous segment's last score MMA has read Q.
      auto load_q = [&](int bq) -> bool {
        if (nseg > 0 && !mbar_wait(&bars->q_empty, (nseg - 1) & 1, p.status, abort_flag))
          return false;
        mbar_arrive_expect_tx(&bars->q_full, 9 * kLSubQ);
        for (int s = 0; s < 8; ++s)
          tma_load_3d_nohint(sQ + s * kLSubQ, &p.tm_q, &bars->q_full, 64 * s, 0, bq);
        tma_load_3d_nohint(sQ + 8 * kLSubQ, &p.tm_qr, &bars->q_full, 0, 0, bq);
        ++nseg;
        return true;
      };
      while (ok && walk.next(p, sg)) {
        for (int j = 0; j < sg.nt && ok; ++j, ++g) {
          const int jt = sg.j0 + j * kLatTile;
          const uint32_t prev = (g - 1) & 1u;
          // A later segment's queries go first: Q is free once the previous segment's last
          // score MMA has run, which is well before its value mixes release the slots.
          if (j == 0 && pi == 0 && nseg > 0) {
            ok = load_q(sg.b);
            if (!ok) break;
          }
          // Latent columns 0-511: sub-tile s into slot s once the previous tile's value
          // block s / 2 has released it.
          for (int sidx = pi; sidx < kLSlots; sidx += 2) {
            if (g > 0) ok = mbar_wait(&bars->empty[sidx], prev, p.status, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars->full[sidx], kLSubK);
            tma_load_3d_nohint(sRing + sidx * kLSubK, &p.tm_c, &bars->full[sidx], 64 * sidx,
                               jt, sg.b);
          }
          if (!ok) break;
          if (j == 0 && pi == 0 && nseg == 0) {
            // The first segment's queries come from the absorb kernel, which may still be
            // running (this grid can start early; the latent loads above do not depend on
            // it).
            grid_dep_wait();
            ok = load_q(sg.b);
            if (!ok) break;
          }
          // Rotary keys into the P buffer once the previous tile's value mixes are done.
          if (pi == 1) {
            if (g > 0) ok = mbar_wait(&bars->pe_free, prev, p.status, abort_flag);
            if (!ok) break;
            mbar_arrive_expect_tx(&bars->pe_full, kLSubK);
            tma_load_3d_nohint(sP, &p.tm_kr, &bars->pe_full, 0, jt, sg.b);
          }
        }
      }
      // Every load issued must land before shared memory is released: each barrier has at
      // most its last phase in flight.  (A tile whose loads were only partly issued after a
      // failed wait leaves its remaining slots one phase behind: their drains end at the
      // wait limit, after the abort that caused them.)
      if (pi == 0 && nseg > 0) ldrain(&bars->q_full, (uint32_t)(nseg - 1) & 1u);
      if (g > 0) {
        for (int sidx = pi; sidx < kLSlots; sidx += 2)
          ldrain(&bars->full[sidx], (g - 1) & 1u);
        if (pi == 1) ldrain(&bars->pe_full, (g - 1) & 1u);
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    constexpr uint32_t kIdQK = tc::idesc_bf16_f32_ab(128, 64, false, false);
    constexpr uint32_t kIdPV = tc::idesc_bf16_f32_ab(128, 64, true, true);
    constexpr uint32_t kIdL = tc::idesc_bf16_f32_ab(128, 64, false, true);
    // P [keys, heads]: one 128-byte row per key, 8-key groups 1024 B apart (N = 64 spans a
    // single swizzle atom, so the leading offset is unused).
    const uint64_t dhi_p = tc::smem_desc_sw128(0, 16, 1024);
    const uint64_t dhi_k = tc::smem_desc_sw128(0, 16, 1024);
    const uint64_t dhi_mn = tc::smem_desc_sw128(0, kLSubK, 1024);  // slots 2q, 2q+1 adjacent
    const uint32_t q_lo = smem_u32(sQ) >> 4;
    const uint32_t ring_lo = smem_u32(sRing) >> 4;
    const uint32_t p_lo = smem_u32(sP) >> 4;
    const uint32_t s_tmem = tbase;            // S^T: 64 columns
    const uint32_t o_tmem = tbase + kLColO;   // O^T: 4 blocks of 64 columns
    const uint32_t l_tmem = tbase + kLColL;   // L: 64 columns
    const uint32_t ones_tmem = tbase + kLColOnes;
    bool ok = true;
    uint32_t g = 0;  // key tiles over the run
    int ns = 0;      // segments
    while (ok && walk.next(p, sg)) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, ns & 1, p.status, abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      for (int j = 0; j < sg.nt && ok; ++j, ++g) {
        const uint32_t ph = g & 1u;
        // S^T = K_tile Q^T over 576 columns: 4 k-steps of 16 per 64-column sub-tile; the
        // rotary-key sub-tile (in the P buffer) last.
        for (int sidx = 0; sidx < 9; ++sidx) {
          uint64_t* fb = sidx < 8 ? &bars->full[sidx] : &bars->pe_full;
          ok = __all_sync(0xffffffffu, mbar_wait(fb, ph, p.status, abort_flag));
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t a_lo = sidx < 8 ? ring_lo + sidx * (kLSubK >> 4) : p_lo;
          if (tc::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t koff = kk * (32 >> 4);
              const uint64_t adesc = dhi_k | (uint64_t)(a_lo + koff);
              const uint64_t bdesc = dhi_k | (uint64_t)(q_lo + sidx * (kLSubQ >> 4) + koff);
              tc::mma_ss(s_tmem, adesc, bdesc, kIdQK, (sidx | kk) != 0 ? 1u : 0u);
            }
            if (sidx == 8) {
              tc::commit(&bars->s_full);
              if (j == sg.nt - 1) tc::commit(&bars->q_empty);  // segment's last read of Q
            }
          }
          __syncwarp();
        }
        if (!ok) break;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_ready, ph, p.status, abort_flag));
        // The segment's first value mix overwrites O^T and L: the previous segment's must
        // have been read out.
        if (ok && j == 0 && ns > 0)
          ok = mbar_wait(&bars->o_free, (ns - 1) & 1, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after_sync();
        // O^T block q (latent columns 128q..128q+127) += C_tile^T P over the tile's keys:
        // A = slots 2q and 2q + 1 read MN-major, B = P; then L += 1 P (A = ones in TMEM).
        if (tc::elect_one()) {
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t adesc =
                  dhi_mn | (uint64_t)(ring_lo + 2 * q * (kLSubK >> 4) + kk * (2048 >> 4));
              const uint64_t bdesc = dhi_p | (uint64_t)(p_lo + kk * (2048 >> 4));
              tc::mma_ss(o_tmem + 64 * q, adesc, bdesc, kIdPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
#ifdef MLA_TEST_DROP_SLOT_RELEASE
            // Test build only: CTA 0 skips the release of slot 0 after its first tile.  The
            // producer's bounded wait to refill it then gives up, which exercises the timeout
            // report and the unwinding (the final commit still covers every MMA in flight).
            const bool withhold = blockIdx.x == 0 && g == 0 && q == 0;
#else
            constexpr bool withhold = false;
#endif
            if (!withhold) tc::commit(&bars->empty[2 * q]);
            tc::commit(&bars->empty[2 * q + 1]);
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bdesc = dhi_p | (uint64_t)(p_lo + kk * (2048 >> 4));
            tc::mma_ts(l_tmem, ones_tmem, bdesc, kIdL, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc::commit(&bars->pe_free);
          if (j == sg.nt - 1) tc::commit(&bars->o_done);
        }
        __syncwarp();
      }
      ++ns;
    }
    if (tc::elect_one()) tc::commit(&bars->mma_done);
    __syncwarp();
    ldrain(&bars->mma_done, 0);
  } else if (warp >= 4) {
    // ================= softmax warps =================
    // Two groups of 4 warps: group g owns heads [32g, 32g + 32).  Thread = key row r of the
    // tile = TMEM lane r (warp % 4 selects the lane quarter); its 32 columns of the S^T row
    // are its group's heads.  For the value pass, lane r is latent column 128q + r of O^T
    // block q (and row r of L), and the group rescales its heads' columns.
    const int grp = (warp - 4) >> 2;
    const int hb = 32 * grp;
    const int sw = warp & 3;
    const int r = sw * 32 + lane;
    const int t = threadIdx.x - 128;  // owner of head t when t < 64 (warps 4, 5)
    const uint32_t lane_off = (uint32_t)(sw * 32) << 16;
    const uint32_t s_t = tbase + lane_off + hb;
    const uint32_t o_t = tbase + lane_off + kLColO + hb;
    const uint32_t l_t = tbase + lane_off + kLColL + hb;
    float* red_max = reinterpret_cast<float*>(smem + kLOffRed);  // [4 quarters][64 heads]
    float* mbase = red_max + 256;                                 // [64] exponent base
    float* alpha_s = mbase + 64;                                  // [64] this tile's rescale
    int* any_rescale = reinterpret_cast<int*>(alpha_s + 64);      // [2], by tile parity
    const float sl2 = p.scale_log2;
    if (t < 2) any_rescale[t] = 0;
    if (grp == 0) {
      // The all-ones A operand of the row-sum MMA (bf16 1.0 pairs), 32 columns.
      uint32_t one[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) one[i] = 0x3F803F80u;
      tc::tmem_st32(tbase + lane_off + kLColOnes, one);
      tc::tmem_wait_st();
    }
    softmax_sync();
    bool ok = true;
    uint32_t g = 0;  // key tiles over the run
    int ns = 0;      // segments
    while (ok && walk.next(p, sg)) {
      float m_own = -INFINITY;  // running max (log2 units) of head t in this segment
      for (int j = 0; j < sg.nt; ++j, ++g) {
        const bool got =
            __all_sync(0xffffffffu, mbar_wait(&bars->s_full, g & 1, p.status, abort_flag));
        float v[32];
        if (got) {
          tc::fence_after_sync();
          uint32_t ra[32];
          tc::tmem_ld32(s_t, ra);
          tc::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = __uint_as_float(ra[h]);
          if (sg.j0 + j * kLatTile + r >= sg.j1) {  // key past the segment or past kv_len
#pragma unroll
            for (int h = 0; h < 32; ++h) v[h] = -INFINITY;
          }
        } else {
#pragma unroll
          for (int h = 0; h < 32; ++h) v[h] = -INFINITY;
        }
        // Per-head maximum over this warp's 32 keys (warp-uniform results).
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 m4 = make_float4(redux_max(v[4 * i]), redux_max(v[4 * i + 1]),
                                        redux_max(v[4 * i + 2]), redux_max(v[4 * i + 3]));
          if (lane == 0) reinterpret_cast<float4*>(red_max + sw * 64 + hb)[i] = m4;
        }
        if (!softmax_and(got)) {  // barrier A; every warp leaves together on a failed wait
          ok = false;
          break;
        }
        if (t < 64) {
          const float tm = fmaxf(fmaxf(red_max[t], red_max[64 + t]),
                                 fmaxf(red_max[128 + t], red_max[192 + t])) * sl2;
          float a = 1.f;
          if (j == 0) {
            m_own = tm;  // key j0 < kv_len is visible: finite
          } else if (tm > m_own + kLRescale) {
            a = ex2_approx(m_own - tm);
            m_own = tm;
          }
          mbase[t] = m_own;
          alpha_s[t] = a;
          if (a != 1.f) any_rescale[g & 1] = 1;
        } else if (t == 64) {
          any_rescale[(g + 1) & 1] = 0;  // everyone read it before barrier A of this tile
        }
        softmax_sync();  // barrier B
        // p = 2^(s * scale * log2(e) - m), two heads per packed fma
        uint32_t pk[16];
#pragma unroll
        for (int h = 0; h < 32; h += 4) {
          const float4 mb = *reinterpret_cast<const float4*>(mbase + hb + h);
          const uint64_t sl2_2 = f2_pack(sl2, sl2);
          float x0, x1, x2, x3;
          f2_unpack(ffma2(f2_pack(v[h], v[h + 1]), sl2_2, f2_pack(-mb.x, -mb.y)), x0, x1);
          f2_unpack(ffma2(f2_pack(v[h + 2], v[h + 3]), sl2_2, f2_pack(-mb.z, -mb.w)), x2, x3);
          pk[h >> 1] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
          pk[(h >> 1) + 1] = pack_bf16x2(ex2_approx(x2), ex2_approx(x3));
        }
        if (any_rescale[g & 1]) {
          // O^T and L columns of this group's heads whose max grew.
#pragma unroll 1
          for (int q = 0; q < 5; ++q) {
            const uint32_t col = q < 4 ? o_t + 64 * q : l_t;
            uint32_t o[32];
            tc::tmem_ld32(col, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e)
              o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha_s[hb + e]);
            tc::tmem_st32(col, o);
          }
          tc::tmem_wait_st();
        }
        // P [128 keys x 64 heads] bf16, 128-byte swizzled like a TMA tile: key r's row holds
        // this group's 32 heads in 16-byte chunks 4g .. 4g + 3.
        {
          uint8_t* row = sP + r * 128;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
            *reinterpret_cast<uint4*>(row + (((4 * grp + cc) ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        }
        fence_proxy_async_smem();  // P written by threads, read by the tensor core
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_ready);
      }
      if (!ok) break;
      // The segment's partial: O^T and the row sums once its last value mix has run, at
      // partial index c + b; then O^T and L are released for the next segment.
      if (__all_sync(0xffffffffu, mbar_wait(&bars->o_done, ns & 1, p.status, abort_flag))) {
        tc::fence_after_sync();
        const size_t row0 = (size_t)(c + sg.b) * p.H;  // (partial, head 0)
        const int nh = min(32, p.H - hb);                // this group's heads present
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t oa[32];
          tc::tmem_ld32(o_t + 64 * q, oa);
          tc::tmem_wait_ld();
          // column 128q + r of heads hb.., one 2 KB row apart
          float* dst = p.part_acc + (row0 + hb) * kLD + 128 * q + r;
#pragma unroll
          for (int h = 0; h < 32; ++h)
            if (h < nh) dst[h * kLD] = __uint_as_float(oa[h]);
        }
        if (t < 64) {  // warps 4 and 5, whole warps (the TMEM load is warp-wide)
          // Every row of L holds the sums; owner t (lane t % 32) takes column t from its own
          // lane quarter.
          uint32_t la[32];
          tc::tmem_ld32(tbase + lane_off + kLColL + (t & ~31), la);
          tc::tmem_wait_ld();
          float l = 0.f;
#pragma unroll
          for (int h = 0; h < 32; ++h) l = (h == (t & 31)) ? __uint_as_float(la[h]) : l;
          if (t < p.H)
            *reinterpret_cast<float2*>(p.part_ml + (row0 + t) * 2) = make_float2(m_own, l);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free);
      }
      ++ns;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, 512);
  }
}

// Warp-level bf16 MMA (m16n8k16, fp32 accumulate) for the two per-head projections: small
// GEMMs (64 sequences x 128 columns x 128, 64 x 32 x 512) whose operands sit in padded
// shared memory and are read with ldmatrix.  Fragments (g = lane / 4, c = lane % 4): A a0
// (row g, cols 2c, 2c+1), a1 (row g+8), a2 (cols + 8), a3 (row g+8, cols + 8); B b0 (rows
// k = 2c, 2c+1, col g), b1 (k + 8); C c0, c1 (row g, cols 2c, 2c+1), c2, c3 (row g+8).
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 bf16 matrices from shared memory; lane l gives the row address of matrix l / 8.
__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// The same, each matrix transposed.
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

constexpr int kPB = 64;            // sequences per projection CTA
constexpr int kAbN = 128;          // latent columns per absorb CTA
constexpr int kAbRow = 128 + 8;    // padded bf16 row (128 values) of the absorb operands
constexpr int kAbsorbSmem = (128 + kPB) * kAbRow * 2;
constexpr int kCuB = 32;           // sequences per merge + up-projection CTA
constexpr int kUpRow = kLD + 8;    // padded bf16 row (512 values)
constexpr int kCuSmem = (128 + kCuB) * kUpRow * 2;

// q_lat[b,h,n] = sum_k W_K[h][k][n] q_nope[b,h,k] for one head, a quarter of the 512 latent
// columns and 64 sequences: [64 x 128] . [128 x 128].  W_K[h] = rows h*256 .. h*256+127 of
// kv_b_proj (k = no-rope key dim, n = latent dim).  Warp w: row tile w % 4 (16 sequences),
// columns 64 (w / 4) .. +63.
__global__ void __launch_bounds__(256) latent_absorb_kernel(const LatentArgs a) {
  grid_dep_launch();
  extern __shared__ __align__(16) uint8_t ab_smem[];
  uint16_t* sw = reinterpret_cast<uint16_t*>(ab_smem);  // W_K slice: 128 rows (k) x 128 (n)
  uint16_t* sq = sw + 128 * kAbRow;                      // q_nope: 64 rows (b) x 128 (k)
  const int h = blockIdx.x;
  const int n0 = blockIdx.y * kAbN;
  const int b0 = blockIdx.z * kPB;
  const int nb = min(kPB, a.B - b0);
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    cp_async16(sw + r * kAbRow + c * 8, a.w_kvb + ((size_t)h * 256 + r) * kLD + n0 + c * 8);
  }
  for (int i = threadIdx.x; i < kPB * 16; i += blockDim.x) {
    const int r = i >> 4, c = i & 15;
    if (r < nb)
      cp_async16(sq + r * kAbRow + c * 8, a.q_nope + ((size_t)(b0 + r) * a.H + h) * 128 + c * 8);
    else
      *reinterpret_cast<uint4*>(sq + r * kAbRow + c * 8) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_wait_all();
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = warp & 3, nh = warp >> 2;
  const int g = lane >> 2, c2 = (lane & 3) * 2;
  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
  for (int k0 = 0; k0 < 128; k0 += 16) {
    uint32_t af[4];
    ldsm4(af, sq + (mt * 16 + (lane & 15)) * kAbRow + k0 + (lane >> 4) * 8);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      // B[k][n] row-major: transposed loads give two n-tiles' (b0, b1)
      uint32_t bf[4];
      ldsm4t(bf, sw + (k0 + (lane & 15)) * kAbRow + nh * 64 + np * 16 + (lane >> 4) * 8);
      mma16816(acc[2 * np], af, bf[0], bf[1]);
      mma16816(acc[2 * np + 1], af, bf[2], bf[3]);
    }
  }
#pragma unroll
  for (int n = 0; n < 8; ++n) {
    const int col = n0 + nh * 64 + n * 8 + c2;
    const int r = mt * 16 + g;
    if (r < nb)
      *reinterpret_cast<uint32_t*>(a.q_lat + ((size_t)(b0 + r) * a.H + h) * kLD + col) =
          pack_bf16x2(acc[n][0], acc[n][1]);
    if (r + 8 < nb)
      *reinterpret_cast<uint32_t*>(a.q_lat + ((size_t)(b0 + r + 8) * a.H + h) * kLD + col) =
          pack_bf16x2(acc[n][2], acc[n][3]);
  }
}

// Merges the split kernel's partials of one (sequence, head) row into bf16 o_lat (the
// up-projection's MMA operand type): o_lat = sum_s 2^(m_s - m) acc_s / sum_s 2^(m_s - m) l_s
// over the CTAs that held the sequence's tiles.  One warp; lane owns columns 4 lane + 128 k.
__device__ __forceinline__ void latent_merge_row(const LatentArgs& a, int b, int h,
                                                 int lane, uint16_t* dst) {
  // The partials of sequence b: CTAs c_lo .. c_hi of the split kernel's partition (with
  // G = min(grid, T) the CTA holding tile x is ceil((x + 1) G / T) - 1), at index c + b.
  const int64_t P0 = a.seq_tile0[b], P1 = a.seq_tile0[b + 1], T = a.seq_tile0[a.B];
  const int64_t G = min((int64_t)a.grid, T);
  const int c_lo = (int)(((P0 + 1) * G - 1) / T);
  const int c_hi = (int)((P1 * G - 1) / T);
  const int n = c_hi - c_lo + 1;
  const size_t row0 = (size_t)(c_lo + b) * a.H + h;  // partial k is row row0 + k H
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml);
  // (max, sum) of partial s0 + lane, read once per pass of 32 partials
  float2 mine = make_float2(-INFINITY, 0.f);
  if (lane < n) mine = ml[row0 + (size_t)lane * a.H];
  float m = mine.x;
  for (int s = 32 + lane; s < n; s += 32) m = fmaxf(m, ml[row0 + (size_t)s * a.H].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f;
  float4 acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* src = reinterpret_cast<const float4*>(a.part_acc + row0 * kLD) + lane;
  const size_t stride = (size_t)a.H * (kLD / 4);  // float4s from one partial to the next
  for (int s0 = 0; s0 < n; s0 += 32) {
    // lane t holds the weight of partial s0 + t
    if (s0 > 0) mine = s0 + lane < n ? ml[row0 + (size_t)(s0 + lane) * a.H]
                                     : make_float2(-INFINITY, 0.f);
    const float f = s0 + lane < n ? ex2_approx(mine.x - m) : 0.f;
    l += f * mine.y;
    const int cnt = min(32, n - s0);
    for (int s = 0; s < cnt; s += 4) {  // up to four partials' rows in flight
      float4 v[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[u][k] = s + u < cnt ? src[(size_t)(s0 + s + u) * stride + 32 * k]
                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float fu = __shfl_sync(0xffffffffu, f, (s + u) & 31);
        if (s + u < cnt) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc[k].x = fmaf(fu, v[u][k].x, acc[k].x);
            acc[k].y = fmaf(fu, v[u][k].y, acc[k].y);
            acc[k].z = fmaf(fu, v[u][k].z, acc[k].z);
            acc[k].w = fmaf(fu, v[u][k].w, acc[k].w);
          }
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    *reinterpret_cast<uint2*>(dst + 4 * lane + 128 * k) =
        make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv),
                   pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
}

// out[b,h,n] = sum_k W_V[h][n][k] o_lat[b,h,k] for one head and 32 sequences:
// [32 x 512] . [512 x 128].  W_V[h] = rows h*256+128 .. h*256+255 of kv_b_proj.  The weight
// is staged before waiting for the split kernel; each of the 16 warps then merges 2
// sequences' rows of o_lat into shared memory, and computes output columns 16 (w % 8) ..
// + 15 of row tile w / 8.
__global__ void __launch_bounds__(512) latent_combine_up_kernel(const LatentArgs a) {
  extern __shared__ __align__(16) uint8_t cu_smem[];
  uint16_t* sw = reinterpret_cast<uint16_t*>(cu_smem);  // W_V[h]: 128 rows (n) x 512 (k)
  uint16_t* so = sw + 128 * kUpRow;                      // o_lat: 32 rows (b) x 512 (k)
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * kCuB;
  const int nb = min(kCuB, a.B - b0);
  for (int i = threadIdx.x; i < 128 * (kLD / 8); i += blockDim.x) {
    const int r = i / (kLD / 8), c = i % (kLD / 8);
    cp_async16(sw + r * kUpRow + c * 8, a.w_kvb + ((size_t)h * 256 + 128 + r) * kLD + c * 8);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  grid_dep_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < kCuB; i += 16) {
    uint16_t* row = so + i * kUpRow;
    if (i < nb) {
      latent_merge_row(a, b0 + i, h, lane, row);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint2*>(row + 4 * lane + 128 * k) = make_uint2(0u, 0u);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  const int g = lane >> 2, c2 = (lane & 3) * 2;
  const int mt = warp >> 3, nw = warp & 7;
  float acc[2][4];  // [column tile]
#pragma unroll
  for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll 4
  for (int k0 = 0; k0 < kLD; k0 += 16) {
    uint32_t af[4], bf[4];
    ldsm4(af, so + (mt * 16 + (lane & 15)) * kUpRow + k0 + (lane >> 4) * 8);
    // W_V rows are n with k contiguous (B column-major): matrices (n 0-7, k0), (n 0-7,
    // k0+8), (n 8-15, k0), (n 8-15, k0+8)
    ldsm4(bf, sw + (nw * 16 + (lane & 7) + ((lane >> 4) << 3)) * kUpRow + k0 +
                   ((lane >> 3) & 1) * 8);
    mma16816(acc[0], af, bf[0], bf[1]);
    mma16816(acc[1], af, bf[2], bf[3]);
  }
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int col = nw * 16 + n * 8 + c2;
    const int r = mt * 16 + g;
    if (r < nb)
      *reinterpret_cast<uint32_t*>(a.out + ((size_t)(b0 + r) * a.H + h) * 128 + col) =
          pack_bf16x2(acc[n][0], acc[n][1]);
    if (r + 8 < nb)
      *reinterpret_cast<uint32_t*>(a.out + ((size_t)(b0 + r + 8) * a.H + h) * 128 + col) =
          pack_bf16x2(acc[n][2], acc[n][3]);
  }
}

// Tensor maps, cached by pointers and sizes (encoding costs microseconds of host time).
struct LMapKey {
  const void* ptr[4];
  int B, H, Tk, kv_rows;
  bool operator==(const LMapKey& o) const {
    for (int i = 0; i < 4; ++i)
      if (ptr[i] != o.ptr[i]) return false;
    return B == o.B && H == o.H && Tk == o.Tk && kv_rows == o.kv_rows;
  }
};
struct LMapEntry {
  LMapKey key;
  CUtensorMap maps[4];
  bool valid;
};
std::mutex g_lmap_mu;
LMapEntry g_lmap[8];
int g_lmap_next = 0;

bool latent_maps(const LatentArgs& a, LatentParams* p) {
  const LMapKey key = {{a.q_lat, a.q_pe, a.c_kv, a.k_pe}, a.B, a.H, a.Tk, a.kv_rows};
  std::lock_guard<std::mutex> lk(g_lmap_mu);
  for (const LMapEntry& e : g_lmap) {
    if (e.valid && e.key == key) {
      p->tm_q = e.maps[0];
      p->tm_qr = e.maps[1];
      p->tm_c = e.maps[2];
      p->tm_kr = e.maps[3];
      return true;
    }
  }
  if (!encode_bf16_3d(&p->tm_q, a.q_lat, kLD, a.H, a.B, a.H, 64) ||
      !encode_bf16_3d(&p->tm_qr, a.q_pe, 64, a.H, a.B, a.H, 64) ||
      !encode_bf16_3d(&p->tm_c, a.c_kv, kLD, a.Tk, a.B, a.kv_rows, 128) ||
      !encode_bf16_3d(&p->tm_kr, a.k_pe, 64, a.Tk, a.B, a.kv_rows, 128))
    return false;
  LMapEntry& e = g_lmap[g_lmap_next];
  g_lmap_next = (g_lmap_next + 1) % 8;
  e.key = key;
  e.maps[0] = p->tm_q;
  e.maps[1] = p->tm_qr;
  e.maps[2] = p->tm_c;
  e.maps[3] = p->tm_kr;
  e.valid = true;
  return true;
}

}  // namespace

cudaError_t launch_latent(const LatentArgs& a, cudaStream_t stream) {
  LatentParams p;
  if (!latent_maps(a, &p)) return cudaErrorInvalidValue;
  p.kv_len = a.kv_len;
  p.part_ml = a.part_ml;
  p.part_acc = a.part_acc;
  p.status = a.status;
  p.B = a.B;
  p.H = a.H;
  p.Tk = a.Tk;
  p.seq_tile0 = a.seq_tile0;
  p.scale_log2 = a.scale_log2;

  static std::atomic<uint64_t> attr_done{0};  // bit per device: smem attributes set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(latent_splitkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kLSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(latent_combine_up_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kCuSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(latent_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAbsorbSmem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  const unsigned bgroups = (unsigned)((a.B + kPB - 1) / kPB);
  latent_absorb_kernel<<<dim3(a.H, kLD / kAbN, bgroups), 256, kAbsorbSmem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // The other two start as programmatic dependents of the kernel before them.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = kLSmem;
  e = cudaLaunchKernelEx(&cfg, latent_splitkv_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(a.H, (unsigned)((a.B + kCuB - 1) / kCuB));
  cfg.blockDim = dim3(512);
  cfg.dynamicSmemBytes = kCuSmem;
  e = cudaLaunchKernelEx(&cfg, latent_combine_up_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
