// prefill.cu -- fused causal MLA attention for Tq >= 1 on sm_103a tensor cores.
//
// Computes, for every sequence b, head h and query row i (position past_len + i),
//   out[b,h,i,:] = sum_j softmax_j( scale * [q_nope|q_pe]_i . [k_nope|k_pe_shared]_j ) v_j
// over the keys j <= i + past_len with j < kv_len[b]: the attention excerpt on the page
// "Kimi K2 · Similarities" (query/key concat, scores, scale, additive causal mask, fp32
// softmax, bf16 weights, weighted sum of values), evaluated flash-style so the [Tq, Tk]
// score matrix never leaves the SM.
//
// Work unit: one (b, h) and a pair of 128-row query tiles (256 rows).  The kernel is
// persistent: one CTA per SM walks its units (heaviest first, snake order across CTAs)
// with TMEM allocated and barriers initialised once, so a unit's query load and the
// previous unit's output stores overlap the tensor-core work of their neighbours.
// Warp roles (384 threads):
//   warp 0      TMA producer: per unit both query tiles (each as soon as the previous
//               unit's last score MMA on it has run), then for every 128-key tile five
//               16 KB sub-tiles (k_nope cols 0-63, k_nope cols 64-127, the shared
//               rotary key, v cols 0-63, v cols 64-127) into an 8-slot ring.
//   warp 1      allocates all 512 TMEM columns; lane 0 issues the MMAs:
//                 S_t  = Q_t K_j^T     12 x (M128 N128 K16), A and B from shared memory,
//                                      the 192-wide contraction split 64 | 64 | 64 so the
//                                      concatenated key is never materialised;
//                 O_t += P_t V_j       8 x (M128 N128 K16), P from TMEM, V from smem.
//               Order per key tile: PV_0(j-1), QK_0(j), PV_1(j-1), QK_1(j), so one
//               softmax warpgroup works while the tensor core runs the other tile.
//   warps 2, 3  only with the fused cache append: the unit that holds a new key tile on
//               its diagonal writes it from shared memory into the caches (warp 2 the
//               key sub-tiles, warp 3 the value sub-tiles, tensor stores issued as soon as
//               the tile lands); the other units' tiles they just pass on.  The ring slots
//               of a tile are released once both its MMAs and its stores have read them.
//   warps 4-7   softmax of query tile 0 (thread = row = TMEM lane);
//   warps 8-11  softmax of query tile 1.  Each reads its S row from TMEM, applies the
//               causal/padding mask only on tiles that straddle the limit, keeps a
//               running max (log2 domain) and sum, writes bf16 P over the S columns, and
//               rescales its O row only when the max grows by more than 2^8 (the stale
//               max cancels exactly in O / l).  At the end of a unit it moves O to
//               registers, releases the O columns for the next unit's first value mix,
//               then normalises and stores the bf16 row.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
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

constexpr int kBM = 128;       // query rows per tile (TMEM lanes)
constexpr int kBN = 128;       // keys per tile
constexpr int kSub = 16384;    // one 128-row x 128-byte (64 bf16) swizzled sub-tile
constexpr int kSlots = 8;      // K/V ring depth in sub-tiles (a power of two)
constexpr int kSubPerKv = 5;   // kn0, kn1, kpe, v0, v1
constexpr int kThreads = 384;
constexpr int kOffQ = 0;                       // 2 tiles x {nope0, nope1, pe}
constexpr int kOffRing = kOffQ + 2 * 3 * kSub;  // 98304
constexpr int kOffBar = kOffRing + kSlots * kSub;  // 229376
constexpr int kSmemBytes = kOffBar + 256 + 1024;   // barriers + 1 KB alignment slack
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if max grows > 2^8

struct PrefillParams {
  CUtensorMap tm_qn;  // q_nope  {128, Tq, B*H}
  CUtensorMap tm_qr;  // q_pe    {64,  Tq, B*H}
  CUtensorMap tm_kn;  // k_nope  {128, Tk, B*H}
  CUtensorMap tm_kr;  // k_pe    {64,  Tk, B}
  CUtensorMap tm_v;   // v       {128, Tk, B*H}
  // Fused cache append only: the new rows (loads) and the caches' rows [0, Tk) (stores).
  CUtensorMap tm_kn_new;  // new k_nope {128, Tq, B*H}
  CUtensorMap tm_kr_new;  // new k_pe   {64,  Tq, B}
  CUtensorMap tm_v_new;   // new v      {128, Tq, B*H}
  CUtensorMap tm_kn_st;   // k_nope cache {128, Tk, B*H}
  CUtensorMap tm_kr_st;   // k_pe cache   {64,  Tk, B}
  CUtensorMap tm_v_st;    // v cache      {128, Tk, B*H}
  int append;  // 1: key tiles n_pre.. come from the new rows and are written to the caches
  int n_pre;   // key tiles of the cached prefix (past_len / 128)
  const int32_t* kv_len;
  const uint32_t* key_bits;  // packed 2D padding mask [B][n_kt][4], or null
  uint16_t* out;
  int* status;
  int B, H, Tq, Tk, past_len, n_qb, n_kt;
  float scale_log2;
};

// Barriers.  K/V tiles are counted over the CTA's whole run (g = 0, 1, ...) and
// double-buffered by tile parity; score steps are counted per query tile over the run;
// Q, O-done and O-free advance once per work unit.
struct Bars {
  uint64_t kfull[2];    // K(g) landed (3 TMA boxes, one transaction count)
  uint64_t vfull[2];    // V(g) landed (2 boxes)
  uint64_t kempty[2];   // K(g) slots released (MMA commit after both score MMAs)
  uint64_t vempty[2];   // V(g) slots released (MMA commit after both value mixes)
  uint64_t q_full[2];   // Q_t of the unit landed
  uint64_t q_empty[2];  // last score MMA of tile t of the unit done: Q_t may be refilled
  uint64_t s_full[2];   // S_t of a step in TMEM
  uint64_t p_ready[2];  // P_t of a step in TMEM (4 warp arrivals)
  uint64_t o_done[2];   // last value mix of tile t of the unit done
  uint64_t o_free[2];   // O_t of the unit read out by the softmax warps (4 warp arrivals)
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Register split of the 384 x 168 registers the block launches with: 88 for the
// producer / MMA warpgroup, 208 for the two softmax warpgroups (128 x 88 + 256 x 208 =
// 64512, the whole pool).
static_assert(128 * 88 + 256 * 208 <= kThreads * 168, "register split");
__device__ __forceinline__ void setmaxnreg_dec_control() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
}
__device__ __forceinline__ void setmaxnreg_inc_softmax() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
}

// Keep the compiler from using tcgen05.ld destinations before tcgen05.wait::ld.
template <int N>
__device__ __forceinline__ void pin(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 8)
    asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]),
                 "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7]));
}
__device__ __forceinline__ void pin32(uint32_t (&r)[32]) { pin<32>(r); }

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Tensor store shared -> global of one 128-byte swizzled box (no negative coordinates; the
// map clips rows past its extent), and the bulk-group bookkeeping around it.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int c0,
                                             int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          tmap),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The source shared memory of every committed store has been read.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One work unit: a pair of 128-row query tiles of one (b, h).  Units are numbered
// heaviest first (the last query tiles see the most keys); CTA c of G takes units
// i G + c in even rounds i and i G + (G - 1 - c) in odd ones, which balances the
// decreasing sizes as well as dynamic assignment would, with no shared counter.
struct Unit {
  int bh, b, r0, kvl, nt0, nt1, n;
  int js;  // key tiles skipped at the front (hidden by the 2D mask); tile j is key tile j + js
  __device__ __forceinline__ int nt(int t) const { return t ? nt1 : nt0; }
};

// Unit index of the CTA's i-th unit, or -1 past the end.
__device__ __forceinline__ int unit_index(const PrefillParams& p, int i) {
  const int G = gridDim.x;
  const int64_t k = (int64_t)i * G + ((i & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return k < (int64_t)p.B * p.H * p.n_qb ? (int)k : -1;
}

// kv_len of a unit's sequence as stored (unclamped), or Tk without kv_len.  The only
// global load of a unit's description: each role fetches it one unit ahead.
__device__ __forceinline__ int unit_kv(const PrefillParams& p, int unit) {
  if (unit < 0 || !p.kv_len) return p.Tk;
  return p.kv_len[(unit % (p.B * p.H)) / p.H];
}

__device__ __forceinline__ Unit unit_make(const PrefillParams& p, int unit, int kv) {
  Unit w;
  const int BH = p.B * p.H;
  const int qb = p.n_qb - 1 - unit / BH;
  w.bh = unit % BH;
  w.b = w.bh / p.H;
  w.r0 = qb * 2 * kBM;
  w.kvl = min(max(kv, 1), p.Tk);
  int nt[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int rt = w.r0 + t * kBM;
    if (rt >= p.Tq) {
      nt[t] = 0;
    } else {
      const int qlast = min(rt + kBM - 1, p.Tq - 1);
      const int lastkey = min(qlast + p.past_len, w.kvl - 1);
      nt[t] = lastkey / kBN + 1;
    }
  }
  w.nt0 = nt[0];
  w.nt1 = nt[1];
  w.n = max(nt[0], nt[1]);
  w.js = 0;
  return w;
}

// Under the 2D mask, a leading key tile whose 128 keys are all hidden adds exactly nothing
// to any row of the unit, so every role starts the unit at the first key tile with a
// visible key.  The skip stops at the first query tile's last key tile, so that each query
// tile keeps at least one key tile; a row left with no visible key at all is rewritten by
// the masked-rows pass.  Each role reads the same packed bits, so all agree on js.
template <bool kMasked>
__device__ __forceinline__ void unit_skip_hidden(const PrefillParams& p, Unit& w) {
  if (!kMasked) return;
  const uint4* kb = reinterpret_cast<const uint4*>(p.key_bits) + (size_t)w.b * p.n_kt;
  int js = 0;
  while (js < w.nt0 - 1) {
    const uint4 k = kb[js];
    if ((k.x | k.y | k.z | k.w) != 0u) break;
    ++js;
  }
  w.js = js;
  w.nt0 -= js;
  if (w.nt1 > 0) w.nt1 -= js;  // nt1 >= nt0 whenever tile 1 has rows
  w.n -= js;
}

// kMasked: the 2D padding mask on keys is applied (p.key_bits); a separate instantiation so
// the unmasked kernel carries none of its per-tile work.
template <bool kMasked>
__global__ void __launch_bounds__(kThreads, 1)
    mla_prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sRing = smem + kOffRing;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kfull[i], 1);
      mbar_init(&bars->vfull[i], 1);
      // With the fused append a tile's slots are also read by the cache writers.
      mbar_init(&bars->kempty[i], p.append ? 2 : 1);
      mbar_init(&bars->vempty[i], p.append ? 2 : 1);
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_ready[i], 4);
      mbar_init(&bars->o_done[i], 1);
      mbar_init(&bars->o_free[i], 4);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
    // Out-of-range kv_len is reported once per CTA that meets it (and clamped).
    for (int i = 0;; ++i) {
      const int u = unit_index(p, i);
      if (u < 0) break;
      const int raw = unit_kv(p, u);
      if (raw < 1 || raw > p.Tk) {
        set_status(p.status, MLA_ERR_KVLEN);
        break;
      }
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = bars->tmem_base;

  if (warp < 4) {
    setmaxnreg_dec_control();
    if (warp == 0 && lane == 0) {
      // ================= TMA producer =================
      prefetch_tmap(&p.tm_qn);
      prefetch_tmap(&p.tm_qr);
      prefetch_tmap(&p.tm_kn);
      prefetch_tmap(&p.tm_kr);
      prefetch_tmap(&p.tm_v);
      if (p.append) {
        prefetch_tmap(&p.tm_kn_new);
        prefetch_tmap(&p.tm_kr_new);
        prefetch_tmap(&p.tm_v_new);
      }
      const uint64_t pol_q = l2_policy_evict_first();
      // Sub-tile u goes to slot u % kSlots, whose previous occupant was sub-tile
      // u - kSlots of key tile (u - kSlots) / 5; that tile's K or V group must have been
      // released by the MMAs before the slot is overwritten.
      auto slot_free = [&](uint32_t u) -> bool {
        if (u < (uint32_t)kSlots) return true;
        const uint32_t prev = u - kSlots;
        const uint32_t st = prev / kSubPerKv;
        uint64_t* bar = (prev % kSubPerKv) < 3 ? &bars->kempty[st & 1] : &bars->vempty[st & 1];
        return mbar_wait(bar, (st >> 1) & 1, p.status, abort_flag);
      };
      // Q_t of unit i: sQ_t is free once the previous unit's last score MMA on tile t has
      // run (one q_empty phase per unit).
      auto load_q = [&](int i, int t, const int r0, const int ntt, const int bh) -> bool {
        if (i > 0 && !mbar_wait(&bars->q_empty[t], (i - 1) & 1, p.status, abort_flag))
          return false;
        if (ntt == 0) {
          mbar_arrive(&bars->q_full[t]);  // nothing to load: complete the phase
          return true;
        }
        mbar_arrive_expect_tx(&bars->q_full[t], 3 * kSub);
        const int rt = r0 + t * kBM;
        uint8_t* dst = sQ + t * 3 * kSub;
        tma_load_3d(dst, &p.tm_qn, &bars->q_full[t], 0, rt, bh, pol_q);
        tma_load_3d(dst + kSub, &p.tm_qn, &bars->q_full[t], 64, rt, bh, pol_q);
        tma_load_3d(dst + 2 * kSub, &p.tm_qr, &bars->q_full[t], 0, rt, bh, pol_q);
        return true;
      };
      uint32_t u = 0;   // ring sub-tiles issued over the run
      uint32_t g = 0;   // key tiles issued over the run
      int q_units = 0;  // units whose Q transactions have been posted
      bool ok = true;
      int kv_next = unit_kv(p, unit_index(p, 0));
      for (int i = 0; ok; ++i) {
        const int unit = unit_index(p, i);
        if (unit < 0) break;
        Unit w = unit_make(p, unit, kv_next);
        unit_skip_hidden<kMasked>(p, w);
        kv_next = unit_kv(p, unit_index(p, i + 1));  // fetched a unit ahead
        ok = load_q(i, 0, w.r0, w.nt0, w.bh);
        q_units = i + 1;
        for (int j = 0; j < w.n && ok; ++j, ++g, u += kSubPerKv) {
          // Key tile j + js; with the fused append the tiles past the cached prefix come from
          // the new rows (row 0 of the new rows is key past_len = 128 n_pre).
          const bool from_new = p.append && j + w.js >= p.n_pre;
          const int jt = from_new ? (j + w.js - p.n_pre) * kBN : (j + w.js) * kBN;
          const CUtensorMap* m_kn = from_new ? &p.tm_kn_new : &p.tm_kn;
          const CUtensorMap* m_kr = from_new ? &p.tm_kr_new : &p.tm_kr;
          const CUtensorMap* m_v = from_new ? &p.tm_v_new : &p.tm_v;
          // K(j): no-rope columns 0-63, 64-127 and the shared rotary tile, one barrier.
          uint64_t* kb = &bars->kfull[g & 1];
          for (int s = 0; s < 3 && ok; ++s) {
            ok = slot_free(u + s);
            if (!ok) break;
            if (s == 0) mbar_arrive_expect_tx(kb, 3 * kSub);
            uint8_t* dst = sRing + ((u + s) & (kSlots - 1)) * kSub;
            if (s < 2)
              tma_load_3d_nohint(dst, m_kn, kb, 64 * s, jt, w.bh);
            else
              tma_load_3d_nohint(dst, m_kr, kb, 0, jt, w.b);
          }
          if (!ok) break;
          // Q of the second tile after the first key tile: the first score MMA needs only
          // Q_0 and K(0).
          if (j == 0) {
            ok = load_q(i, 1, w.r0, w.nt1, w.bh);
            if (!ok) break;
          }
          // V(j): columns 0-63 go to the lower-addressed of its two slots, so one MMA with
          // a positive leading-byte offset covers all 128 value columns.
          uint64_t* vb = &bars->vfull[g & 1];
          const uint32_t sa = (u + 3) & (kSlots - 1), sb = (u + 4) & (kSlots - 1);
          ok = slot_free(u + 3) && slot_free(u + 4);
          if (!ok) break;
          mbar_arrive_expect_tx(vb, 2 * kSub);
          tma_load_3d_nohint(sRing + min(sa, sb) * kSub, m_v, vb, 0, jt, w.bh);
          tma_load_3d_nohint(sRing + max(sa, sb) * kSub, m_v, vb, 64, jt, w.bh);
        }
      }
      // Every load this thread issued must land before shared memory is released.  Each
      // barrier has at most one phase in flight (the next one is posted only after the
      // consumer released the previous), so waiting for the last posted phases suffices.
      if (q_units > 0) {
        drain_wait(&bars->q_full[0], (q_units - 1) & 1);
        drain_wait(&bars->q_full[1], (q_units - 1) & 1);
      }
      for (uint32_t k = (g >= 2 ? g - 2 : 0); k < g; ++k) {
        drain_wait(&bars->kfull[k & 1], (k >> 1) & 1);
        drain_wait(&bars->vfull[k & 1], (k >> 1) & 1);
      }
    } else if ((warp == 2 || warp == 3) && lane == 0 && p.append) {
      // ================= cache writers (fused append) =================
      // warp 2: the key sub-tiles of every tile (kfull / kempty), warp 3: the value
      // sub-tiles (vfull / vempty).  Each waits for a tile to land before it releases it,
      // so a release of tile g + 2 implies both releases of tile g (its slots were refilled),
      // and a store's source has been read before the release.  Owner of new key tile m:
      // the unit whose query tile m holds it on its diagonal (query rows 128 m ...), which
      // reads it whenever there is no kv_len; the rotary key (one per sequence) is written
      // by head 0's owner.
      const bool keys = warp == 2;
      uint32_t u = 0, g = 0;
      bool ok = true;
      int kv_next = unit_kv(p, unit_index(p, 0));
      for (int i = 0; ok; ++i) {
        const int unit = unit_index(p, i);
        if (unit < 0) break;
        Unit w = unit_make(p, unit, kv_next);
        unit_skip_hidden<kMasked>(p, w);
        kv_next = unit_kv(p, unit_index(p, i + 1));
        const int qt0 = w.r0 / kBM;  // the unit's first query tile
        for (int j = 0; j < w.n && ok; ++j, ++g, u += kSubPerKv) {
          const int kt = j + w.js;          // key tile
          const int m = kt - p.n_pre;       // new-row tile, if >= 0
          const bool own = m >= 0 && (m == qt0 || m == qt0 + 1) && m * kBM < p.Tq;
          uint64_t* full = keys ? &bars->kfull[g & 1] : &bars->vfull[g & 1];
          ok = mbar_wait(full, (g >> 1) & 1, p.status, abort_flag);
          if (!ok) break;
          if (own) {
            fence_proxy_async_smem();
            if (keys) {
              for (int s = 0; s < 2; ++s)
                tma_store_3d(&p.tm_kn_st, sRing + ((u + s) & (kSlots - 1)) * kSub, 64 * s,
                             kt * kBN, w.bh);
              if (w.bh % p.H == 0)
                tma_store_3d(&p.tm_kr_st, sRing + ((u + 2) & (kSlots - 1)) * kSub, 0,
                             kt * kBN, w.b);
            } else {
              const uint32_t sa = (u + 3) & (kSlots - 1), sb = (u + 4) & (kSlots - 1);
              tma_store_3d(&p.tm_v_st, sRing + min(sa, sb) * kSub, 0, kt * kBN, w.bh);
              tma_store_3d(&p.tm_v_st, sRing + max(sa, sb) * kSub, 64, kt * kBN, w.bh);
            }
            bulk_commit_group();
            bulk_wait_read_all();
          }
          mbar_arrive(keys ? &bars->kempty[g & 1] : &bars->vempty[g & 1]);
        }
      }
      bulk_wait_all();  // the cache rows are written before the kernel ends
    } else if (warp == 1) {
      // ================= MMA issuer =================
      // The whole warp runs this loop (waits, descriptor arithmetic: warp-uniform values);
      // one elected lane issues each batch of MMAs and commits.  Descriptors are built once
      // (their high word is constant) and per MMA only the start-address field moves.
      constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(128, 128, false);
      constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(128, 128, true);
      constexpr uint32_t kSubLo = kSub >> 4;  // one sub-tile in descriptor address units
      // K-major operands: leading offset unused, 8-row groups 1024 B apart.  V (MN-major):
      // the two 64-column halves are one slot apart, or kSlots - 1 slots when the pair
      // wraps around the ring; 8-key groups 1024 B apart.
      const uint64_t dhi_k = tc::smem_desc_sw128(0, 16, 1024);
      const uint64_t dhi_v_near = tc::smem_desc_sw128(0, kSub, 1024);
      const uint64_t dhi_v_far = tc::smem_desc_sw128(0, (kSlots - 1) * kSub, 1024);
      const uint32_t q_lo = smem_u32(sQ) >> 4;
      const uint32_t ring_lo = smem_u32(sRing) >> 4;
      uint32_t g = 0;             // key tiles consumed over the run
      uint32_t stp[2] = {0, 0};   // value mixes issued per tile over the run
      bool ok = true;
      int kv_next = unit_kv(p, unit_index(p, 0));
      for (int i = 0; ok; ++i) {
        const int unit = unit_index(p, i);
        if (unit < 0) break;
        Unit w = unit_make(p, unit, kv_next);
        unit_skip_hidden<kMasked>(p, w);
        kv_next = unit_kv(p, unit_index(p, i + 1));  // fetched a unit ahead
        for (int j = 0; j <= w.n && ok; ++j) {
          const uint32_t gk = g + (uint32_t)j;           // key tile j of this unit
          const uint32_t uk = gk * kSubPerKv;            // its sub-tiles: uk .. uk+2
          const uint32_t uv = uk - 2u;                   // sub-tiles of V(j-1): uv, uv+1
          uint32_t klo[3];
#pragma unroll
          for (int s = 0; s < 3; ++s) klo[s] = ring_lo + ((uk + s) & (kSlots - 1)) * kSubLo;
          const uint32_t va = uv & (kSlots - 1), vb2 = (uv + 1) & (kSlots - 1);
          const uint32_t vlo = ring_lo + min(va, vb2) * kSubLo;
          const uint64_t dhi_v = vb2 > va ? dhi_v_near : dhi_v_far;
          // V(j-1) first: the value mix of tile 0 can start while K(j) is still landing.
          if (j > 0)
            ok = mbar_wait(&bars->vfull[(gk - 1) & 1], ((gk - 1) >> 1) & 1, p.status,
                           abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc::fence_after_sync();
          bool k_landed = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t s_tmem = tbase + t * 128;
            const uint32_t o_tmem = tbase + 256 + t * 128;
            if (j > 0 && j - 1 < w.nt(t)) {
              // O_t += P_t(j-1) V(j-1): P from TMEM (aliasing S_t), V MN-major from smem.
              ok = mbar_wait(&bars->p_ready[t], stp[t] & 1, p.status, abort_flag);
              // The unit's first value mix overwrites O_t: the previous unit's O_t must
              // have been read out.
              if (ok && j == 1 && i > 0)
                ok = mbar_wait(&bars->o_free[t], (i - 1) & 1, p.status, abort_flag);
              ok = __all_sync(0xffffffffu, ok);
              if (!ok) break;
              tc::fence_after_sync();
              const uint32_t acc0 = (j > 1) ? 1u : 0u;
              if (tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint64_t bdesc = dhi_v | (uint64_t)(vlo + kk * (2048 >> 4));
                  tc::mma_ts(o_tmem, s_tmem + kk * 8, bdesc, kIdescPV, kk > 0 ? 1u : acc0);
                }
                if (j - 1 == w.nt(t) - 1) tc::commit(&bars->o_done[t]);
              }
              __syncwarp();
              ++stp[t];
            }
            if (t == 1 && j > 0) {
              // V(j-1) is no longer needed once both value mixes have run.
              if (tc::elect_one()) tc::commit(&bars->vempty[(gk - 1) & 1]);
              __syncwarp();
            }
            if (j < w.nt(t)) {
              if (j == 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bars->q_full[t], i & 1, p.status, abort_flag));
                if (!ok) break;
              }
              if (!k_landed) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bars->kfull[gk & 1], (gk >> 1) & 1,
                                                       p.status, abort_flag));
                if (!ok) break;
                k_landed = true;
              }
              tc::fence_after_sync();
              // S_t = Q_t K(j)^T over 192 columns: 4 k-steps per 64-column sub-tile.
              const uint32_t qlo = q_lo + t * 3 * kSubLo;
              if (tc::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 12; ++kk) {
                  const uint32_t koff = (kk & 3) * (32 >> 4);
                  const uint64_t adesc = dhi_k | (uint64_t)(qlo + (kk >> 2) * kSubLo + koff);
                  const uint64_t bdesc = dhi_k | (uint64_t)(klo[kk >> 2] + koff);
                  tc::mma_ss(s_tmem, adesc, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars->s_full[t]);
                if (j == w.nt(t) - 1) tc::commit(&bars->q_empty[t]);
              }
              __syncwarp();
            }
          }
          if (!ok) break;
          if (j < w.n) {
            if (tc::elect_one()) tc::commit(&bars->kempty[gk & 1]);
            __syncwarp();
          }
        }
        if (!ok) break;
        // A tile with no rows in this unit still completes its per-unit phases.
        if (w.nt1 == 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full[1], i & 1, p.status, abort_flag));
          if (!ok) break;
          if (tc::elect_one()) {
            tc::commit(&bars->q_empty[1]);
            tc::commit(&bars->o_done[1]);
          }
          __syncwarp();
        }
        g += (uint32_t)w.n;
      }
      // No MMA may still be running when TMEM is released.
      if (tc::elect_one()) tc::commit(&bars->mma_done);
      __syncwarp();
      drain_wait(&bars->mma_done, 0);
    }
    __syncwarp();
  } else {
    // ================= softmax warpgroups =================
    setmaxnreg_inc_softmax();
    const int t = (warp >> 2) - 1;  // query tile 0 or 1
    const int tw = threadIdx.x - 128 * (t + 1);
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tmem = tbase + lane_off + t * 128;
    const uint32_t o_tmem = tbase + lane_off + 256 + t * 128;
    const float sl2 = p.scale_log2;
    uint32_t st = 0;  // score steps of this tile over the run
    bool ok = true;
    int kv_next = unit_kv(p, unit_index(p, 0));
    for (int i = 0; ok; ++i) {
      const int unit = unit_index(p, i);
      if (unit < 0) break;
      Unit w = unit_make(p, unit, kv_next);
      unit_skip_hidden<kMasked>(p, w);
      kv_next = unit_kv(p, unit_index(p, i + 1));  // fetched a unit ahead
      const int ntt = w.nt(t);
      const int qi = w.r0 + t * kBM + tw;  // query row within the sequence
      const int limit = min(qi + p.past_len + 1, w.kvl);  // keys [0, limit) are visible
      float m = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < ntt; ++j, ++st) {
        // 2D padding mask bits of this key tile (same for every row of the CTA), fetched
        // before the wait so the load overlaps it.
        uint4 kbits = make_uint4(~0u, ~0u, ~0u, ~0u);
        if (kMasked)
          kbits = *reinterpret_cast<const uint4*>(p.key_bits +
                                                  ((size_t)w.b * p.n_kt + j + w.js) * 4);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], st & 1, p.status, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        uint32_t r[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tc::tmem_ld32(s_tmem + c * 32, r[c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) pin32(r[c]);

        const int jt = (j + w.js) * kBN;
        if (jt + kBN > limit) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (jt + c * 32 + e >= limit) r[c][e] = __float_as_uint(-INFINITY);
        }
        if (kMasked && (kbits.x & kbits.y & kbits.z & kbits.w) != ~0u) {
          const uint32_t kw[4] = {kbits.x, kbits.y, kbits.z, kbits.w};
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!((kw[c] >> e) & 1u)) r[c][e] = __float_as_uint(-INFINITY);
        }
        // Row max: 8 independent chains of three-input maxima (64 instructions for 128
        // scores; a single 128-long chain would be latency-bound).
        float mxp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mxp[k] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            mxp[(e >> 1) & 7] = fmax3(mxp[(e >> 1) & 7], __uint_as_float(r[c][e]),
                                      __uint_as_float(r[c][e + 1]));
        const float mx = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]),
                               fmaxf(mxp[6], mxp[7]));
        const float m_tile = mx * sl2;
        if (j == 0) {
          m = m_tile;
        } else {
          const bool need = m_tile > m + kRescaleThreshold;
          if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2_approx(m - m_tile) : 1.0f;
            if (need) {
              m = m_tile;
              l *= alpha;
            }
            // 16 columns at a time in a loop that is not unrolled: this rare branch runs
            // while the tile's 128 scores are live, and wider or unrolled chunks made the
            // softmax spill registers (3% on the long prefill).
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t o[16];
              tc::tmem_ld16(o_tmem + c * 16, o);
              tc::tmem_wait_ld();
              pin<16>(o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tc::tmem_st16(o_tmem + c * 16, o);
            }
          }
        }
        // p = 2^(s * scale * log2(e) - m): the scale-and-subtract and the row sum run on
        // fp32 pairs (one instruction per two scores), the exponentials on the MUFU.
        // While every key so far is hidden (only under a 2D padding mask) the running max is
        // -inf; exponents are then taken against 0, giving exactly 0 for hidden keys.
        const float m_base = (kMasked && m == -INFINITY) ? 0.f : m;
        const uint64_t sl2_2 = f2_pack(sl2, sl2);
        const uint64_t negm_2 = f2_pack(-m_base, -m_base);
        uint64_t sp2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t xv = ffma2(
                f2_pack(__uint_as_float(r[c][e]), __uint_as_float(r[c][e + 1])), sl2_2, negm_2);
            float x0, x1;
            f2_unpack(xv, x0, x1);
            x0 = ex2_approx(x0);
            x1 = ex2_approx(x1);
            sp2[(e >> 1) & 3] = fadd2(sp2[(e >> 1) & 3], f2_pack(x0, x1));
            pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16x2(x0, x1);
          }
        }
        float sa, sb;
        f2_unpack(fadd2(fadd2(sp2[0], sp2[1]), fadd2(sp2[2], sp2[3])), sa, sb);
        l += sa + sb;
        tc::tmem_st32(s_tmem, pk[0]);
        tc::tmem_st32(s_tmem + 32, pk[1]);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
#ifdef MLA_TEST_DROP_P_READY
        // Test build only: the first softmax warp of CTA 0 withholds its P-ready arrival on
        // the second key tile of its first unit.  The MMA warp's bounded wait for it then
        // gives up, which exercises the timeout report and the CTA's unwinding (no copy or
        // MMA left in flight, TMEM released).  The arrival carries no transaction bytes.
        const bool withhold = blockIdx.x == 0 && i == 0 && j == 1 && warp == 4;
#else
        constexpr bool withhold = false;
#endif
        if (lane == 0 && !withhold) mbar_arrive(&bars->p_ready[t]);
      }
      if (!ok) break;
      // The unit's output: wait for the last value mix, move O_t to registers, release
      // O_t for the next unit, then normalise and store.
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_done[t], i & 1, p.status, abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      if (ntt == 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->o_free[t]);
        continue;
      }
      uint32_t o[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(o_tmem + c * 32, o[c]);
      tc::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) pin32(o[c]);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[t]);
      // l = 0 only when the 2D padding mask hides every key of the row; that row is
      // rewritten afterwards as the mean of all value rows.
      const float inv = l > 0.f ? 1.0f / l : 0.f;
      if (qi < p.Tq) {
        uint16_t* row = p.out + ((size_t)w.bh * p.Tq + qi) * 128;
        auto pk = [&](int c, int e) {
          return pack_bf16x2(__uint_as_float(o[c][e]) * inv, __uint_as_float(o[c][e + 1]) * inv);
        };
        if ((reinterpret_cast<uintptr_t>(p.out) & 31u) == 0) {
          // 32-byte stores: each fills one whole sector of the row.
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const int e = v * 16;
              asm volatile(
                  "st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                      row + c * 32 + e),
                  "r"(pk(c, e)), "r"(pk(c, e + 2)), "r"(pk(c, e + 4)), "r"(pk(c, e + 6)),
                  "r"(pk(c, e + 8)), "r"(pk(c, e + 10)), "r"(pk(c, e + 12)), "r"(pk(c, e + 14))
                  : "memory");
            }
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(row);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 q;
              q.x = pk(c, v * 8 + 0);
              q.y = pk(c, v * 8 + 2);
              q.z = pk(c, v * 8 + 4);
              q.w = pk(c, v * 8 + 6);
              dst[c * 4 + v] = q;
            }
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, 512);
  }
}

// ---- host side: tensor maps and launch -------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// bf16 tensor viewed as {inner, rows, planes} (planes plane_rows rows apart) with 128-byte
// swizzled {64, 128, 1} boxes; rows past `rows` read as zeros.
bool encode_3d(EncodeTiledFn fn, CUtensorMap* m, const void* base, uint64_t inner,
               uint64_t rows, uint64_t planes, uint64_t plane_rows) {
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner * 2, inner * 2 * plane_rows};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host-side cache of encoded tensor maps, keyed by the five input pointers and the sizes:
// a serving loop calls the same buffers over and over, and encoding costs microseconds.
struct MapKey {
  const void* ptr[8];  // q_nope, q_pe, k_nope, k_pe, v, then the new rows (append only)
  int B, H, Tq, Tk, kv_rows;
  bool operator==(const MapKey& o) const {
    for (int i = 0; i < 8; ++i)
      if (ptr[i] != o.ptr[i]) return false;
    return B == o.B && H == o.H && Tq == o.Tq && Tk == o.Tk && kv_rows == o.kv_rows;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap maps[11];
  bool valid;
};
constexpr int kMapCacheSize = 16;
std::mutex g_map_mu;
MapEntry g_map_cache[kMapCacheSize];
int g_map_next = 0;

bool tensor_maps(const PrefillArgs& a, PrefillParams* p) {
  const MapKey key = {{a.q_nope, a.q_pe, a.k_nope, a.k_pe, a.v, a.new_k_nope, a.new_k_pe,
                       a.new_v},
                      a.B, a.H, a.Tq, a.Tk, a.kv_rows};
  CUtensorMap* dst[11] = {&p->tm_qn,     &p->tm_qr,     &p->tm_kn,    &p->tm_kr,
                          &p->tm_v,      &p->tm_kn_new, &p->tm_kr_new, &p->tm_v_new,
                          &p->tm_kn_st,  &p->tm_kr_st,  &p->tm_v_st};
  const int n_maps = a.new_k_nope ? 11 : 5;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (const MapEntry& e : g_map_cache) {
      if (e.valid && e.key == key) {
        for (int k = 0; k < n_maps; ++k) *dst[k] = e.maps[k];
        return true;
      }
    }
  }
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const uint64_t BH = (uint64_t)a.B * a.H;
  if (!encode_3d(fn, &p->tm_qn, a.q_nope, 128, a.Tq, BH, a.Tq) ||
      !encode_3d(fn, &p->tm_qr, a.q_pe, 64, a.Tq, BH, a.Tq) ||
      !encode_3d(fn, &p->tm_kn, a.k_nope, 128, a.Tk, BH, a.kv_rows) ||
      !encode_3d(fn, &p->tm_kr, a.k_pe, 64, a.Tk, a.B, a.kv_rows) ||
      !encode_3d(fn, &p->tm_v, a.v, 128, a.Tk, BH, a.kv_rows))
    return false;
  if (a.new_k_nope) {
    // New rows [B,H,Tq,*] / [B,Tq,64]; the stores go to the caches' rows [0, Tk) (the
    // maps clip a tile's rows past Tk).
    if (!encode_3d(fn, &p->tm_kn_new, a.new_k_nope, 128, a.Tq, BH, a.Tq) ||
        !encode_3d(fn, &p->tm_kr_new, a.new_k_pe, 64, a.Tq, a.B, a.Tq) ||
        !encode_3d(fn, &p->tm_v_new, a.new_v, 128, a.Tq, BH, a.Tq) ||
        !encode_3d(fn, &p->tm_kn_st, a.k_nope, 128, a.Tk, BH, a.kv_rows) ||
        !encode_3d(fn, &p->tm_kr_st, a.k_pe, 64, a.Tk, a.B, a.kv_rows) ||
        !encode_3d(fn, &p->tm_v_st, a.v, 128, a.Tk, BH, a.kv_rows))
      return false;
  }
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry& e = g_map_cache[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCacheSize;
  e.key = key;
  for (int k = 0; k < n_maps; ++k) e.maps[k] = *dst[k];
  e.valid = true;
  return true;
}

}  // namespace

// Cache append for Tq > 1 (the cache update of the attention excerpt: the new rows follow
// the cached prefix).  One thread per 16-byte chunk; rows of k_nope / v are 16 chunks, rows
// of the shared rotary key 8.
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const size_t bh_rows = (size_t)a.B * a.H * a.Tq;  // k_nope and v rows
  const size_t pe_rows = (size_t)a.B * a.Tq;        // k_pe rows
  const size_t n16 = bh_rows * 16 * 2 + pe_rows * 8;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x) {
    if (i < bh_rows * 32) {
      const bool is_v = i >= bh_rows * 16;
      const size_t k = is_v ? i - bh_rows * 16 : i;
      const size_t row = k >> 4, c = k & 15;      // row = (b*H + h)*Tq + t
      const size_t bh = row / a.Tq, t = row % a.Tq;
      const uint4* src = reinterpret_cast<const uint4*>((is_v ? a.new_v : a.new_k_nope) + row * 128);
      uint4* dst = reinterpret_cast<uint4*>((is_v ? a.cache_v : a.cache_k_nope) +
                                            (bh * a.kv_rows + a.past_len + t) * 128);
      dst[c] = src[c];
    } else {
      const size_t k = i - bh_rows * 32;
      const size_t row = k >> 3, c = k & 7;       // row = b*Tq + t
      const size_t b = row / a.Tq, t = row % a.Tq;
      reinterpret_cast<uint4*>(a.cache_k_pe + (b * a.kv_rows + a.past_len + t) * 64)[c] =
          reinterpret_cast<const uint4*>(a.new_k_pe + row * 64)[c];
    }
  }
}

cudaError_t launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
  const size_t n16 = (size_t)a.B * a.H * a.Tq * 32 + (size_t)a.B * a.Tq * 8;
  const int sms = device_sm_count();
  const size_t blocks = std::min<size_t>((n16 + 255) / 256, (size_t)(sms > 0 ? sms : 152) * 8);
  kv_append_kernel<<<(unsigned)std::max<size_t>(blocks, 1), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

bool encode_bf16_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t planes, uint64_t plane_rows, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, planes};
  cuuint64_t strides[2] = {inner * 2, inner * 2 * plane_rows};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_tiled(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d,
            st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  PrefillParams p{};
  if (!tensor_maps(a, &p)) return cudaErrorInvalidValue;
  const uint64_t BH = (uint64_t)a.B * a.H;
  p.kv_len = a.kv_len;
  p.key_bits = a.key_bits;
  p.n_kt = (a.Tk + kBN - 1) / kBN;
  p.out = a.out;
  p.status = a.status;
  p.B = a.B;
  p.H = a.H;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.past_len = a.past_len;
  p.append = a.new_k_nope != nullptr ? 1 : 0;
  p.n_pre = a.past_len / kBN;
  if (p.append && (a.past_len % kBN != 0 || a.kv_len != nullptr || a.key_bits != nullptr))
    return cudaErrorInvalidValue;
  p.n_qb = (a.Tq + 2 * kBM - 1) / (2 * kBM);
  p.scale_log2 = a.scale_log2;
  const uint64_t units = BH * (uint64_t)p.n_qb;
  if (units > 0x7fffffffull) return cudaErrorInvalidValue;

  static std::atomic<uint64_t> attr_done{0};  // bit per device: smem attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(mla_prefill_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(mla_prefill_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  // Persistent: one CTA per SM (at most one per unit), each walking its units.
  const int sms = device_sm_count();
  const uint64_t grid = std::min<uint64_t>(units, (uint64_t)(sms > 0 ? sms : 152));
  if (p.key_bits)
    mla_prefill_kernel<true><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(p);
  else
    mla_prefill_kernel<false><<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
