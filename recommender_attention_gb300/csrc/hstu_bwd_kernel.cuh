// Backward of the HSTU attention forward for sm_103a: the gradients dQ, dK, dV
// of the forward's output for an output gradient dO (the exact derivative of
// the forward in composable_kernel 18_hstu_attention README, "Forward
// computation"; its training mode saves the softmax LSE for this pass).
//
// With s = alpha Q K^T, the mask M, c = attn_scale and g = dO:
//   SiLU:     a = M . SiLU(s)                  dV = c a^T g
//             dS = M . (c g V^T) . SiLU'(s)    (SiLU'(x) = sig(x) (1 + x (1 - sig(x))))
//   softmax:  p = M . exp(s - lse)             dV = c p^T g
//             dS = p . (c g V^T - delta),  delta = rowsum(g . O)
//   both:     dQ = alpha dS K,  dK = alpha dS^T Q
//
// Two persistent kernels with one warp of TMA loads (which also claims work
// units from a global counter, longest first, and publishes them to the other
// roles through a two-slot ring), one MMA warp (the whole warp runs the loop,
// one elected lane issues) and two elementwise warpgroups.  Work goes in half
// tiles of 64 columns with two or three TMEM buffers, so the tensor core
// computes the next half tiles' score products while the elementwise warps
// process the current one:
//   dQ kernel, one unit per (sequence, head, query tile): for every key tile of
//     the tile's set and each half of it, S = Q K_h^T and dP = dO V_h^T (N = 64)
//     into buffer t % (DQ_LAG + 1), dS (16-bit) packed over S, dQ += dS K_h
//     with K read MN-major from its tile, issued DQ_LAG half tiles behind the
//     score products (K and V in rings of their own); the elementwise warps
//     then scale dQ by alpha.
//   dK/dV kernel, one unit per (sequence, head, key tile): for every query tile
//     whose key-tile set holds this key tile (a bit word per 32 query tiles,
//     written by the scheduler) and each half of it, S^T = K Q_h^T and
//     dP^T = V dO_h^T, P^T and dS^T packed over them, dV += P^T dO_h and
//     dK += dS^T Q_h with dO and Q read MN-major; then dV * attn_scale and
//     dK * alpha.
// TMEM: buffer b at columns [128 b, 128 b + 128) (scores, then the score
// gradients at +64), accumulators after the buffers (dQ kernel: from column
// 128 (DQ_LAG + 1); dK/dV kernel: from column 256).  Query tiles follow the
// forward's layout (q_layout): context rows may sit on the top lanes of a
// sequence's last query tile, and that tile's Q and dO then arrive as 8-row
// TMA boxes.  Every wait is bounded (2 s); a timeout sets the device error word
// and every role stops.
#pragma once
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"
#include "hstu_rab.cuh"

namespace hstu {

constexpr int kBwdThreads = 320;   // producer, MMA, two elementwise warpgroups
constexpr int kHalf = 64;          // columns of a half tile
constexpr int kHalfBytes = kHalf * 128;   // rows of a half tile inside a 128-row swizzled chunk

template <int D, int DV, bool RAB = false>
struct BwdCfg {
  static constexpr int KCH = (D + 63) / 64;
  static constexpr int VCH = (DV + 63) / 64;
  static constexpr int CHUNK = kBlockN * 128;   // one 128-row x 128-byte swizzle box
  static constexpr int TQ = KCH * CHUNK;        // a Q or K tile
  static constexpr int TV = VCH * CHUNK;        // a V or dO tile
  static constexpr int STAGES = 2;             // dK/dV kernel: the Q + dO ring
  static constexpr int RAB_OFFSET = (TQ + TV) * (1 + STAGES);   // relative attention bias tables, per warp
  // then, per elementwise warp, the gradients of the bias tables over a unit (dQ kernel)
  static constexpr int RAB_GRAD_OFFSET = RAB_OFFSET + (RAB ? 8 * static_cast<int>(sizeof(RabWarp)) : 0);
  static constexpr int SMEM_BYTES = RAB_GRAD_OFFSET + (RAB ? 8 * static_cast<int>(sizeof(RabGradWarp)) : 0) + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t ACC = 256;          // first accumulator column (dK/dV kernel)
  static_assert(D % 32 == 0 && DV % 32 == 0 && ACC + D + DV <= TMEM_COLS, "backward head dimensions");
  // dQ kernel: the dQ product of half tile i is issued after the score
  // products of half tile i + DQ_LAG, so the elementwise pass of a half tile
  // has DQ_LAG half tiles of tensor work to hide behind.  That takes
  // DQ_LAG + 1 score buffers in TMEM and DQ_LAG + 1 stages in the K ring (K
  // feeds the dQ product too); V, read by the score products only, has a ring
  // of its own.  With the bias, whose tables take the third K stage's room,
  // DQ_LAG is 1.
  static constexpr int DQ_LAG = RAB ? 1 : 2;
  static constexpr int DQ_BUFS = DQ_LAG + 1;
  static constexpr int DQ_KST = DQ_LAG + 1;
  static constexpr int DQ_VST = 2;
  static constexpr uint32_t DQ_ACC = 128u * DQ_BUFS;   // dQ accumulator's first column
  static constexpr int DQ_TILES_BYTES = TQ + TV + DQ_KST * TQ + DQ_VST * TV;
  static constexpr int DQ_SMEM_BYTES = RAB ? SMEM_BYTES : DQ_TILES_BYTES + 1024;
  static_assert(DQ_ACC + D <= TMEM_COLS && DQ_BUFS <= 3, "dQ kernel TMEM");
  static_assert(!RAB || DQ_TILES_BYTES == RAB_OFFSET, "the bias tables follow the dQ kernel's rings");
};

constexpr int kBwdEwWarps = 8;

struct BwdCtl {
  uint64_t one_full, one_empty;           // dQ kernel: Q + dO of the unit; dK/dV kernel: K + V
  uint64_t ring_full[2], ring_empty[2];   // dK/dV kernel: Q + dO per query tile
  uint64_t k_full[3], k_empty[3];         // dQ kernel: K per key tile
  uint64_t v_full[2], v_empty[2];         // dQ kernel: V per key tile
  uint64_t s_full[3], p_full[3];          // per TMEM buffer: score products ready / 16-bit operands written
  uint64_t acc_full, acc_empty;           // accumulators complete / read out
  uint64_t sched_full[2], sched_empty[2];   // claimed units: published by the producer / taken by all
  int sched[2];                             // unit index, or -1 after the last
  uint32_t tmem_base;
  volatile int abort_flag;
};

// dK/dV elementwise warps: per warp, its 32 query columns' softmax statistics
// (lse in log2 units, delta / attn_scale) and allowed key intervals (lo, hi,
// diagonal key), read back as broadcasts
struct BwdColInfo {
  int4 col_rng[kBwdEwWarps][32];
  alignas(16) float2 col_stat[kBwdEwWarps][32];   // read two columns at a time as float4
};

__device__ __forceinline__ bool bwd_wait(BwdCtl& ctl, const BwdParams& p, uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_wait(bar, parity, kWaitLimitNs)) return true;
  ctl.abort_flag = 1;
  atomicOr(&p.ws_header[kWsError], kErrTimeout);
  return false;
}
__device__ __forceinline__ bool bwd_warp_wait(BwdCtl& ctl, const BwdParams& p, uint64_t* bar, uint32_t parity) {
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, kWaitLimitNs));
  if (!ok) {
    ctl.abort_flag = 1;
    atomicOr(&p.ws_header[kWsError], kErrTimeout);
  }
  return ok;
}

struct BwdUnit {
  SeqGeom s;
  QLayout L;
  int b, t, h, g;   // t: query tile (dQ kernel) or key tile (dK/dV kernel)
  float scale;
};
__device__ __forceinline__ BwdUnit decode_bwd_unit(const BwdParams& p, int4 w) {
  BwdUnit u;
  u.b = w.x;
  u.t = w.y;
  u.h = w.z;
  u.g = u.b / p.batch_per_group;
  u.s = make_geom(p.off_q, p.off_kv, p.targets, u.b, p.ctx[u.g], p.loc[u.g], p.mf[u.g], p.causal,
                  p.self_attn, p.kv_targets);
  u.L = q_layout(u.s);
  u.scale = p.group_scale[u.g];
  return u;
}

// Producer: claims the next unit from the global counter and publishes its
// index (-1 once the queue is drained) into the ring.
__device__ __forceinline__ bool sched_publish(BwdCtl& ctl, const BwdParams& p, int* counter, int n_units,
                                              int& s_it, int& ui) {
  const int slot = s_it & 1;
  if (!bwd_wait(ctl, p, &ctl.sched_empty[slot], ((s_it >> 1) & 1) ^ 1)) return false;
  const int x = atomicAdd(counter, 1);
  ui = x < n_units ? x : -1;
  ctl.sched[slot] = ui;
  ptx::mbar_arrive(&ctl.sched_full[slot]);
  ++s_it;
  return true;
}
// MMA and elementwise warps: the next published unit (-1: none left).
__device__ __forceinline__ bool sched_take(BwdCtl& ctl, const BwdParams& p, int lane, int& s_it, int& ui) {
  const int slot = s_it & 1;
  if (!bwd_warp_wait(ctl, p, &ctl.sched_full[slot], (s_it >> 1) & 1)) return false;
  ui = *reinterpret_cast<volatile int*>(&ctl.sched[slot]);
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(&ctl.sched_empty[slot]);
  ++s_it;
  return true;
}

// Member words of a key-tile unit: bit m % 32 of word m / 32 is query tile m.
struct MemberWords {
  const unsigned* w;
  int n;   // words
};
__device__ __forceinline__ MemberWords member_words(const BwdParams& p, const BwdUnit& u) {
  MemberWords mw;
  mw.n = (u.L.nq + 31) / 32;
  mw.w = p.kv_mask + p.kv_mask_base[u.b] + static_cast<long long>(u.t) * mw.n;
  return mw;
}
__device__ __forceinline__ int member_count(const MemberWords& mw) {
  int c = 0;
  for (int i = 0; i < mw.n; ++i) c += __popc(mw.w[i]);
  return c;
}

// Full-tile bounds of query tile m of sequence b, as the scheduler recorded them.
__device__ __forceinline__ TileBounds load_qtile_bounds(const BwdParams& p, int b, int m) {
  const int* r = p.qtiles + static_cast<long long>(p.qtile_base[b] + m) * kQTileInts;
  const int4 c = *reinterpret_cast<const int4*>(r + 4);
  const int4 d = *reinterpret_cast<const int4*>(r + 8);
  TileBounds tb;
  tb.LO = c.w;
  tb.HI = d.x;
  tb.maxLO = d.y;
  tb.minHI = d.z;
  return tb;
}

// TMA of a query-side tile (Q or dO) of query tile m in the forward's lane layout.
__device__ __forceinline__ void load_query_tile(const CUtensorMap* m128, const CUtensorMap* m8, uint8_t* dst,
                                                uint64_t* bar, const SeqGeom& s, const QLayout& L, int m,
                                                int x0, int nchunks) {
  const int qrow = m * kBlockM;
  if (!(L.ctx_lane0 >= 0 && m == L.nq - 1)) {
    for (int kc = 0; kc < nchunks; ++kc)
      ptx::tma_load_2d(dst + kc * (kBlockN * 128), m128, bar, x0 + kc * 64, s.q0 + qrow);
  } else {
    for (int g = 0; g < kBlockM / 8; ++g) {
      const int row = g * 8 < L.ctx_lane0 ? qrow + g * 8 : (g * 8 - L.ctx_lane0);
      for (int kc = 0; kc < nchunks; ++kc)
        ptx::tma_load_2d(dst + kc * (kBlockN * 128) + g * 1024, m8, bar, x0 + kc * 64, s.q0 + row);
    }
  }
}

// C[tmem] = A B^T over KS k-steps: A a 128-row tile, B 64 rows starting at
// b_base (a half of a 128-row tile), both K-major 128-byte-swizzled chunks.
template <int KS>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
  const uint64_t ad0 = ptx::sdesc_sw128(a_base, 16, 1024), bd0 = ptx::sdesc_sw128(b_base, 16, 1024);
  auto off = [](int ks) { return static_cast<uint64_t>(((ks >> 2) * (kBlockN * 128) + (ks & 3) * 32) >> 4); };
#pragma unroll
  for (int g = 0; g + 8 <= KS; g += 8) {
    uint64_t ad[8], bd[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { ad[j] = ad0 + off(g + j); bd[j] = bd0 + off(g + j); }
    ptx::umma_ss_x8(d_tmem, ad, bd, idesc, g > 0 ? 1u : 0u);
  }
  if constexpr (KS % 8 >= 4) {
    constexpr int g = KS / 8 * 8;
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) { ad[j] = ad0 + off(g + j); bd[j] = bd0 + off(g + j); }
    ptx::umma_ss_x4(d_tmem, ad, bd, idesc, g > 0 ? 1u : 0u);
  }
#pragma unroll
  for (int ks = KS / 4 * 4; ks < KS; ++ks)   // hdim 96: the last two k-steps
    ptx::umma_ss(d_tmem, ad0 + off(ks), bd0 + off(ks), idesc, ks > 0 ? 1u : 0u);
}
// C[tmem] (+)= A B over one half tile: A (128 x 64, 16-bit) packed in TMEM by
// the elementwise warps (warpgroup w's 32 columns at a_tmem + 32 w, 16 columns
// each), B 64 rows of a tile from b_base read MN-major (K = its rows).
__device__ __forceinline__ void mma_half_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, uint32_t idesc,
                                            bool accumulate) {
  const uint64_t bd0 = ptx::sdesc_sw128(b_base, kBlockN * 128, 1024);
  uint32_t pa[4];
  uint64_t bd[4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    pa[kk] = a_tmem + (kk >> 1) * 32 + (kk & 1) * 8;
    bd[kk] = bd0 + static_cast<uint64_t>((kk * 2048) >> 4);
  }
  ptx::umma_ts_x4(d_tmem, pa, bd, idesc, accumulate ? 1u : 0u);
}

// SiLU and its derivative for the 32 scores of one row, in fp32 (packed f32x2
// products, tanh.approx.f32 per element): with h = alpha s / 2, t = tanh(h),
// sig = (1 + t) / 2, SiLU(x) = h (1 + t) and SiLU'(x) = sig + SiLU(x) (1 - sig).
// pa receives SiLU(x) (when WANT_A), pr receives dp * SiLU'(x), each rounded
// once to the storage type; pairs whose bit in `allow` is clear give 0
// (MASKED).  PRESCALED: sv already holds h (with a relative attention bias,
// alpha s / 2 + rab / 2).  ds_f32 (optional) receives dp * SiLU'(x) in fp32.
template <bool BF16, bool WANT_A, bool MASKED, bool PRESCALED = false>
__device__ __forceinline__ void silu_bwd_f32(const uint32_t (&sv)[32], const uint32_t (&dv)[32], float half_alpha,
                                             uint32_t allow, uint32_t (&pa)[16], uint32_t (&pr)[16],
                                             float* ds_f32 = nullptr) {
  const uint64_t ha = ptx::f32x2(half_alpha, half_alpha);
  const uint64_t half = ptx::f32x2(0.5f, 0.5f), neg_half = ptx::f32x2(-0.5f, -0.5f);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    uint64_t h = ptx::f32x2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]));
    if constexpr (!PRESCALED) h = ptx::mul_f32x2(h, ha);
    float h0, h1;
    ptx::f32x2_split(h, h0, h1);
    const uint64_t t = ptx::f32x2(ptx::tanh_approx(h0), ptx::tanh_approx(h1));
    const uint64_t sg = ptx::fma_f32x2(t, half, half);        // sig
    const uint64_t a = ptx::fma_f32x2(h, t, h);               // SiLU(x)
    const uint64_t om = ptx::fma_f32x2(t, neg_half, half);    // 1 - sig
    const uint64_t d = ptx::fma_f32x2(a, om, sg);             // SiLU'(x)
    const uint64_t g = ptx::f32x2(__uint_as_float(dv[2 * k]), __uint_as_float(dv[2 * k + 1]));
    uint32_t a16 = 0;
    if constexpr (WANT_A) a16 = ptx::cvt_pack16<BF16>(a);
    const uint64_t r32 = ptx::mul_f32x2(g, d);
    uint32_t r16 = ptx::cvt_pack16<BF16>(r32);
    if (ds_f32 != nullptr) {   // the fp32 values too (masked: 0)
      float r0, r1;
      ptx::f32x2_split(r32, r0, r1);
      ds_f32[2 * k] = (!MASKED || ((allow >> (2 * k)) & 1u)) ? r0 : 0.f;
      ds_f32[2 * k + 1] = (!MASKED || ((allow >> (2 * k + 1)) & 1u)) ? r1 : 0.f;
    }
    if constexpr (MASKED) {
      const uint32_t lo = static_cast<uint32_t>(static_cast<int32_t>(allow << (31 - 2 * k)) >> 31);
      const uint32_t hi = static_cast<uint32_t>(static_cast<int32_t>(allow << (30 - 2 * k)) >> 31);
      const uint32_t keep = (lo & 0x0000FFFFu) | (hi & 0xFFFF0000u);
      a16 &= keep;
      r16 &= keep;
    }
    if constexpr (WANT_A) pa[k] = a16;
    pr[k] = r16;
  }
}

// Teardown shared by both kernels: after an abort let copies and MMAs in
// flight land, then free TMEM.
__device__ __forceinline__ void bwd_teardown(BwdCtl& ctl, int tid, int warp, uint32_t tmem, uint32_t cols) {
  if (ctl.abort_flag && tid == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, cols);
  }
}

__device__ __forceinline__ void bwd_init(BwdCtl& ctl, int tid, int warp) {
  if (tid == 0) {
    ptx::mbar_init(&ctl.one_full, 1);
    ptx::mbar_init(&ctl.one_empty, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl.ring_full[i], 1);
      ptx::mbar_init(&ctl.ring_empty[i], 1);
      ptx::mbar_init(&ctl.v_full[i], 1);
      ptx::mbar_init(&ctl.v_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&ctl.k_full[i], 1);
      ptx::mbar_init(&ctl.k_empty[i], 1);
      ptx::mbar_init(&ctl.s_full[i], 1);
      ptx::mbar_init(&ctl.p_full[i], kEwThreads);
    }
    ptx::mbar_init(&ctl.acc_full, 1);
    ptx::mbar_init(&ctl.acc_empty, kEwThreads);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl.sched_full[i], 1);
      ptx::mbar_init(&ctl.sched_empty[i], 1 + kBwdEwWarps);   // the MMA warp and the elementwise warps
    }
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
}

}  // namespace hstu

namespace hstu {

// ---------------------------------------------------------------------------------- dQ
template <int D, int DV, bool BF16, bool SOFTMAX, bool RAB = false, bool RAB_GRAD = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    hstu_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_q8, const __grid_constant__ CUtensorMap tm_do8,
                       const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<D, DV, RAB>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                    // Q then dO of the unit's query tile
  uint8_t* sDO = smem + Cfg::TQ;
  uint8_t* sK = sDO + Cfg::TV;           // K ring (DQ_KST stages), then the V ring (DQ_VST)
  uint8_t* sV = sK + Cfg::DQ_KST * Cfg::TQ;
  constexpr int NB = Cfg::DQ_BUFS, KST = Cfg::DQ_KST, VST = Cfg::DQ_VST, LAG = Cfg::DQ_LAG;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  bwd_init(ctl, tid, warp);
  const uint32_t tmem = ctl.tmem_base;   // score buffers [0, 128 NB), dQ [128 NB, 128 NB + D)
  ptx::grid_dependency_wait();
  const int n_units = p.ws_header[kWsUnits];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer + unit claims
    if (lane == 0) {
      int s_it = 0, one_it = 0, kv_it = 0, ui = -1;
      bool ok = sched_publish(ctl, p, p.ws_header + kWsCounter, n_units, s_it, ui);
      BwdUnit u;
      if (ok && ui >= 0) u = decode_bwd_unit(p, p.units[ui]);
      while (ok && ui >= 0 && !ctl.abort_flag) {
        const TileSet ts = query_tile_kv_tiles(u.s, u.L, u.t);
        if (ts.count > 0) {
          if (!bwd_wait(ctl, p, &ctl.one_empty, (one_it & 1) ^ 1)) break;
          ptx::mbar_arrive_expect_tx(&ctl.one_full, Cfg::TQ + Cfg::TV);
          load_query_tile(&tm_q, &tm_q8, sQ, &ctl.one_full, u.s, u.L, u.t, u.h * D, Cfg::KCH);
          load_query_tile(&tm_do, &tm_do8, sDO, &ctl.one_full, u.s, u.L, u.t, u.h * DV, Cfg::VCH);
          ++one_it;
          for (int k = 0; k < ts.count; ++k) {
            const int ks = kv_it % KST, vs = kv_it % VST;
            const int krow = u.s.kv0 + tileset_at(ts, k) * kBlockN;
            if (!bwd_wait(ctl, p, &ctl.k_empty[ks], ((kv_it / KST) & 1) ^ 1)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(&ctl.k_full[ks], Cfg::TQ);
            for (int kc = 0; kc < Cfg::KCH; ++kc)
              ptx::tma_load_2d(sK + ks * Cfg::TQ + kc * Cfg::CHUNK, &tm_k, &ctl.k_full[ks], u.h * D + kc * 64, krow);
            if (!bwd_wait(ctl, p, &ctl.v_empty[vs], ((kv_it / VST) & 1) ^ 1)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(&ctl.v_full[vs], Cfg::TV);
            for (int kc = 0; kc < Cfg::VCH; ++kc)
              ptx::tma_load_2d(sV + vs * Cfg::TV + kc * Cfg::CHUNK, &tm_v, &ctl.v_full[vs], u.h * DV + kc * 64,
                               krow);
            ++kv_it;
          }
          if (!ok) break;
        }
        // the next unit: claimed now, its Q and dO prefetched into L2 while
        // this unit's last tiles run
        if (!sched_publish(ctl, p, p.ws_header + kWsCounter, n_units, s_it, ui)) break;
        if (ui >= 0) {
          u = decode_bwd_unit(p, p.units[ui]);
          if (!(u.L.ctx_lane0 >= 0 && u.t == u.L.nq - 1)) {
            for (int kc = 0; kc < Cfg::KCH; ++kc)
              ptx::tma_prefetch_2d(&tm_q, u.h * D + kc * 64, u.s.q0 + u.t * kBlockM);
            for (int kc = 0; kc < Cfg::VCH; ++kc)
              ptx::tma_prefetch_2d(&tm_do, u.h * DV + kc * 64, u.s.q0 + u.t * kBlockM);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Half tile i of the unit (key tile i / 2, rows 64 (i % 2) of it) goes to
    // buffer t % NB.  Its score products are issued before the dQ product of
    // half tile i - LAG, so the elementwise warps find the next scores ready
    // and the tensor pipe has LAG half tiles of work queued behind them.
    const bool leader = ptx::elect_one_sync();
    constexpr uint32_t idesc_s = ptx::idesc_f16_f32acc(BF16, false, kBlockM, kHalf);
    constexpr uint32_t idesc_dq = ptx::idesc_f16_f32acc(BF16, true, kBlockM, D);
    const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sDO);
    const uint32_t k_ring = ptx::smem_u32(sK), v_ring = ptx::smem_u32(sV);
    int s_it = 0, one_it = 0, kv_it = 0, t_it = 0, u_it = 0, ui = -1;
    bool ok = true;
    while (ok && !ctl.abort_flag) {
      if (!sched_take(ctl, p, lane, s_it, ui) || ui < 0) break;
      const BwdUnit u = decode_bwd_unit(p, p.units[ui]);
      const int nt = query_tile_kv_tiles(u.s, u.L, u.t).count;
      if (nt == 0) continue;
      if (!bwd_warp_wait(ctl, p, &ctl.one_full, one_it & 1)) break;
      ptx::tc_fence_after();
      const int n_sub = 2 * nt;
      // dQ += dS K for half tile i (TMEM buffer of half tile t)
      auto dq_step = [&](int i, int t) -> bool {
        const int b = t % NB, kt = kv_it + (i >> 1), ks = kt % KST, hh = i & 1;
        if (!bwd_warp_wait(ctl, p, &ctl.p_full[b], (t / NB) & 1)) return false;
        ptx::tc_fence_after();
        if (i == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.acc_empty, (u_it & 1) ^ 1)) return false;
          ptx::tc_fence_after();
        }
        if (leader) {
          const uint32_t k_base = k_ring + ks * Cfg::TQ + hh * kHalfBytes;
          mma_half_ts(tmem + Cfg::DQ_ACC, tmem + 128 * b, k_base, idesc_dq, i > 0);
          if (hh == 1) ptx::umma_commit(&ctl.k_empty[ks]);   // the key tile's last read
        }
        __syncwarp();
        return true;
      };
      for (int i = 0; i < n_sub && ok; ++i) {
        const int t = t_it + i, b = t % NB, kt = kv_it + (i >> 1), ks = kt % KST, vs = kt % VST, hh = i & 1;
        if (hh == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.k_full[ks], (kt / KST) & 1)) { ok = false; break; }
          if (!bwd_warp_wait(ctl, p, &ctl.v_full[vs], (kt / VST) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        if (leader) {
          const uint32_t k_base = k_ring + ks * Cfg::TQ + hh * kHalfBytes;
          const uint32_t v_base = v_ring + vs * Cfg::TV + hh * kHalfBytes;
          mma_scores<D / 16>(tmem + 128 * b, q_base, k_base, idesc_s);         // S = Q K_h^T
          mma_scores<DV / 16>(tmem + 128 * b + 64, do_base, v_base, idesc_s);  // dP = dO V_h^T
          if (hh == 1) ptx::umma_commit(&ctl.v_empty[vs]);          // V is read by dP only
          if (i == n_sub - 1) ptx::umma_commit(&ctl.one_empty);   // Q and dO are no longer read
          ptx::umma_commit(&ctl.s_full[b]);
        }
        __syncwarp();
        if (i >= LAG && !dq_step(i - LAG, t - LAG)) { ok = false; break; }
      }
      if (!ok) break;
      for (int i = n_sub > LAG ? n_sub - LAG : 0; i < n_sub && ok; ++i)
        if (!dq_step(i, t_it + i)) ok = false;
      if (!ok) break;
      if (leader) ptx::umma_commit(&ctl.acc_full);
      __syncwarp();
      t_it += n_sub;
      kv_it += nt;
      ++one_it;
      ++u_it;
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    // Warpgroup wg takes columns [32 wg, 32 wg + 32) of each half tile; lanes
    // are query rows.  dS is kept without attn_scale (the epilogue applies
    // alpha * attn_scale).
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float alpha = p.alpha;
    const float half_alpha = 0.5f * p.alpha;
    constexpr float kLog2e = 1.4426950408889634f;
    int s_it = 0, t_it = 0, u_it = 0, ui = -1;
    bool ok = true;
    while (ok && !ctl.abort_flag) {
      if (!sched_take(ctl, p, lane, s_it, ui) || ui < 0) break;
      const BwdUnit u = decode_bwd_unit(p, p.units[ui]);
      const TileSet ts = query_tile_kv_tiles(u.s, u.L, u.t);
      const int nt = ts.count;
      const int qr = q_row(u.s, u.L, u.t, rloc);
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      const long long grow = static_cast<long long>(u.s.q0) + row;
      uint16_t* dq_row = reinterpret_cast<uint16_t*>(p.dq) + grow * p.dq_stride + u.h * D + wg * (D / 2);
      if (nt == 0) {   // no key reaches this tile: dQ = 0
        if (valid) {
#pragma unroll
          for (int c = 0; c < D / 2; c += 8) *reinterpret_cast<uint4*>(dq_row + c) = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      int r_lo, r_hi;
      row_uih_keys(u.s, row, r_lo, r_hi);
      int r_diag = row_diag_key(u.s, row);
      int r_ctx = u.s.c;
      if (!valid) { r_lo = r_hi = 0; r_diag = -1; r_ctx = 0; }
      float lse2 = 0.f, dlt = 0.f;   // softmax: lse (log2 units), delta / attn_scale
      if constexpr (SOFTMAX) {
        if (valid) {
          lse2 = p.lse[static_cast<long long>(u.h) * p.total_q + grow] * kLog2e;
          dlt = p.delta[static_cast<long long>(u.h) * p.total_q + grow] / u.scale;
        }
      }
      // relative attention bias: this warp's tables, the row's timestamp and
      // position, and each key tile's timestamps (one per lane and half) loaded
      // a key tile ahead
      RabWarp* rw = reinterpret_cast<RabWarp*>(smem + Cfg::RAB_OFFSET) + (warp - 2);
      long long ts_row = 0, nk0 = 0, nk1 = 0;
      int pos_row = 0;
      auto load_keys = [&](int nn) {
        if constexpr (RAB) {
          if (p.ts_q != nullptr) {
            nk0 = p.ts_kv[u.s.kv0 + min(nn * kBlockN + 32 * wg + lane, u.s.Lkv - 1)];
            nk1 = p.ts_kv[u.s.kv0 + min(nn * kBlockN + kHalf + 32 * wg + lane, u.s.Lkv - 1)];
          }
        }
      };
      // gradients of the bias tables (when asked for): this warp's sums over the unit
      RabGradWarp* rg = reinterpret_cast<RabGradWarp*>(smem + Cfg::RAB_GRAD_OFFSET) + (warp - 2);
      RabGradAcc racc{-1, 0.f, 0.f};
      // (RAB_GRAD: the instantiation that computes them, launched only when asked)
      const bool grad_time = RAB_GRAD && p.d_rab_time != nullptr && p.ts_q != nullptr && p.rab_time != nullptr;
      const bool grad_pos = RAB_GRAD && p.d_rab_pos != nullptr && p.rab_pos != nullptr;
      if constexpr (RAB) {
        __syncwarp();   // the previous unit's lookups are done
        rab_build(*rw, p.ts_q != nullptr ? p.rab_time : nullptr, p.rab_pos, p.rab_np, u.h,
                  SOFTMAX ? kLog2e : 0.5f, lane);
        if (grad_time || grad_pos) {
          for (int i = lane; i < kRabTimeBuckets + 1; i += 32) rg->t[i] = 0.f;
          for (int i = lane; i < p.rab_np; i += 32) rg->pos[i] = 0.f;
          racc = RabGradAcc{-1, 0.f, 0.f};
        }
        __syncwarp();
        if (p.ts_q != nullptr) ts_row = p.ts_q[u.s.q0 + row];
        pos_row = row < u.s.c ? row : row + (u.s.ukv - u.s.u);
        load_keys(tileset_at(ts, 0));
      }
      const FullTiles ft = full_tile_ranges(u.s, q_tile_bounds(u.s, u.L, u.t));
      for (int idx = 0; idx < nt && ok; ++idx) {
        const int n = tileset_at(ts, idx);
        const long long ck0 = nk0, ck1 = nk1;
        if (RAB && idx + 1 < nt) load_keys(tileset_at(ts, idx + 1));
        const bool full = n < ft.ctx_hi || (n >= ft.lo && n < ft.hi);
        const int j0 = n * kBlockN;
        RowMask rm;
        rm.ctx = r_ctx - j0;
        rm.lo = r_lo - j0;
        rm.span = static_cast<uint32_t>(r_hi - r_lo);
        rm.diag = r_diag >= 0 ? r_diag - j0 : -1000000;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          const int t = t_it++, b = t % NB;
          const uint32_t sb = tmem + lane_base + 128 * b + 32 * wg;
          const uint32_t mb = full ? 0xFFFFFFFFu : rm.bits32(kHalf * hh + 32 * wg);
          if (!bwd_warp_wait(ctl, p, &ctl.s_full[b], (t / NB) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          uint32_t sv[32], dv[32], pk[16];
          ptx::tmem_ld32(sb, sv);
          ptx::tmem_ld32(sb + 64, dv);
          ptx::tmem_ld_wait(sv);
          ptx::tmem_ld_wait(dv);
          RabRow rr{0, 0};
          RabCols rc{};
          RabChunk rk{};
          const bool has_time = p.ts_q != nullptr && p.rab_time != nullptr;
          if constexpr (RAB) {   // sv becomes alpha s + rab, scaled (SiLU: / 2, softmax: * log2 e)
            const long long ck = hh ? ck1 : ck0;
            const long long base = __shfl_sync(0xffffffffu, ck, 0);
            rr = RabRow{p.ts_q != nullptr ? rab_rel_ts(ts_row, base) : 0, pos_row};
            rc = rab_cols(p.ts_q != nullptr ? rab_rel_ts(ck, base) : 0, j0 + kHalf * hh + 32 * wg + lane, true);
            rk = rab_apply32<true>(sv, SOFTMAX ? alpha * kLog2e : half_alpha, *rw, p.rab_np, has_time, rr, rc);
          }
          float dsf[32];   // dS in fp32, for the bias tables' gradients
          const bool want_ds = RAB_GRAD && (grad_time || grad_pos);
          if constexpr (!SOFTMAX) {
            if (full) silu_bwd_f32<BF16, false, false, RAB>(sv, dv, half_alpha, mb, pk, pk, want_ds ? dsf : nullptr);
            else silu_bwd_f32<BF16, false, true, RAB>(sv, dv, half_alpha, mb, pk, pk, want_ds ? dsf : nullptr);
          } else {
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              float ds[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float s = __uint_as_float(sv[k + e]);
                const float g = __uint_as_float(dv[k + e]);
                const float r = ex2_approx((RAB ? s : s * (alpha * kLog2e)) - lse2) * (g - dlt);
                ds[e] = ((mb >> (k + e)) & 1u) ? r : 0.f;
                dsf[k + e] = ds[e];
              }
              pk[k >> 1] = pack2<BF16>(ds[0], ds[1]);
            }
          }
          if constexpr (RAB) {
            if (want_ds) {
              // a lane with no row of the sequence (past a ragged last query
              // tile) computed dS from rows that are not this sequence's: in a
              // full tile nothing masked it, and its dQ is never stored
              if (!valid) {
#pragma unroll
                for (int k = 0; k < 32; ++k) dsf[k] = 0.f;
              }
              rab_grad32<true>(dsf, rk, *rg, racc, *rw, p.rab_np, grad_time, grad_pos, rr, rc);
            }
          }
          ptx::tmem_st16(sb, pk);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&ctl.p_full[b]);
        }
      }
      if (!ok) break;
      if constexpr (RAB) {
        // this warp's table gradients of the unit, x attn_scale (dS above is kept
        // without it), into the outputs
        if (grad_time || grad_pos) {
          rab_grad_flush(racc, *rg, p.rab_np, grad_time, grad_pos);
          __syncwarp();
          if (grad_time && lane < kRabTimeBuckets) {
            const float v = rg->t[lane] + (lane == kRabTimeBuckets - 1 ? rg->t[kRabTimeBuckets] : 0.f);
            if (v != 0.f) atomicAdd(p.d_rab_time + u.h * kRabTimeBuckets + lane, v * u.scale);
          }
          if (grad_pos) {
            for (int i = lane; i < p.rab_np; i += 32) {
              const float v = rg->pos[i];
              if (v != 0.f) atomicAdd(p.d_rab_pos + static_cast<long long>(u.h) * p.rab_np + i, v * u.scale);
            }
          }
        }
      }
      // dQ * alpha * attn_scale out of TMEM: this warpgroup's half of the D columns
      if (!bwd_warp_wait(ctl, p, &ctl.acc_full, u_it & 1)) break;
      ptx::tc_fence_after();
      const float mul = alpha * u.scale;
#pragma unroll 1
      for (int c = 0; c < D / 2; c += 16) {   // 16 columns at a time (hdim 96: 48 per warpgroup)
        uint32_t o[16];
        ptx::tmem_ld16(tmem + lane_base + Cfg::DQ_ACC + wg * (D / 2) + c, o);
        ptx::tmem_ld_wait(o);
        if (valid) {
          uint32_t q2[8];
#pragma unroll
          for (int k = 0; k < 16; k += 2)
            q2[k >> 1] = pack2<BF16>(__uint_as_float(o[k]) * mul, __uint_as_float(o[k + 1]) * mul);
          *reinterpret_cast<uint4*>(dq_row + c) = make_uint4(q2[0], q2[1], q2[2], q2[3]);
          *reinterpret_cast<uint4*>(dq_row + c + 8) = make_uint4(q2[4], q2[5], q2[6], q2[7]);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl.acc_empty);
      ++u_it;
    }
  }
  bwd_teardown(ctl, tid, warp, tmem, Cfg::TMEM_COLS);
}

}  // namespace hstu

namespace hstu {

// ---------------------------------------------------------------------------------- dK, dV
template <int D, int DV, bool BF16, bool SOFTMAX, bool RAB = false>
__global__ void __launch_bounds__(kBwdThreads, 1)
    hstu_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_q8, const __grid_constant__ CUtensorMap tm_do8,
                         const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<D, DV, RAB>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  __shared__ BwdColInfo cinfo;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;                    // K then V of the unit's key tile
  uint8_t* sV = smem + Cfg::TQ;
  uint8_t* sQD = sV + Cfg::TV;           // ring: Q then dO of a member query tile per stage
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  bwd_init(ctl, tid, warp);
  // buffers [0, 256), dV [256, 256 + DV), dK [256 + DV, 256 + DV + D)
  const uint32_t tmem = ctl.tmem_base;
  ptx::grid_dependency_wait();
  const int n_units = p.ws_header[kWsKvUnits];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer + unit claims
    if (lane == 0) {
      int s_it = 0, u_it = 0, q_it = 0, ui = -1;
      bool ok = sched_publish(ctl, p, p.ws_header + kWsKvCounter, n_units, s_it, ui);
      BwdUnit u;
      if (ok && ui >= 0) u = decode_bwd_unit(p, p.kv_units[ui]);
      while (ok && ui >= 0 && !ctl.abort_flag) {
        const MemberWords mw = member_words(p, u);
        if (member_count(mw) > 0) {
          if (!bwd_wait(ctl, p, &ctl.one_empty, (u_it & 1) ^ 1)) break;
          ptx::mbar_arrive_expect_tx(&ctl.one_full, Cfg::TQ + Cfg::TV);
          const int krow = u.s.kv0 + u.t * kBlockN;
          for (int kc = 0; kc < Cfg::KCH; ++kc)
            ptx::tma_load_2d(sK + kc * Cfg::CHUNK, &tm_k, &ctl.one_full, u.h * D + kc * 64, krow);
          for (int kc = 0; kc < Cfg::VCH; ++kc)
            ptx::tma_load_2d(sV + kc * Cfg::CHUNK, &tm_v, &ctl.one_full, u.h * DV + kc * 64, krow);
          ++u_it;
          for (int w = 0; w < mw.n && ok; ++w) {
            unsigned bits = mw.w[w];
            while (bits != 0u) {
              const int m = w * 32 + __ffs(bits) - 1;
              bits &= bits - 1u;
              const int st = q_it & 1;
              if (!bwd_wait(ctl, p, &ctl.ring_empty[st], ((q_it >> 1) & 1) ^ 1)) { ok = false; break; }
              uint8_t* dst = sQD + st * (Cfg::TQ + Cfg::TV);
              ptx::mbar_arrive_expect_tx(&ctl.ring_full[st], Cfg::TQ + Cfg::TV);
              load_query_tile(&tm_q, &tm_q8, dst, &ctl.ring_full[st], u.s, u.L, m, u.h * D, Cfg::KCH);
              load_query_tile(&tm_do, &tm_do8, dst + Cfg::TQ, &ctl.ring_full[st], u.s, u.L, m, u.h * DV,
                              Cfg::VCH);
              ++q_it;
            }
          }
          if (!ok) break;
        }
        // the next unit: claimed now, its K and V prefetched into L2
        if (!sched_publish(ctl, p, p.ws_header + kWsKvCounter, n_units, s_it, ui)) break;
        if (ui >= 0) {
          u = decode_bwd_unit(p, p.kv_units[ui]);
          for (int kc = 0; kc < Cfg::KCH; ++kc)
            ptx::tma_prefetch_2d(&tm_k, u.h * D + kc * 64, u.s.kv0 + u.t * kBlockN);
          for (int kc = 0; kc < Cfg::VCH; ++kc)
            ptx::tma_prefetch_2d(&tm_v, u.h * DV + kc * 64, u.s.kv0 + u.t * kBlockN);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Half tile i of the unit (member query tile i / 2, rows 64 (i % 2) of it)
    // goes to buffer t & 1; its score products are issued before the gradient
    // products of half tile i - 1.
    const bool leader = ptx::elect_one_sync();
    constexpr uint32_t idesc_s = ptx::idesc_f16_f32acc(BF16, false, kBlockM, kHalf);
    constexpr uint32_t idesc_dv = ptx::idesc_f16_f32acc(BF16, true, kBlockM, DV);
    constexpr uint32_t idesc_dk = ptx::idesc_f16_f32acc(BF16, true, kBlockM, D);
    const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV), qd_base = ptx::smem_u32(sQD);
    int s_it = 0, u_it = 0, q_it = 0, t_it = 0, ui = -1;
    bool ok = true;
    while (ok && !ctl.abort_flag) {
      if (!sched_take(ctl, p, lane, s_it, ui) || ui < 0) break;
      const BwdUnit u = decode_bwd_unit(p, p.kv_units[ui]);
      const int nm = member_count(member_words(p, u));
      if (nm == 0) continue;
      if (!bwd_warp_wait(ctl, p, &ctl.one_full, u_it & 1)) break;
      ptx::tc_fence_after();
      const int n_sub = 2 * nm;
      // dV += P^T dO_h and dK += dS^T Q_h for half tile i (buffer of half tile t)
      auto grad_step = [&](int i, int t) -> bool {
        const int b = t & 1, qt = q_it + (i >> 1), st = qt & 1, hh = i & 1;
        if (!bwd_warp_wait(ctl, p, &ctl.p_full[b], (t >> 1) & 1)) return false;
        ptx::tc_fence_after();
        if (i == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.acc_empty, (u_it & 1) ^ 1)) return false;
          ptx::tc_fence_after();
        }
        if (leader) {
          const uint32_t q_b = qd_base + st * (Cfg::TQ + Cfg::TV) + hh * kHalfBytes;
          mma_half_ts(tmem + Cfg::ACC, tmem + 128 * b, q_b + Cfg::TQ, idesc_dv, i > 0);
          mma_half_ts(tmem + Cfg::ACC + DV, tmem + 128 * b + 64, q_b, idesc_dk, i > 0);
          if (hh == 1) ptx::umma_commit(&ctl.ring_empty[st]);
        }
        __syncwarp();
        return true;
      };
      for (int i = 0; i < n_sub && ok; ++i) {
        const int t = t_it + i, b = t & 1, qt = q_it + (i >> 1), st = qt & 1, hh = i & 1;
        if (hh == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.ring_full[st], (qt >> 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        if (leader) {
          const uint32_t q_b = qd_base + st * (Cfg::TQ + Cfg::TV) + hh * kHalfBytes;
          mma_scores<D / 16>(tmem + 128 * b, k_base, q_b, idesc_s);                    // S^T = K Q_h^T
          mma_scores<DV / 16>(tmem + 128 * b + 64, v_base, q_b + Cfg::TQ, idesc_s);     // dP^T = V dO_h^T
          if (i == n_sub - 1) ptx::umma_commit(&ctl.one_empty);   // K and V are no longer read
          ptx::umma_commit(&ctl.s_full[b]);
        }
        __syncwarp();
        if (i > 0 && !grad_step(i - 1, t - 1)) { ok = false; break; }
      }
      if (!ok || !grad_step(n_sub - 1, t_it + n_sub - 1)) break;
      if (leader) ptx::umma_commit(&ctl.acc_full);
      __syncwarp();
      t_it += n_sub;
      q_it += nm;
      ++u_it;
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    // Lanes are key rows; warpgroup wg takes query columns [32 wg, 32 wg + 32)
    // of each half tile.  Lane l works out column l's row, validity, allowed
    // key interval (partial tiles) and softmax statistics into this warp's
    // slots of ctl.col_*, which every lane then reads as broadcasts.  dS^T is
    // kept without attn_scale (the epilogue applies alpha * attn_scale).
    const int wg = (warp - 2) >> 2;
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float alpha = p.alpha;
    const float half_alpha = 0.5f * p.alpha;
    constexpr float kLog2e = 1.4426950408889634f;
    const float4* stat4 = reinterpret_cast<const float4*>(&cinfo.col_stat[ew][0]);
    int s_it = 0, t_it = 0, a_it = 0, ui = -1;
    bool ok = true;
    while (ok && !ctl.abort_flag) {
      if (!sched_take(ctl, p, lane, s_it, ui) || ui < 0) break;
      const BwdUnit u = decode_bwd_unit(p, p.kv_units[ui]);
      const MemberWords mw = member_words(p, u);
      const int nm = member_count(mw);
      const int j = u.t * kBlockN + rloc;   // this lane's key row
      const bool kvalid = j < u.s.Lkv;
      const long long krow = static_cast<long long>(u.s.kv0) + j;
      uint16_t* dv_row = reinterpret_cast<uint16_t*>(p.dv) + krow * p.dv_stride + u.h * DV + wg * (DV / 2);
      uint16_t* dk_row = reinterpret_cast<uint16_t*>(p.dk) + krow * p.dk_stride + u.h * D + wg * (D / 2);
      if (nm == 0) {   // no query sees this key tile: dK = dV = 0
        if (kvalid) {
#pragma unroll
          for (int c = 0; c < DV / 2; c += 8) *reinterpret_cast<uint4*>(dv_row + c) = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int c = 0; c < D / 2; c += 8) *reinterpret_cast<uint4*>(dk_row + c) = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const bool ctx_key = j < u.s.c;   // context keys are seen by every query row
      // relative attention bias: this warp's tables; the key row's timestamp,
      // relative to the unit's first key, and position
      RabWarp* rw = reinterpret_cast<RabWarp*>(smem + Cfg::RAB_OFFSET) + ew;
      long long ts_base = 0;
      RabRow krow_rab{0, j};
      if constexpr (RAB) {
        __syncwarp();   // the previous unit's lookups are done
        rab_build(*rw, p.ts_q != nullptr ? p.rab_time : nullptr, p.rab_pos, p.rab_np, u.h,
                  SOFTMAX ? kLog2e : 0.5f, lane);
        __syncwarp();
        if (p.ts_q != nullptr) {
          ts_base = p.ts_kv[u.s.kv0 + u.t * kBlockN];
          krow_rab.ts = rab_rel_ts(p.ts_kv[u.s.kv0 + min(j, u.s.Lkv - 1)], ts_base);
        }
      }
      for (int w = 0; w < mw.n && ok; ++w) {
        unsigned bits = mw.w[w];
        while (bits != 0u && ok) {
          const int m = w * 32 + __ffs(bits) - 1;
          bits &= bits - 1u;
          const FullTiles ft = full_tile_ranges(u.s, load_qtile_bounds(p, u.b, m));
          const bool full = u.t < ft.ctx_hi || (u.t >= ft.lo && u.t < ft.hi);
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            const int t = t_it++, b = t & 1;
            const uint32_t sb = tmem + lane_base + 128 * b + 32 * wg;
            // this lane's column: row, validity, interval, statistics
            const int qi = q_row(u.s, u.L, m, kHalf * hh + 32 * wg + lane);
            const uint32_t cvalid = __ballot_sync(0xffffffffu, qi >= 0);
            __syncwarp();   // the previous half tile's broadcasts are all read
            if (!full) {
              int lo = 0, hi = 0, dg = -1;
              if (qi >= 0) {
                row_uih_keys(u.s, qi, lo, hi);
                dg = row_diag_key(u.s, qi);
              }
              cinfo.col_rng[ew][lane] = make_int4(lo, hi, dg, 0);
            }
            int c_ts = 0;   // bias: this lane's column's timestamp
            if constexpr (RAB) {
              if (p.ts_q != nullptr && qi >= 0) c_ts = rab_rel_ts(p.ts_q[u.s.q0 + qi], ts_base);
            }
            if constexpr (SOFTMAX) {
              float l2 = 0.f, dl = 0.f;
              if (qi >= 0) {
                const long long gq = static_cast<long long>(u.h) * p.total_q + u.s.q0 + qi;
                l2 = p.lse[gq] * kLog2e;
                dl = p.delta[gq] / u.scale;
              }
              cinfo.col_stat[ew][lane] = make_float2(l2, dl);
            }
            __syncwarp();
            uint32_t allow = cvalid;
            if (!full && !ctx_key) {
              uint32_t seen = 0u;
#pragma unroll
              for (int kk = 0; kk < 32; ++kk) {
                const int4 r = cinfo.col_rng[ew][kk];
                seen |= static_cast<uint32_t>((j >= r.x && j < r.y) || j == r.z) << kk;
              }
              allow &= seen;
            }
            const bool masked = !full || cvalid != 0xFFFFFFFFu;   // warp-uniform
            if (!bwd_warp_wait(ctl, p, &ctl.s_full[b], (t >> 1) & 1)) { ok = false; break; }
            ptx::tc_fence_after();
            uint32_t sv[32], dv[32], pp[16], pd[16];
            ptx::tmem_ld32(sb, sv);
            ptx::tmem_ld32(sb + 64, dv);
            ptx::tmem_ld_wait(sv);
            ptx::tmem_ld_wait(dv);
            if constexpr (RAB) {   // sv becomes alpha s + rab, scaled (SiLU: / 2, softmax: * log2 e)
              const int c_pos = qi < 0 ? 0 : (qi < u.s.c ? qi : qi + (u.s.ukv - u.s.u));
              rab_apply32<false>(sv, SOFTMAX ? alpha * kLog2e : half_alpha, *rw, p.rab_np,
                                 p.ts_q != nullptr && p.rab_time != nullptr, krow_rab,
                                 rab_cols(c_ts, c_pos, qi >= 0));
            }
            if constexpr (!SOFTMAX) {
              if (masked) silu_bwd_f32<BF16, true, true, RAB>(sv, dv, half_alpha, allow, pp, pd);
              else silu_bwd_f32<BF16, true, false, RAB>(sv, dv, half_alpha, allow, pp, pd);
            } else {
#pragma unroll
              for (int k = 0; k < 32; k += 2) {
                float pv[2], ds[2];
                const float4 st4 = stat4[k >> 1];   // columns k, k + 1
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const float s = __uint_as_float(sv[k + e]);
                  const float g = __uint_as_float(dv[k + e]);
                  const float l2 = e ? st4.z : st4.x;
                  const float dl = e ? st4.w : st4.y;
                  const float a = ex2_approx((RAB ? s : s * (alpha * kLog2e)) - l2);
                  const float r = a * (g - dl);
                  const bool al = (allow >> (k + e)) & 1u;
                  pv[e] = al ? a : 0.f;
                  ds[e] = al ? r : 0.f;
                }
                pp[k >> 1] = pack2<BF16>(pv[0], pv[1]);
                pd[k >> 1] = pack2<BF16>(ds[0], ds[1]);
              }
            }
            ptx::tmem_st16(sb, pp);
            ptx::tmem_st16(sb + 64, pd);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctl.p_full[b]);
          }
        }
      }
      if (!ok) break;
      // dV * attn_scale and dK * alpha * attn_scale: this warpgroup's half of each
      if (!bwd_warp_wait(ctl, p, &ctl.acc_full, a_it & 1)) break;
      ptx::tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int W = part == 0 ? DV : D;
        const float mul = part == 0 ? u.scale : alpha * u.scale;
        const uint32_t col0 = Cfg::ACC + (part == 0 ? 0 : DV) + wg * (W / 2);
        uint16_t* dst = part == 0 ? dv_row : dk_row;
#pragma unroll 1
        for (int c = 0; c < W / 2; c += 16) {   // 16 columns at a time (hdim 96: 48 per warpgroup)
          uint32_t o[16];
          ptx::tmem_ld16(tmem + lane_base + col0 + c, o);
          ptx::tmem_ld_wait(o);
          if (kvalid) {
            uint32_t pk[8];
#pragma unroll
            for (int k = 0; k < 16; k += 2)
              pk[k >> 1] = pack2<BF16>(__uint_as_float(o[k]) * mul, __uint_as_float(o[k + 1]) * mul);
            *reinterpret_cast<uint4*>(dst + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(dst + c + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl.acc_empty);
      ++a_it;
    }
  }
  bwd_teardown(ctl, tid, warp, tmem, Cfg::TMEM_COLS);
}

// Host side: both backward kernels of one head dimension, the dQ kernel first.
template <int D, int DV, bool BF16, bool SOFTMAX, bool RAB>
cudaError_t launch_bwd_pair(const BwdMaps& m, const BwdParams& p, int grid_q, int grid_kv, cudaStream_t stream) {
  constexpr int smem = BwdCfg<D, DV, RAB>::SMEM_BYTES;        // dK/dV kernel
  constexpr int smem_q = BwdCfg<D, DV, RAB>::DQ_SMEM_BYTES;   // dQ kernel
  // the dQ kernel that also sums the bias tables' gradients, when they are asked for
  const bool grad = RAB && (p.d_rab_time != nullptr || p.d_rab_pos != nullptr);
  auto kq = grad ? hstu_bwd_dq_kernel<D, DV, BF16, SOFTMAX, RAB, RAB> : hstu_bwd_dq_kernel<D, DV, BF16, SOFTMAX, RAB>;
  auto kkv = hstu_bwd_dkdv_kernel<D, DV, BF16, SOFTMAX, RAB>;
  static_assert(smem + sizeof(BwdCtl) + sizeof(BwdColInfo) <= 232448, "shared memory over the 227 KB a CTA may use");
  static_assert(smem_q + sizeof(BwdCtl) <= 232448, "shared memory over the 227 KB a CTA may use");
  static std::atomic<unsigned long long> q_attr_set{0}, qg_attr_set{0}, kv_attr_set{0};
  cudaError_t e = ensure_smem_attr(kq, smem_q, grad ? qg_attr_set : q_attr_set);
  if (e == cudaSuccess) e = ensure_smem_attr(kkv, smem, kv_attr_set);
  if (e != cudaSuccess) return e;
  kq<<<grid_q, kBwdThreads, smem_q, stream>>>(m.q, m.k, m.v, m.d_o, m.q8, m.d_o8, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kkv<<<grid_kv, kBwdThreads, smem, stream>>>(m.q, m.k, m.v, m.d_o, m.q8, m.d_o8, p);
  return cudaGetLastError();
}

template <int D, int DV, bool RAB>
cudaError_t launch_bwd_dispatch(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q,
                                int grid_kv, cudaStream_t stream) {
  if (bf16) return softmax ? launch_bwd_pair<D, DV, true, true, RAB>(m, p, grid_q, grid_kv, stream)
                           : launch_bwd_pair<D, DV, true, false, RAB>(m, p, grid_q, grid_kv, stream);
  return softmax ? launch_bwd_pair<D, DV, false, true, RAB>(m, p, grid_q, grid_kv, stream)
                 : launch_bwd_pair<D, DV, false, false, RAB>(m, p, grid_q, grid_kv, stream);
}

}  // namespace hstu
