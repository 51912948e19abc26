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
// Two persistent kernels, each a static round-robin over its work units, with
// one warp of TMA loads, one MMA warp (the whole warp runs the loop, one
// elected lane issues) and two elementwise warpgroups that split each score
// row's 128 columns:
//   dQ kernel, one unit per (sequence, head, query tile): for every key tile of
//     the tile's set, S = Q K^T and dP = dO V^T into TMEM, dS (16-bit, packed
//     over S) back into TMEM, dQ += dS K with K read MN-major from its tile;
//     the elementwise warps then scale dQ by alpha and store it.
//   dK/dV kernel, one unit per (sequence, head, key tile): for every query tile
//     whose key-tile set holds this key tile, S^T = K Q^T and dP^T = V dO^T,
//     P^T and dS^T (packed over S^T and dP^T), dV += P^T dO and dK += dS^T Q
//     with dO and Q read MN-major; then dV * attn_scale and dK * alpha.
// Query tiles follow the forward's layout (q_layout): context rows may sit on
// the top lanes of a sequence's last query tile, and that tile's Q and dO then
// arrive as 8-row TMA boxes.  Every wait is bounded (2 s); a timeout sets the
// device error word and every role stops.
#pragma once
#include "hstu_fwd_kernel.cuh"
#include "hstu_launch.h"

namespace hstu {

constexpr int kBwdThreads = 320;   // producer, MMA, two elementwise warpgroups

template <int D, int DV>
struct BwdCfg {
  static constexpr int KCH = (D + 63) / 64;
  static constexpr int VCH = (DV + 63) / 64;
  static constexpr int CHUNK = kBlockN * 128;   // one 128-row x 128-byte swizzle box
  static constexpr int TQ = KCH * CHUNK;        // a Q or K tile
  static constexpr int TV = VCH * CHUNK;        // a V or dO tile
  static constexpr int STAGES = 2;
  static constexpr int SMEM_BYTES = (TQ + TV) * (1 + STAGES) + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(D % 16 == 0 && DV % 32 == 0 && 256 + D + DV <= TMEM_COLS, "backward head dimensions");
};

struct BwdCtl {
  uint64_t one_full, one_empty;        // dQ kernel: Q + dO of the unit; dK/dV kernel: K + V
  uint64_t ring_full[2], ring_empty[2];   // dQ kernel: K + V per key tile; dK/dV kernel: Q + dO
  uint64_t s_full, p_full;             // both score products ready / the 16-bit operands written
  uint64_t acc_full, acc_empty;        // accumulators complete / read out
  uint32_t tmem_base;
  volatile int abort_flag;
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

// The query-tile record the scheduler wrote for tile m of sequence b.
struct QTileRec {
  TileSet ts;
  TileBounds tb;
};
__device__ __forceinline__ QTileRec load_qtile(const BwdParams& p, int b, int m) {
  const int4* r = reinterpret_cast<const int4*>(p.qtiles + static_cast<long long>(p.qtile_base[b] + m) * kQTileInts);
  const int4 a = r[0], c = r[1], d = r[2];
  QTileRec q;
  q.ts.lo0 = a.x; q.ts.hi0 = a.y; q.ts.lo1 = a.z; q.ts.hi1 = a.w;
  q.ts.lo2 = c.x; q.ts.hi2 = c.y; q.ts.count = c.z;
  q.tb.LO = c.w; q.tb.HI = d.x; q.tb.maxLO = d.y; q.tb.minHI = d.z;
  return q;
}
__device__ __forceinline__ bool tileset_has(const TileSet& ts, int n) {
  return (n >= ts.lo0 && n < ts.hi0) | (n >= ts.lo1 && n < ts.hi1) | (n >= ts.lo2 && n < ts.hi2);
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

// C[tmem] (+)= A B^T, both K-major 128-row tiles in shared memory, KS k-steps.
template <int KS>
__device__ __forceinline__ void mma_ss_kmajor(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
  const uint64_t ad0 = ptx::sdesc_sw128(a_base, 16, 1024), bd0 = ptx::sdesc_sw128(b_base, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint64_t off = static_cast<uint64_t>(((ks >> 2) * (kBlockN * 128) + (ks & 3) * 32) >> 4);
    ptx::umma_ss(d_tmem, ad0 + off, bd0 + off, idesc, ks > 0 ? 1u : 0u);
  }
}
// C[tmem] (+)= A B with A (128 x 128, 16-bit) packed in TMEM at a_tmem the way
// the elementwise warps write it, and B a 128-row tile in shared memory read
// MN-major (K = its rows, N = its columns).
__device__ __forceinline__ void mma_ts_mnmajor(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, uint32_t idesc,
                                               bool accumulate) {
  const uint64_t bd0 = ptx::sdesc_sw128(b_base, kBlockN * 128, 1024);
  uint32_t pa[8];
  uint64_t vd[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    pa[kk] = a_tmem + (kk >> 2) * 64 + (kk & 3) * 8;
    vd[kk] = bd0 + static_cast<uint64_t>((kk * 2048) >> 4);
  }
  ptx::umma_ts_x8(d_tmem, pa, vd, idesc, accumulate ? 1u : 0u);
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------------- dQ
template <int D, int DV, bool BF16, bool SOFTMAX>
__global__ void __launch_bounds__(kBwdThreads, 1)
    hstu_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_q8, const __grid_constant__ CUtensorMap tm_do8,
                       const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<D, DV>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                    // Q then dO of the unit's query tile
  uint8_t* sDO = smem + Cfg::TQ;
  uint8_t* sKV = sDO + Cfg::TV;          // ring: K then V of a key tile per stage
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    ptx::mbar_init(&ctl.one_full, 1);
    ptx::mbar_init(&ctl.one_empty, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl.ring_full[i], 1);
      ptx::mbar_init(&ctl.ring_empty[i], 1);
    }
    ptx::mbar_init(&ctl.s_full, 1);
    ptx::mbar_init(&ctl.p_full, kEwThreads);
    ptx::mbar_init(&ctl.acc_full, 1);
    ptx::mbar_init(&ctl.acc_empty, kEwThreads);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;   // S [0,128), dP [128,256), dQ [256, 256 + D)
  ptx::grid_dependency_wait();
  const int n_units = p.ws_header[kWsUnits];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int one_it = 0, kv_it = 0;
      bool ok = true;
      for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
        const BwdUnit u = decode_bwd_unit(p, p.units[ui]);
        const TileSet ts = query_tile_kv_tiles(u.s, u.L, u.t);
        if (ts.count == 0) continue;
        if (!bwd_wait(ctl, p, &ctl.one_empty, (one_it & 1) ^ 1)) break;
        ptx::mbar_arrive_expect_tx(&ctl.one_full, Cfg::TQ + Cfg::TV);
        load_query_tile(&tm_q, &tm_q8, sQ, &ctl.one_full, u.s, u.L, u.t, u.h * D, Cfg::KCH);
        load_query_tile(&tm_do, &tm_do8, sDO, &ctl.one_full, u.s, u.L, u.t, u.h * DV, Cfg::VCH);
        ++one_it;
        for (int k = 0; k < ts.count; ++k) {
          const int st = kv_it & 1;
          if (!bwd_wait(ctl, p, &ctl.ring_empty[st], ((kv_it >> 1) & 1) ^ 1)) { ok = false; break; }
          const int krow = u.s.kv0 + tileset_at(ts, k) * kBlockN;
          uint8_t* dst = sKV + st * (Cfg::TQ + Cfg::TV);
          ptx::mbar_arrive_expect_tx(&ctl.ring_full[st], Cfg::TQ + Cfg::TV);
          for (int kc = 0; kc < Cfg::KCH; ++kc)
            ptx::tma_load_2d(dst + kc * Cfg::CHUNK, &tm_k, &ctl.ring_full[st], u.h * D + kc * 64, krow);
          for (int kc = 0; kc < Cfg::VCH; ++kc)
            ptx::tma_load_2d(dst + Cfg::TQ + kc * Cfg::CHUNK, &tm_v, &ctl.ring_full[st], u.h * DV + kc * 64, krow);
          ++kv_it;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = ptx::elect_one_sync();
    constexpr uint32_t idesc_s = ptx::idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);
    constexpr uint32_t idesc_dq = ptx::idesc_f16_f32acc(BF16, true, kBlockM, D);
    const uint32_t q_base = ptx::smem_u32(sQ), do_base = ptx::smem_u32(sDO), kv_base = ptx::smem_u32(sKV);
    int one_it = 0, kv_it = 0, t_it = 0, u_it = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
      const BwdUnit u = decode_bwd_unit(p, p.units[ui]);
      const int nt = query_tile_kv_tiles(u.s, u.L, u.t).count;
      if (nt == 0) continue;
      if (!bwd_warp_wait(ctl, p, &ctl.one_full, one_it & 1)) break;
      ptx::tc_fence_after();
      for (int t = 0; t < nt; ++t) {
        const int st = kv_it & 1;
        if (!bwd_warp_wait(ctl, p, &ctl.ring_full[st], (kv_it >> 1) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t k_base = kv_base + st * (Cfg::TQ + Cfg::TV);
        if (leader) {
          mma_ss_kmajor<D / 16>(tmem, q_base, k_base, idesc_s);                  // S = Q K^T
          mma_ss_kmajor<DV / 16>(tmem + 128, do_base, k_base + Cfg::TQ, idesc_s);  // dP = dO V^T
          ptx::umma_commit(&ctl.s_full);
        }
        __syncwarp();
        if (!bwd_warp_wait(ctl, p, &ctl.p_full, t_it & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        if (t == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.acc_empty, (u_it & 1) ^ 1)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        if (leader) {
          mma_ts_mnmajor(tmem + 256, tmem, k_base, idesc_dq, t > 0);   // dQ += dS K
          ptx::umma_commit(&ctl.ring_empty[st]);
          if (t == nt - 1) {
            ptx::umma_commit(&ctl.one_empty);
            ptx::umma_commit(&ctl.acc_full);
          }
        }
        __syncwarp();
        ++kv_it;
        ++t_it;
      }
      ++one_it;
      ++u_it;
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const int c0 = wg * 64;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float alpha = p.alpha;
    constexpr float kLog2e = 1.4426950408889634f;
    int t_it = 0, u_it = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
      const BwdUnit u = decode_bwd_unit(p, p.units[ui]);
      const TileSet ts = query_tile_kv_tiles(u.s, u.L, u.t);
      const TileBounds tb = q_tile_bounds(u.s, u.L, u.t);
      const int nt = ts.count;
      const int qr = q_row(u.s, u.L, u.t, rloc);
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      const long long grow = static_cast<long long>(u.s.q0) + row;
      uint16_t* dq_row = reinterpret_cast<uint16_t*>(p.dq) + grow * p.dq_stride + u.h * D;
      if (nt == 0) {   // no key reaches this tile: dQ = 0
        if (valid) {
#pragma unroll
          for (int c = 0; c < D / 2; c += 8)
            *reinterpret_cast<uint4*>(dq_row + wg * (D / 2) + c) = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      int r_lo, r_hi;
      row_uih_keys(u.s, row, r_lo, r_hi);
      int r_diag = row_diag_key(u.s, row);
      int r_ctx = u.s.c;
      if (!valid) { r_lo = r_hi = 0; r_diag = -1; r_ctx = 0; }
      float lse2 = 0.f, dlt = 0.f;
      if constexpr (SOFTMAX) {
        if (valid) {
          lse2 = p.lse[static_cast<long long>(u.h) * p.total_q + grow] * kLog2e;
          dlt = p.delta[static_cast<long long>(u.h) * p.total_q + grow];
        }
      }
      const FullTiles ft = full_tile_ranges(u.s, tb);
      for (int idx = 0; idx < nt && ok; ++idx) {
        const int n = tileset_at(ts, idx);
        const bool full = n < ft.ctx_hi || (n >= ft.lo && n < ft.hi);
        const int j0 = n * kBlockN;
        RowMask rm;
        rm.ctx = r_ctx - j0;
        rm.lo = r_lo - j0;
        rm.span = static_cast<uint32_t>(r_hi - r_lo);
        rm.diag = r_diag >= 0 ? r_diag - j0 : -1000000;
        if (!bwd_warp_wait(ctl, p, &ctl.s_full, t_it & 1)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tmem + lane_base + c0 + 32 * q, sv);
          ptx::tmem_ld32(tmem + lane_base + 128 + c0 + 32 * q, dv);
          ptx::tmem_ld_wait(sv);
          ptx::tmem_ld_wait(dv);
          const uint32_t mb = full ? 0xFFFFFFFFu : rm.bits32(c0 + 32 * q);
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float s = __uint_as_float(sv[k + e]);
              const float dp = __uint_as_float(dv[k + e]);
              float r;
              if constexpr (SOFTMAX) {
                const float pr = ex2_approx(fmaf(s, alpha * kLog2e, -lse2));
                r = pr * fmaf(dp, u.scale, -dlt);
              } else {
                const float x = alpha * s;
                const float sig = fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);
                r = dp * u.scale * sig * fmaf(x, 1.f - sig, 1.f);
              }
              ds[e] = ((mb >> (k + e)) & 1u) ? r : 0.f;
            }
            pk[k >> 1] = pack2<BF16>(ds[0], ds[1]);
          }
          ptx::tmem_st16(tmem + lane_base + c0 + 16 * q, pk);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.p_full);
        ++t_it;
      }
      if (!ok) break;
      // dQ * alpha out of TMEM: this warpgroup's half of the D columns
      if (!bwd_warp_wait(ctl, p, &ctl.acc_full, u_it & 1)) break;
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 2; c += 32) {
        uint32_t o[32];
        ptx::tmem_ld32(tmem + lane_base + 256 + wg * (D / 2) + c, o);
        ptx::tmem_ld_wait(o);
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2)
            pk[k >> 1] = pack2<BF16>(__uint_as_float(o[k]) * alpha, __uint_as_float(o[k + 1]) * alpha);
#pragma unroll
          for (int k = 0; k < 16; k += 4)
            *reinterpret_cast<uint4*>(dq_row + wg * (D / 2) + c + 2 * k) =
                make_uint4(pk[k], pk[k + 1], pk[k + 2], pk[k + 3]);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl.acc_empty);
      ++u_it;
    }
  }

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
    ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------- dK, dV
template <int D, int DV, bool BF16, bool SOFTMAX>
__global__ void __launch_bounds__(kBwdThreads, 1)
    hstu_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_q8, const __grid_constant__ CUtensorMap tm_do8,
                         const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<D, DV>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;                    // K then V of the unit's key tile
  uint8_t* sV = smem + Cfg::TQ;
  uint8_t* sQD = sV + Cfg::TV;           // ring: Q then dO of a query tile per stage
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    ptx::mbar_init(&ctl.one_full, 1);
    ptx::mbar_init(&ctl.one_empty, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl.ring_full[i], 1);
      ptx::mbar_init(&ctl.ring_empty[i], 1);
    }
    ptx::mbar_init(&ctl.s_full, 1);
    ptx::mbar_init(&ctl.p_full, kEwThreads);
    ptx::mbar_init(&ctl.acc_full, 1);
    ptx::mbar_init(&ctl.acc_empty, kEwThreads);
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // S^T [0,128), dP^T [128,256), dV [256, 256 + DV), dK [256 + DV, 256 + DV + D)
  const uint32_t tmem = ctl.tmem_base;
  ptx::grid_dependency_wait();
  const int n_units = p.ws_header[kWsKvUnits];

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int u_it = 0, q_it = 0;
      bool ok = true;
      for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
        const BwdUnit u = decode_bwd_unit(p, p.kv_units[ui]);
        if (!bwd_wait(ctl, p, &ctl.one_empty, (u_it & 1) ^ 1)) break;
        ptx::mbar_arrive_expect_tx(&ctl.one_full, Cfg::TQ + Cfg::TV);
        const int krow = u.s.kv0 + u.t * kBlockN;
        for (int kc = 0; kc < Cfg::KCH; ++kc)
          ptx::tma_load_2d(sK + kc * Cfg::CHUNK, &tm_k, &ctl.one_full, u.h * D + kc * 64, krow);
        for (int kc = 0; kc < Cfg::VCH; ++kc)
          ptx::tma_load_2d(sV + kc * Cfg::CHUNK, &tm_v, &ctl.one_full, u.h * DV + kc * 64, krow);
        ++u_it;
        for (int m = 0; m < u.L.nq; ++m) {
          if (!tileset_has(load_qtile(p, u.b, m).ts, u.t)) continue;
          const int st = q_it & 1;
          if (!bwd_wait(ctl, p, &ctl.ring_empty[st], ((q_it >> 1) & 1) ^ 1)) { ok = false; break; }
          uint8_t* dst = sQD + st * (Cfg::TQ + Cfg::TV);
          ptx::mbar_arrive_expect_tx(&ctl.ring_full[st], Cfg::TQ + Cfg::TV);
          load_query_tile(&tm_q, &tm_q8, dst, &ctl.ring_full[st], u.s, u.L, m, u.h * D, Cfg::KCH);
          load_query_tile(&tm_do, &tm_do8, dst + Cfg::TQ, &ctl.ring_full[st], u.s, u.L, m, u.h * DV, Cfg::VCH);
          ++q_it;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = ptx::elect_one_sync();
    constexpr uint32_t idesc_s = ptx::idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);
    constexpr uint32_t idesc_dv = ptx::idesc_f16_f32acc(BF16, true, kBlockM, DV);
    constexpr uint32_t idesc_dk = ptx::idesc_f16_f32acc(BF16, true, kBlockM, D);
    const uint32_t k_base = ptx::smem_u32(sK), v_base = ptx::smem_u32(sV), qd_base = ptx::smem_u32(sQD);
    int u_it = 0, q_it = 0, t_it = 0, a_it = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
      const BwdUnit u = decode_bwd_unit(p, p.kv_units[ui]);
      if (!bwd_warp_wait(ctl, p, &ctl.one_full, u_it & 1)) break;
      ptx::tc_fence_after();
      int nm = 0;
      for (int m = 0; m < u.L.nq; ++m) {
        if (!tileset_has(load_qtile(p, u.b, m).ts, u.t)) continue;
        const int st = q_it & 1;
        if (!bwd_warp_wait(ctl, p, &ctl.ring_full[st], (q_it >> 1) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t q_b = qd_base + st * (Cfg::TQ + Cfg::TV);
        if (leader) {
          mma_ss_kmajor<D / 16>(tmem, k_base, q_b, idesc_s);                    // S^T = K Q^T
          mma_ss_kmajor<DV / 16>(tmem + 128, v_base, q_b + Cfg::TQ, idesc_s);   // dP^T = V dO^T
          ptx::umma_commit(&ctl.s_full);
        }
        __syncwarp();
        if (!bwd_warp_wait(ctl, p, &ctl.p_full, t_it & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        if (nm == 0) {
          if (!bwd_warp_wait(ctl, p, &ctl.acc_empty, (a_it & 1) ^ 1)) { ok = false; break; }
          ptx::tc_fence_after();
        }
        if (leader) {
          mma_ts_mnmajor(tmem + 256, tmem, q_b + Cfg::TQ, idesc_dv, nm > 0);         // dV += P^T dO
          mma_ts_mnmajor(tmem + 256 + DV, tmem + 128, q_b, idesc_dk, nm > 0);       // dK += dS^T Q
          ptx::umma_commit(&ctl.ring_empty[st]);
        }
        __syncwarp();
        ++q_it;
        ++t_it;
        ++nm;
      }
      if (!ok) break;
      if (leader) {
        ptx::umma_commit(&ctl.one_empty);
        if (nm > 0) ptx::umma_commit(&ctl.acc_full);
      }
      __syncwarp();
      if (nm > 0) ++a_it;
      ++u_it;
    }
  } else {
    // ------------------------------------------------------------ elementwise warpgroups
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const int c0 = wg * 64;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float alpha = p.alpha;
    constexpr float kLog2e = 1.4426950408889634f;
    int t_it = 0, a_it = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < n_units && ok && !ctl.abort_flag; ui += gridDim.x) {
      const BwdUnit u = decode_bwd_unit(p, p.kv_units[ui]);
      const int j = u.t * kBlockN + rloc;   // this lane's key row
      const bool kvalid = j < u.s.Lkv;
      const long long krow = static_cast<long long>(u.s.kv0) + j;
      uint16_t* dv_row = reinterpret_cast<uint16_t*>(p.dv) + krow * p.dv_stride + u.h * DV;
      uint16_t* dk_row = reinterpret_cast<uint16_t*>(p.dk) + krow * p.dk_stride + u.h * D;
      int nm = 0;
      for (int m = 0; m < u.L.nq && ok; ++m) {
        const QTileRec rec = load_qtile(p, u.b, m);
        if (!tileset_has(rec.ts, u.t)) continue;
        const FullTiles ft = full_tile_ranges(u.s, rec.tb);
        const bool full = u.t < ft.ctx_hi || (u.t >= ft.lo && u.t < ft.hi);
        if (!bwd_warp_wait(ctl, p, &ctl.s_full, t_it & 1)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll 1
        for (int q = 0; q < 2; ++q) {
          // column (query) of this lane: its row, validity and, for a partial
          // block, its allowed key interval, shared with the other lanes
          const int col = c0 + 32 * q + lane;
          const int qi = q_row(u.s, u.L, m, col);
          const uint32_t cvalid = __ballot_sync(0xffffffffu, qi >= 0);
          int c_lo = 0, c_hi = 0, c_dg = -1;
          if (!full && qi >= 0) {
            row_uih_keys(u.s, qi, c_lo, c_hi);
            c_dg = row_diag_key(u.s, qi);
          }
          float c_lse2 = 0.f, c_dlt = 0.f;
          if constexpr (SOFTMAX) {
            if (qi >= 0) {
              const long long gq = static_cast<long long>(u.h) * p.total_q + u.s.q0 + qi;
              c_lse2 = p.lse[gq] * kLog2e;
              c_dlt = p.delta[gq];
            }
          }
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tmem + lane_base + c0 + 32 * q, sv);
          ptx::tmem_ld32(tmem + lane_base + 128 + c0 + 32 * q, dv);
          ptx::tmem_ld_wait(sv);
          ptx::tmem_ld_wait(dv);
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float pv[2], ds[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int kk = k + e;
              bool allowed = (cvalid >> kk) & 1u;
              if (!full) {
                const int lo = __shfl_sync(0xffffffffu, c_lo, kk);
                const int hi = __shfl_sync(0xffffffffu, c_hi, kk);
                const int dg = __shfl_sync(0xffffffffu, c_dg, kk);
                allowed = allowed && (j < u.s.c || (j >= lo && j < hi) || j == dg);
              }
              const float s = __uint_as_float(sv[kk]);
              const float dp = __uint_as_float(dv[kk]);
              float a, r;
              if constexpr (SOFTMAX) {
                const float l2 = __shfl_sync(0xffffffffu, c_lse2, kk);
                const float dl = __shfl_sync(0xffffffffu, c_dlt, kk);
                a = ex2_approx(fmaf(s, alpha * kLog2e, -l2));
                r = a * fmaf(dp, u.scale, -dl);
              } else {
                const float x = alpha * s;
                const float sig = fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);
                a = x * sig;
                r = dp * u.scale * sig * fmaf(x, 1.f - sig, 1.f);
              }
              pv[e] = allowed ? a : 0.f;
              ds[e] = allowed ? r : 0.f;
            }
            pp[k >> 1] = pack2<BF16>(pv[0], pv[1]);
            pd[k >> 1] = pack2<BF16>(ds[0], ds[1]);
          }
          ptx::tmem_st16(tmem + lane_base + c0 + 16 * q, pp);
          ptx::tmem_st16(tmem + lane_base + 128 + c0 + 16 * q, pd);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.p_full);
        ++t_it;
        ++nm;
      }
      if (!ok) break;
      // dV * attn_scale and dK * alpha: this warpgroup's half of each
      if (nm > 0) {
        if (!bwd_warp_wait(ctl, p, &ctl.acc_full, a_it & 1)) break;
        ptx::tc_fence_after();
      }
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {
        const int W = part == 0 ? DV : D;
        const float mul = part == 0 ? u.scale : alpha;
        const uint32_t col0 = 256 + (part == 0 ? 0 : DV) + wg * (W / 2);
        uint16_t* dst = (part == 0 ? dv_row : dk_row) + wg * (W / 2);
#pragma unroll 1
        for (int c = 0; c < W / 2; c += 32) {
          uint32_t o[32];
          if (nm > 0) {
            ptx::tmem_ld32(tmem + lane_base + col0 + c, o);
            ptx::tmem_ld_wait(o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
          if (kvalid) {
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2)
              pk[k >> 1] = pack2<BF16>(__uint_as_float(o[k]) * mul, __uint_as_float(o[k + 1]) * mul);
#pragma unroll
            for (int k = 0; k < 16; k += 4)
              *reinterpret_cast<uint4*>(dst + c + 2 * k) = make_uint4(pk[k], pk[k + 1], pk[k + 2], pk[k + 3]);
          }
        }
      }
      if (nm > 0) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.acc_empty);
        ++a_it;
      }
    }
  }

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
    ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

}  // namespace hstu

namespace hstu {

// Host side: both backward kernels of one head dimension, the dQ kernel first.
template <int D, bool BF16, bool SOFTMAX>
cudaError_t launch_bwd_pair(const BwdMaps& m, const BwdParams& p, int grid_q, int grid_kv, cudaStream_t stream) {
  constexpr int smem = BwdCfg<D, D>::SMEM_BYTES;
  auto kq = hstu_bwd_dq_kernel<D, D, BF16, SOFTMAX>;
  auto kkv = hstu_bwd_dkdv_kernel<D, D, BF16, SOFTMAX>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_done[64] = {};
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  kq<<<grid_q, kBwdThreads, smem, stream>>>(m.q, m.k, m.v, m.d_o, m.q8, m.d_o8, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kkv<<<grid_kv, kBwdThreads, smem, stream>>>(m.q, m.k, m.v, m.d_o, m.q8, m.d_o8, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dispatch(const BwdMaps& m, const BwdParams& p, bool bf16, bool softmax, int grid_q,
                                int grid_kv, cudaStream_t stream) {
  if (bf16) return softmax ? launch_bwd_pair<D, true, true>(m, p, grid_q, grid_kv, stream)
                           : launch_bwd_pair<D, true, false>(m, p, grid_q, grid_kv, stream);
  return softmax ? launch_bwd_pair<D, false, true>(m, p, grid_q, grid_kv, stream)
                 : launch_bwd_pair<D, false, false>(m, p, grid_q, grid_kv, stream);
}

}  // namespace hstu
