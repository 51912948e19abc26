// HSTU attention forward on CTA pairs (hdim 128, no bias) for sm_103a.
//
// The same computation as hstu_fwd_kernel (composable_kernel
// 18_hstu_attention README, "Forward computation"), with the work unit widened
// to two query tiles of one (sequence, head, split): the higher tile on the
// even CTA of a two-CTA cluster, the one below it on the odd CTA, both run
// against the union of their key tiles.  Both products of a key tile are one
// tcgen05.mma of cta_group::2 with M = 256, issued by the even CTA:
//     S = Q K^T    A = each CTA's own 128 query rows, B = K split by key:
//                  keys [0, 64) of the tile in the even CTA, [64, 128) in the odd
//     O += P V     A = each CTA's P in its own TMEM, B = V split by column:
//                  hdim columns [0, 64) in the even CTA, [64, 128) in the odd
// Each CTA therefore loads half of every K and V tile and its tensor core reads
// 6 KB of shared memory per 128x128x16 step instead of 8 KB: the single-CTA
// kernel's tile is bound by shared-memory bandwidth (operand reads plus the TMA
// writes of K and V), not by the MMA rate.
//
// A key tile outside one CTA's own tile set is fully masked for its rows and
// contributes nothing; a unit whose lower tile does not exist (the first tile of
// a sequence with an odd number of tiles) runs the odd CTA on no rows.
//
// Roles per CTA: warp 0 loads Q and this CTA's half of K (lane 0) and its half
// of V (lane 1); warps 2..5 the epilogue, warps 6..13 the elementwise groups
// (own rows, own TMEM), as in hstu_fwd_kernel.  The even CTA also runs the
// scheduler (warp 14), which publishes each unit to both CTAs, and two MMA
// issuers: Q K^T (warp 1) and P V (warp 15).  TMEM holds three score buffers
// and one O accumulator, so the scores run up to three tiles ahead of P V;
// the epilogue reads a unit's whole O row before storing it, to hand the
// single buffer back early.  Barriers the issuers wait on live in the even
// CTA: the odd CTA's copies complete on them and its warps arrive on them
// through shared::cluster addresses.  Commits reach the barriers of both CTAs
// (multicast).  Every wait is bounded.
//
// Measured on the large jagged workload it is slower than the single-CTA
// kernel (the tile is bound by the elementwise pass and the MMA hand-offs, not
// by shared-memory bandwidth), so the library runs it only when asked
// (hstu_fwd_args::cta_pairs = 1).
#pragma once
#include "hstu_fwd_kernel.cuh"

namespace hstu {

template <bool SOFTMAX>
struct PairCfg {
  static constexpr int D = 128, DV = 128;
  static constexpr int CHUNK_BYTES = kBlockM * 128;       // 128 rows x 128 bytes (64 columns)
  static constexpr int QTILE_BYTES = 2 * CHUNK_BYTES;     // this CTA's 128 query rows
  static constexpr int KHALF_CHUNK = (kBlockN / 2) * 128; // 64 key rows x 128 bytes
  static constexpr int KHALF_BYTES = 2 * KHALF_CHUNK;     // this CTA's 64 keys of a K tile
  static constexpr int VHALF_BYTES = CHUNK_BYTES;         // 128 keys x this CTA's 64 V columns
  static constexpr int QBUF = 2, KSTAGES = 4, VSTAGES = 3;
  static constexpr int TILES_BYTES = QBUF * QTILE_BYTES + KSTAGES * KHALF_BYTES + VSTAGES * VHALF_BYTES;
  static constexpr int STAGE_BOX_BYTES = 32 * 128;
  static constexpr int STAGE_BUFS = 2;
  static constexpr int STAGE_BYTES = STAGE_BUFS * kFwdEpiWarps * STAGE_BOX_BYTES;
  static constexpr int SOFTMAX_BYTES = SOFTMAX ? static_cast<int>(sizeof(SoftmaxScratch)) : 0;
  static constexpr int SMEM_BYTES = TILES_BYTES + STAGE_BYTES + SOFTMAX_BYTES + 1024;
  // TMEM: three 128-column score buffers (P packed over each, as in the
  // single-CTA kernel), then one O accumulator
  static constexpr int SBUF = 3;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = SBUF * 128;
  static_assert(O_COL + DV <= TMEM_COLS, "TMEM budget");
};

// Units published ahead of the slowest consumer (the pair kernel's ring).
constexpr int kPairSchedDepth = 2;

// One CTA's view of a pair unit.
struct alignas(16) PairView {
  UnitView u;      // u.m: this CTA's query tile, < 0 for none; u.ts, k0, k1: the pair's key tiles
  int live;        // 0: no more units
  int peer_rows;   // (even CTA) the odd CTA holds a query tile in this unit
};

struct PairSmemCtl {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[3], p_full[3], pv_done[3];
  uint64_t o_full, o_empty;
  uint64_t sched_full[kPairSchedDepth], sched_empty[kPairSchedDepth];
  uint64_t xch[2];
  uint64_t rs_full, rs_empty;
  PairView view[kPairSchedDepth];
  uint32_t tmem_base;
  volatile int abort_flag;
  uint8_t f_order[kFusedMaxBatch];
  int f_ubase[kFusedMaxBatch + 1];
  float f_pscale[kFusedMaxBatch];
  int f_err;
};

// Consumers of a published unit: Q/K and V producers (lanes 0 and 1 of warp
// 0), epilogue and elementwise warps in both CTAs, and the two MMA issuers in
// the even one.
constexpr int kPairSchedArrivals = 2 * (2 + kEpiWarps + kEwThreads / 32) + 2;

// The union of two tile sets as a tile set: sorted, disjoint, empty slots last.
// When more than three ranges remain, the third grows to cover the rest (its
// extra tiles are fully masked for every row and add nothing).
__device__ __forceinline__ TileSet tileset_union(const TileSet& a, const TileSet& b) {
  int lo[6] = {a.lo0, a.lo1, a.lo2, b.lo0, b.lo1, b.lo2};
  int hi[6] = {a.hi0, a.hi1, a.hi2, b.hi0, b.hi1, b.hi2};
#pragma unroll
  for (int i = 1; i < 6; ++i)
#pragma unroll
    for (int j = i; j > 0; --j)
      if (lo[j] < lo[j - 1]) {
        const int tl = lo[j], th = hi[j];
        lo[j] = lo[j - 1]; hi[j] = hi[j - 1];
        lo[j - 1] = tl; hi[j - 1] = th;
      }
  int rl[3] = {kNoTile, kNoTile, kNoTile}, rh[3] = {kNoTile, kNoTile, kNoTile};
  int n = 0;
#pragma unroll
  for (int i = 0; i < 6; ++i) {
    if (lo[i] == kNoTile || hi[i] <= lo[i]) continue;
    if (n > 0 && lo[i] <= rh[n - 1]) {
      rh[n - 1] = hi[i] > rh[n - 1] ? hi[i] : rh[n - 1];
    } else if (n == 3) {
      rh[2] = hi[i] > rh[2] ? hi[i] : rh[2];
    } else {
      rl[n] = lo[i];
      rh[n] = hi[i];
      ++n;
    }
  }
  TileSet t;
  t.lo0 = rl[0]; t.hi0 = rh[0];
  t.lo1 = rl[1]; t.hi1 = rh[1];
  t.lo2 = rl[2]; t.hi2 = rh[2];
  t.count = (t.hi0 - t.lo0) + (t.hi1 - t.lo1) + (t.hi2 - t.lo2);
  return t;
}

// Pair unit `unit` of the in-kernel schedule: per sequence position, heads
// outer, tile pairs (nq-1, nq-2), (nq-3, nq-4), ... and splits innermost.
__device__ __forceinline__ void decode_pair_unit(const FwdParams& p, const PairSmemCtl& ctl, int unit,
                                                 PairView& even, PairView& odd) {
  const int pos = seg_find(ctl.f_ubase, p.batch, unit);
  const int b = ctl.f_order[pos];
  UnitView u;
  u.g = b / p.batch_per_group;
  u.s = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[u.g], p.loc[u.g], p.mf[u.g], p.causal, p.self_attn,
                  p.kv_targets);
  u.L = q_layout(u.s);
  const int local = unit - ctl.f_ubase[pos];
  const int per_h = ((u.L.nq + 1) >> 1) * p.splits;
  u.h = local / per_h;
  const int rem = local - u.h * per_h;
  const int pi = rem / p.splits;
  u.sp = rem - pi * p.splits;
  const int m0 = u.L.nq - 1 - 2 * pi, m1 = m0 - 1;
  const TileBounds tb0 = q_tile_bounds(u.s, u.L, m0);
  const TileBounds tb1 = m1 >= 0 ? q_tile_bounds(u.s, u.L, m1) : tb0;
  TileSet ts = query_tile_kv_tiles(u.s, u.L, m0, tb0);
  if (m1 >= 0) ts = tileset_union(ts, query_tile_kv_tiles(u.s, u.L, m1, tb1));
  u.ts = ts;
  split_range(ts.count, u.sp, p.splits, u.k0, u.k1);
  u.scale = ctl.f_pscale[pos];
  even.u = u;
  even.u.m = m0;
  even.u.tb = tb0;
  odd.u = u;
  odd.u.m = m1;
  odd.u.tb = tb1;
  even.live = odd.live = 1;
  even.peer_rows = m1 >= 0 ? 1 : 0;
  odd.peer_rows = 1;
}

template <typename Ctl>
__device__ __forceinline__ bool wait_cl_or_abort(Ctl& ctl, const FwdParams& p, uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_wait_cluster(bar, parity, kWaitLimitNs)) return true;
  ctl.abort_flag = 1;
  atomicOr(&p.ws_header[kWsError], kErrTimeout);
  return false;
}
// warp_wait_or_abort for a barrier that the other CTA arrives on.
template <typename Ctl>
__device__ __forceinline__ bool warp_wait_cl_or_abort(Ctl& ctl, const FwdParams& p, uint64_t* bar,
                                                      uint32_t parity) {
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_cluster(bar, parity, kWaitLimitNs));
  if (!ok) {
    ctl.abort_flag = 1;
    atomicOr(&p.ws_header[kWsError], kErrTimeout);
  }
  return ok;
}

// The shared::cluster address of a barrier of the even CTA (the same offset in both).
__device__ __forceinline__ uint32_t even_bar(uint64_t* bar) { return ptx::mapa(ptx::smem_u32(bar), 0); }

template <bool BF16, bool SOFTMAX>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFwdThreads, 1)
    hstu_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k64,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q8,
                         const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ FwdParams p) {
  using Cfg = PairCfg<SOFTMAX>;
  constexpr int D = Cfg::D;
  constexpr int DV = Cfg::DV;
  constexpr int KST = Cfg::KSTAGES;
  constexpr int VST = Cfg::VSTAGES;
  constexpr int SB = Cfg::SBUF;
  constexpr int QB = Cfg::QBUF;
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairSmemCtl ctl;
  // the same offsets in both CTAs: the MMA's descriptors address both
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + QB * Cfg::QTILE_BYTES;
  uint8_t* sV = sK + KST * Cfg::KHALF_BYTES;
  uint8_t* sStage = smem + Cfg::TILES_BYTES;
  SoftmaxScratch* sx = reinterpret_cast<SoftmaxScratch*>(smem + Cfg::TILES_BYTES + Cfg::STAGE_BYTES);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int rank = static_cast<int>(ptx::cluster_ctarank());
  const bool even = rank == 0;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&ctl.q_full[s], 1);
      ptx::mbar_init(&ctl.q_empty[s], 1);
    }
    for (int s = 0; s < KST; ++s) {
      ptx::mbar_init(&ctl.k_full[s], 1);
      ptx::mbar_init(&ctl.k_empty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      ptx::mbar_init(&ctl.v_full[s], 1);
      ptx::mbar_init(&ctl.v_empty[s], 1);
    }
    for (int s = 0; s < SB; ++s) {
      ptx::mbar_init(&ctl.s_full[s], 1);
      ptx::mbar_init(&ctl.p_full[s], 2 * (kEwThreads / 32));   // one per elementwise warp of each CTA
      ptx::mbar_init(&ctl.pv_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) ptx::mbar_init(&ctl.xch[s], kEwThreads);
    ptx::mbar_init(&ctl.o_full, 1);
    ptx::mbar_init(&ctl.o_empty, 2 * kEpiWarps);                 // one per epilogue warp of each CTA
    ptx::mbar_init(&ctl.rs_full, kEwThreads);
    ptx::mbar_init(&ctl.rs_empty, 32 * kEpiWarps);
    for (int s = 0; s < kPairSchedDepth; ++s) {
      ptx::mbar_init(&ctl.sched_full[s], 1);
      ptx::mbar_init(&ctl.sched_empty[s], kPairSchedArrivals);
    }
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k64);
    ptx::prefetch_tensormap(&tm_v);
    ptx::prefetch_tensormap(&tm_o);
  }
  // both CTAs' barriers exist before any copy or arrival reaches them
  ptx::cluster_sync();
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl.tmem_base, Cfg::TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // The even CTA orders the units (FwdParams::fused: the host uses this kernel
  // only for batches it schedules in-kernel); the dynamic claims wait for the
  // header reset that precedes this kernel on the stream.
  int n_units = 0;
  if (even) {
    n_units = fused_schedule<2>(p, ctl, reinterpret_cast<int*>(sK), tid, kFwdThreads);
    if (tid == 64 && (ctl.f_err != 0 || ptx::cluster_id_x() == 0)) {
      ptx::grid_dependency_wait();
      if (ctl.f_err != 0) atomicOr(&p.ws_header[kWsError], ctl.f_err);
      else p.ws_header[kWsUnits] = n_units;   // read by the combine kernel
    }
  }

  // reads the next published unit of ring slot (it % kPairSchedDepth) and frees the slot
  auto take = [&](int& sched_it, PairView& v, bool whole_warp) -> bool {
    const int slot = sched_it % kPairSchedDepth;
    const uint32_t par = (sched_it / kPairSchedDepth) & 1;
    const bool ok = whole_warp ? warp_wait_cl_or_abort(ctl, p, &ctl.sched_full[slot], par)
                               : wait_cl_or_abort(ctl, p, &ctl.sched_full[slot], par);
    if (!ok) return false;
    v = ctl.view[slot];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) ptx::mbar_arrive_remote(even_bar(&ctl.sched_empty[slot]));
    ++sched_it;
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ Q / K producer
    if (lane == 0) {
      int q_it = 0, kv_it = 0, sched_it = 0;
      while (!ctl.abort_flag) {
        PairView cur;
        if (!take(sched_it, cur, false) || !cur.live) break;
        const UnitView& u = cur.u;
        if (u.k1 <= u.k0) continue;
        const int qb = q_it % QB;
        if (!wait_or_abort(ctl, p, &ctl.q_empty[qb], ((q_it / QB) & 1) ^ 1)) break;
        if (even) ptx::mbar_arrive_expect_tx(&ctl.q_full[qb], Cfg::QTILE_BYTES * (1 + cur.peer_rows));
        const uint32_t qbar = even_bar(&ctl.q_full[qb]);
        if (u.m >= 0) {
          const int qrow = u.m * kBlockM;
          uint8_t* qdst = sQ + qb * Cfg::QTILE_BYTES;
          if (!(u.L.ctx_lane0 >= 0 && u.m == u.L.nq - 1)) {
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
              ptx::tma_load_2d_pair(qdst + kc * Cfg::CHUNK_BYTES, &tm_q, qbar, u.h * D + kc * 64, u.s.q0 + qrow);
          } else {
            // own rows on lanes [0, ctx_lane0), the context rows above: 8-row boxes
            const int lane0 = u.L.ctx_lane0;
            for (int g = 0; g < kBlockM / 8; ++g) {
              const int row = g * 8 < lane0 ? qrow + g * 8 : (g * 8 - lane0);
#pragma unroll
              for (int kc = 0; kc < 2; ++kc)
                ptx::tma_load_2d_pair(qdst + kc * Cfg::CHUNK_BYTES + g * 1024, &tm_q8, qbar, u.h * D + kc * 64,
                                      u.s.q0 + row);
            }
          }
        }
        ++q_it;
        bool ok = true;
        for (int k = u.k0; k < u.k1; ++k) {
          const int krow = u.s.kv0 + tileset_at(u.ts, k) * kBlockN + rank * (kBlockN / 2);
          const int ks = kv_it % KST;
          if (!wait_or_abort(ctl, p, &ctl.k_empty[ks], ((kv_it / KST) & 1) ^ 1)) { ok = false; break; }
          if (even) ptx::mbar_arrive_expect_tx(&ctl.k_full[ks], 2 * Cfg::KHALF_BYTES);
          const uint32_t kbar = even_bar(&ctl.k_full[ks]);
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
            ptx::tma_load_2d_pair(sK + ks * Cfg::KHALF_BYTES + kc * Cfg::KHALF_CHUNK, &tm_k64, kbar,
                                  u.h * D + kc * 64, krow);
          ++kv_it;
        }
        if (!ok) break;
      }
    }
    if (lane == 1) {
      // ---------------------------------------------------------- V producer (lane 1)
      int kv_it = 0, sched_it = 0;
      while (!ctl.abort_flag) {
        PairView cur;
        if (!take(sched_it, cur, false) || !cur.live) break;
        const UnitView& u = cur.u;
        bool ok = true;
        for (int k = u.k0; k < u.k1; ++k) {
          const int vs = kv_it % VST;
          const int vrow = u.s.kv0 + tileset_at(u.ts, k) * kBlockN;
          if (!wait_or_abort(ctl, p, &ctl.v_empty[vs], ((kv_it / VST) & 1) ^ 1)) { ok = false; break; }
          if (even) ptx::mbar_arrive_expect_tx(&ctl.v_full[vs], 2 * Cfg::VHALF_BYTES);
          ptx::tma_load_2d_pair(sV + vs * Cfg::VHALF_BYTES, &tm_v, even_bar(&ctl.v_full[vs]), u.h * DV + rank * 64,
                                vrow);
          ++kv_it;
        }
        if (!ok) break;
      }
    }
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler (even CTA)
    // Claims pair units (the cluster's first is its own index, the queue hands
    // out the rest from the cluster count on), decodes both CTAs' views and
    // publishes them into the same ring slot of each CTA.
    if (even) {
      int sched_it = 0;
      bool first = true, waited = false;
      const int n_clusters = static_cast<int>(ptx::nclusters_x());
      while (!ctl.abort_flag) {
        bool ok = true, live = false;
        if (lane == 0) {
          int id;
          if (first) {
            id = static_cast<int>(ptx::cluster_id_x());
          } else {
            if (!waited) {
              ptx::grid_dependency_wait();
              waited = true;
            }
            id = atomicAdd(&p.ws_header[kWsCounter], 1) + n_clusters;
          }
          live = id < n_units;
          PairView ev, od;
          if (live) decode_pair_unit(p, ctl, id, ev, od);
          ev.live = od.live = live ? 1 : 0;
          const int slot = sched_it % kPairSchedDepth;
          ok = wait_or_abort(ctl, p, &ctl.sched_empty[slot], ((sched_it / kPairSchedDepth) & 1) ^ 1);
          if (ok) {
            ctl.view[slot] = ev;
            const uint32_t dst = ptx::mapa(ptx::smem_u32(&ctl.view[slot]), 1);
            const uint4* src = reinterpret_cast<const uint4*>(&od);
#pragma unroll
            for (int i = 0; i < static_cast<int>(sizeof(PairView) / 16); ++i)
              ptx::st_cluster_v4(dst + 16 * i, src[i].x, src[i].y, src[i].z, src[i].w);
            ptx::mbar_arrive(&ctl.sched_full[slot]);
            // the odd CTA's view, written above, before its consumers see the slot
            ptx::fence_acq_rel_cluster();
            ptx::mbar_arrive_cluster(ptx::mapa(ptx::smem_u32(&ctl.sched_full[slot]), 1));
          }
        }
        first = false;
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        if (!__shfl_sync(0xffffffffu, live ? 1 : 0, 0)) break;
        ++sched_it;
      }
    }
  } else if (warp == 1 || warp == kVProdWarp) {
    // ------------------------------------------------------------ MMA issuers (even CTA)
    // Two warps walk the same stream of tiles (the units' key tiles, in
    // order): warp 1 issues Q K^T, warp 15 issues P V, so neither warp's waits
    // sit in the other's way.  Q K^T of tile t goes into S buffer t % 3 once
    // the P V that read that buffer (tile t - 3) has completed (its commit):
    // the scores run up to three tiles ahead of P V.
    if (even) {
      const bool is_qk = warp == 1;
      const bool leader = ptx::elect_one_sync();
      constexpr uint32_t idesc_qk = ptx::idesc_f16_f32acc(BF16, false, 2 * kBlockM, kBlockN);
      constexpr uint32_t idesc_pv = ptx::idesc_f16_f32acc(BF16, true, 2 * kBlockM, DV);
      constexpr uint16_t kBoth = 3;
      const uint64_t q_desc = ptx::sdesc_sw128(ptx::smem_u32(sQ), 16, 1024);
      const uint32_t k_base = ptx::smem_u32(sK);
      const uint32_t v_base = ptx::smem_u32(sV);
      int sched_it = 0, q_it = 0, kv_it = 0, t_in = 0, nt = 0, qb = 0, q_round = 0;
      bool ok = true;
      for (int si = 0; ok && !ctl.abort_flag; ++si) {
        // the next tile of the stream (empty split units have none)
        bool end = false;
        while (t_in >= nt) {
          PairView v;
          if (!take(sched_it, v, true)) { ok = false; break; }
          if (!v.live) { end = true; break; }
          nt = v.u.k1 - v.u.k0;
          t_in = 0;
          if (nt > 0) {
            qb = q_it % QB;
            q_round = q_it++;
          }
        }
        if (!ok || end) break;
        const int kvi = kv_it++;
        const bool first = t_in == 0, last = t_in == nt - 1;
        ++t_in;
        const int sb = si % SB;
        if (is_qk) {
          if (si >= SB && !warp_wait_or_abort(ctl, p, &ctl.pv_done[sb], ((si - SB) / SB) & 1)) { ok = false; break; }
          if (first && !warp_wait_or_abort(ctl, p, &ctl.q_full[qb], (q_round / QB) & 1)) { ok = false; break; }
          const int st = kvi % KST;
          if (!warp_wait_or_abort(ctl, p, &ctl.k_full[st], (kvi / KST) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t k_desc = ptx::sdesc_sw128(k_base + st * Cfg::KHALF_BYTES, 16, 1024);
          uint64_t ad[8], bd[8];
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            ad[ks] = q_desc + static_cast<uint64_t>((qb * Cfg::QTILE_BYTES) >> 4) +
                     static_cast<uint64_t>(((ks >> 2) * Cfg::CHUNK_BYTES + (ks & 3) * 32) >> 4);
            bd[ks] = k_desc + static_cast<uint64_t>(((ks >> 2) * Cfg::KHALF_CHUNK + (ks & 3) * 32) >> 4);
          }
          if (leader) {
            ptx::umma_ss_x8_pair(tmem + sb * 128, ad, bd, idesc_qk, 0u);
            ptx::umma_commit_pair(&ctl.k_empty[st], kBoth);
            ptx::umma_commit_pair(&ctl.s_full[sb], kBoth);
            if (last) ptx::umma_commit_pair(&ctl.q_empty[qb], kBoth);   // the unit's Q may be replaced
          }
          __syncwarp();
        } else {
          const int st = kvi % VST;
          if (!warp_wait_or_abort(ctl, p, &ctl.v_full[st], (kvi / VST) & 1)) { ok = false; break; }
          if (first && !warp_wait_or_abort(ctl, p, &ctl.o_empty, (q_round & 1) ^ 1)) { ok = false; break; }
          if (!warp_wait_or_abort(ctl, p, &ctl.p_full[sb], (si / SB) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint64_t v_desc = ptx::sdesc_sw128(v_base + st * Cfg::VHALF_BYTES, Cfg::CHUNK_BYTES, 1024);
          uint32_t pa[8];
          uint64_t vd[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            pa[kk] = tmem + sb * 128 + (kk >> 2) * 64 + (kk & 3) * 8;
            vd[kk] = v_desc + static_cast<uint64_t>((kk * 2048) >> 4);
          }
          if (leader) {
            ptx::umma_ts_x8_pair(tmem + Cfg::O_COL, pa, vd, idesc_pv, first ? 0u : 1u);
            ptx::umma_commit_pair(&ctl.v_empty[st], kBoth);
            ptx::umma_commit_pair(&ctl.pv_done[sb], kBoth);   // frees S buffer sb for Q K^T of tile si + 3
            if (last) ptx::umma_commit_pair(&ctl.o_full, kBoth);
          }
          __syncwarp();
        }
      }
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue warpgroup
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t stage_warp = ptx::smem_u32(sStage) + (warp - 2) * Cfg::STAGE_BUFS * Cfg::STAGE_BOX_BYTES;
    int st_it = 0;
    int q_it = 0, sched_it = 0;
    while (!ctl.abort_flag) {
      PairView cur;
      if (!take(sched_it, cur, true) || !cur.live) break;
      const UnitView& u = cur.u;
      const int nt = u.k1 - u.k0;
      const int qr = u.m >= 0 ? q_row(u.s, u.L, u.m, rloc) : -1;
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      const long long grow = static_cast<long long>(u.s.q0) + row;
      const uint32_t o_tmem = tmem + lane_base + Cfg::O_COL;
      float m_run = -INFINITY, l_run = 0.f;
      if (nt > 0) {
        if (!warp_wait_or_abort(ctl, p, &ctl.o_full, q_it & 1)) break;
        if constexpr (SOFTMAX) {
          if (!warp_wait_or_abort(ctl, p, &ctl.rs_full, q_it & 1)) break;
          m_run = sx->rs_m[0][rloc];
          l_run = sx->rs_l[0][0][rloc] + sx->rs_l[0][1][rloc];
        }
        ptx::tc_fence_after();
      }
      const bool write_part = p.splits > 1;
      const long long grow0 = __shfl_sync(0xffffffffu, grow, 0);
      const bool tma_rows = !write_part && __all_sync(0xffffffffu, valid && grow == grow0 + lane);
      float mul = u.scale;
      if constexpr (SOFTMAX) mul = l_run > 0.f ? u.scale / l_run : 0.f;
      // hands the O buffer (and the softmax statistics) back to the MMA issuer
      auto release_o = [&]() {
        ptx::tc_fence_before();
        if constexpr (SOFTMAX) ptx::mbar_arrive(&ctl.rs_empty);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(even_bar(&ctl.o_empty));
      };
      if (write_part) {
        // split partials: fp32 x attn_scale (softmax: not yet / row sum), 32 columns at a time
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          if (nt > 0) {
            ptx::tmem_ld32(o_tmem + c * 32, o);
            ptx::tmem_ld_wait(o);
            if (c == DV / 32 - 1) release_o();
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
          if (valid) {
            float* dst =
                p.o_part + ((static_cast<long long>(u.sp) * p.total_q + grow) * p.nhead + u.h) * DV + c * 32;
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              *reinterpret_cast<float4*>(dst + k) =
                  make_float4(__uint_as_float(o[k]) * u.scale, __uint_as_float(o[k + 1]) * u.scale,
                              __uint_as_float(o[k + 2]) * u.scale, __uint_as_float(o[k + 3]) * u.scale);
          }
        }
      } else {
        // the whole row of O, scaled and packed to the storage type, is read
        // before anything is stored, so the single O buffer goes back to the
        // next unit's P V products as early as possible
        uint32_t pk[DV / 2];
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          if (nt > 0) {
            ptx::tmem_ld32(o_tmem + c * 32, o);
            ptx::tmem_ld_wait(o);
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = 0u;
          }
#pragma unroll
          for (int k = 0; k < 32; k += 2)
            pk[c * 16 + (k >> 1)] = pack2<BF16>(__uint_as_float(o[k]) * mul, __uint_as_float(o[k + 1]) * mul);
        }
        if (nt > 0) release_o();
        if (tma_rows) {
          // 64-column boxes: piece j of row r sits at r * 128 + ((j ^ (r & 7)) * 16)
#pragma unroll
          for (int bx = 0; bx < DV / 64; ++bx) {
            const uint32_t buf = stage_warp + (st_it % Cfg::STAGE_BUFS) * Cfg::STAGE_BOX_BYTES;
            if (st_it >= Cfg::STAGE_BUFS) {   // that buffer's last store has read it
              if (lane == 0) ptx::bulk_wait_group_read<Cfg::STAGE_BUFS - 1>();
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              ptx::st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), pk[bx * 32 + 4 * j],
                                pk[bx * 32 + 4 * j + 1], pk[bx * 32 + 4 * j + 2], pk[bx * 32 + 4 * j + 3]);
            ptx::fence_proxy_async_smem();   // the generic-proxy writes, before the bulk copy reads them
            __syncwarp();
            if (lane == 0) {
              ptx::tma_store_2d(&tm_o, buf, u.h * DV + bx * 64, static_cast<int>(grow0));
              ptx::bulk_commit_group();
            }
            ++st_it;
          }
        } else if (valid) {
          uint16_t* dst = reinterpret_cast<uint16_t*>(p.o) + grow * p.o_stride + u.h * DV;
#pragma unroll
          for (int k = 0; k < DV / 2; k += 4)
            *reinterpret_cast<uint4*>(dst + 2 * k) = make_uint4(pk[k], pk[k + 1], pk[k + 2], pk[k + 3]);
        }
      }
      if (nt > 0) ++q_it;
      if (valid) {
        if (write_part) {
          if constexpr (SOFTMAX) {
            float* ml = p.ml_part + ((static_cast<long long>(u.sp) * p.nhead + u.h) * p.total_q + grow) * 2;
            ml[0] = m_run;
            ml[1] = l_run;
          }
        } else if (SOFTMAX && p.lse != nullptr) {
          p.lse[static_cast<long long>(u.h) * p.total_q + grow] =
              l_run > 0.f ? m_run * 0.6931471805599453f + logf(l_run) : -INFINITY;
        }
      }
    }
  } else if (warp < kSchedWarp) {
    // ------------------------------------------------------------ elementwise warpgroups
    const int wg = (warp - 2 - kEpiWarps) >> 2;
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const int c0 = wg * 64;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float half_alpha = 0.5f * p.alpha;
    const float scale_log2 = p.alpha * 1.4426950408889634f;
    int s_it = 0, q_it = 0, sched_it = 0;
    while (!ctl.abort_flag) {
      PairView cur;
      if (!take(sched_it, cur, true) || !cur.live) break;
      const UnitView& u = cur.u;
      const int nt = u.k1 - u.k0;
      const bool own = u.m >= 0;   // this CTA holds a query tile in the unit
      const int qr = own ? q_row(u.s, u.L, u.m, rloc) : -1;
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      int r_lo, r_hi;
      row_uih_keys(u.s, row, r_lo, r_hi);
      int r_diag = row_diag_key(u.s, row);
      int r_ctx = u.s.c;
      if (!valid) { r_lo = r_hi = 0; r_diag = -1; r_ctx = 0; }
      const uint32_t o_tmem = tmem + lane_base + Cfg::O_COL;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      int n, n_end, n_lo1, n_hi1, n_lo2, n_hi2;
      {
        const int n0c = u.ts.hi0 - u.ts.lo0, n1c = u.ts.hi1 - u.ts.lo1;
        const int k = u.k0;
        if (k < n0c) {
          n = u.ts.lo0 + k; n_end = u.ts.hi0;
          n_lo1 = u.ts.lo1; n_hi1 = u.ts.hi1; n_lo2 = u.ts.lo2; n_hi2 = u.ts.hi2;
        } else if (k - n0c < n1c) {
          n = u.ts.lo1 + (k - n0c); n_end = u.ts.hi1;
          n_lo1 = u.ts.lo2; n_hi1 = u.ts.hi2; n_lo2 = n_hi2 = kNoTile;
        } else {
          n = u.ts.lo2 + (k - n0c - n1c); n_end = u.ts.hi2;
          n_lo1 = n_hi1 = n_lo2 = n_hi2 = kNoTile;
        }
      }
      FullTiles ft = full_tile_ranges(u.s, u.tb);
      if (!own) ft.ctx_hi = ft.lo = ft.hi = 0;   // no rows: every tile takes the masked path (P = 0)
      for (int idx = 0; idx < nt; ++idx) {
        const bool full = n < ft.ctx_hi || (n >= ft.lo && n < ft.hi);
        const int j0 = n * kBlockN;
        if (++n == n_end) {
          n = n_lo1; n_end = n_hi1;
          n_lo1 = n_lo2; n_hi1 = n_hi2;
        }
        RowMask rm;
        rm.ctx = r_ctx - j0;
        rm.lo = r_lo - j0;
        rm.span = static_cast<uint32_t>(r_hi - r_lo);
        rm.diag = r_diag >= 0 ? r_diag - j0 : -1000000;
        const int si = s_it + idx;
        if (!warp_wait_or_abort(ctl, p, &ctl.s_full[si % SB], (si / SB) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t s_tmem = tmem + lane_base + (si % SB) * 128 + c0;
        uint32_t r[64];
        ptx::tmem_ld64(s_tmem, r);
        ptx::tmem_ld_wait(r);
        if constexpr (!SOFTMAX) {
          // P packed over this warpgroup's S columns (the scores are in registers)
          if (full) silu_pack<BF16, false>(r, s_tmem, half_alpha, rm, c0);
          else silu_pack<BF16, true>(r, s_tmem, half_alpha, rm, c0);
        } else {
          float mx = -INFINITY;
          if (full) {
#pragma unroll
            for (int k = 0; k < 64; ++k) mx = fmaxf(mx, __uint_as_float(r[k]));
          } else {
            const uint32_t mb0 = rm.bits32(c0), mb1 = rm.bits32(c0 + 32);
#pragma unroll
            for (int k = 0; k < 64; ++k) {
              const uint32_t mb = k < 32 ? mb0 : mb1;
              const uint32_t keep = static_cast<uint32_t>(static_cast<int32_t>(mb << (31 - (k & 31))) >> 31);
              r[k] = (r[k] & keep) | (0xFF800000u & ~keep);   // masked scores become -inf
              mx = fmaxf(mx, __uint_as_float(r[k]));
            }
          }
          sx->xmax[si & 1][wg][rloc] = mx;
          ptx::mbar_arrive(&ctl.xch[si & 1]);
          if (!warp_wait_or_abort(ctl, p, &ctl.xch[si & 1], (si >> 1) & 1)) { ok = false; break; }
          mx = fmaxf(mx, sx->xmax[si & 1][wg ^ 1][rloc]);
          mx *= scale_log2;
          // the P V that last read this buffer (done: this tile's scores were computed
          // after it); keeps the phase tracking of pv_done unambiguous
          if (si >= SB) {
            if (!warp_wait_or_abort(ctl, p, &ctl.pv_done[si % SB], ((si - SB) / SB) & 1)) { ok = false; break; }
          }
          const bool grow = mx > m_run + 8.0f;
          const bool rescale = grow && idx > 0 && m_run != -INFINITY;
          if (__any_sync(0xffffffffu, rescale)) {
            const int sp = si - 1;
            if (!warp_wait_or_abort(ctl, p, &ctl.pv_done[sp % SB], (sp / SB) & 1)) { ok = false; break; }
            ptx::tc_fence_after();
            const float corr = rescale ? ex2_approx(m_run - mx) : 1.0f;
#pragma unroll 1
            for (int c = wg; c < DV / 32; c += 2) {
              uint32_t o[32];
              ptx::tmem_ld32(o_tmem + c * 32, o);
              ptx::tmem_ld_wait(o);
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * corr);
              ptx::tmem_st32(o_tmem + c * 32, o);
            }
            l_run *= corr;
          }
          if (grow) m_run = mx;
          const float nm = m_run == -INFINITY ? 0.f : -m_run;
          float lsum0 = 0.f, lsum1 = 0.f;
          uint32_t pk[32];
#pragma unroll
          for (int k = 0; k < 64; ++k) r[k] = __float_as_uint(fmaf(__uint_as_float(r[k]), scale_log2, nm));
#pragma unroll
          for (int k = 0; k < 64; ++k) r[k] = __float_as_uint(ex2_approx(__uint_as_float(r[k])));
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float e0 = __uint_as_float(r[2 * k]), e1 = __uint_as_float(r[2 * k + 1]);
            lsum0 += e0;
            lsum1 += e1;
            pk[k] = pack2<BF16>(e0, e1);
          }
          ptx::tmem_st32(s_tmem, pk);
          l_run += lsum0 + lsum1;
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_remote(even_bar(&ctl.p_full[si % SB]));
      }
      if (!ok) break;
      if constexpr (SOFTMAX) {
        if (nt > 0) {
          if (!warp_wait_or_abort(ctl, p, &ctl.rs_empty, (q_it & 1) ^ 1)) break;
          if (wg == 0) sx->rs_m[0][rloc] = m_run;
          sx->rs_l[0][wg][rloc] = l_run;
          ptx::mbar_arrive(&ctl.rs_full);
        }
      }
      if (nt > 0) ++q_it;
      s_it += nt;
    }
  }

  // ---------------------------------------------------------------- teardown
  if (warp >= 2 && warp < 2 + kEpiWarps && lane == 0) ptx::bulk_wait_group<0>();
  if (ctl.abort_flag && tid == 0) {
    // let copies and MMAs already in flight land before either CTA releases its memory
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ptx::globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still arrive on its barriers or the
  // pair's MMAs may still use its shared memory or TMEM
  ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host launch
// Grid: 2 x clusters (a multiple of the cluster size), a programmatic
// dependent of the header reset that precedes it on the stream.
template <bool BF16, bool SOFTMAX>
cudaError_t launch_fwd_pair_inst(const FwdMaps& m, const FwdParams& p, int clusters, cudaStream_t stream) {
  constexpr int smem = PairCfg<SOFTMAX>::SMEM_BYTES;
  static_assert(smem + sizeof(PairSmemCtl) <= 232448, "shared memory over the 227 KB a CTA may use");
  auto kern = hstu_fwd_pair_kernel<BF16, SOFTMAX>;
  static std::atomic<unsigned long long> attr_set{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_set);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.k64, m.v, m.q8, m.o, p);
}

// Clusters of the pair kernel that fit on the device at once (0: none, or the
// query failed); cached per device.
template <bool BF16, bool SOFTMAX>
int fwd_pair_max_clusters() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  constexpr int smem = PairCfg<SOFTMAX>::SMEM_BYTES;
  auto kern = hstu_fwd_pair_kernel<BF16, SOFTMAX>;
  static std::atomic<unsigned long long> attr_set{0};
  if (ensure_smem_attr(kern, smem, attr_set) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (n > 0 && dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_release);
  return n;
}

}  // namespace hstu
