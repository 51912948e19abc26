// Persistent, warp-specialised HSTU attention forward for sm_103a.
//
// Per work unit (batch b, query tile m of 128 rows, head h, KV split sp) the
// kernel computes, for the key tiles the functional mask does not fully
// exclude (composable_kernel 18_hstu_attention README, "Forward computation"):
//     S = Q K^T                       tcgen05.mma, A = Q and B = K from shared memory, D in TMEM
//     P = SiLU(alpha S) on allowed entries, 0 elsewhere        (SiLU mode)
//       = exp(alpha S - m) with a running max m                 (softmax mode, online)
//     O += P V                        tcgen05.mma, A = P from TMEM (aliasing S), B = V (MN-major)
// and writes O * attn_scale (softmax: / rowsum, plus LSE) or, with split-KV,
// fp32 partials (x attn_scale) and row statistics for the combine kernel.
//
// Roles (512 threads, one CTA per SM, all waits time-bounded):
//   warp 0       Q/K producer: TMA loads of Q once per unit (the next unit's Q
//                prefetched into L2) and of K tiles into their ring
//   warp 15      V producer: TMA loads of V tiles into their own ring
//   warp 1       TMEM owner + MMA issuer (the whole warp runs the loop, one
//                elected lane issues)
//   warps 2..5   epilogue warpgroup, one query row per thread: reads a unit's O
//                out of TMEM once its last P V product is done, hands the
//                buffer back, scales (softmax: by 1/rowsum) and stores O / LSE
//   warps 6..13  elementwise groups: warpgroup g (warps 6+4g .. 9+4g) owns key
//                columns [64g, 64g+64) of every score row, one row per thread:
//                TMEM S -> registers, mask + SiLU/softmax, P -> TMEM
//   warp 14      scheduler: takes units from the global queue, decodes them and
//                publishes them to the other roles through a shared-memory ring
//
// TMEM (512 columns): S0 [0,128), S1 [128,256) double-buffered scores; the
// 16-bit P of key columns [64g, 64g+64) is packed into S columns
// [64g, 64g+32) of the same buffer;
// O [256, 256 + DV) and, for DV <= 128, a second O buffer right after it so the
// epilogue of one unit overlaps the next unit's P V products.
//
// Head dimensions: D (of q and k) in {64, 96, 128, 256}, DV (of v and o) equal
// to D or, for D = 96, 64.  A 96-wide row occupies two 64-element swizzle
// chunks; Q K^T runs 6 k-steps, so the unused half chunk (the next head's
// columns, or TMA zero fill past the last head) is never read, and P V with
// N = 96 reads only the first 96 columns of the V tile.
//
// The mask and SiLU run in fp32 on the fp32 scores read out of TMEM:
// SiLU(x) = h + h tanh(h) with h = x / 2, the products in packed f32x2
// arithmetic and tanh.approx.f32 per element.  P is rounded once, to the
// storage type, as the A operand of the second product; attn_scale multiplies
// the fp32 O accumulator in the epilogue (it is linear in P).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hstu_common.cuh"
#include "hstu_launch.h"
#include "hstu_rab.cuh"
#include "ptx.cuh"

namespace hstu {

// Softmax-only exchange buffers (after the tiles in dynamic shared memory).
struct SoftmaxScratch {
  float xmax[2][2][128];      // [tile parity][warpgroup][row] row-max exchange
  float rs_m[2][128];         // [O buffer][row] running max (log2 units)
  float rs_l[2][2][128];      // [O buffer][warpgroup][row] row sum over the warpgroup's columns
};

template <int D, int DV, bool SOFTMAX, bool RAB = false>
struct FwdCfg {
  static constexpr int KCH = (D + 63) / 64;           // 128-byte column chunks per Q / K row
  static constexpr int VCH = (DV + 63) / 64;          // ... per V row
  static constexpr int CHUNK_BYTES = kBlockN * 128;   // one 128-row x 128-byte TMA box
  static constexpr int TILE_BYTES = KCH * CHUNK_BYTES;    // one Q or K tile
  static constexpr int VTILE_BYTES = VCH * CHUNK_BYTES;   // one V tile
  // Q is double-buffered where it fits so the next unit's Q streams in early.
  static constexpr int QBUF = D <= 128 ? 2 : 1;
  // K ring depth: two stages at hdim 128 (the O staging of the TMA-store
  // epilogue, the softmax scratch and the bias tables take the third's room);
  // three at hdim 96, four at hdim 64
  static constexpr int KSTAGES = D == 64 ? 4 : (D <= 128 ? ((SOFTMAX || RAB || D == 128) ? 2 : 3) : 1);
  static constexpr int VSTAGES = D == 64 ? 4 : (D <= 128 ? 2 : 1);                   // V ring depth
  static constexpr int TILES_BYTES = (QBUF + KSTAGES) * TILE_BYTES + VSTAGES * VTILE_BYTES;
  static constexpr int SOFTMAX_BYTES = SOFTMAX ? static_cast<int>(sizeof(SoftmaxScratch)) : 0;
  static constexpr int RAB_BYTES = RAB ? static_cast<int>(sizeof(RabWarp)) * 8 : 0;   // one per elementwise warp
  // TMA-store epilogue (output widths that are whole 64-column boxes): per
  // epilogue warp, STAGE_BUFS buffers of one 32-row x 64-column box (4 KB,
  // 128-byte swizzle); two when they fit in the 227 KB a CTA may use (with
  // 2 KB kept for the static control block), else one
  static constexpr int STAGE_BOX_BYTES = 32 * 128;
  static constexpr int BASE_BYTES = TILES_BYTES + SOFTMAX_BYTES + RAB_BYTES + 1024;
  static constexpr int STAGE_BUFS =
      DV % 64 != 0 ? 0 : (BASE_BYTES + 2 * kFwdEpiWarps * STAGE_BOX_BYTES + 2048 <= 232448 ? 2 : 1);
  static constexpr int STAGE_BYTES = STAGE_BUFS * kFwdEpiWarps * STAGE_BOX_BYTES;
  static constexpr int SMEM_BYTES = BASE_BYTES + STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t O_COL = 256;
  static constexpr int O_BUFS = DV <= 128 ? 2 : 1;
  static_assert(O_COL + O_BUFS * DV <= TMEM_COLS, "TMEM budget");
  static_assert(D % 16 == 0 && DV % 32 == 0 && DV <= 256, "head dimensions");
};

constexpr int kEpiWarps = kFwdEpiWarps;   // epilogue warpgroup
constexpr int kEwThreads = 256;    // two elementwise warpgroups
constexpr int kFwdThreads = 64 + 32 * kEpiWarps + kEwThreads + 64;   // 512: 128 registers per thread
constexpr int kSchedWarp = kFwdThreads / 32 - 2;
constexpr int kVProdWarp = kFwdThreads / 32 - 1;
constexpr int kSchedDepth = 2;   // published-unit ring (deeper claims ahead hurt the tail balance)
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait, then give up



template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bits [0, x) of a word, x clamped to [0, 32].
__device__ __forceinline__ uint32_t low_bits(int x) {
  return x <= 0 ? 0u : (x >= 32 ? 0xFFFFFFFFu : (1u << x) - 1u);
}

// Per-row mask in tile-local column terms: key column c (0..127) of the tile
// is allowed iff c < ctx || (unsigned)(c - lo) < span || c == diag.
struct RowMask {
  int ctx, lo, diag;
  uint32_t span;
  // whether column cb + i is allowed, as bit i (i = 0..31)
  __device__ __forceinline__ uint32_t bits32(int cb) const {
    const int d = diag - cb;
    return low_bits(ctx - cb) | (low_bits(lo + static_cast<int>(span) - cb) & ~low_bits(lo - cb)) |
           (static_cast<uint32_t>(d) < 32u ? 1u << d : 0u);
  }
};

struct UnitView {
  SeqGeom s;
  QLayout L;     // the sequence's query-tile layout (which rows tile m holds)
  TileSet ts;
  TileBounds tb;
  int m, h, g, sp, k0, k1;
  float scale;   // resolved attn_scale of the unit's group
};

__device__ __forceinline__ UnitView decode_unit(const FwdParams& p, int unit) {
  const int4 w = p.units[unit];
  UnitView u;
  const int b = w.x;
  u.m = w.y;
  u.h = w.z;
  u.sp = w.w;
  u.g = b / p.batch_per_group;
  u.s = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[u.g], p.loc[u.g], p.mf[u.g], p.causal,
                  p.self_attn, p.kv_targets);
  u.L = q_layout(u.s);
  u.tb = q_tile_bounds(u.s, u.L, u.m);
  u.ts = query_tile_kv_tiles(u.s, u.L, u.m, u.tb);
  split_range(u.ts.count, u.sp, p.splits, u.k0, u.k1);
  u.scale = p.group_scale[u.g];
  return u;
}

struct FwdSmemCtl {
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t sched_full[kSchedDepth], sched_empty[kSchedDepth];
  uint64_t xch[2];            // softmax row-max exchange between the warpgroups, per tile parity
  uint64_t rs_full[2], rs_empty[2];   // softmax row statistics of O buffer ob: ready / consumed
  UnitView sched_view[kSchedDepth];   // decoded units published by the producer
  int sched_live[kSchedDepth];        // 0: no more units
  uint32_t tmem_base;
  volatile int abort_flag;
  // in-kernel schedule (FwdParams::fused): position -> sequence (longest
  // first), first unit of each position, attn_scale of each position's group,
  // and the device error bits the offsets raised
  uint8_t f_order[kFusedMaxBatch];
  int f_ubase[kFusedMaxBatch + 1];
  float f_pscale[kFusedMaxBatch];
  int f_err;
};

// Largest k in [0, n) with a[k] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int seg_find(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Exclusive prefix sum of v[0, n) (n <= 32 * 4) by one warp, in place; v[n]
// receives the total.
__device__ __forceinline__ void warp_exclusive_scan(int* v, int n, int lane) {
  constexpr int kPer = kFusedMaxBatch / 32;
  int loc[kPer], sum = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = lane * kPer + k;
    loc[k] = i < n ? v[i] : 0;
    sum += loc[k];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  int run = incl - sum;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int i = lane * kPer + k;
    if (i < n) v[i] = run;
    run += loc[k];
  }
  if (lane == 31) v[n] = incl;
}

// The scheduler's work, done by every CTA for itself (FwdParams::fused, batch
// <= kFusedMaxBatch), by all threads of the CTA before any role starts, so
// that no separate scheduler kernel runs before the forward.  The same
// validation and order as hstu_prep_kernel: each sequence's offsets are
// checked (errors go to ctl.f_err and leave no units), its query tiles and
// executed key tiles are counted, the sequences are ranked by executed tiles
// (most first, ties by index) and the units are numbered per position with
// heads outer, query tiles from the last down and splits innermost.
// `scratch` (3 batch + 2 ints) is shared memory no TMA load uses yet.
// TPU: query tiles per unit (2: the CTA-pair kernel, whose unit is two query
// tiles of one head, from the last down).  Returns the number of units.
template <int TPU = 1, typename Ctl>
__device__ __forceinline__ int fused_schedule(const FwdParams& p, Ctl& ctl, int* scratch, int tid, int nthreads) {
  const int B = p.batch;
  const int G = p.num_groups;
  int* tb = scratch;        // [B + 1] query tiles per sequence, then their exclusive prefix
  int* cost = tb + B + 1;   // [B] executed key tiles per sequence
  int* gmax = cost + B;     // [G] largest query UIH length of each group
  for (int i = tid; i < B; i += nthreads) cost[i] = 0;
  for (int g = tid; g < G; g += nthreads) gmax[g] = 0;
  if (tid == 0) ctl.f_err = 0;
  __syncthreads();
  for (int b = tid; b < B; b += nthreads) {
    const int g = b / p.batch_per_group;
    const int c = p.ctx[g];
    int err = 0;
    const int q0 = p.off_q[b], q1 = p.off_q[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.total_q) err |= kErrOffsets;
    const int t = p.targets ? p.targets[b] : 0;
    if (t < 0 || q1 - q0 < c + t) err |= kErrQLayout;
    int Lkv = q1 - q0;
    if (!p.self_attn) {
      const int k0 = p.off_kv[b], k1 = p.off_kv[b + 1];
      if (k0 < 0 || k1 < k0 || k1 > p.total_kv) err |= kErrOffsets;
      Lkv = k1 - k0;
      if (Lkv < c + (p.kv_targets ? t : 0)) err |= kErrKvLayout;
    }
    if (q1 - q0 > p.max_seqlen_q || Lkv > p.max_seqlen_kv) err |= kErrMaxSeqlen;
    if (err) atomicOr(&ctl.f_err, err);
    else atomicMax(&gmax[g], q1 - q0 - c - t);
    tb[b] = err ? 0 : q_layout(q1 - q0, c).nq;
  }
  __syncthreads();
  if (ctl.f_err != 0) return 0;
  if (tid < 32) warp_exclusive_scan(tb, B, tid);
  __syncthreads();
  const int n_items = tb[B];
  for (int i = tid; i < n_items; i += nthreads) {
    const int b = seg_find(tb, B, i);
    const int g = b / p.batch_per_group;
    const SeqGeom sg = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[g], p.loc[g], p.mf[g], p.causal,
                                 p.self_attn, p.kv_targets);
    atomicAdd(&cost[b], query_tile_kv_tiles(sg, q_layout(sg), i - tb[b]).count);
  }
  __syncthreads();
  for (int b = tid; b < B; b += nthreads) {
    const int cb = cost[b];
    int r = 0;
    for (int b2 = 0; b2 < B; ++b2) {
      const int c2 = cost[b2];
      r += (c2 > cb) | ((c2 == cb) & (b2 < b));
    }
    ctl.f_order[r] = static_cast<uint8_t>(b);
  }
  __syncthreads();
  for (int pos = tid; pos < B; pos += nthreads) {
    const int b = ctl.f_order[pos];
    ctl.f_ubase[pos] = ((tb[b + 1] - tb[b] + TPU - 1) / TPU) * p.nhead * p.splits;
    const int g = b / p.batch_per_group;
    float sc = p.attn_scale[g];
    if (sc == 0.f) {   // 0 means 1 / max UIH length of the group
      const int mu = p.max_uih[g] > 0 ? p.max_uih[g] : gmax[g];
      sc = mu > 0 ? 1.f / static_cast<float>(mu) : 1.f;
    }
    ctl.f_pscale[pos] = sc;
  }
  __syncthreads();
  if (tid < 32) warp_exclusive_scan(ctl.f_ubase, B, tid);
  __syncthreads();
  return ctl.f_ubase[B];
}

// decode_unit for the in-kernel schedule.
__device__ __forceinline__ UnitView decode_fused_unit(const FwdParams& p, const FwdSmemCtl& ctl, int unit) {
  const int pos = seg_find(ctl.f_ubase, p.batch, unit);
  const int b = ctl.f_order[pos];
  UnitView u;
  u.g = b / p.batch_per_group;
  u.s = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[u.g], p.loc[u.g], p.mf[u.g], p.causal, p.self_attn,
                  p.kv_targets);
  u.L = q_layout(u.s);
  const int local = unit - ctl.f_ubase[pos];
  const int per_h = u.L.nq * p.splits;
  u.h = local / per_h;
  const int rem = local - u.h * per_h;
  u.m = u.L.nq - 1 - rem / p.splits;
  u.sp = rem % p.splits;
  u.tb = q_tile_bounds(u.s, u.L, u.m);
  u.ts = query_tile_kv_tiles(u.s, u.L, u.m, u.tb);
  split_range(u.ts.count, u.sp, p.splits, u.k0, u.k1);
  u.scale = ctl.f_pscale[pos];
  return u;
}

// Bounded wait; on timeout flags the error word and asks every role to stop.
template <typename Ctl>
__device__ __forceinline__ bool wait_or_abort(Ctl& ctl, const FwdParams& p, uint64_t* bar, uint32_t parity) {
  if (ptx::mbar_wait(bar, parity, kWaitLimitNs)) return true;
  ctl.abort_flag = 1;
  atomicOr(&p.ws_header[kWsError], kErrTimeout);
  return false;
}

// Warp-uniform bounded wait for the elementwise group: every lane waits, then
// the warp agrees (and reconverges) before the next .sync.aligned tcgen05 op.
template <typename Ctl>
__device__ __forceinline__ bool warp_wait_or_abort(Ctl& ctl, const FwdParams& p, uint64_t* bar, uint32_t parity) {
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, kWaitLimitNs));
  if (!ok) {
    ctl.abort_flag = 1;
    atomicOr(&p.ws_header[kWsError], kErrTimeout);
  }
  return ok;
}

// SiLU of the 2 NP scores of key columns [c0, c0 + 2 NP) of one row (fp32 bit
// patterns in r), in fp32: h = alpha s / 2 (one packed f32x2 multiply per
// pair), t = tanh(h) (tanh.approx.f32 per element), SiLU(alpha s) = h + h t
// (one packed f32x2 fma per pair).  Each pair is rounded once, to the storage
// type, when it is packed into its P word pk[k] (masked columns: 0).
// PRESCALED: r already holds alpha s / 2 (plus the halved bias).
template <bool BF16, bool MASKED, bool PRESCALED = false, int NP = 32>
__device__ __forceinline__ void silu_words(const uint32_t (&r)[2 * NP], uint32_t (&pk)[NP], float half_alpha,
                                           const RowMask& rm, int c0) {
  static_assert(NP == 16 || NP == 32, "16 or 32 pairs");
  // all pairs stage by stage, so the NP tanh pairs are in flight together
  const uint64_t ha = ptx::f32x2(half_alpha, half_alpha);
  uint64_t h[NP];
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    h[k] = ptx::f32x2(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
    if constexpr (!PRESCALED) h[k] = ptx::mul_f32x2(h[k], ha);
  }
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    float h0, h1;
    ptx::f32x2_split(h[k], h0, h1);
    h[k] = ptx::fma_f32x2(h[k], ptx::f32x2(ptx::tanh_approx(h0), ptx::tanh_approx(h1)), h[k]);
  }
#pragma unroll
  for (int k = 0; k < NP; ++k) pk[k] = ptx::cvt_pack16<BF16>(h[k]);
  if constexpr (MASKED) {
    // bit 2k (2k+1) of a chunk's mask keeps the low (high) half of its pair k
    const uint32_t mb0 = rm.bits32(c0), mb1 = NP > 16 ? rm.bits32(c0 + 32) : 0u;
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      const uint32_t mb = k < 16 ? mb0 : mb1;
      const int kk = k & 15;
      const uint32_t lo = static_cast<uint32_t>(static_cast<int32_t>(mb << (31 - 2 * kk)) >> 31);
      const uint32_t hi = static_cast<uint32_t>(static_cast<int32_t>(mb << (30 - 2 * kk)) >> 31);
      pk[k] &= (lo & 0x0000FFFFu) | (hi & 0xFFFF0000u);
    }
  }
}

// silu_words, then the NP words to the TMEM columns at p_tmem (one store).
template <bool BF16, bool MASKED, bool PRESCALED = false, int NP = 32>
__device__ __forceinline__ void silu_pack(const uint32_t (&r)[2 * NP], uint32_t p_tmem, float half_alpha,
                                          const RowMask& rm, int c0) {
  uint32_t pk[NP];
  silu_words<BF16, MASKED, PRESCALED, NP>(r, pk, half_alpha, rm, c0);
  if constexpr (NP == 32) ptx::tmem_st32(p_tmem, pk);
  else ptx::tmem_st16(p_tmem, pk);
}

template <int D, int DV, bool BF16, bool SOFTMAX, bool RAB = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    hstu_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q8,
                    const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ FwdParams p) {
  using Cfg = FwdCfg<D, DV, SOFTMAX, RAB>;
  constexpr int KCH = Cfg::KCH;
  constexpr int VCH = Cfg::VCH;
  constexpr int KST = Cfg::KSTAGES;
  constexpr int VST = Cfg::VSTAGES;
  constexpr int OB = Cfg::O_BUFS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int QB = Cfg::QBUF;
  uint8_t* sQ = smem;
  uint8_t* sK = smem + QB * Cfg::TILE_BYTES;
  uint8_t* sV = sK + KST * Cfg::TILE_BYTES;
  uint8_t* sStage = smem + Cfg::TILES_BYTES;   // O staging of the TMA-store epilogue (1024-byte aligned)
  SoftmaxScratch* sx = reinterpret_cast<SoftmaxScratch*>(smem + Cfg::TILES_BYTES + Cfg::STAGE_BYTES);   // softmax only
  RabWarp* rabw =
      reinterpret_cast<RabWarp*>(smem + Cfg::TILES_BYTES + Cfg::STAGE_BYTES + Cfg::SOFTMAX_BYTES);   // bias only

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

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
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&ctl.s_full[s], 1);
      ptx::mbar_init(&ctl.p_full[s], kEwThreads);
      ptx::mbar_init(&ctl.pv_done[s], 1);
      ptx::mbar_init(&ctl.o_full[s], 1);
      ptx::mbar_init(&ctl.o_empty[s], 32 * kEpiWarps);
      ptx::mbar_init(&ctl.xch[s], kEwThreads);
      ptx::mbar_init(&ctl.rs_full[s], kEwThreads);
      ptx::mbar_init(&ctl.rs_empty[s], 32 * kEpiWarps);
    }
    for (int s = 0; s < kSchedDepth; ++s) {
      ptx::mbar_init(&ctl.sched_full[s], 1);
      // Q/K producer, V producer, MMA, epilogue and elementwise warps
      ptx::mbar_init(&ctl.sched_empty[s], 3 + kEpiWarps + kEwThreads / 32);
    }
    ctl.abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
    if constexpr (Cfg::STAGE_BUFS > 0) ptx::prefetch_tensormap(&tm_o);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, Cfg::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  // Launched as a programmatic dependent of the kernel before it on the stream
  // (the scheduler, or with the in-kernel schedule the header reset): the
  // work list and the header are read only after it has completed.  With the
  // in-kernel schedule, every CTA orders the units itself first (reading only
  // the offsets and targets, which that kernel does not write), in shared
  // memory no TMA load uses yet; only the dynamic claims wait for the reset.
  int n_units;
  if (p.fused) {
    n_units = fused_schedule(p, ctl, reinterpret_cast<int*>(sK), tid, kFwdThreads);
    // the first epilogue warp (idle until the first unit's O) reports
    if (tid == 64 && (ctl.f_err != 0 || blockIdx.x == 0)) {
      ptx::grid_dependency_wait();
      if (ctl.f_err != 0) atomicOr(&p.ws_header[kWsError], ctl.f_err);
      else p.ws_header[kWsUnits] = n_units;   // read by the combine kernel
    }
  } else {
    ptx::grid_dependency_wait();
    n_units = p.ws_header[kWsUnits];
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Only the next unit's Q tile is prefetched into L2: K/V tiles are mostly
      // L2 hits (every query tile of a head re-reads them), and prefetching them
      // as well doubled the L2 lookups of a path already near the L2 limit.
      auto prefetch_unit = [&](const UnitView& u) {
        if (u.k1 <= u.k0) return;
#pragma unroll
        for (int kc = 0; kc < KCH; ++kc)
          ptx::tma_prefetch_2d(&tm_q, u.h * D + kc * 64, u.s.q0 + u.m * kBlockM);
      };
      int q_it = 0, kv_it = 0, sched_it = 0;
      // reads the next published unit from the scheduler ring
      auto take = [&](UnitView& u) -> int {   // 1 live, 0 end, -1 abort
        const int slot = sched_it % kSchedDepth;
        if (!wait_or_abort(ctl, p, &ctl.sched_full[slot], (sched_it / kSchedDepth) & 1)) return -1;
        const int live = ctl.sched_live[slot];
        u = ctl.sched_view[slot];
        ptx::mbar_arrive(&ctl.sched_empty[slot]);
        ++sched_it;
        return live;
      };
      UnitView cur, nxt;
      int cur_live = take(cur);
      if (cur_live > 0) prefetch_unit(cur);
      while (cur_live > 0 && !ctl.abort_flag) {
        int nxt_live = 0;
        bool have_nxt = false;
        // the next unit is read (and its Q tile prefetched into L2) about three
        // tiles before this unit's last loads
        auto look_ahead = [&]() -> bool {
          if (have_nxt) return true;
          have_nxt = true;
          nxt_live = take(nxt);
          if (nxt_live < 0) return false;
          if (nxt_live > 0) prefetch_unit(nxt);
          return true;
        };
        bool ok = true;
        if (cur.k1 > cur.k0) {
          const int qb = q_it % QB;
          if (!wait_or_abort(ctl, p, &ctl.q_empty[qb], ((q_it / QB) & 1) ^ 1)) break;
          ptx::mbar_arrive_expect_tx(&ctl.q_full[qb], Cfg::TILE_BYTES);
          const int qrow = cur.m * kBlockM;   // the tile's rows, lane r = row qrow + r
          uint8_t* qdst = sQ + qb * Cfg::TILE_BYTES;
          if (!(cur.L.ctx_lane0 >= 0 && cur.m == cur.L.nq - 1)) {   // one 128-row box per chunk
#pragma unroll
            for (int kc = 0; kc < KCH; ++kc)
              ptx::tma_load_2d(qdst + kc * Cfg::CHUNK_BYTES, &tm_q, &ctl.q_full[qb], cur.h * D + kc * 64,
                               cur.s.q0 + qrow);
          } else {
            // the tile's own rows on lanes [0, ctx_lane0), the context rows on
            // lanes [ctx_lane0, 128): 8-row boxes (one swizzle atom each), 16 per chunk
            const int lane0 = cur.L.ctx_lane0;
            for (int g = 0; g < kBlockM / 8; ++g) {
              const int row = g * 8 < lane0 ? qrow + g * 8 : (g * 8 - lane0);
#pragma unroll
              for (int kc = 0; kc < KCH; ++kc)
                ptx::tma_load_2d(qdst + kc * Cfg::CHUNK_BYTES + g * 1024, &tm_q8, &ctl.q_full[qb],
                                 cur.h * D + kc * 64, cur.s.q0 + row);
            }
          }
          ++q_it;
          const int k_ahead = cur.k1 - 3 > cur.k0 ? cur.k1 - 3 : cur.k0;
          for (int k = cur.k0; k < cur.k1 && ok; ++k) {
            if (k == k_ahead && !look_ahead()) { ok = false; break; }
            const int n = tileset_at(cur.ts, k);
            const int krow = cur.s.kv0 + n * kBlockN;
            const int ks = kv_it % KST;
            if (!wait_or_abort(ctl, p, &ctl.k_empty[ks], ((kv_it / KST) & 1) ^ 1)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(&ctl.k_full[ks], Cfg::TILE_BYTES);
#pragma unroll
            for (int kc = 0; kc < KCH; ++kc)
              ptx::tma_load_2d(sK + ks * Cfg::TILE_BYTES + kc * Cfg::CHUNK_BYTES, &tm_k, &ctl.k_full[ks],
                               cur.h * D + kc * 64, krow);
            ++kv_it;
          }
        }
        if (!ok || !look_ahead()) break;
        cur = nxt;
        cur_live = nxt_live;
      }
    }
  } else if (warp == kVProdWarp) {
    // ------------------------------------------------------------ V producer
    // Streams V tiles into their ring independently of the K ring, so that a
    // K tile never waits behind a V slot (and vice versa).
    if (lane == 0) {
      int kv_it = 0, sched_it = 0;
      while (!ctl.abort_flag) {
        const int slot = sched_it % kSchedDepth;
        if (!wait_or_abort(ctl, p, &ctl.sched_full[slot], (sched_it / kSchedDepth) & 1)) break;
        const bool live = ctl.sched_live[slot] != 0;
        const UnitView u = ctl.sched_view[slot];
        ptx::mbar_arrive(&ctl.sched_empty[slot]);
        ++sched_it;
        if (!live) break;
        bool ok = true;
        for (int k = u.k0; k < u.k1; ++k) {
          const int vs = kv_it % VST;
          const int vrow = u.s.kv0 + tileset_at(u.ts, k) * kBlockN;
          if (!wait_or_abort(ctl, p, &ctl.v_empty[vs], ((kv_it / VST) & 1) ^ 1)) { ok = false; break; }
          ptx::mbar_arrive_expect_tx(&ctl.v_full[vs], Cfg::VTILE_BYTES);
#pragma unroll
          for (int kc = 0; kc < VCH; ++kc)
            ptx::tma_load_2d(sV + vs * Cfg::VTILE_BYTES + kc * Cfg::CHUNK_BYTES, &tm_v, &ctl.v_full[vs],
                             u.h * DV + kc * 64, vrow);
          ++kv_it;
        }
        if (!ok) break;
      }
    }
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------ scheduler
    // Takes units from the global queue (lane 0), decodes them and publishes
    // each into its own ring slot, running up to kSchedDepth units ahead.  With
    // the in-kernel schedule each CTA's first unit is its own index (no wait
    // for the header reset, so its loads start at once) and the queue hands out
    // the units from the grid size on.
    int sched_it = 0;
    bool first = true, waited = !p.fused;
    while (!ctl.abort_flag) {
      bool ok = true, live = false;
      if (lane == 0) {
        int id;
        if (p.fused && first) {
          id = static_cast<int>(blockIdx.x);
        } else {
          if (!waited) {
            ptx::grid_dependency_wait();
            waited = true;
          }
          id = atomicAdd(&p.ws_header[kWsCounter], 1) + (p.fused ? static_cast<int>(gridDim.x) : 0);
        }
        live = id < n_units;
        UnitView u;
        if (live) u = p.fused ? decode_fused_unit(p, ctl, id) : decode_unit(p, id);
        const int slot = sched_it % kSchedDepth;
        ok = wait_or_abort(ctl, p, &ctl.sched_empty[slot], ((sched_it / kSchedDepth) & 1) ^ 1);
        if (ok) {
          if (live) ctl.sched_view[slot] = u;
          ctl.sched_live[slot] = live ? 1 : 0;
          ptx::mbar_arrive(&ctl.sched_full[slot]);
        }
      }
      first = false;
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (!__shfl_sync(0xffffffffu, live ? 1 : 0, 0)) break;   // the queue is drained: end marker published
      ++sched_it;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, so every descriptor is warp-uniform;
    // one elected lane issues the tcgen05 instructions and barrier arrivals.
    const bool leader = ptx::elect_one_sync();
    {
      constexpr uint32_t idesc_qk = ptx::idesc_f16_f32acc(BF16, false, kBlockM, kBlockN);
      constexpr uint32_t idesc_pv = ptx::idesc_f16_f32acc(BF16, true, kBlockM, DV);
      const uint32_t q_base = ptx::smem_u32(sQ);
      const uint32_t k_base = ptx::smem_u32(sK);
      const uint32_t v_base = ptx::smem_u32(sV);
      int q_it = 0, kv_it = 0, s_it = 0, sched_it = 0;
      bool ok = true;
      // The K-major operands of Q K^T advance by 32 bytes per 16-element step
      // inside a 128-byte swizzle row and by one 128-row chunk every 4 steps;
      // the descriptors are the stage's base plus that offset (16-byte units).
      const uint64_t q_desc = ptx::sdesc_sw128(q_base, 16, 1024);
      // S = Q K^T for the tile held in K stage (kvi % KST), into S buffer (si & 1).
      auto issue_qk = [&](int kvi, int si, int qb) -> bool {
        const int st = kvi % KST;
        if (!warp_wait_or_abort(ctl, p, &ctl.k_full[st], (kvi / KST) & 1)) return false;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + (si & 1) * 128;
        const uint64_t k_desc = ptx::sdesc_sw128(k_base + st * Cfg::TILE_BYTES, 16, 1024);
        // k-steps in asm blocks of 8 while 8 remain, then of 4, then single (D = 96: 4 + 2)
        constexpr int KS = D / 16;
        auto desc_a = [&](int ks) {
          return q_desc + static_cast<uint64_t>((qb * Cfg::TILE_BYTES) >> 4) +
                 static_cast<uint64_t>(((ks >> 2) * Cfg::CHUNK_BYTES + (ks & 3) * 32) >> 4);
        };
        auto desc_b = [&](int ks) {
          return k_desc + static_cast<uint64_t>(((ks >> 2) * Cfg::CHUNK_BYTES + (ks & 3) * 32) >> 4);
        };
#pragma unroll
        for (int g = 0; g + 8 <= KS; g += 8) {
          uint64_t ad[8], bd[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) { ad[j] = desc_a(g + j); bd[j] = desc_b(g + j); }
          if (leader) ptx::umma_ss_x8(d_tmem, ad, bd, idesc_qk, g > 0 ? 1u : 0u);
        }
        if constexpr (KS % 8 >= 4) {
          constexpr int g = KS / 8 * 8;
          uint64_t ad[4], bd[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) { ad[j] = desc_a(g + j); bd[j] = desc_b(g + j); }
          if (leader) ptx::umma_ss_x4(d_tmem, ad, bd, idesc_qk, g > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = KS / 4 * 4; ks < KS; ++ks)
          if (leader) ptx::umma_ss(d_tmem, desc_a(ks), desc_b(ks), idesc_qk, ks > 0 ? 1u : 0u);
        if (leader) {
          ptx::umma_commit(&ctl.k_empty[st]);
          ptx::umma_commit(&ctl.s_full[si & 1]);
        }
        __syncwarp();
        return true;
      };
      // O += P V for tile index si (K/V index kvi) into O buffer ob; `first`
      // starts the accumulation, `last` hands the buffer to the epilogue.
      auto issue_pv = [&](int si, int kvi, int ob, int o_round, bool first, bool last) -> bool {
        if (!warp_wait_or_abort(ctl, p, &ctl.p_full[si & 1], (si >> 1) & 1)) return false;
        ptx::tc_fence_after();
        if (first) {
          if (!warp_wait_or_abort(ctl, p, &ctl.o_empty[ob], (o_round & 1) ^ 1)) return false;
          ptx::tc_fence_after();
        }
        const int st = kvi % VST;
        if (!warp_wait_or_abort(ctl, p, &ctl.v_full[st], (kvi / VST) & 1)) return false;
        ptx::tc_fence_after();
        // P of key columns [64 g, 64 g + 64) is packed at S columns [64 g, 64 g + 32);
        // V (MN-major) advances 2048 bytes per step.
        const uint64_t v_desc = ptx::sdesc_sw128(v_base + st * Cfg::VTILE_BYTES, Cfg::CHUNK_BYTES, 1024);
        uint32_t pa[8];
        uint64_t vd[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          pa[kk] = tmem + (si & 1) * 128 + (kk >> 2) * 64 + (kk & 3) * 8;
          vd[kk] = v_desc + static_cast<uint64_t>((kk * 2048) >> 4);
        }
        if (leader) {
          ptx::umma_ts_x8(tmem + Cfg::O_COL + ob * DV, pa, vd, idesc_pv, first ? 0u : 1u);
          ptx::umma_commit(&ctl.v_empty[st]);
          if constexpr (SOFTMAX) ptx::umma_commit(&ctl.pv_done[si & 1]);
          if (last) ptx::umma_commit(&ctl.o_full[ob]);
        }
        __syncwarp();
        return true;
      };
      // Tiles of consecutive units form one stream: Q K^T of tile t is issued
      // before the P V product of tile t-1, across unit boundaries too, so the
      // elementwise warps find the next scores ready when a unit ends.  (P is
      // packed over its S buffer: Q K^T of tile t overwrites the buffer that the
      // already-issued P V product of tile t-2 read.)  With one Q buffer the
      // next unit's Q load waits for this unit's last Q K^T, so the pending
      // P V product is issued first.
      bool pend = false;
      int pend_si = 0, pend_kvi = 0, pend_ob = 0, pend_round = 0;
      bool pend_first = false, pend_last = false;
      auto flush = [&]() -> bool {
        if (!pend) return true;
        pend = false;
        return issue_pv(pend_si, pend_kvi, pend_ob, pend_round, pend_first, pend_last);
      };
      while (ok && !ctl.abort_flag) {
        const int slot = sched_it % kSchedDepth;
        if (!warp_wait_or_abort(ctl, p, &ctl.sched_full[slot], (sched_it / kSchedDepth) & 1)) { ok = false; break; }
        const bool live = ctl.sched_live[slot] != 0;
        const UnitView u = ctl.sched_view[slot];
        __syncwarp();
        if (leader) ptx::mbar_arrive(&ctl.sched_empty[slot]);
        ++sched_it;
        if (!live) break;
        const int nt = u.k1 - u.k0;
        if (nt <= 0) {
          // An empty split unit: issue the pending P V now.  Holding it across
          // empty units would stall the epilogue on that unit's O, and with
          // it the scheduler ring this loop is waiting on.
          if (!flush()) { ok = false; break; }
          continue;
        }
        if (QB == 1 && !flush()) { ok = false; break; }
        const int ob = q_it % OB;
        const int qb = q_it % QB;
        if (!warp_wait_or_abort(ctl, p, &ctl.q_full[qb], (q_it / QB) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        for (int t = 0; t < nt; ++t) {
          if (!issue_qk(kv_it + t, s_it + t, qb)) { ok = false; break; }
          if (t == nt - 1 && leader) ptx::umma_commit(&ctl.q_empty[qb]);   // Q may be replaced
          if (!flush()) { ok = false; break; }
          pend = true;
          pend_si = s_it + t;
          pend_kvi = kv_it + t;
          pend_ob = ob;
          pend_round = q_it / OB;
          pend_first = t == 0;
          pend_last = t == nt - 1;
        }
        if (!ok) break;
        kv_it += nt;
        s_it += nt;
        ++q_it;
      }
      if (ok) flush();
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue warpgroup
    // One query row per thread, all DV output columns: waits for the unit's last
    // P V product, reads O out of TMEM, hands the buffer back, scales and stores.
    // A warp whose 32 rows are consecutive rows of one sequence stages each
    // 64-column box of its rows in shared memory (128-byte swizzle) and writes
    // it with one TMA store; warps holding a ragged tail or the context rows of
    // the last query tile store their rows with plain 16-byte stores.
    const int quarter = warp & 3;
    const int rloc = quarter * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t stage_warp = ptx::smem_u32(sStage) + (warp - 2) * Cfg::STAGE_BUFS * Cfg::STAGE_BOX_BYTES;
    int st_it = 0;   // boxes this warp has stored with TMA (selects the staging buffer)
    int q_it = 0, sched_it = 0;
    while (!ctl.abort_flag) {
      const int slot = sched_it % kSchedDepth;
      if (!warp_wait_or_abort(ctl, p, &ctl.sched_full[slot], (sched_it / kSchedDepth) & 1)) break;
      const bool live = ctl.sched_live[slot] != 0;
      const UnitView u = ctl.sched_view[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl.sched_empty[slot]);
      ++sched_it;
      if (!live) break;
      const int nt = u.k1 - u.k0;
      const int qr = q_row(u.s, u.L, u.m, rloc);   // this lane's row of the sequence, or -1
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      const long long grow = static_cast<long long>(u.s.q0) + row;   // global token row
      const int ob = q_it % OB;
      const uint32_t o_tmem = tmem + lane_base + Cfg::O_COL + ob * DV;
      float m_run = -INFINITY, l_run = 0.f;
      if (nt > 0) {
        if (!warp_wait_or_abort(ctl, p, &ctl.o_full[ob], (q_it / OB) & 1)) break;
        if constexpr (SOFTMAX) {
          if (!warp_wait_or_abort(ctl, p, &ctl.rs_full[ob], (q_it / OB) & 1)) break;
          m_run = sx->rs_m[ob][rloc];
          l_run = sx->rs_l[ob][0][rloc] + sx->rs_l[ob][1][rloc];
        }
        ptx::tc_fence_after();
      }
      const bool write_part = p.splits > 1;
      const long long grow0 = __shfl_sync(0xffffffffu, grow, 0);
      const bool tma_rows = Cfg::STAGE_BUFS > 0 && !write_part &&
                            __all_sync(0xffffffffu, valid && grow == grow0 + lane);   // warp-uniform
      float mul = u.scale;
      if constexpr (SOFTMAX) mul = l_run > 0.f ? u.scale / l_run : 0.f;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        if (nt > 0) {
          ptx::tmem_ld32(o_tmem + c * 32, o);
          ptx::tmem_ld_wait(o);
          if (c == DV / 32 - 1) {   // all of O read: the buffer (and statistics) may be reused
            ptx::tc_fence_before();
            ptx::mbar_arrive(&ctl.o_empty[ob]);
            if constexpr (SOFTMAX) ptx::mbar_arrive(&ctl.rs_empty[ob]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0u;
        }
        // unused lanes store nothing (a branch, not a `continue`: the warp stays
        // converged for the next collective TMEM load)
        if (valid && write_part) {
          // fp32 partial, already x attn_scale (softmax: not yet / row sum)
          float* dst = p.o_part + ((static_cast<long long>(u.sp) * p.total_q + grow) * p.nhead + u.h) * DV + c * 32;
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + k) =
                make_float4(__uint_as_float(o[k]) * u.scale, __uint_as_float(o[k + 1]) * u.scale,
                            __uint_as_float(o[k + 2]) * u.scale, __uint_as_float(o[k + 3]) * u.scale);
        } else if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2)
            pk[k >> 1] = pack2<BF16>(__uint_as_float(o[k]) * mul, __uint_as_float(o[k + 1]) * mul);
          bool staged = false;
          if constexpr (Cfg::STAGE_BUFS > 0) {
            if (tma_rows) {
              // columns [32 c, 32 c + 32) are 16-byte pieces 4 (c & 1) .. 4 (c & 1) + 3 of
              // the row in box c / 2; piece j of row r sits at r * 128 + ((j ^ (r & 7)) * 16)
              staged = true;
              const uint32_t buf = stage_warp + (st_it % Cfg::STAGE_BUFS) * Cfg::STAGE_BOX_BYTES;
              if ((c & 1) == 0 && st_it >= Cfg::STAGE_BUFS) {   // that buffer's last store has read it
                if (lane == 0) ptx::bulk_wait_group_read<Cfg::STAGE_BUFS - 1>();
                __syncwarp();
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int j = (c & 1) * 4 + q;
                ptx::st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), pk[4 * q], pk[4 * q + 1],
                                  pk[4 * q + 2], pk[4 * q + 3]);
              }
              if (c & 1) {
                ptx::fence_proxy_async_smem();   // the generic-proxy writes, before the bulk copy reads them
                __syncwarp();
                if (lane == 0) {
                  ptx::tma_store_2d(&tm_o, buf, u.h * DV + (c >> 1) * 64, static_cast<int>(grow0));
                  ptx::bulk_commit_group();
                }
                ++st_it;
              }
            }
          }
          if (!staged) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(p.o) + grow * p.o_stride + u.h * DV + c * 32;
#pragma unroll
            for (int k = 0; k < 16; k += 4)
              *reinterpret_cast<uint4*>(dst + 2 * k) = make_uint4(pk[k], pk[k + 1], pk[k + 2], pk[k + 3]);
          }
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
    const int wg = (warp - 2 - kEpiWarps) >> 2;   // warpgroup: key columns [64 wg, 64 wg + 64)
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int rloc = quarter * 32 + lane;    // row within the query tile
    const int c0 = wg * 64;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const float half_alpha = 0.5f * p.alpha;   // SiLU's argument halved: h = alpha s / 2
    const float scale_log2 = p.alpha * 1.4426950408889634f;
    int s_it = 0, q_it = 0, sched_it = 0;
    while (!ctl.abort_flag) {
      const int slot = sched_it % kSchedDepth;
      if (!warp_wait_or_abort(ctl, p, &ctl.sched_full[slot], (sched_it / kSchedDepth) & 1)) break;
      const bool live = ctl.sched_live[slot] != 0;
      const UnitView u = ctl.sched_view[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&ctl.sched_empty[slot]);
      ++sched_it;
      if (!live) break;
      const int nt = u.k1 - u.k0;
      const int qr = q_row(u.s, u.L, u.m, rloc);   // this lane's row of the sequence, or -1
      const bool valid = qr >= 0;
      const int row = valid ? qr : 0;
      int r_lo, r_hi;
      row_uih_keys(u.s, row, r_lo, r_hi);
      int r_diag = row_diag_key(u.s, row);
      int r_ctx = u.s.c;
      if (!valid) { r_lo = r_hi = 0; r_diag = -1; r_ctx = 0; }
      // relative attention bias: this warp's tables for the unit's head, and the
      // row's timestamp (relative to the sequence's first key) and position
      RabRow rrow{0, 0};
      long long ts_row = 0;   // the row's timestamp; made relative to each key tile's first key
      if constexpr (RAB) {
        RabWarp& rw = rabw[warp - 2 - kEpiWarps];
        __syncwarp();   // the previous unit's lookups are done
        rab_build(rw, p.ts_q != nullptr ? p.rab_time : nullptr, p.rab_pos, p.rab_np, u.h,
                  SOFTMAX ? 1.4426950408889634f : 0.5f, lane);
        __syncwarp();
        if (p.ts_q != nullptr) ts_row = p.ts_q[u.s.q0 + row];
        rrow.pos = row < u.s.c ? row : row + (u.s.ukv - u.s.u);
      }
      const int ob = q_it % OB;
      const uint32_t o_tmem = tmem + lane_base + Cfg::O_COL + ob * DV;   // softmax rescale:
                                                                        // 32-column chunks wg, wg+2, ...

      float m_run = -INFINITY, l_run = 0.f;   // softmax row state (log2 domain); l over own columns
      bool ok = true;
      // Walk tiles [k0, k1) of the unit's tile set: n is the current key tile,
      // n_end the end of its range, (n_lo1, n_hi1) the next range.  Ranges are
      // sorted and empty ones come last, so one step to the next range suffices.
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
      const FullTiles ft = full_tile_ranges(u.s, u.tb);
      // bias: raw timestamps of this warpgroup's 64 keys of the next tile, one
      // per lane and chunk (keys past the sequence repeat its last one), loaded
      // a tile ahead so their latency hides behind the current tile
      long long nk0 = 0, nk1 = 0;
      auto load_keys = [&](int jt0) {
        if constexpr (RAB) {
          if (p.ts_q != nullptr) {
            nk0 = p.ts_kv[u.s.kv0 + min(jt0 + c0 + lane, u.s.Lkv - 1)];
            nk1 = p.ts_kv[u.s.kv0 + min(jt0 + c0 + 32 + lane, u.s.Lkv - 1)];
          }
        }
      };
      if (nt > 0) load_keys(n * kBlockN);
      for (int idx = 0; idx < nt; ++idx) {
        const bool full = n < ft.ctx_hi || (n >= ft.lo && n < ft.hi);
        const int j0 = n * kBlockN;
        if (++n == n_end) {
          n = n_lo1; n_end = n_hi1;
          n_lo1 = n_lo2; n_hi1 = n_hi2;
        }
        const long long ck0 = nk0, ck1 = nk1;
        if (idx + 1 < nt) load_keys(n * kBlockN);
        RowMask rm;
        rm.ctx = r_ctx - j0;
        rm.lo = r_lo - j0;
        rm.span = static_cast<uint32_t>(r_hi - r_lo);
        rm.diag = r_diag >= 0 ? r_diag - j0 : -1000000;
        const int si = s_it + idx;
        // bias: the keys' timestamps (loaded a tile ahead) and the row's, relative
        // to the warpgroup's first key of the tile
        int tsk0 = 0, tsk1 = 0;
        if constexpr (RAB) {
          if (p.ts_q != nullptr) {
            const long long base = __shfl_sync(0xffffffffu, ck0, 0);
            tsk0 = rab_rel_ts(ck0, base);
            tsk1 = rab_rel_ts(ck1, base);
            rrow.ts = rab_rel_ts(ts_row, base);
          }
        }
        if (!warp_wait_or_abort(ctl, p, &ctl.s_full[si & 1], (si >> 1) & 1)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t s_tmem = tmem + lane_base + (si & 1) * 128 + c0;
        uint32_t r[64];
        float rab_mx = -INFINITY;   // softmax with the bias: the row max of the biased scores
        if constexpr (RAB && !SOFTMAX) {
          // SiLU with the bias: a runtime loop over the two 32-column halves,
          // so the bias code is inlined once per tile.  Each half is loaded,
          // becomes (alpha s + rab) / 2, and packs into its 16 P words at the
          // columns the one-store form uses (word k holds columns 2k, 2k+1):
          // half 0 over its own first 16 S columns, half 1 over half 0's
          // last 16, all already in registers.
          const RabWarp& rw = rabw[warp - 2 - kEpiWarps];
          const bool has_time = p.ts_q != nullptr && p.rab_time != nullptr;
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t x[32];
            ptx::tmem_ld32(s_tmem + 32 * hh, x);
            ptx::tmem_ld_wait(x);
            // keys past the sequence repeat its last one: every column counts in the ranges
            rab_apply32<true>(x, 0.5f * p.alpha, rw, p.rab_np, has_time, rrow,
                              rab_cols(hh ? tsk1 : tsk0, j0 + c0 + 32 * hh + lane, true));
            if (full) silu_pack<BF16, false, true, 16>(x, s_tmem + 16 * hh, half_alpha, rm, c0 + 32 * hh);
            else silu_pack<BF16, true, true, 16>(x, s_tmem + 16 * hh, half_alpha, rm, c0 + 32 * hh);
          }
        } else {
          if constexpr (RAB && SOFTMAX) {
            // softmax with the bias: the same runtime loop over the halves,
            // each half's (alpha s + rab) * log2 e, masked scores -inf, written
            // back over its own scores and folded into the row max; the
            // exponentials below take the halves again (32 score registers live
            // at a time instead of 64)
            const RabWarp& rw = rabw[warp - 2 - kEpiWarps];
            const bool has_time = p.ts_q != nullptr && p.rab_time != nullptr;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t x[32];
              ptx::tmem_ld32(s_tmem + 32 * hh, x);
              ptx::tmem_ld_wait(x);
              // keys past the sequence repeat its last one: every column counts in the ranges
              rab_apply32<true>(x, scale_log2, rw, p.rab_np, has_time, rrow,
                                rab_cols(hh ? tsk1 : tsk0, j0 + c0 + 32 * hh + lane, true));
              if (!full) {
                const uint32_t mb = rm.bits32(c0 + 32 * hh);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                  const uint32_t keep = static_cast<uint32_t>(static_cast<int32_t>(mb << (31 - k)) >> 31);
                  x[k] = (x[k] & keep) | (0xFF800000u & ~keep);   // masked scores become -inf
                }
              }
#pragma unroll
              for (int k = 0; k < 32; ++k) rab_mx = fmaxf(rab_mx, __uint_as_float(x[k]));
              ptx::tmem_st32(s_tmem + 32 * hh, x);
            }
            ptx::tmem_st_wait();
          } else {
            ptx::tmem_ld64(s_tmem, r);
            ptx::tmem_ld_wait(r);
          }
        }
        if constexpr (!SOFTMAX) {
          if constexpr (!RAB) {
            // P is packed over this warpgroup's S columns (already in registers)
            if (full) silu_pack<BF16, false>(r, s_tmem, half_alpha, rm, c0);
            else silu_pack<BF16, true>(r, s_tmem, half_alpha, rm, c0);
          }
        } else {
          float mx = RAB ? rab_mx : -INFINITY;
          if (RAB) {
            // (max and mask already taken in the bias pass)
          } else if (full) {
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
          // row max over both halves
          sx->xmax[si & 1][wg][rloc] = mx;
          ptx::mbar_arrive(&ctl.xch[si & 1]);
          if (!warp_wait_or_abort(ctl, p, &ctl.xch[si & 1], (si >> 1) & 1)) { ok = false; break; }
          mx = fmaxf(mx, sx->xmax[si & 1][wg ^ 1][rloc]);
          if constexpr (!RAB) mx *= scale_log2;   // with a bias the scores are already in log2 units
          // PV of the tile before last must be complete before this tile; keeps the
          // parity tracking of pv_done unambiguous.
          if (si >= 2) {
            if (!warp_wait_or_abort(ctl, p, &ctl.pv_done[si & 1], ((si - 2) >> 1) & 1)) { ok = false; break; }
          }
          // A new running max more than 2^8 above the old one: rescale what O
          // already holds (only after a previous tile of this unit, whose PV
          // must have completed).  The need is per row, but the wait and the
          // TMEM accesses are warp-collective, so a warp rescales when any of
          // its rows needs it and the other rows multiply by 1.  Both
          // warpgroups see the same maxima, so the same warps of each take
          // the branch.
          const bool grow = mx > m_run + 8.0f;
          const bool rescale = grow && idx > 0 && m_run != -INFINITY;
          if (__any_sync(0xffffffffu, rescale)) {
            const int sp = si - 1;
            if (!warp_wait_or_abort(ctl, p, &ctl.pv_done[sp & 1], (sp >> 1) & 1)) { ok = false; break; }
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
          if constexpr (RAB) {
            // the halves again: half 0's P words over its own first 16
            // columns, half 1's over half 0's last 16 (both already read)
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t x[32], pk[16];
              ptx::tmem_ld32(s_tmem + 32 * hh, x);
              ptx::tmem_ld_wait(x);
#pragma unroll
              for (int k = 0; k < 32; ++k)   // masked scores are -inf and give 0
                x[k] = __float_as_uint(ex2_approx(__uint_as_float(x[k]) + nm));
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float e0 = __uint_as_float(x[2 * k]), e1 = __uint_as_float(x[2 * k + 1]);
                lsum0 += e0;
                lsum1 += e1;
                pk[k] = pack2<BF16>(e0, e1);
              }
              ptx::tmem_st16(s_tmem + 16 * hh, pk);
            }
          } else {
            uint32_t pk[32];
            // stage by stage so the exponentials of the 64 scores overlap
#pragma unroll
            for (int k = 0; k < 64; ++k)   // masked scores are -inf and give 0
              r[k] = __float_as_uint(fmaf(__uint_as_float(r[k]), scale_log2, nm));
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
          }
          l_run += lsum0 + lsum1;
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&ctl.p_full[si & 1]);
      }
      if (!ok) break;

      if constexpr (SOFTMAX) {
        // hand this unit's row statistics to the epilogue warpgroup
        if (nt > 0) {
          if (!warp_wait_or_abort(ctl, p, &ctl.rs_empty[ob], ((q_it / OB) & 1) ^ 1)) break;
          if (wg == 0) sx->rs_m[ob][rloc] = m_run;
          sx->rs_l[ob][wg][rloc] = l_run;
          ptx::mbar_arrive(&ctl.rs_full[ob]);
        }
      }
      if (nt > 0) ++q_it;
      s_it += nt;
    }
  }

  // ---------------------------------------------------------------- teardown
  if constexpr (Cfg::STAGE_BUFS > 0) {
    // epilogue warps: their TMA stores have read the staging buffers and landed
    if (warp >= 2 && warp < 2 + kEpiWarps && lane == 0) ptx::bulk_wait_group<0>();
  }
  if (ctl.abort_flag && tid == 0) {
    // let copies / MMAs already in flight land before the CTA releases its memory
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

// ---------------------------------------------------------------- host launch
// One instantiation of the forward: its shared-memory limit set once per
// device, launched as a programmatic dependent of the scheduler kernel that
// precedes it on the stream.
template <int D, int DV, bool BF16, bool SOFTMAX, bool RAB>
cudaError_t launch_fwd_inst(const FwdMaps& m, const FwdParams& p, int grid, cudaStream_t stream) {
  constexpr int smem = FwdCfg<D, DV, SOFTMAX, RAB>::SMEM_BYTES;
  static_assert(smem + sizeof(FwdSmemCtl) <= 232448, "shared memory over the 227 KB a CTA may use");
  auto kern = hstu_fwd_kernel<D, DV, BF16, SOFTMAX, RAB>;
  static std::atomic<unsigned long long> attr_set{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_set);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, m.q8, m.o, p);
}

// The four dtype x nonlinearity instantiations of one head-dimension pair.
template <int D, int DV, bool RAB>
cudaError_t launch_fwd_dispatch(const FwdMaps& m, const FwdParams& p, bool bf16, bool softmax, int grid,
                                cudaStream_t stream) {
  if (bf16) return softmax ? launch_fwd_inst<D, DV, true, true, RAB>(m, p, grid, stream)
                           : launch_fwd_inst<D, DV, true, false, RAB>(m, p, grid, stream);
  return softmax ? launch_fwd_inst<D, DV, false, true, RAB>(m, p, grid, stream)
                 : launch_fwd_inst<D, DV, false, false, RAB>(m, p, grid, stream);
}

}  // namespace hstu
