// Relative attention bias of the HSTU layer ("From transformer parallelism to
// HSTU", sections 2.4 and 3.5): added to the scaled score of every (query row
// i, key j) before the nonlinearity,
//
//   rab[i, j] = rab_time[h, bucket(|ts_i - ts_j|)] + rab_pos[h, min(|pos_i - j|, P - 1)]
//
// with the section's time-gap buckets (lower edges 0, 1, 5, 30, 60, 300, 1800,
// 3600, 86400, 604800, 2.6e6 seconds; the last bucket open-ended) and pos_i the
// query row's position in key coordinates (i for a context row, i + (u_kv - u)
// for UIH and target rows: the mask's bottom-right alignment).
//
// Device side, per elementwise warp:
//   * once per unit, a 33-entry table indexed by clz(gap): a gap's leading bit
//     fixes its power-of-two octave, and no octave holds more than one bucket
//     edge, so an entry packs the bucket at the octave's low end (bits 27-30)
//     and the edge inside it (bits 0-26; all ones when there is none, which
//     only gaps of 2^27 s and more reach, and those are in the last bucket,
//     whose weight is repeated one slot further); the head's 11 time weights
//     and its positional table, all fp32;
//   * per key tile, the warpgroup's 64 keys' timestamps, loaded one tile ahead,
//     and the row's, relative to the first of those keys and clamped to
//     +-2^30 s so every gap fits 32 bits (a row clamped there is at least
//     2^29 s from every key of a tile spanning less than 2^29 s: the last
//     bucket either way), the keys' in two registers per lane, read by the
//     other lanes with shuffles;
//   * per 32-column chunk and row, each term is one constant when the row's
//     timestamp lies outside the columns' range and both ends fall in the same
//     bucket (the extreme gaps are at the range's ends), and when every column
//     is at least P - 1 away; otherwise it is looked up column by column.
// Weights are stored pre-multiplied by the factor the caller's arithmetic
// wants (1/2 for the SiLU half-argument, log2 e for the softmax exponent).
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "hstu_common.cuh"
#include "ptx.cuh"

namespace hstu {

constexpr int kRabTimeBuckets = 11;
constexpr int kRabMaxPos = 256;               // largest positional table per head
constexpr int kRabTsClamp = 1 << 30;          // relative timestamps are clamped to +-2^30 s
constexpr int kRabNoEdge = (1 << 27) - 1;

// Lower edges of the time-gap buckets in seconds ("From transformer parallelism
// to HSTU", section 3.5).
__host__ __device__ constexpr int rab_time_edge(int k) {
  return k == 0 ? 0 : k == 1 ? 1 : k == 2 ? 5 : k == 3 ? 30 : k == 4 ? 60 : k == 5 ? 300
       : k == 6 ? 1800 : k == 7 ? 3600 : k == 8 ? 86400 : k == 9 ? 604800 : 2600000;
}
// Bucket of a gap >= 0: the last bucket whose lower edge it reaches.
__host__ __device__ inline int rab_time_bucket(long long gap) {
  int b = 0;
  for (int k = 1; k < kRabTimeBuckets; ++k) b += gap >= rab_time_edge(k) ? 1 : 0;
  return b;
}

// Per elementwise warp.
struct RabWarp {
  int tab[33];                       // by clz(gap): bucket at the octave's low end << 27 | edge inside it
  float wt[kRabTimeBuckets + 1];     // time weights (pre-scaled); the last repeated
  float pos[kRabMaxPos];             // positional weights (pre-scaled)
};

__device__ __forceinline__ int rab_rel_ts(long long t, long long base) {
  long long d = t - base;
  d = d < -static_cast<long long>(kRabTsClamp - 1) ? -static_cast<long long>(kRabTsClamp - 1) : d;
  d = d > static_cast<long long>(kRabTsClamp - 1) ? static_cast<long long>(kRabTsClamp - 1) : d;
  return static_cast<int>(d);
}

// Builds the warp's tables for head h (all lanes call it); `scale` multiplies
// every weight.  Null tables give zero terms.
__device__ __forceinline__ void rab_build(RabWarp& w, const float* rab_time, const float* rab_pos, int np, int h,
                                          float scale, int lane) {
  for (int idx = lane; idx <= 32; idx += 32) {
    // octave of clz == idx: gaps [2^(31 - idx), 2^(32 - idx)); idx 32: gap 0
    const long long lo = idx == 32 ? 0 : (1LL << (31 - idx));
    const long long hi = idx == 32 ? 1 : (1LL << (32 - idx));
    const int b = rab_time_bucket(lo);
    int edge = kRabNoEdge;
    if (b + 1 < kRabTimeBuckets && rab_time_edge(b + 1) < hi) edge = rab_time_edge(b + 1);
    w.tab[idx] = (b << 27) | edge;
  }
  if (lane < kRabTimeBuckets + 1) {
    const int b = lane < kRabTimeBuckets ? lane : kRabTimeBuckets - 1;
    w.wt[lane] = rab_time != nullptr ? rab_time[h * kRabTimeBuckets + b] * scale : 0.f;
  }
  for (int d = lane; d < np; d += 32) w.pos[d] = rab_pos != nullptr ? rab_pos[h * np + d] * scale : 0.f;
}

// Bucket slot of one gap (0 <= gap < 2^31); slot 11 stands for bucket 10.
__device__ __forceinline__ int rab_time_slot(const RabWarp& w, int gap) {
  const int e = w.tab[__clz(gap)];
  return (e >> 27) + (gap >= (e & kRabNoEdge) ? 1 : 0);
}
// Temporal weight of one gap.
__device__ __forceinline__ float rab_time_weight(const RabWarp& w, int gap) { return w.wt[rab_time_slot(w, gap)]; }

// This lane's row: relative timestamp and key-coordinate position.
struct RabRow {
  int ts, pos;
};

// The 32 columns of a chunk, lane l describing column l: its relative
// timestamp and key-coordinate position, and over the valid columns the
// extremes of both (invalid columns are ignored there and their scores
// masked later).
struct RabCols {
  int ts, pos;
  int tmin, tmax, pmin, pmax;
};
__device__ __forceinline__ RabCols rab_cols(int ts, int pos, bool valid) {
  RabCols c;
  c.ts = ts;
  c.pos = pos;
  c.tmin = __reduce_min_sync(0xffffffffu, valid ? ts : 0x7fffffff);
  c.tmax = __reduce_max_sync(0xffffffffu, valid ? ts : -0x7fffffff);
  c.pmin = __reduce_min_sync(0xffffffffu, valid ? pos : 0x7fffffff);
  c.pmax = __reduce_max_sync(0xffffffffu, valid ? pos : -0x7fffffff);
  return c;
}

// How a chunk's two terms vary, for one row: the distance term is one constant
// (the table's last entry) when every column is at least np - 1 away; the time
// term is one constant when the row's timestamp lies outside the columns'
// range and both ends fall in the same bucket (the extreme gaps are at the
// range's ends).  all_* are the warp's agreement (warp-collective).
struct RabChunk {
  bool time_const;   // this row
  int slot;          // this row's time slot at the columns' near end (the constant when time_const)
  bool all_pos, all_time;
};
__device__ __forceinline__ RabChunk rab_classify(const RabWarp& w, int np, bool has_time, const RabRow& row,
                                                 const RabCols& c) {
  RabChunk k;
  const int dmin = row.pos <= c.pmin ? c.pmin - row.pos : (row.pos >= c.pmax ? row.pos - c.pmax : 0);
  const bool pos_const = dmin >= np - 1;
  k.time_const = !has_time;
  k.slot = -1;
  if (has_time && (row.ts >= c.tmax || row.ts <= c.tmin)) {
    const int g0 = abs(row.ts - c.tmin), g1 = abs(row.ts - c.tmax);
    const int s0 = rab_time_slot(w, g0), s1 = rab_time_slot(w, g1);
    k.time_const = s0 == s1 || (s0 >= kRabTimeBuckets - 1 && s1 >= kRabTimeBuckets - 1);
    k.slot = s0;
  }
  k.all_pos = __all_sync(0xffffffffu, pos_const);
  k.all_time = __all_sync(0xffffffffu, k.time_const);
  return k;
}

// r[k] (a raw score, fp32 bits) becomes fma(s, mul, scaled bias) for the 32
// columns of the chunk: bias(row, column k) = time weight of |row.ts - ts_k|
// plus distance weight of min(|row.pos - pos_k|, np - 1).  CONTIG: column k's
// position is c.pmin + k (keys of a tile), else it comes from lane k.  The
// whole warp takes one of three forms (rab_classify), so every lane runs the
// same shuffles: both terms constant, only the distance looked up key by key,
// or both looked up (a constant distance term then reads the table's last
// entry).  Fewer unrolled forms keep the code small enough to stay in the
// instruction cache.  Returns the chunk's classification.  Warp-collective.
template <bool CONTIG>
__device__ __forceinline__ RabChunk rab_apply32(uint32_t* r, float mul, const RabWarp& w, int np, bool has_time,
                                                const RabRow& row, const RabCols& c) {
  const RabChunk k = rab_classify(w, np, has_time, row, c);
  const float wt_const = k.slot >= 0 ? w.wt[k.slot] : 0.f;
  if (k.all_pos && k.all_time) {
    const float b = w.pos[np - 1] + wt_const;
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(fmaf(__uint_as_float(r[j]), mul, b));
  } else if (k.all_time) {   // the distance varies over the chunk, the time bucket does not
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int pk = CONTIG ? c.pmin + j : __shfl_sync(0xffffffffu, c.pos, j);
      int d = abs(row.pos - pk);
      d = d < np - 1 ? d : np - 1;
      r[j] = __float_as_uint(fmaf(__uint_as_float(r[j]), mul, w.pos[d] + wt_const));
    }
  } else {   // the time bucket varies (and the distance may)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int tk = __shfl_sync(0xffffffffu, c.ts, j);
      const int pk = CONTIG ? c.pmin + j : __shfl_sync(0xffffffffu, c.pos, j);
      float b = k.time_const ? wt_const : rab_time_weight(w, abs(row.ts - tk));
      int d = abs(row.pos - pk);
      d = d < np - 1 ? d : np - 1;
      b += w.pos[d];
      r[j] = __float_as_uint(fmaf(__uint_as_float(r[j]), mul, b));
    }
  }
  return k;
}

// Per elementwise warp: the gradients of the two tables over the current
// unit (slot 11 of t stands for bucket 10, as in RabWarp::wt).
struct RabGradWarp {
  float t[kRabTimeBuckets + 1];
  float pos[kRabMaxPos];
};

// One lane's running sums of score gradients between flushes: the time
// bucket it is adding to (-1: none yet) and that sum, and the sum for the
// distance table's last entry (every column at least np - 1 away).  A row's
// bucket changes only a few times along a unit's key tiles, so most chunks
// add in registers.
struct RabGradAcc {
  int t_slot;
  float t_sum;
  float far_pos;
};
__device__ __forceinline__ void rab_grad_time_add(RabGradAcc& a, RabGradWarp& g, int slot, float v) {
  if (slot != a.t_slot) {
    if (a.t_slot >= 0) atomicAdd(&g.t[a.t_slot], a.t_sum);
    a.t_slot = slot;
    a.t_sum = 0.f;
  }
  a.t_sum += v;
}

// Adds the score gradients ds[k] of one row's chunk (the columns rab_apply32
// took, with the classification k it returned) to the entries of the two
// tables they read:
// time-bucket sums and the far distance entry in the lane's registers (acc),
// nearer distances per column into the warp's shared sums (neighbouring rows
// are at different distances, so those adds rarely collide).  has_time /
// has_pos: the tables exist.  Warp-collective.
template <bool CONTIG>
__device__ __forceinline__ void rab_grad32(const float (&ds)[32], const RabChunk& k, RabGradWarp& g, RabGradAcc& acc,
                                           const RabWarp& w, int np, bool has_time, bool has_pos, const RabRow& row,
                                           const RabCols& c) {
  float sum;
  {
    uint64_t s2 = ptx::f32x2(ds[0], ds[1]);
#pragma unroll
    for (int j = 2; j < 32; j += 2) s2 = ptx::fma_f32x2(ptx::f32x2(ds[j], ds[j + 1]), ptx::f32x2(1.f, 1.f), s2);
    float lo, hi;
    ptx::f32x2_split(s2, lo, hi);
    sum = lo + hi;
  }
  if (has_pos) {
    if (k.all_pos) {
      acc.far_pos += sum;
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int pk = CONTIG ? c.pmin + j : __shfl_sync(0xffffffffu, c.pos, j);
        const int d = abs(row.pos - pk);
        if (d < np - 1) atomicAdd(&g.pos[d], ds[j]);
        else acc.far_pos += ds[j];
      }
    }
  }
  if (has_time) {
    if (k.all_time) {
      rab_grad_time_add(acc, g, k.slot, sum);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int tk = __shfl_sync(0xffffffffu, c.ts, j);
        if (!k.time_const) rab_grad_time_add(acc, g, rab_time_slot(w, abs(row.ts - tk)), ds[j]);
      }
      if (k.time_const) rab_grad_time_add(acc, g, k.slot, sum);
    }
  }
}

// The lane's register sums into the warp's shared sums (the far distance
// entry summed over the warp first).  Warp-collective.
__device__ __forceinline__ void rab_grad_flush(RabGradAcc& acc, RabGradWarp& g, int np, bool has_time, bool has_pos) {
  if (has_time && acc.t_slot >= 0) atomicAdd(&g.t[acc.t_slot], acc.t_sum);
  if (has_pos) {
    float tot = acc.far_pos;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&g.pos[np - 1], tot);
  }
  acc = RabGradAcc{-1, 0.f, 0.f};
}

}  // namespace hstu
