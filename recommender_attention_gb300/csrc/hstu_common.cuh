// Shared definitions of the HSTU forward kernels: launch parameters, the
// per-sequence geometry and the functional mask in interval form.
//
// Mask (composable_kernel 18_hstu_attention README, "Masking" table and the
// phy_seqlen formulas).  A sequence is laid out [context c | UIH u | targets t]
// on the query side and [context c | UIH u_kv | targets t] (self-attention) or
// [context c | UIH u_kv] (cross-attention) on the key side.  For a query row i
// the allowed keys are exactly
//     [0, c)                    context keys, visible to every query
//   U [lo_i, hi_i)              the row's UIH keys (one interval, see below)
//   U {i} if i is a target row  (self-attention: a target key is seen only by itself)
// where, with UIH coordinates x_i = (i - c) + (u_kv - u) for a UIH row
// (bottom-right aligned for cross-attention), x_i = u_kv for a target row and
// x_j = j - c for a key:
//   context rows: every UIH key;
//   other rows:   x_j <= x_i when causal; when a local window W > 0 applies and
//                 the row is not in the min-full tail (F > 0 and x_i >= u_kv - F),
//                 |x_i - x_j| <= W.
// Because consecutive rows' intervals overlap or nest, the union over any run
// of rows is again one interval; tile skipping relies on that.
#pragma once
#include <cstdint>
#include <climits>

#ifdef __CUDACC__
#define HSTU_HD __host__ __device__ __forceinline__
#else
#define HSTU_HD inline
#endif

namespace hstu {

constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 128;      // keys per tile
constexpr int kFwdEpiWarps = 4;   // epilogue warps of the forward kernel (32 query rows each)
constexpr int kFusedMaxBatch = 128;   // largest batch the forward kernel schedules by itself
constexpr int kMaxGroups = 256;   // per-group parameter slots in the launch parameters
constexpr int kMaxSplits = 16;

// Device error word bits (also returned by hstu_attn_fwd_check).
enum : int {
  kErrOffsets = 1,       // offsets not monotone or beyond the token totals
  kErrQLayout = 2,       // query length < context + targets
  kErrKvLayout = 4,      // key length < context (cross) / != query length (self)
  kErrMaxSeqlen = 8,     // a length exceeds the max_seqlen hint the workspace was sized for
  kErrTimeout = 16,      // a pipeline wait gave up (the kernel returned early)
};

// Workspace header (int32 slots).
enum : int {
  kWsUnits = 0,      // number of work units written by the scheduler
  kWsError = 1,      // device error word
  kWsCounter = 2,    // dynamic work counter of the persistent kernel
  kWsTilesLo = 4,    // executed (b, h, q-tile, kv-tile) blocks, int64 in slots 4-5
  kWsPairsLo = 6,    // allowed (b, h, i, j) pairs, int64 in slots 6-7 (stats only)
  kWsKvUnits = 8,    // backward: number of key-tile work units
  kWsKvCounter = 9,  // backward: dynamic work counter of the dK/dV kernel
  kWsHeaderInts = 64,
};

struct SeqGeom {
  int q0, kv0;     // first token of the sequence in the flattened Q / KV tensors
  int Lq, Lkv;     // physical lengths
  int c, u, ukv;   // context, query UIH, key UIH lengths
  int W, F;        // local window, min-full tail
  int causal, self_attn;
  int tkv;         // the key side ends with the targets' own keys (self-attention, or
                   // cross-attention over a cached history: M-FALCON)
};

// UIH coordinate of query row i (meaningful for i >= c).
HSTU_HD int uih_coord(const SeqGeom& s, int i) {
  return i < s.c + s.u ? (i - s.c) + (s.ukv - s.u) : s.ukv;
}

// Allowed UIH keys of query row i as the key interval [lo, hi); hi == lo when none.
HSTU_HD void row_uih_keys(const SeqGeom& s, int i, int& lo, int& hi) {
  if (i < s.c) {
    lo = s.c;
    hi = s.c + s.ukv;
    return;
  }
  const int x = uih_coord(s, i);
  int xlo = 0, xhi = s.ukv - 1;
  if (s.causal) xhi = xhi < x ? xhi : x;
  const bool full = s.F > 0 && x >= s.ukv - s.F;
  if (s.W > 0 && !full) {
    xlo = xlo > x - s.W ? xlo : x - s.W;
    if (!s.causal) xhi = xhi < x + s.W ? xhi : x + s.W;
  }
  lo = s.c + xlo;
  hi = s.c + xhi + 1;
  if (hi < lo) hi = lo;
}

// The single target key row i may see (its own), or -1.  Target r is query row
// c + u + r and key row c + ukv + r.
HSTU_HD int row_diag_key(const SeqGeom& s, int i) {
  return (s.tkv && i >= s.c + s.u && i < s.Lq) ? i + (s.ukv - s.u) : -1;
}

// Number of allowed keys of row i (0 <= i < Lq).
HSTU_HD int row_pair_count(const SeqGeom& s, int i) {
  int lo, hi;
  row_uih_keys(s, i, lo, hi);
  return s.c + (hi - lo) + (row_diag_key(s, i) >= 0 ? 1 : 0);
}

// Over the valid rows of [i0, i1): the hull [LO, HI) of their UIH-key intervals
// (LO >= HI: no row has one), the largest lo and the smallest hi.  The interval
// ends are monotone on each of the pieces context / UIH before the min-full
// tail / min-full tail / targets, so evaluating the rows at piece boundaries
// gives the exact extremes.
struct TileBounds {
  int LO, HI, maxLO, minHI;
};
HSTU_HD TileBounds tile_uih_bounds(const SeqGeom& s, int i0, int i1) {
  if (i1 > s.Lq) i1 = s.Lq;
  TileBounds t{INT_MAX, INT_MIN, INT_MIN, INT_MAX};
  const int ff = s.c + (s.u - s.F > 0 ? s.u - s.F : 0);
  int shift = s.u - s.ukv;
  if (!s.causal && s.W > 0) shift -= s.W;
  const int fne = s.c + (shift > 0 ? shift : 0);
  const int cand[10] = {i0, i1 - 1, s.c - 1, s.c, s.c + s.u - 1, s.c + s.u, ff - 1, ff, fne - 1, fne};
#pragma unroll
  for (int k = 0; k < 10; ++k) {
    int r = cand[k];
    r = r < i0 ? i0 : r;
    r = r > i1 - 1 ? i1 - 1 : r;
    int lo, hi;
    row_uih_keys(s, r, lo, hi);
    t.maxLO = t.maxLO > lo ? t.maxLO : lo;
    t.minHI = t.minHI < hi ? t.minHI : hi;
    if (hi > lo) {
      t.LO = t.LO < lo ? t.LO : lo;
      t.HI = t.HI > hi ? t.HI : hi;
    }
  }
  return t;
}

HSTU_HD TileBounds merge_bounds(TileBounds a, const TileBounds& b) {
  a.LO = a.LO < b.LO ? a.LO : b.LO;
  a.HI = a.HI > b.HI ? a.HI : b.HI;
  a.maxLO = a.maxLO > b.maxLO ? a.maxLO : b.maxLO;
  a.minHI = a.minHI < b.minHI ? a.minHI : b.minHI;
  return a;
}

// Query-tile layout of a sequence.  Query tile m holds rows [128 m, 128 m + 128)
// on lanes 0..127, aligned with the key tiles so a causal diagonal stays within
// one key tile.  Context rows see every UIH key, so the tile holding them runs
// all of the sequence's key tiles; when the sequence has more than one query
// tile and the context rows fit on the spare top lanes of the last tile (from
// lane 128 - ceil8(c), so each 8-row group is a whole swizzle atom), they move
// there: that tile already runs every UIH key tile in the common causal case,
// and tile 0 then runs only its own diagonal.  Lanes [0, c) of tile 0 are then
// unused.
struct QLayout {
  int nq;          // query tiles of the sequence
  int ctx_lane0;   // >= 0: the context rows sit on lanes [ctx_lane0, ctx_lane0 + c) of tile nq - 1
};
HSTU_HD QLayout q_layout(int Lq, int c) {
  QLayout L;
  L.nq = (Lq + kBlockM - 1) / kBlockM;
  L.ctx_lane0 = -1;
  if (c > 0 && L.nq > 1) {
    const int cpad = (c + 7) & ~7;
    const int last_rows = Lq - (L.nq - 1) * kBlockM;
    if (cpad <= kBlockM - last_rows) L.ctx_lane0 = kBlockM - cpad;
  }
  return L;
}
HSTU_HD QLayout q_layout(const SeqGeom& s) { return q_layout(s.Lq, s.c); }
// Row of the sequence on lane r of query tile m, or -1 (an unused lane).
HSTU_HD int q_row(const SeqGeom& s, const QLayout& L, int m, int r) {
  if (L.ctx_lane0 >= 0) {
    if (m == L.nq - 1 && r >= L.ctx_lane0) {
      const int cr = r - L.ctx_lane0;
      return cr < s.c ? cr : -1;
    }
    if (m == 0 && r < s.c) return -1;   // moved to the last tile
  }
  const int v = m * kBlockM + r;
  return v < s.Lq ? v : -1;
}
// The rows of query tile m as up to two runs: [a0, a1) on lanes a0 - 128 m ..,
// and the moved context rows [c0, c1) (empty unless m is the last tile).
HSTU_HD void q_tile_runs(const SeqGeom& s, const QLayout& L, int m, int& a0, int& a1, int& c0, int& c1) {
  a0 = m * kBlockM;
  a1 = a0 + kBlockM < s.Lq ? a0 + kBlockM : s.Lq;
  c0 = c1 = 0;
  if (L.ctx_lane0 >= 0) {
    if (m == 0) a0 = s.c;
    if (m == L.nq - 1) c1 = s.c;
  }
}
// tile_uih_bounds over all rows of query tile m.
HSTU_HD TileBounds q_tile_bounds(const SeqGeom& s, const QLayout& L, int m) {
  int a0, a1, c0, c1;
  q_tile_runs(s, L, m, a0, a1, c0, c1);
  TileBounds b = tile_uih_bounds(s, a0, a1);
  if (c1 > c0) b = merge_bounds(b, tile_uih_bounds(s, c0, c1));
  return b;
}

// Key tiles (of kBlockN keys) a query tile touches, as up to three sorted,
// disjoint tile-index ranges: the context keys, the UIH hull, the target
// diagonal.  Empty slots hold [kNoTile, kNoTile).  Written with fixed slots and
// a compare-swap network (no runtime array indexing) so it stays in registers.
constexpr int kNoTile = 0x3fffffff;
struct TileSet {
  int lo0, hi0, lo1, hi1, lo2, hi2;
  int count;   // number of tiles
};

HSTU_HD void tile_range_swap_if(int& alo, int& ahi, int& blo, int& bhi) {
  if (blo < alo) {
    const int tl = alo, th = ahi;
    alo = blo; ahi = bhi;
    blo = tl; bhi = th;
  }
}

// b: q_tile_bounds(s, L, m), when the caller has it already.
HSTU_HD TileSet query_tile_kv_tiles(const SeqGeom& s, const QLayout& L, int m, const TileBounds& b) {
  int i0, i1, c0, c1;   // [i0, i1): the run that may hold target rows
  q_tile_runs(s, L, m, i0, i1, c0, c1);
  TileSet t;
  t.lo0 = t.hi0 = t.lo1 = t.hi1 = t.lo2 = t.hi2 = kNoTile;
  if (s.c > 0 && (i1 > i0 || c1 > c0)) {
    t.lo0 = 0;
    t.hi0 = (s.c + kBlockN - 1) / kBlockN;
  }
  if (b.HI > b.LO) {
    t.lo1 = b.LO / kBlockN;
    t.hi1 = (b.HI + kBlockN - 1) / kBlockN;
  }
  if (s.tkv) {   // the target rows' own keys
    const int d0 = i0 > s.c + s.u ? i0 : s.c + s.u;
    const int sh = s.ukv - s.u;
    if (i1 > d0) {
      t.lo2 = (d0 + sh) / kBlockN;
      t.hi2 = (i1 + sh + kBlockN - 1) / kBlockN;
    }
  }
  // sort the three slots by start (empty slots sort last)
  tile_range_swap_if(t.lo0, t.hi0, t.lo1, t.hi1);
  tile_range_swap_if(t.lo1, t.hi1, t.lo2, t.hi2);
  tile_range_swap_if(t.lo0, t.hi0, t.lo1, t.hi1);
  // merge overlapping or adjacent ranges into the earlier slot
  if (t.lo1 != kNoTile && t.lo1 <= t.hi0) {
    t.hi0 = t.hi1 > t.hi0 ? t.hi1 : t.hi0;
    t.lo1 = t.lo2; t.hi1 = t.hi2;
    t.lo2 = t.hi2 = kNoTile;
  }
  if (t.lo2 != kNoTile) {
    if (t.lo2 <= t.hi1) {
      t.hi1 = t.hi2 > t.hi1 ? t.hi2 : t.hi1;
      t.lo2 = t.hi2 = kNoTile;
    }
  }
  if (t.lo1 != kNoTile && t.lo1 <= t.hi0) {
    t.hi0 = t.hi1 > t.hi0 ? t.hi1 : t.hi0;
    t.lo1 = t.lo2; t.hi1 = t.hi2;
    t.lo2 = t.hi2 = kNoTile;
  }
  t.count = (t.hi0 - t.lo0) + (t.hi1 - t.lo1) + (t.hi2 - t.lo2);
  return t;
}
HSTU_HD TileSet query_tile_kv_tiles(const SeqGeom& s, const QLayout& L, int m) {
  return query_tile_kv_tiles(s, L, m, q_tile_bounds(s, L, m));
}

// The k-th tile (0-based) of a tile set.
HSTU_HD int tileset_at(const TileSet& ts, int k) {
  const int n0 = ts.hi0 - ts.lo0;
  if (k < n0) return ts.lo0 + k;
  k -= n0;
  const int n1 = ts.hi1 - ts.lo1;
  if (k < n1) return ts.lo1 + k;
  return ts.lo2 + (k - n1);
}

// Tiles [k0, k1) of the set belong to split `sp` of `splits`.
HSTU_HD void split_range(int count, int sp, int splits, int& k0, int& k1) {
  k0 = static_cast<int>((static_cast<long long>(count) * sp) / splits);
  k1 = static_cast<int>((static_cast<long long>(count) * (sp + 1)) / splits);
}

// True when every valid row of query tile m sees every key of key tile n, so
// the per-element predicate can be skipped.  Conservative: may say false for a
// tile that happens to be fully allowed, never true for one that is not.
// `b` is tile_uih_bounds of the query tile.
HSTU_HD bool tile_fully_allowed(const SeqGeom& s, const TileBounds& b, int n) {
  const int j0 = n * kBlockN, j1 = j0 + kBlockN;
  if (j1 > s.Lkv) return false;
  if (j1 <= s.c) return true;
  if (j1 > s.c + s.ukv) return false;   // holds target keys
  const int jlo = j0 > s.c ? j0 : s.c;
  return b.maxLO <= jlo && b.minHI >= j1;
}


// tile_fully_allowed(s, b, n) as index ranges: true exactly when n < ctx_hi
// (key tiles inside the context prefix) or lo <= n < hi (UIH tiles every row
// of the query tile sees in full).
struct FullTiles {
  int ctx_hi, lo, hi;
};
HSTU_HD FullTiles full_tile_ranges(const SeqGeom& s, const TileBounds& b) {
  FullTiles f;
  f.ctx_hi = (s.c < s.Lkv ? s.c : s.Lkv) / kBlockN;
  int e = s.Lkv;
  if (s.c + s.ukv < e) e = s.c + s.ukv;
  if (b.minHI < e) e = b.minHI;
  f.hi = e > 0 ? e / kBlockN : 0;
  f.lo = s.c >= b.maxLO ? 0 : (b.maxLO + kBlockN - 1) / kBlockN;
  return f;
}

// Launch parameters of the persistent forward kernel.
struct FwdParams {
  void* o;                 // [total_q, o_stride] outputs (fp16/bf16)
  float* lse;              // [nhead, total_q] or null
  float* o_part;           // split partials [splits, total_q, nhead, hdim_v] fp32
  float* ml_part;          // split row stats [splits, nhead, total_q, 2] fp32
  const int* off_q;
  const int* off_kv;       // == off_q for self-attention
  const int* targets;      // null = no targets
  const int4* units;       // work units {b, m, h, split}
  int* ws_header;          // workspace header (kWs*)
  const float* group_scale;  // resolved attn_scale per group
  long long o_stride;      // elements between consecutive output tokens
  int total_q;
  int batch, nhead, num_groups, batch_per_group;
  int causal, self_attn, kv_targets, splits;
  float alpha;             // resolved QK scale
  // relative attention bias (the kernels built with it only): per-token
  // timestamps (seconds; ts_kv == ts_q for self-attention; null = no temporal
  // term), per-head tables [nhead, 11] and [nhead, rab_np] (null = zero term)
  const long long* ts_q;
  const long long* ts_kv;
  const float* rab_time;
  const float* rab_pos;
  int rab_np;
  // in-kernel scheduling (fused != 0, batch <= kFusedMaxBatch): every CTA
  // validates the offsets and orders the units itself; units and
  // group_scale above are then unused
  int fused;
  int total_kv, max_seqlen_q, max_seqlen_kv;
  int ctx[kMaxGroups], loc[kMaxGroups], mf[kMaxGroups];
  int max_uih[kMaxGroups];        // per-group override of the attn_scale default (0 = automatic)
  float attn_scale[kMaxGroups];   // per-group attn_scale (0 = 1 / max UIH length of the group)
};

// Per query tile, for the backward's key-tile units: its TileSet (6 range ends
// and the count) and TileBounds (4), padded to 12 ints.
constexpr int kQTileInts = 12;

// Launch parameters of the scheduler (prep) kernel.
struct PrepParams {
  const int* off_q;
  const int* off_kv;
  const int* targets;
  int4* units;
  int* ws_header;
  float* group_scale;
  int* batch_scratch;      // [5 * batch + 3] ints (used when batch is large)
  // backward scheduling (null for the forward): the first query tile of each
  // sequence [batch + 1], every query tile's key-tile set and bounds
  // [query tiles][kQTileInts], and the key-tile units {b, n, h, 0}
  int* qtile_base;
  int* qtiles;
  int4* kv_units;
  int max_kv_units;
  unsigned* kv_mask;       // member query tiles of every (sequence, key tile), as bit words
  int* kv_mask_base;       // [batch + 1] first word of each sequence
  int max_mask_words;
  int batch, nhead, num_groups, batch_per_group, splits;
  int total_q, total_kv, max_seqlen_q, max_seqlen_kv, max_units;
  int causal, self_attn, kv_targets;
  int ctx[kMaxGroups], loc[kMaxGroups], mf[kMaxGroups], max_uih[kMaxGroups];
  float attn_scale[kMaxGroups];
};

// Backward kernel parameters (dQ and dK/dV kernels).
struct BwdParams {
  void* dq;                // [total_q, dq_stride] gradients (storage type)
  void* dk;                // [total_kv, dk_stride]
  void* dv;                // [total_kv, dv_stride]
  const float* lse;        // [nhead, total_q] natural-log LSE of the forward (softmax)
  const float* delta;      // [nhead, total_q] rowsum(dO . O) (softmax)
  const int* off_q;
  const int* off_kv;       // == off_q for self-attention
  const int* targets;
  const int4* units;       // dQ units {b, m, h, 0}
  const int4* kv_units;    // dK/dV units {b, n, h, 0}
  const int* qtile_base;   // [batch + 1] first query tile of each sequence
  const int* qtiles;       // [query tiles][kQTileInts]
  const unsigned* kv_mask;       // member query tiles per (sequence, key tile) as bit words
  const int* kv_mask_base;       // [batch + 1] first word of each sequence
  int* ws_header;
  const float* group_scale;
  long long dq_stride, dk_stride, dv_stride;
  int total_q, batch, nhead, batch_per_group, causal, self_attn, kv_targets;
  float alpha;
  // relative attention bias (the kernels built with it only), as in FwdParams
  const long long* ts_q;
  const long long* ts_kv;
  const float* rab_time;
  const float* rab_pos;
  int rab_np;
  // gradients of the bias tables, [nhead, 11] and [nhead, rab_np] (null = not
  // wanted); zeroed by the host, summed into by the dQ kernel
  float* d_rab_time;
  float* d_rab_pos;
  int ctx[kMaxGroups], loc[kMaxGroups], mf[kMaxGroups];
};

// Combine kernel parameters (split-KV).
// Split-KV combine kernel parameters.  The partials are already x attn_scale.
struct CombineParams {
  void* o;
  float* lse;
  const float* o_part;     // [splits, total_q, nhead, hdim_v]
  const float* ml_part;    // [splits, nhead, total_q, 2]: running max (log2 units), row sum
  const int* off_q;
  const int* ws_header;
  long long o_stride;
  int total_q, nhead, batch, splits;
};

// Fills the geometry of sequence b from the device/host offset arrays.
HSTU_HD SeqGeom make_geom(const int* off_q, const int* off_kv, const int* targets, int b,
                          int c, int W, int F, int causal, int self_attn, int kv_targets) {
  SeqGeom s;
  s.q0 = off_q[b];
  s.Lq = off_q[b + 1] - s.q0;
  s.kv0 = self_attn ? s.q0 : off_kv[b];
  s.Lkv = self_attn ? s.Lq : off_kv[b + 1] - s.kv0;
  const int t = targets ? targets[b] : 0;
  s.c = c;
  s.u = s.Lq - c - t;
  s.ukv = self_attn ? s.u : s.Lkv - c - (kv_targets ? t : 0);
  s.W = W;
  s.F = F;
  s.causal = causal;
  s.self_attn = self_attn;
  s.tkv = self_attn || kv_targets;
  return s;
}

}  // namespace hstu
