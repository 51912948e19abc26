// Scheduler (prep), header reset, pair-count, split-KV combine, softmax row-sum and self-test kernels.
//
// The scheduler runs as one CTA before the forward kernel, on the same stream
// (for batches above kFusedMaxBatch, for the stats call and for the backward;
// smaller forwards order their units inside the forward kernel, after a
// one-block kernel that zeroes the workspace header):
// it validates the jagged offsets, counts for every query tile the key tiles
// the functional mask does not fully exclude, orders the sequences longest
// first (most executed tiles first, so the persistent kernel's dynamic queue
// is a longest-processing-time schedule and a sequence's heads and query tiles
// run close together in time for L2 reuse of its K/V) and writes one work unit
// per (sequence, head, query tile, KV split).  It also resolves the per-group
// attn_scale default (composable_kernel 18_hstu_attention README, "Command-line
// arguments": attn_scale 0 means 1/max_seqlen, the maximum UIH length).
//
// The combine kernel merges split-KV partials ("Split-KV" section of the same
// README): SiLU partials add; softmax partials are weighted by their running
// maxima, divided by the merged row sum, and the LSE is written.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hstu_common.cuh"
#include "hstu_launch.h"
#include "ptx.cuh"

namespace hstu {

namespace {

constexpr int kPrepThreads = 1024;
constexpr int kSortMaxBatch = 2048;   // above this the sequences keep their input order
constexpr int kPrepSmemBatch = 2048;  // scratch arrays live in shared memory up to this batch

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Exclusive prefix sum of data[0, n) in place; data[n] receives the total.
// Every thread of the block must call it.
__device__ int block_exclusive_scan(int* data, int n, int* s_wsum) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
  const int per = (n + nth - 1) / nth;
  const int beg = min(tid * per, n), end = min(beg + per, n);
  int local = 0;
  for (int i = beg; i < end; ++i) local += data[i];
  const int incl = warp_incl_scan(local);
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < nwarps ? s_wsum[lane] : 0;
    v = warp_incl_scan(v);
    s_wsum[lane] = v;
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? s_wsum[warp - 1] : 0);
  for (int i = beg; i < end; ++i) {
    const int v = data[i];
    data[i] = run;
    run += v;
  }
  const int total = s_wsum[nwarps - 1];
  if (tid == 0) data[n] = total;
  __syncthreads();
  return total;
}

// Largest index k in [0, n) with a[k] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int find_segment(const int* a, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPrepThreads) hstu_prep_kernel(const __grid_constant__ PrepParams p) {
  extern __shared__ int dsm[];
  __shared__ int s_gmax[kMaxGroups];
  __shared__ int s_err;
  __shared__ unsigned long long s_tiles;
  __shared__ int s_wsum[32];
  ptx::grid_launch_dependents();   // the forward kernel may start its prologue now
  const int tid = threadIdx.x, nth = blockDim.x;
  const int B = p.batch;
  int* tbase = B <= kPrepSmemBatch ? dsm : p.batch_scratch;   // [B+1] query-tile offsets
  int* cost = tbase + (B + 1);                                 // [B] key tiles per sequence
  int* order = cost + B;                                       // [B] sequences, longest first
  int* ubase = order + B;                                      // [B+1] unit offsets by position
  int* kbase = ubase + (B + 1);                                // [B+1] key-tile unit offsets (backward)
  for (int g = tid; g < kMaxGroups; g += nth) s_gmax[g] = 0;
  if (tid == 0) {
    s_err = 0;
    s_tiles = 0ull;
  }
  __syncthreads();

  // 1. validate every sequence; query tiles per sequence
  for (int b = tid; b < B; b += nth) {
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
    if (err) atomicOr(&s_err, err);
    else atomicMax(&s_gmax[g], q1 - q0 - c - t);
    tbase[b] = err ? 0 : q_layout(q1 - q0, c).nq;
    cost[b] = 0;
  }
  __syncthreads();
  if (s_err != 0) {
    if (tid == 0) {
      p.ws_header[kWsError] = s_err;
      p.ws_header[kWsUnits] = 0;
      p.ws_header[kWsKvUnits] = 0;
      p.ws_header[kWsCounter] = 0;
      p.ws_header[kWsKvCounter] = 0;
      reinterpret_cast<long long*>(p.ws_header + kWsTilesLo)[0] = 0;
    }
    return;
  }
  const int n_items = block_exclusive_scan(tbase, B, s_wsum);

  // 2. key tiles of every (sequence, query tile)
  unsigned long long tiles = 0ull;
  for (int i = tid; i < n_items; i += nth) {
    const int b = find_segment(tbase, B, i);
    const int g = b / p.batch_per_group;
    const SeqGeom s = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[g], p.loc[g], p.mf[g], p.causal,
                                p.self_attn, p.kv_targets);
    const QLayout L = q_layout(s);
    const TileSet ts = query_tile_kv_tiles(s, L, i - tbase[b]);
    const int cnt = ts.count;
    if (p.qtiles) {
      const TileBounds tb = q_tile_bounds(s, L, i - tbase[b]);
      int* o = p.qtiles + static_cast<long long>(i) * kQTileInts;
      o[0] = ts.lo0; o[1] = ts.hi0; o[2] = ts.lo1; o[3] = ts.hi1; o[4] = ts.lo2; o[5] = ts.hi2;
      o[6] = ts.count;
      o[7] = tb.LO; o[8] = tb.HI; o[9] = tb.maxLO; o[10] = tb.minHI;
    }
    atomicAdd(&cost[b], cnt);
    tiles += cnt;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tiles += __shfl_down_sync(0xffffffffu, tiles, o);
  if ((tid & 31) == 0 && tiles) atomicAdd(&s_tiles, tiles * static_cast<unsigned long long>(p.nhead));
  __syncthreads();

  // 3. longest sequence first (stable rank sort on the executed-tile count)
  const bool sort = B <= kSortMaxBatch;
  for (int b = tid; b < B; b += nth) {
    int r = b;
    if (sort) {
      const int cb = cost[b];
      r = 0;
      for (int b2 = 0; b2 < B; ++b2) {
        const int c2 = cost[b2];
        r += (c2 > cb) | ((c2 == cb) & (b2 < b));
      }
    }
    order[r] = b;
  }
  __syncthreads();
  for (int pos = tid; pos < B; pos += nth) {
    const int b = order[pos];
    ubase[pos] = (tbase[b + 1] - tbase[b]) * p.nhead * p.splits;
  }
  __syncthreads();
  const int total = block_exclusive_scan(ubase, B, s_wsum);
  if (total > p.max_units) {
    if (tid == 0) {
      p.ws_header[kWsError] = kErrMaxSeqlen;
      p.ws_header[kWsUnits] = 0;
      p.ws_header[kWsKvUnits] = 0;
      p.ws_header[kWsCounter] = 0;
      p.ws_header[kWsKvCounter] = 0;
      reinterpret_cast<long long*>(p.ws_header + kWsTilesLo)[0] = 0;
    }
    return;
  }

  // 4. units: per sequence, heads outer, splits innermost, query tiles from
  //    the last down: the tiles holding context rows (which see every key)
  //    come last in the layout, and under a causal mask later tiles run more
  //    key tiles, so the queue ends on the smallest units.
  for (int u = tid; u < total; u += nth) {
    const int pos = find_segment(ubase, B, u);
    const int b = order[pos];
    const int nq = tbase[b + 1] - tbase[b];
    const int per_h = nq * p.splits;
    const int local = u - ubase[pos];
    const int h = local / per_h;
    const int rem = local - h * per_h;
    const int m = nq - 1 - rem / p.splits;
    p.units[u] = make_int4(b, m, h, rem % p.splits);
  }

  // 4b. backward: the query-tile base of each sequence, and key-tile units in
  //     the same sequence order, heads outer, key tiles from the first (seen
  //     by most query tiles under a causal mask) up
  int total_kv_units = 0;
  if (p.qtiles) {
    for (int b = tid; b <= B; b += nth) p.qtile_base[b] = tbase[b];
    for (int pos = tid; pos < B; pos += nth) {
      const int b = order[pos];
      const int k0 = p.self_attn ? p.off_q[b] : p.off_kv[b];
      const int k1 = p.self_attn ? p.off_q[b + 1] : p.off_kv[b + 1];
      kbase[pos] = ((k1 - k0 + kBlockN - 1) / kBlockN) * p.nhead;   // every key row gets its gradient
    }
    __syncthreads();
    total_kv_units = block_exclusive_scan(kbase, B, s_wsum);
    if (total_kv_units > p.max_kv_units) {
      if (tid == 0) {
        p.ws_header[kWsError] = kErrMaxSeqlen;
        p.ws_header[kWsUnits] = 0;
        p.ws_header[kWsKvUnits] = 0;
        p.ws_header[kWsCounter] = 0;
        p.ws_header[kWsKvCounter] = 0;
        reinterpret_cast<long long*>(p.ws_header + kWsTilesLo)[0] = 0;
      }
      return;
    }
    for (int u = tid; u < total_kv_units; u += nth) {
      const int pos = find_segment(kbase, B, u);
      const int b = order[pos];
      const int per_h = (kbase[pos + 1] - kbase[pos]) / p.nhead;
      const int local = u - kbase[pos];
      p.kv_units[u] = make_int4(b, local % per_h, local / per_h, 0);
    }
    // member masks: bit (m % 32) of word kv_mask_base[b] + n * words_b + m / 32
    // is set when query tile m of sequence b runs key tile n (words_b =
    // ceil(query tiles / 32)); the dK/dV kernel walks these words instead of
    // testing every query tile's record
    int* mb = p.kv_mask_base;
    for (int b = tid; b < B; b += nth) {
      const int k0 = p.self_attn ? p.off_q[b] : p.off_kv[b];
      const int k1 = p.self_attn ? p.off_q[b + 1] : p.off_kv[b + 1];
      mb[b] = ((k1 - k0 + kBlockN - 1) / kBlockN) * ((tbase[b + 1] - tbase[b] + 31) / 32);
    }
    __syncthreads();
    const int total_words = block_exclusive_scan(mb, B, s_wsum);
    if (total_words > p.max_mask_words) {
      if (tid == 0) {
        p.ws_header[kWsError] = kErrMaxSeqlen;
        p.ws_header[kWsUnits] = 0;
        p.ws_header[kWsKvUnits] = 0;
        p.ws_header[kWsCounter] = 0;
        p.ws_header[kWsKvCounter] = 0;
        reinterpret_cast<long long*>(p.ws_header + kWsTilesLo)[0] = 0;
      }
      return;
    }
    for (int i = tid; i < total_words; i += nth) p.kv_mask[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n_items; i += nth) {
      const int b = find_segment(tbase, B, i);
      const int m = i - tbase[b];
      const int words = (tbase[b + 1] - tbase[b] + 31) / 32;
      const int nk = words > 0 ? (mb[b + 1] - mb[b]) / words : 0;
      const int* r = p.qtiles + static_cast<long long>(i) * kQTileInts;
      unsigned* base = p.kv_mask + mb[b] + m / 32;
      const unsigned bit = 1u << (m & 31);
      for (int k = 0; k < 3; ++k) {
        const int lo = r[2 * k], hi = r[2 * k + 1] < nk ? r[2 * k + 1] : nk;
        for (int n = lo; n < hi; ++n) atomicOr(base + static_cast<long long>(n) * words, bit);
      }
    }
  }

  // 5. attn_scale per group: 0 means 1 / (max UIH length of the group)
  for (int g = tid; g < p.num_groups; g += nth) {
    float sc = p.attn_scale[g];
    if (sc == 0.f) {
      const int mu = p.max_uih[g] > 0 ? p.max_uih[g] : s_gmax[g];
      sc = mu > 0 ? 1.f / static_cast<float>(mu) : 1.f;
    }
    p.group_scale[g] = sc;
  }
  __syncthreads();
  if (tid == 0) {
    p.ws_header[kWsError] = 0;
    p.ws_header[kWsUnits] = total;
    p.ws_header[kWsKvUnits] = total_kv_units;
    p.ws_header[kWsCounter] = 0;
    p.ws_header[kWsKvCounter] = 0;
    reinterpret_cast<long long*>(p.ws_header + kWsTilesLo)[0] = static_cast<long long>(s_tiles);
  }
}

// Allowed (b, h, i, j) pairs: one CTA per sequence.
__global__ void __launch_bounds__(256) hstu_pairs_kernel(const __grid_constant__ PrepParams p) {
  const int b = blockIdx.x;
  const int g = b / p.batch_per_group;
  const SeqGeom s = make_geom(p.off_q, p.off_kv, p.targets, b, p.ctx[g], p.loc[g], p.mf[g], p.causal,
                              p.self_attn, p.kv_targets);
  long long sum = 0;
  for (int i = threadIdx.x; i < s.Lq; i += blockDim.x) sum += row_pair_count(s, i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_down_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0 && sum)
    atomicAdd(reinterpret_cast<unsigned long long*>(p.ws_header + kWsPairsLo),
              static_cast<unsigned long long>(sum) * p.nhead);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2c(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Groups of R (token row, head) pairs per warp iteration (R = 4; 2 for
// softmax and D = 256), lanes across the D columns (one float4 each, two for
// D = 256; coalesced rows), over a grid of three resident blocks per SM that
// strides through the groups.  Every load of an iteration (the statistics and the
// partials of two splits at a time) is issued before any is used, and
// validity is tested after the loads (all addresses stay inside the
// workspace), so an iteration waits for about one memory round trip per two
// splits.  Softmax: lane s holds split s's running max and row sum; the merged
// max, weights and row sum come from warp reductions.  Launched as a
// programmatic dependent of the forward kernel: it waits for the forward's
// completion before reading.  Rows outside every sequence and calls whose
// scheduler found a device error are left untouched.
constexpr int kCombineBlocksPerSm = 3;

template <int D, bool BF16, bool SOFTMAX>
__global__ void __launch_bounds__(256, kCombineBlocksPerSm) hstu_combine_kernel(const __grid_constant__ CombineParams p) {
  constexpr int NV4 = (D / 4 + 31) / 32;
  constexpr int R = (D > 128 || SOFTMAX) ? 2 : 4;   // pairs per warp iteration
  constexpr int SU = 2;                // splits per round of loads
  ptx::grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long npairs = static_cast<long long>(p.total_q) * p.nhead;
  const int units = p.ws_header[kWsUnits];
  const int row_lo = p.off_q[0], row_hi = p.off_q[p.batch];
  const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long g = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); g * R < npairs;
       g += nwarps) {
    const long long pair0 = g * R;
    long long row[R];
    int hh[R];
    bool live[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      live[r] = pair0 + r < npairs;
      const long long pr = live[r] ? pair0 + r : pair0;
      row[r] = pr / p.nhead;
      hh[r] = static_cast<int>(pr % p.nhead);
    }
    float wl[R], mul[R], lse[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wl[r] = 1.f;
      mul[r] = 1.f;
      lse[r] = 0.f;
    }
    if constexpr (SOFTMAX) {
      float m[R], l[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
        if (lane < p.splits) {
          const float2 ml = *reinterpret_cast<const float2*>(
              p.ml_part + ((static_cast<long long>(lane) * p.nhead + hh[r]) * p.total_q + row[r]) * 2);
          m[r] = ml.x;
          l[r] = ml.y;
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float M = m[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        wl[r] = m[r] == -INFINITY ? 0.f : exp2f(m[r] - M);
        float L = wl[r] * l[r];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        mul[r] = L > 0.f ? 1.f / L : 0.f;
        lse[r] = L > 0.f ? M * 0.6931471805599453f + logf(L) : -INFINITY;
      }
    }
    float4 acc[R][NV4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int k = 0; k < NV4; ++k) acc[r][k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < p.splits; s0 += SU) {
      float4 v[SU][R][NV4];
#pragma unroll
      for (int j = 0; j < SU; ++j)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4* src = reinterpret_cast<const float4*>(
              p.o_part + ((static_cast<long long>(s0 + j) * p.total_q + row[r]) * p.nhead + hh[r]) * D);
#pragma unroll
          for (int k = 0; k < NV4; ++k) {
            const int c4 = lane + 32 * k;
            v[j][r][k] = (s0 + j < p.splits && 4 * c4 < D) ? src[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
      for (int j = 0; j < SU; ++j)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float w = SOFTMAX ? __shfl_sync(0xffffffffu, wl[r], (s0 + j) & 31) : 1.f;
#pragma unroll
          for (int k = 0; k < NV4; ++k) {
            acc[r][k].x = fmaf(w, v[j][r][k].x, acc[r][k].x);
            acc[r][k].y = fmaf(w, v[j][r][k].y, acc[r][k].y);
            acc[r][k].z = fmaf(w, v[j][r][k].z, acc[r][k].z);
            acc[r][k].w = fmaf(w, v[j][r][k].w, acc[r][k].w);
          }
        }
    }
    if (units == 0) continue;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (!live[r] || row[r] < row_lo || row[r] >= row_hi) continue;
      uint16_t* dst = reinterpret_cast<uint16_t*>(p.o) + row[r] * p.o_stride + static_cast<long long>(hh[r]) * D;
#pragma unroll
      for (int k = 0; k < NV4; ++k) {
        const int c4 = lane + 32 * k;
        if (4 * c4 < D)
          *reinterpret_cast<uint2*>(dst + 4 * c4) =
              make_uint2(pack2c<BF16>(acc[r][k].x * mul[r], acc[r][k].y * mul[r]),
                         pack2c<BF16>(acc[r][k].z * mul[r], acc[r][k].w * mul[r]));
      }
      if (SOFTMAX && lane == 0 && p.lse != nullptr) p.lse[static_cast<long long>(hh[r]) * p.total_q + row[r]] = lse[r];
    }
  }
}

// Zeroes the forward's workspace header (work counter, error word, unit count)
// before a forward that schedules itself; the forward kernel, its programmatic
// dependent, starts as soon as this kernel has begun.
__global__ void __launch_bounds__(kWsHeaderInts) hstu_fwd_reset_kernel(int* ws_header) {
  ptx::grid_launch_dependents();
  ws_header[threadIdx.x] = 0;
}

// One thread waits on a barrier that nothing arrives on; the bounded wait must
// give up after timeout_ns and let the kernel finish.
__global__ void hstu_wait_selftest_kernel(int* result, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) *result = ptx::mbar_wait(&bar, 0, timeout_ns) ? 0 : 1;
}

// delta[h, i] = sum_e dO[i, h, e] O[i, h, e] (fp32), the row term of the
// softmax backward.  TPR threads per (row, head), 8 elements (16 bytes) each.
template <bool BF16, int TPR>
__global__ void __launch_bounds__(256) hstu_bwd_delta_kernel(const uint16_t* __restrict__ o, long long o_stride,
                                                             const uint16_t* __restrict__ d_o, long long do_stride,
                                                             float* __restrict__ delta, int total_q, int nhead,
                                                             int hdim_v) {
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long pair = gid / TPR;
  const int sub = static_cast<int>(gid % TPR);
  const bool live = pair < static_cast<long long>(total_q) * nhead;
  const int row = live ? static_cast<int>(pair / nhead) : 0;
  const int h = live ? static_cast<int>(pair % nhead) : 0;
  float acc = 0.f;
  if (live && sub * 8 < hdim_v) {
    const long long col = static_cast<long long>(h) * hdim_v + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * o_stride + col);
    const uint4 b = *reinterpret_cast<const uint4*>(d_o + row * do_stride + col);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float a0, a1, b0, b1;
      if constexpr (BF16) {
        a0 = __uint_as_float(av[k] << 16);
        a1 = __uint_as_float(av[k] & 0xFFFF0000u);
        b0 = __uint_as_float(bv[k] << 16);
        b1 = __uint_as_float(bv[k] & 0xFFFF0000u);
      } else {
        a0 = __half2float(__ushort_as_half(static_cast<unsigned short>(av[k] & 0xFFFFu)));
        a1 = __half2float(__ushort_as_half(static_cast<unsigned short>(av[k] >> 16)));
        b0 = __half2float(__ushort_as_half(static_cast<unsigned short>(bv[k] & 0xFFFFu)));
        b1 = __half2float(__ushort_as_half(static_cast<unsigned short>(bv[k] >> 16)));
      }
      acc = fmaf(a0, b0, acc);
      acc = fmaf(a1, b1, acc);
    }
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0) delta[static_cast<long long>(h) * total_q + row] = acc;
}

template <bool BF16, int TPR>
cudaError_t launch_delta_t(const void* o, long long o_stride, const void* d_o, long long do_stride, float* delta,
                           int total_q, int nhead, int hdim_v, cudaStream_t stream) {
  const long long threads = static_cast<long long>(total_q) * nhead * TPR;
  const long long blocks = (threads + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  hstu_bwd_delta_kernel<BF16, TPR><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(o), o_stride, static_cast<const uint16_t*>(d_o), do_stride, delta, total_q,
      nhead, hdim_v);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_delta(const void* o, long long o_stride, const void* d_o, long long do_stride, float* delta,
                             int total_q, int nhead, int hdim_v, bool bf16, cudaStream_t stream) {
  const int per = (hdim_v + 7) / 8;
  if (per <= 8) return bf16 ? launch_delta_t<true, 8>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream)
                            : launch_delta_t<false, 8>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream);
  if (per <= 16) return bf16 ? launch_delta_t<true, 16>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream)
                             : launch_delta_t<false, 16>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream);
  if (per <= 32) return bf16 ? launch_delta_t<true, 32>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream)
                             : launch_delta_t<false, 32>(o, o_stride, d_o, do_stride, delta, total_q, nhead, hdim_v, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_selftest(int* result, unsigned long long timeout_ns, cudaStream_t stream) {
  hstu_wait_selftest_kernel<<<1, 32, 0, stream>>>(result, timeout_ns);
  return cudaGetLastError();
}

template <int D, bool BF16, bool SOFTMAX>
cudaError_t launch_combine_t(const CombineParams& p, unsigned grid, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, hstu_combine_kernel<D, BF16, SOFTMAX>, p);
}

template <int D>
cudaError_t launch_combine_d(const CombineParams& p, bool bf16, bool softmax, unsigned grid, cudaStream_t stream) {
  if (bf16) return softmax ? launch_combine_t<D, true, true>(p, grid, stream)
                           : launch_combine_t<D, true, false>(p, grid, stream);
  return softmax ? launch_combine_t<D, false, true>(p, grid, stream) : launch_combine_t<D, false, false>(p, grid, stream);
}

cudaError_t launch_fwd_reset(int* ws_header, cudaStream_t stream) {
  hstu_fwd_reset_kernel<<<1, kWsHeaderInts, 0, stream>>>(ws_header);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream) {
  const size_t dsmem = p.batch <= kPrepSmemBatch ? (5 * static_cast<size_t>(p.batch) + 3) * sizeof(int) : 0;
  hstu_prep_kernel<<<1, kPrepThreads, dsmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_pairs(const PrepParams& p, cudaStream_t stream) {
  hstu_pairs_kernel<<<p.batch, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, int hdim, bool bf16, bool softmax, int sms, cudaStream_t stream) {
  const int per_warp = (hdim > 128 || softmax) ? 2 : 4;
  const long long warps = (static_cast<long long>(p.total_q) * p.nhead + per_warp - 1) / per_warp;
  long long blocks = (warps + 7) / 8;
  const long long resident = static_cast<long long>(kCombineBlocksPerSm) * (sms > 0 ? sms : 148);
  if (blocks > resident) blocks = resident;
  const unsigned grid = static_cast<unsigned>(blocks);
  if (grid == 0) return cudaSuccess;
  switch (hdim) {
    case 64: return launch_combine_d<64>(p, bf16, softmax, grid, stream);
    case 96: return launch_combine_d<96>(p, bf16, softmax, grid, stream);
    case 128: return launch_combine_d<128>(p, bf16, softmax, grid, stream);
    case 256: return launch_combine_d<256>(p, bf16, softmax, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
