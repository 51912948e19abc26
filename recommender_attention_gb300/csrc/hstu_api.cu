// C ABI of the HSTU forward and backward: argument validation, workspace
// planning, TMA tensor-map encoding and the launches (scheduler -> forward
// [-> split-KV combine]; scheduler -> row sums -> dQ -> dK/dV).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "hstu_attn.h"
#include "hstu_common.cuh"
#include "hstu_launch.h"
#include "hstu_rab.cuh"

// The ABI's bias limits size the kernels' shared-memory tables.
static_assert(HSTU_RAB_MAX_POS == hstu::kRabMaxPos, "positional table size differs from the ABI limit");
static_assert(HSTU_RAB_TIME_BUCKETS == hstu::kRabTimeBuckets, "time-bucket count differs from the ABI");

using namespace hstu;

namespace {

static_assert(HSTU_MAX_GROUPS == kMaxGroups, "group slots");
static_assert(HSTU_MAX_SPLITS == kMaxSplits, "split slots");

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// SM count of the current device, cached per device (devices 0..63); safe from
// several host threads (racing first calls store the same value).
int sm_count_current() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int64_t packed_or(int64_t stride, int64_t packed) { return stride == 0 ? packed : stride; }

hstu_status validate(const hstu_fwd_args* a) {
  if (!a) return HSTU_ERR_INVALID_ARG;
  if (a->dtype != HSTU_DTYPE_FP16 && a->dtype != HSTU_DTYPE_BF16) return HSTU_ERR_UNSUPPORTED;
  if (a->batch < 1 || a->nhead < 1 || a->total_q < 1 || a->total_kv < 1) return HSTU_ERR_INVALID_ARG;
  if (a->hdim_qk != 64 && a->hdim_qk != 96 && a->hdim_qk != 128 && a->hdim_qk != 256)
    return HSTU_ERR_UNSUPPORTED;
  if (a->hdim_v != a->hdim_qk && !(a->hdim_qk == 96 && a->hdim_v == 64)) return HSTU_ERR_UNSUPPORTED;
  if (a->num_groups < 1 || a->batch % a->num_groups != 0) return HSTU_ERR_INVALID_ARG;
  if (a->num_groups > kMaxGroups) return HSTU_ERR_UNSUPPORTED;
  if (a->num_splits < 0) return HSTU_ERR_INVALID_ARG;
  if (a->num_splits > kMaxSplits) return HSTU_ERR_UNSUPPORTED;
  if (a->max_seqlen_q < 0 || a->max_seqlen_kv < 0) return HSTU_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return HSTU_ERR_INVALID_ARG;
  if (a->softmax != 0 && a->softmax != 1) return HSTU_ERR_INVALID_ARG;
  if (!std::isfinite(a->alpha) || a->alpha < 0.f) return HSTU_ERR_INVALID_ARG;
  if (a->seq_offsets_kv == nullptr && a->total_kv != a->total_q) return HSTU_ERR_INVALID_ARG;
  if (a->kv_targets != 0 && a->kv_targets != 1) return HSTU_ERR_INVALID_ARG;
  if (a->cta_pairs < -1 || a->cta_pairs > 1) return HSTU_ERR_INVALID_ARG;
  if (a->kv_targets && a->seq_offsets_kv == nullptr) return HSTU_ERR_INVALID_ARG;
  if (a->rab_time != nullptr || a->rab_pos != nullptr) {
    if (a->rab_time != nullptr &&
        (a->timestamps_q == nullptr || (a->seq_offsets_kv != nullptr && a->timestamps_kv == nullptr)))
      return HSTU_ERR_INVALID_ARG;
    if (a->rab_pos != nullptr && (a->rab_pos_buckets < 1 || a->rab_pos_buckets > HSTU_RAB_MAX_POS))
      return HSTU_ERR_INVALID_ARG;
  }
  const int64_t wq = static_cast<int64_t>(a->nhead) * a->hdim_qk;
  const int64_t wv = static_cast<int64_t>(a->nhead) * a->hdim_v;
  const int64_t qs = packed_or(a->q_row_stride, wq), ks = packed_or(a->k_row_stride, wq);
  const int64_t vs = packed_or(a->v_row_stride, wv), os = packed_or(a->o_row_stride, wv);
  if (qs < wq || ks < wq || vs < wv || os < wv) return HSTU_ERR_INVALID_ARG;
  if ((qs * 2) % 16 || (ks * 2) % 16 || (vs * 2) % 16 || (os * 2) % 16) return HSTU_ERR_INVALID_ARG;
  for (int g = 0; g < a->num_groups; ++g) {
    if (a->local_len && a->local_len[g] < 0) return HSTU_ERR_INVALID_ARG;
    if (a->context_len && a->context_len[g] < 0) return HSTU_ERR_INVALID_ARG;
    if (a->minfull_len && a->minfull_len[g] < 0) return HSTU_ERR_INVALID_ARG;
    if (a->max_uih_len && a->max_uih_len[g] < 0) return HSTU_ERR_INVALID_ARG;
    if (a->attn_scale && !std::isfinite(a->attn_scale[g])) return HSTU_ERR_INVALID_ARG;
  }
  return HSTU_OK;
}

hstu_status validate_pointers(const hstu_fwd_args* a) {
  if (!a->q || !a->k || !a->v || !a->o || !a->seq_offsets_q) return HSTU_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(a->q) | reinterpret_cast<uintptr_t>(a->k) |
                        reinterpret_cast<uintptr_t>(a->v) | reinterpret_cast<uintptr_t>(a->o);
  if (mis & 15) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->timestamps_q) | reinterpret_cast<uintptr_t>(a->timestamps_kv)) & 7)
    return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->rab_time) | reinterpret_cast<uintptr_t>(a->rab_pos)) & 3)
    return HSTU_ERR_INVALID_ARG;
  if (a->workspace == nullptr || (reinterpret_cast<uintptr_t>(a->workspace) & 255))
    return HSTU_ERR_WORKSPACE;
  return HSTU_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int splits;
  int max_seq_q, max_seq_kv;
  int max_units;
  size_t off_scale, off_scratch, off_units, off_opart, off_mlpart, total;
};

int choose_splits(const hstu_fwd_args* a, int max_seq_q, int max_seq_kv, int sms) {
  if (a->num_splits > 0) return a->num_splits;
  const long long q_tiles = (max_seq_q + kBlockM - 1) / kBlockM;
  const long long units = static_cast<long long>(a->batch) * q_tiles * a->nhead;
  const int kv_tiles = (max_seq_kv + kBlockN - 1) / kBlockN;
  // about 8 units per SM: the splits of long key ranges balance the persistent
  // queue; each split keeps at least 12 key tiles, so the partials' extra
  // traffic (written, then merged by the combine kernel) stays small
  const long long target = 8LL * (sms > 0 ? sms : 148);
  if (units >= target || kv_tiles < 24) return 1;
  long long s = (target + units - 1) / units;
  if (s > kv_tiles / 12) s = kv_tiles / 12;
  if (s > kMaxSplits) s = kMaxSplits;
  return s < 1 ? 1 : static_cast<int>(s);
}

Plan make_plan(const hstu_fwd_args* a, int sms) {
  Plan pl{};
  pl.max_seq_q = a->max_seqlen_q > 0 ? a->max_seqlen_q : a->total_q;
  pl.max_seq_kv = a->max_seqlen_kv > 0 ? a->max_seqlen_kv : a->total_kv;
  pl.splits = choose_splits(a, pl.max_seq_q, pl.max_seq_kv, sms);
  // query tiles per sequence: ceil((L - c) / 128) main tiles plus at most
  // ceil(c / 128) <= ceil(L / 128) context tiles (see q_layout)
  const long long tiles_a = static_cast<long long>(a->batch) * (2 * ((pl.max_seq_q + kBlockM - 1) / kBlockM));
  const long long tiles_b = 2 * ((static_cast<long long>(a->total_q) + kBlockM - 1) / kBlockM) + 2LL * a->batch;
  const long long q_tiles = tiles_a < tiles_b ? tiles_a : tiles_b;
  long long units = q_tiles * a->nhead * pl.splits;
  if (units > (1LL << 30)) units = 1LL << 30;
  pl.max_units = static_cast<int>(units);
  size_t off = align256(kWsHeaderInts * sizeof(int));
  pl.off_scale = off;
  off = align256(off + kMaxGroups * sizeof(float));
  pl.off_scratch = off;
  off = align256(off + (5ull * a->batch + 3) * sizeof(int));
  pl.off_units = off;
  off = align256(off + static_cast<size_t>(pl.max_units) * sizeof(int4));
  pl.off_opart = pl.off_mlpart = 0;
  if (pl.splits > 1) {
    pl.off_opart = off;
    off = align256(off + static_cast<size_t>(pl.splits) * a->total_q * a->nhead * a->hdim_v * sizeof(float));
    pl.off_mlpart = off;
    off = align256(off + static_cast<size_t>(pl.splits) * a->nhead * a->total_q * 2 * sizeof(float));
  }
  pl.total = off;
  return pl;
}

bool encode_map(CUtensorMap* m, const void* base, bool bf16, int64_t inner, int64_t rows,
                int64_t row_stride_elems, uint32_t box_rows = kBlockN) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_elems * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void fill_group_params(const hstu_fwd_args* a, int* ctx, int* loc, int* mf) {
  for (int g = 0; g < kMaxGroups; ++g) {
    const bool in = g < a->num_groups;
    ctx[g] = (in && a->context_len) ? a->context_len[g] : 0;
    loc[g] = (in && a->local_len) ? a->local_len[g] : 0;
    mf[g] = (in && a->minfull_len) ? a->minfull_len[g] : 0;
  }
}

PrepParams make_prep(const hstu_fwd_args* a, const Plan& pl) {
  PrepParams pp;
  std::memset(&pp, 0, sizeof(pp));
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  pp.off_q = a->seq_offsets_q;
  pp.off_kv = a->seq_offsets_kv ? a->seq_offsets_kv : a->seq_offsets_q;
  pp.targets = a->num_targets;
  pp.units = reinterpret_cast<int4*>(ws + pl.off_units);
  pp.ws_header = reinterpret_cast<int*>(ws);
  pp.group_scale = reinterpret_cast<float*>(ws + pl.off_scale);
  pp.batch_scratch = reinterpret_cast<int*>(ws + pl.off_scratch);
  pp.batch = a->batch;
  pp.nhead = a->nhead;
  pp.num_groups = a->num_groups;
  pp.batch_per_group = a->batch / a->num_groups;
  pp.splits = pl.splits;
  pp.total_q = a->total_q;
  pp.total_kv = a->total_kv;
  pp.max_seqlen_q = pl.max_seq_q;
  pp.max_seqlen_kv = pl.max_seq_kv;
  pp.max_units = pl.max_units;
  pp.causal = a->causal;
  pp.self_attn = a->seq_offsets_kv == nullptr;
  pp.kv_targets = a->kv_targets;
  fill_group_params(a, pp.ctx, pp.loc, pp.mf);
  for (int g = 0; g < kMaxGroups; ++g) {
    const bool in = g < a->num_groups;
    pp.max_uih[g] = (in && a->max_uih_len) ? a->max_uih_len[g] : 0;
    pp.attn_scale[g] = (in && a->attn_scale) ? a->attn_scale[g] : 0.f;
  }
  return pp;
}

// ---------------------------------------------------------------- backward
// The forward's layout with one split (header, group scales, batch scratch,
// query-tile units), then the query-tile records, the key-tile units and, in
// softmax mode, the row sums delta [H, total_q].
struct BwdPlan {
  Plan fwd;
  int q_tiles, max_kv_units, max_mask_words;
  size_t off_qbase, off_qtiles, off_kvunits, off_maskbase, off_mask, off_delta, total;
};

hstu_fwd_args bwd_fwd_view(const hstu_bwd_args* a) {
  hstu_fwd_args f = a->fwd;
  f.num_splits = 1;
  return f;
}

hstu_status validate_bwd(const hstu_bwd_args* a) {
  if (!a) return HSTU_ERR_INVALID_ARG;
  const hstu_fwd_args f = bwd_fwd_view(a);
  const hstu_status st = validate(&f);
  if (st != HSTU_OK) return st;
  // hdim 64 and 128 (hdim_v equal), 96 with hdim_v 96 or 64; a bias only with 64 / 128 (validate)
  const bool pair_ok = (f.hdim_v == f.hdim_qk && (f.hdim_qk == 64 || f.hdim_qk == 96 || f.hdim_qk == 128)) ||
                       (f.hdim_qk == 96 && f.hdim_v == 64);
  if (!pair_ok) return HSTU_ERR_UNSUPPORTED;
  const int64_t w = static_cast<int64_t>(f.nhead) * f.hdim_qk;
  const int64_t wv = static_cast<int64_t>(f.nhead) * f.hdim_v;
  const int64_t sq[2] = {packed_or(a->dq_row_stride, w), packed_or(a->dk_row_stride, w)};
  const int64_t sv[2] = {packed_or(a->do_row_stride, wv), packed_or(a->dv_row_stride, wv)};
  for (int i = 0; i < 2; ++i) {
    if (sq[i] < w || (sq[i] * 2) % 16) return HSTU_ERR_INVALID_ARG;
    if (sv[i] < wv || (sv[i] * 2) % 16) return HSTU_ERR_INVALID_ARG;
  }
  return HSTU_OK;
}

BwdPlan make_bwd_plan(const hstu_bwd_args* a, int sms) {
  const hstu_fwd_args f = bwd_fwd_view(a);
  BwdPlan bp{};
  bp.fwd = make_plan(&f, sms);
  bp.q_tiles = bp.fwd.max_units / f.nhead;
  const long long kv_a = static_cast<long long>(f.batch) * ((bp.fwd.max_seq_kv + kBlockN - 1) / kBlockN);
  const long long kv_b = (static_cast<long long>(f.total_kv) + kBlockN - 1) / kBlockN + f.batch;
  long long kv_units = (kv_a < kv_b ? kv_a : kv_b) * f.nhead;
  if (kv_units > (1LL << 30)) kv_units = 1LL << 30;
  bp.max_kv_units = static_cast<int>(kv_units);
  size_t off = bp.fwd.total;
  bp.off_qbase = off;
  off = align256(off + (static_cast<size_t>(f.batch) + 1) * sizeof(int));
  bp.off_qtiles = off;
  off = align256(off + static_cast<size_t>(bp.q_tiles) * kQTileInts * sizeof(int));
  bp.off_kvunits = off;
  off = align256(off + static_cast<size_t>(bp.max_kv_units) * sizeof(int4));
  // member masks: (key tiles) x ceil(query tiles of the longest sequence / 32) words
  const long long words_per_tile = ((bp.fwd.max_seq_q + kBlockM - 1) / kBlockM + 31) / 32;
  long long mask_words = static_cast<long long>(bp.max_kv_units / f.nhead) * (words_per_tile > 0 ? words_per_tile : 1);
  if (mask_words > (1LL << 30)) mask_words = 1LL << 30;
  bp.max_mask_words = static_cast<int>(mask_words);
  bp.off_maskbase = off;
  off = align256(off + (static_cast<size_t>(f.batch) + 1) * sizeof(int));
  bp.off_mask = off;
  off = align256(off + static_cast<size_t>(bp.max_mask_words) * sizeof(unsigned));
  bp.off_delta = 0;
  if (f.softmax) {
    bp.off_delta = off;
    off = align256(off + static_cast<size_t>(f.nhead) * f.total_q * sizeof(float));
  }
  bp.total = off;
  return bp;
}

}  // namespace

extern "C" {

int32_t hstu_abi_version(void) { return HSTU_ABI_VERSION; }

const char* hstu_status_string(hstu_status s) {
  switch (s) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported configuration";
    case HSTU_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case HSTU_ERR_CUDA: return "CUDA error";
    case HSTU_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

int32_t hstu_device_sm_count(void) { return sm_count_current(); }

size_t hstu_fwd_args_size(void) { return sizeof(hstu_fwd_args); }

hstu_status hstu_selftest_wait_timeout(int32_t* result_dev, uint64_t timeout_ns, void* stream_ptr,
                                       int32_t* timed_out) {
  if (!result_dev || !timed_out) return HSTU_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (launch_wait_selftest(result_dev, timeout_ns, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (cudaMemcpy(timed_out, result_dev, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return HSTU_ERR_CUDA;
  return HSTU_OK;
}

hstu_status hstu_attn_fwd_workspace_size(const hstu_fwd_args* a, size_t* bytes) {
  if (!bytes) return HSTU_ERR_INVALID_ARG;
  const hstu_status st = validate(a);
  if (st != HSTU_OK) return st;
  *bytes = make_plan(a, sm_count_current()).total;
  return HSTU_OK;
}

hstu_status hstu_attn_fwd(const hstu_fwd_args* a, void* stream_ptr) {
  hstu_status st = validate(a);
  if (st != HSTU_OK) return st;
  st = validate_pointers(a);
  if (st != HSTU_OK) return st;
  const int sms = sm_count_current();
  if (sms <= 0) return HSTU_ERR_CUDA;
  const Plan pl = make_plan(a, sms);
  if (a->workspace_bytes < pl.total) return HSTU_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const bool bf16 = a->dtype == HSTU_DTYPE_BF16;
  const int D = a->hdim_qk;
  const int64_t wq = static_cast<int64_t>(a->nhead) * D;
  const int64_t wv = static_cast<int64_t>(a->nhead) * a->hdim_v;
  FwdMaps maps;
  if (!encode_map(&maps.q, a->q, bf16, wq, a->total_q, packed_or(a->q_row_stride, wq)) ||
      !encode_map(&maps.q8, a->q, bf16, wq, a->total_q, packed_or(a->q_row_stride, wq), 8) ||
      !encode_map(&maps.k, a->k, bf16, wq, a->total_kv, packed_or(a->k_row_stride, wq)) ||
      !encode_map(&maps.v, a->v, bf16, wv, a->total_kv, packed_or(a->v_row_stride, wv)) ||
      !encode_map(&maps.o, a->o, bf16, wv, a->total_q, packed_or(a->o_row_stride, wv), 32))
    return HSTU_ERR_CUDA;
  const bool rab = a->rab_time != nullptr || a->rab_pos != nullptr;
  const bool fused = a->batch <= kFusedMaxBatch;
  const bool sm = a->softmax != 0;
  // CTA pairs when asked for (hdim 128 without a bias, in-kernel schedule)
  int pair_clusters = 0;
  if (D == 128 && a->hdim_v == 128 && !rab && fused && a->cta_pairs > 0) {
    const int mc = fwd_pair_max_clusters_d128(bf16, sm);
    pair_clusters = mc < pl.max_units ? mc : pl.max_units;
    if (pair_clusters > 0 &&
        !encode_map(&maps.k64, a->k, bf16, wq, a->total_kv, packed_or(a->k_row_stride, wq), kBlockN / 2))
      return HSTU_ERR_CUDA;
  }

  const PrepParams pp = make_prep(a, pl);
  // Batches up to kFusedMaxBatch sequences are scheduled inside the forward
  // kernel, after a one-block reset of the header; larger ones by the
  // scheduler kernel.
  if ((fused ? launch_fwd_reset(pp.ws_header, stream) : launch_prep(pp, stream)) != cudaSuccess)
    return HSTU_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  FwdParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.o = a->o;
  fp.lse = a->softmax ? a->lse : nullptr;
  fp.o_part = pl.splits > 1 ? reinterpret_cast<float*>(ws + pl.off_opart) : nullptr;
  fp.ml_part = pl.splits > 1 ? reinterpret_cast<float*>(ws + pl.off_mlpart) : nullptr;
  fp.off_q = a->seq_offsets_q;
  fp.off_kv = a->seq_offsets_kv ? a->seq_offsets_kv : a->seq_offsets_q;
  fp.targets = a->num_targets;
  fp.units = pp.units;
  fp.ws_header = pp.ws_header;
  fp.group_scale = pp.group_scale;
  fp.o_stride = packed_or(a->o_row_stride, wv);
  fp.total_q = a->total_q;
  fp.batch = a->batch;
  fp.nhead = a->nhead;
  fp.num_groups = a->num_groups;
  fp.batch_per_group = a->batch / a->num_groups;
  fp.causal = a->causal;
  fp.self_attn = a->seq_offsets_kv == nullptr;
  fp.kv_targets = a->kv_targets;
  fp.splits = pl.splits;
  fp.alpha = a->alpha != 0.f ? a->alpha : 1.f / std::sqrt(static_cast<float>(a->hdim_qk));
  if (rab) {
    fp.ts_q = a->rab_time != nullptr ? reinterpret_cast<const long long*>(a->timestamps_q) : nullptr;
    fp.ts_kv = fp.ts_q == nullptr ? nullptr
               : reinterpret_cast<const long long*>(a->seq_offsets_kv ? a->timestamps_kv : a->timestamps_q);
    fp.rab_time = a->rab_time;
    fp.rab_pos = a->rab_pos;
    fp.rab_np = a->rab_pos != nullptr ? a->rab_pos_buckets : 1;
  }
  fill_group_params(a, fp.ctx, fp.loc, fp.mf);
  fp.fused = fused ? 1 : 0;
  fp.total_kv = a->total_kv;
  fp.max_seqlen_q = pl.max_seq_q;
  fp.max_seqlen_kv = pl.max_seq_kv;
  for (int g = 0; g < kMaxGroups; ++g) {
    fp.max_uih[g] = pp.max_uih[g];
    fp.attn_scale[g] = pp.attn_scale[g];
  }
  const int grid = pl.max_units < sms ? (pl.max_units > 0 ? pl.max_units : 1) : sms;
  if (a->event_fwd_begin &&
      cudaEventRecord(static_cast<cudaEvent_t>(a->event_fwd_begin), stream) != cudaSuccess)
    return HSTU_ERR_CUDA;
  cudaError_t e;
  if (pair_clusters > 0) e = launch_fwd_pair_d128(maps, fp, bf16, sm, pair_clusters, stream);
  else if (rab) e = D == 64  ? launch_fwd_rab_d64(maps, fp, bf16, sm, grid, stream)
                  : D == 96  ? launch_fwd_rab_d96(maps, fp, a->hdim_v, bf16, sm, grid, stream)
                  : D == 128 ? launch_fwd_rab_d128(maps, fp, bf16, sm, grid, stream)
                             : launch_fwd_rab_d256(maps, fp, bf16, sm, grid, stream);
  else if (D == 64) e = launch_fwd_d64(maps, fp, bf16, sm, grid, stream);
  else if (D == 96) e = launch_fwd_d96(maps, fp, a->hdim_v, bf16, sm, grid, stream);
  else if (D == 128) e = launch_fwd_d128(maps, fp, bf16, sm, grid, stream);
  else e = launch_fwd_d256(maps, fp, bf16, sm, grid, stream);
  if (e != cudaSuccess) return HSTU_ERR_CUDA;
  if (a->event_fwd_end &&
      cudaEventRecord(static_cast<cudaEvent_t>(a->event_fwd_end), stream) != cudaSuccess)
    return HSTU_ERR_CUDA;

  if (pl.splits > 1) {
    CombineParams cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.o = a->o;
    cp.lse = fp.lse;
    cp.o_part = fp.o_part;
    cp.ml_part = fp.ml_part;
    cp.off_q = a->seq_offsets_q;
    cp.ws_header = pp.ws_header;
    cp.o_stride = fp.o_stride;
    cp.total_q = a->total_q;
    cp.nhead = a->nhead;
    cp.batch = a->batch;
    cp.splits = pl.splits;
    if (launch_combine(cp, a->hdim_v, bf16, sm, sms, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  }

  return HSTU_OK;
}

hstu_status hstu_attn_fwd_check(const void* workspace, void* stream_ptr, int32_t* device_error) {
  if (!workspace) return HSTU_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return HSTU_ERR_CUDA;
  int32_t err = 0;
  if (cudaMemcpy(&err, static_cast<const int*>(workspace) + kWsError, sizeof(int32_t),
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (device_error) *device_error = err;
  return err ? HSTU_ERR_DEVICE : HSTU_OK;
}

hstu_status hstu_attn_fwd_stats(const hstu_fwd_args* a, void* stream_ptr, hstu_fwd_stats* out) {
  if (!out) return HSTU_ERR_INVALID_ARG;
  hstu_status st = validate(a);
  if (st != HSTU_OK) return st;
  if (!a->seq_offsets_q) return HSTU_ERR_INVALID_ARG;
  if (a->workspace == nullptr || (reinterpret_cast<uintptr_t>(a->workspace) & 255)) return HSTU_ERR_WORKSPACE;
  const int sms = sm_count_current();
  if (sms <= 0) return HSTU_ERR_CUDA;
  const Plan pl = make_plan(a, sms);
  if (a->workspace_bytes < pl.total) return HSTU_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const PrepParams pp = make_prep(a, pl);
  if (launch_prep(pp, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (cudaMemsetAsync(pp.ws_header + kWsPairsLo, 0, 2 * sizeof(int), stream) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (launch_pairs(pp, stream) != cudaSuccess) return HSTU_ERR_CUDA;
  int hdr[kWsHeaderInts];
  if (cudaStreamSynchronize(stream) != cudaSuccess) return HSTU_ERR_CUDA;
  if (cudaMemcpy(hdr, pp.ws_header, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return HSTU_ERR_CUDA;
  long long tiles, pairs;
  std::memcpy(&tiles, hdr + kWsTilesLo, sizeof(tiles));
  std::memcpy(&pairs, hdr + kWsPairsLo, sizeof(pairs));
  out->executed_tiles = tiles;
  out->allowed_pairs = pairs;
  out->work_units = hdr[kWsUnits];
  out->num_splits = pl.splits;
  out->device_error = hdr[kWsError];
  out->reserved = 0;
  return hdr[kWsError] ? HSTU_ERR_DEVICE : HSTU_OK;
}

size_t hstu_bwd_args_size(void) { return sizeof(hstu_bwd_args); }

hstu_status hstu_attn_bwd_workspace_size(const hstu_bwd_args* a, size_t* bytes) {
  if (!bytes) return HSTU_ERR_INVALID_ARG;
  const hstu_status st = validate_bwd(a);
  if (st != HSTU_OK) return st;
  *bytes = make_bwd_plan(a, sm_count_current()).total;
  return HSTU_OK;
}

hstu_status hstu_attn_bwd(const hstu_bwd_args* a, void* stream_ptr) {
  hstu_status st = validate_bwd(a);
  if (st != HSTU_OK) return st;
  const hstu_fwd_args f = bwd_fwd_view(a);
  if (!f.q || !f.k || !f.v || !f.seq_offsets_q || !a->d_o || !a->dq || !a->dk || !a->dv)
    return HSTU_ERR_INVALID_ARG;
  if (f.softmax && (!f.o || !f.lse)) return HSTU_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(f.q) | reinterpret_cast<uintptr_t>(f.k) |
                        reinterpret_cast<uintptr_t>(f.v) | reinterpret_cast<uintptr_t>(f.o) |
                        reinterpret_cast<uintptr_t>(a->d_o) | reinterpret_cast<uintptr_t>(a->dq) |
                        reinterpret_cast<uintptr_t>(a->dk) | reinterpret_cast<uintptr_t>(a->dv);
  if (mis & 15) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(f.timestamps_q) | reinterpret_cast<uintptr_t>(f.timestamps_kv)) & 7)
    return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(f.rab_time) | reinterpret_cast<uintptr_t>(f.rab_pos)) & 3)
    return HSTU_ERR_INVALID_ARG;
  // gradients of the bias tables: only of a table the call uses (the time table
  // needs its timestamps), 4-byte aligned
  if (a->d_rab_time != nullptr && (f.rab_time == nullptr || f.timestamps_q == nullptr)) return HSTU_ERR_INVALID_ARG;
  if (a->d_rab_pos != nullptr && f.rab_pos == nullptr) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->d_rab_time) | reinterpret_cast<uintptr_t>(a->d_rab_pos)) & 3)
    return HSTU_ERR_INVALID_ARG;
  if (f.workspace == nullptr || (reinterpret_cast<uintptr_t>(f.workspace) & 255)) return HSTU_ERR_WORKSPACE;
  const int sms = sm_count_current();
  if (sms <= 0) return HSTU_ERR_CUDA;
  const BwdPlan bp = make_bwd_plan(a, sms);
  if (f.workspace_bytes < bp.total) return HSTU_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const bool bf16 = f.dtype == HSTU_DTYPE_BF16;
  const int D = f.hdim_qk;
  const int64_t w = static_cast<int64_t>(f.nhead) * D;
  const int64_t wv = static_cast<int64_t>(f.nhead) * f.hdim_v;
  const int64_t do_stride = packed_or(a->do_row_stride, wv);
  BwdMaps maps;
  if (!encode_map(&maps.q, f.q, bf16, w, f.total_q, packed_or(f.q_row_stride, w)) ||
      !encode_map(&maps.q8, f.q, bf16, w, f.total_q, packed_or(f.q_row_stride, w), 8) ||
      !encode_map(&maps.k, f.k, bf16, w, f.total_kv, packed_or(f.k_row_stride, w)) ||
      !encode_map(&maps.v, f.v, bf16, wv, f.total_kv, packed_or(f.v_row_stride, wv)) ||
      !encode_map(&maps.d_o, a->d_o, bf16, wv, f.total_q, do_stride) ||
      !encode_map(&maps.d_o8, a->d_o, bf16, wv, f.total_q, do_stride, 8))
    return HSTU_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(f.workspace);
  PrepParams pp = make_prep(&f, bp.fwd);
  pp.qtile_base = reinterpret_cast<int*>(ws + bp.off_qbase);
  pp.qtiles = reinterpret_cast<int*>(ws + bp.off_qtiles);
  pp.kv_units = reinterpret_cast<int4*>(ws + bp.off_kvunits);
  pp.max_kv_units = bp.max_kv_units;
  pp.kv_mask = reinterpret_cast<unsigned*>(ws + bp.off_mask);
  pp.kv_mask_base = reinterpret_cast<int*>(ws + bp.off_maskbase);
  pp.max_mask_words = bp.max_mask_words;
  if (launch_prep(pp, stream) != cudaSuccess) return HSTU_ERR_CUDA;

  float* delta = f.softmax ? reinterpret_cast<float*>(ws + bp.off_delta) : nullptr;
  if (f.softmax && launch_bwd_delta(f.o, packed_or(f.o_row_stride, wv), a->d_o, do_stride, delta, f.total_q,
                                    f.nhead, f.hdim_v, bf16, stream) != cudaSuccess)
    return HSTU_ERR_CUDA;

  BwdParams bw;
  std::memset(&bw, 0, sizeof(bw));
  bw.dq = a->dq;
  bw.dk = a->dk;
  bw.dv = a->dv;
  bw.lse = f.softmax ? f.lse : nullptr;
  bw.delta = delta;
  bw.off_q = f.seq_offsets_q;
  bw.off_kv = f.seq_offsets_kv ? f.seq_offsets_kv : f.seq_offsets_q;
  bw.targets = f.num_targets;
  bw.units = pp.units;
  bw.kv_units = pp.kv_units;
  bw.qtile_base = pp.qtile_base;
  bw.qtiles = pp.qtiles;
  bw.kv_mask = pp.kv_mask;
  bw.kv_mask_base = pp.kv_mask_base;
  bw.ws_header = pp.ws_header;
  bw.group_scale = pp.group_scale;
  bw.dq_stride = packed_or(a->dq_row_stride, w);
  bw.dk_stride = packed_or(a->dk_row_stride, w);
  bw.dv_stride = packed_or(a->dv_row_stride, wv);
  bw.total_q = f.total_q;
  bw.batch = f.batch;
  bw.nhead = f.nhead;
  bw.batch_per_group = f.batch / f.num_groups;
  bw.causal = f.causal;
  bw.self_attn = f.seq_offsets_kv == nullptr;
  bw.kv_targets = f.kv_targets;
  bw.alpha = f.alpha != 0.f ? f.alpha : 1.f / std::sqrt(static_cast<float>(D));
  const bool rab = f.rab_time != nullptr || f.rab_pos != nullptr;
  if (rab) {
    bw.ts_q = f.rab_time != nullptr ? reinterpret_cast<const long long*>(f.timestamps_q) : nullptr;
    bw.ts_kv = bw.ts_q == nullptr ? nullptr
               : reinterpret_cast<const long long*>(f.seq_offsets_kv ? f.timestamps_kv : f.timestamps_q);
    bw.rab_time = f.rab_time;
    bw.rab_pos = f.rab_pos;
    bw.rab_np = f.rab_pos != nullptr ? f.rab_pos_buckets : 1;
    bw.d_rab_time = a->d_rab_time;
    bw.d_rab_pos = a->d_rab_pos;
    // the dQ kernel sums into them
    if (a->d_rab_time != nullptr &&
        cudaMemsetAsync(a->d_rab_time, 0, sizeof(float) * f.nhead * HSTU_RAB_TIME_BUCKETS, stream) != cudaSuccess)
      return HSTU_ERR_CUDA;
    if (a->d_rab_pos != nullptr &&
        cudaMemsetAsync(a->d_rab_pos, 0, sizeof(float) * f.nhead * f.rab_pos_buckets, stream) != cudaSuccess)
      return HSTU_ERR_CUDA;
  }
  fill_group_params(&f, bw.ctx, bw.loc, bw.mf);
  const int mu = bp.fwd.max_units, mk = bp.max_kv_units;
  const int grid_q = mu < sms ? (mu > 0 ? mu : 1) : sms;
  const int grid_kv = mk < sms ? (mk > 0 ? mk : 1) : sms;
  cudaError_t e;
  if (rab) e = D == 64 ? launch_bwd_rab_d64(maps, bw, bf16, f.softmax != 0, grid_q, grid_kv, stream)
               : D == 96 ? launch_bwd_rab_d96(maps, bw, f.hdim_v, bf16, f.softmax != 0, grid_q, grid_kv, stream)
                         : launch_bwd_rab_d128(maps, bw, bf16, f.softmax != 0, grid_q, grid_kv, stream);
  else if (D == 64) e = launch_bwd_d64(maps, bw, bf16, f.softmax != 0, grid_q, grid_kv, stream);
  else if (D == 96) e = launch_bwd_d96(maps, bw, f.hdim_v, bf16, f.softmax != 0, grid_q, grid_kv, stream);
  else e = launch_bwd_d128(maps, bw, bf16, f.softmax != 0, grid_q, grid_kv, stream);
  return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

}  // extern "C"
