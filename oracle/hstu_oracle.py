"""fp64 CPU oracle for the HSTU attention forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm use it.  It shares no code with the CUDA path.

What it computes (composable_kernel ``18_hstu_attention`` README, section
"Forward computation"; same operator in the older README's "HSTU-attention
operator" description), for every batch b, head h, query row i, key row j:

    s[i, j]  = alpha * <q[i, h, :], k[j, h, :]>                 (QK projection)
    masked s is set to zero                                      (Functional masking)
    SiLU:    p = SiLU(s) on allowed entries, 0 elsewhere
             o[i, h, :] = attn_scale * sum_j p[i, j] * v[j, h, :]
    softmax: p = attn_scale * softmax(s) over the allowed j only
             lse[h, i] = log(sum_{allowed j} exp(s[i, j]))        ("LSE saved")

in float64 from the already-rounded fp16/bf16 inputs, with the dense mask
materialised per sequence.  The mask follows the README's "Masking" table and
its physical-length formulas; where the text is silent the readings below are
used (each one a named constant or a commented branch):

  * ctx keys (j < c) are visible to every query ("always visible to all
    queries").
  * target keys are visible only to the target row itself (targets are
    "excluded from attending": read as "not attended by other rows"; the
    M-FALCON description in "From transformer parallelism to HSTU", section
    5.3, has candidates that do not attend to one another).
  * ctx query rows see ctx keys and every UIH key (the causal and local
    components are defined on UIH positions only).
  * UIH and target rows: UIH coordinates x_i = (i - c) + (u_kv - u) for a UIH
    row (bottom-right alignment for cross-attention), x_i = u_kv for a target
    row; key coordinate x_j = j - c; d = x_i - x_j.  Causal removes d < 0.  A
    row is "min-full" when F > 0 and x_i >= u_kv - F; a row that is not
    min-full and has W > 0 keeps only |d| <= W (WINDOW_KEEPS_DISTANCE_EQUAL_W).
  * M-FALCON ("From transformer parallelism to HSTU", section 5.3): a
    microbatch of candidates attends to the cached keys/values of the user's
    history, candidates never to each other.  As a cross-attention call whose
    key sequence is [context | history | the candidates' own keys] and whose
    query sequence is [context | the candidates] (targets on both sides,
    ``kv_targets``), candidate r sees exactly what it sees as a target row of
    the self-attention over [context | history | candidates]: the context
    keys, the history under the usual rules, and its own key.
  * softmax mode excludes masked entries (weight 0) rather than giving them
    exp(0); a row with no allowed key has o = 0 and lse = -inf.
  * alpha = 0 means 1/sqrt(hdim_qk); attn_scale = 0 means 1/max_uih where
    max_uih is the override when positive, else the largest Q UIH length of
    the batch's group; a group whose largest UIH length is 0 uses 1.0.
  * groups are consecutive blocks of batch/num_groups batches.

Relative attention bias ("From transformer parallelism to HSTU", sections
2.4 and 3.5; the rab term of the HSTU layer's spatial aggregation), when the
parameters carry one: s[i, j] gains, before the nonlinearity and the mask,

    rab[i, j] = rab_time[h, bucket(|ts_i - ts_j|)] + rab_pos[h, min(|pos_i - j|, P - 1)]

with the section 3.5 bucket edges (seconds) 0, 1, 5, 30, 60, 300, 1800, 3600,
86400, 604800, 2.6e6 (bucket k holds [edge_k, edge_k+1), bucket 10 everything
from 2.6e6 up), one learned scalar per head and bucket.  The pages name a
positional half without defining it; the reading here is one scalar per head
and clamped distance, pos_i being query row i's position in key coordinates
(i for a context row, i + (u_kv - u) otherwise: the mask's bottom-right
alignment, and a target row's own key at distance 0).

The backward (``hstu_attention_backward``) is the exact gradient of that
forward (the README's training mode keeps the softmax LSE for it); it is
pinned against central finite differences of the forward.

Parity of every function here is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

# Reading of "attend only to the N most recent keys": a key at UIH distance
# d = x_i - x_j is kept when d <= N (the row itself plus N earlier keys).
WINDOW_KEEPS_DISTANCE_EQUAL_W = True


# ----------------------------------------------------------------------------
# Physical lengths ("Masking": phy_seqlen formulas)
# ----------------------------------------------------------------------------
def phy_seqlen_q(uih_seqlen: int, num_targets: int, context_len: int) -> int:
    """phy_seqlen_q = uih_seqlen + num_targets + context_len."""
    return uih_seqlen + num_targets + context_len


def phy_seqlen_kv(uih_seqlen_kv: int, num_targets: int, context_len: int, cross: bool,
                  kv_targets: bool = False) -> int:
    """Self-attention: uih + targets + context; cross-attention: uih_kv + context,
    plus the targets' own keys when the key sequence carries them (M-FALCON)."""
    if cross and not kv_targets:
        return uih_seqlen_kv + context_len
    return uih_seqlen_kv + num_targets + context_len


def group_of_batch(b: int, batch: int, num_groups: int) -> int:
    """Group HSTU: batch must be a multiple of G; groups are consecutive blocks
    of batch/G batches (the README's 18-batch, 3-group example is only
    consistent with this)."""
    if num_groups < 1 or batch % num_groups != 0:
        raise ValueError("batch must be a multiple of num_groups")
    return b // (batch // num_groups)


# ----------------------------------------------------------------------------
# Mask ("Masking" table)
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class SeqMaskParams:
    """Mask parameters of one sequence (already resolved for its group)."""

    L_q: int          # physical query length  c + u + t
    L_kv: int         # physical key length     c + u + t (self), c + u_kv (cross),
                      # c + u_kv + t (cross with the targets' own keys)
    context: int      # c
    targets: int      # t
    causal: bool
    local: int        # W, 0 = no local window
    minfull: int      # F, 0 = no min-full tail
    cross: bool
    kv_targets: bool = False   # cross-attention key sequence ends with the t targets' keys

    @property
    def uih_q(self) -> int:
        return self.L_q - self.context - self.targets

    @property
    def uih_kv(self) -> int:
        if not self.cross:
            return self.uih_q
        return self.L_kv - self.context - (self.targets if self.kv_targets else 0)


def mask_rows(p: SeqMaskParams, rows: np.ndarray) -> np.ndarray:
    """Boolean allowed[r, j] for the query rows ``rows`` and every key j < L_kv.

    The rules are taken in order; the first rule that speaks for (i, j) decides.
    """
    c, u, u_kv = p.context, p.uih_q, p.uih_kv
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(p.L_kv, dtype=np.int64)[None, :]
    shape = (i.shape[0], j.shape[1])
    allowed = np.zeros(shape, dtype=bool)
    decided = np.zeros(shape, dtype=bool)

    # 1. contextual key: visible to every query.
    rule = np.broadcast_to(j < c, shape)
    allowed |= rule & ~decided
    decided |= rule

    # 2. target key (self-attention, or cross-attention carrying the targets'
    #    keys): visible to its own row only.  Target r sits at query row c+u+r
    #    and key row c+u_kv+r, so "own" means j - u_kv == i - u.
    rule = np.broadcast_to(j >= c + u_kv, shape)
    allowed |= rule & ~decided & (j - u_kv == i - u)
    decided |= rule

    # 3. contextual query with a UIH key: no causal/local rule applies to it.
    rule = np.broadcast_to(i < c, shape)
    allowed |= rule & ~decided
    decided |= rule

    # 4. UIH or target query with a UIH key.
    x_i = np.where(i < c + u, (i - c) + (u_kv - u), u_kv)
    x_j = j - c
    d = x_i - x_j
    ok = np.ones(shape, dtype=bool)
    if p.causal:
        ok &= d >= 0
    if p.local > 0:
        full = (p.minfull > 0) & (x_i >= u_kv - p.minfull)
        if WINDOW_KEEPS_DISTANCE_EQUAL_W:
            in_window = np.abs(d) <= p.local
        else:
            in_window = np.abs(d) < p.local
        ok &= full | in_window
    allowed |= ok & ~decided
    return allowed


def dense_mask(p: SeqMaskParams) -> np.ndarray:
    """The materialised [L_q, L_kv] mask of one sequence."""
    return mask_rows(p, np.arange(p.L_q))


# ----------------------------------------------------------------------------
# Non-linearities ("Forward computation": Non-linearity)
# ----------------------------------------------------------------------------
def silu(s: np.ndarray) -> np.ndarray:
    """SiLU(s) = s * sigmoid(s) = s / (1 + exp(-s)), elementwise, fp64."""
    with np.errstate(over="ignore"):
        return s / (1.0 + np.exp(-s))


# ----------------------------------------------------------------------------
# Relative attention bias ("From transformer parallelism to HSTU", section 3.5)
# ----------------------------------------------------------------------------
# Lower edges of the time-gap buckets, in seconds (the section's table).
TIME_BUCKET_EDGES = (0.0, 1.0, 5.0, 30.0, 60.0, 300.0, 1800.0, 3600.0, 86400.0, 604800.0, 2.6e6)


def time_gap_bucket(gap) -> np.ndarray:
    """Bucket of a time gap >= 0 (seconds): the largest k with gap >= edge_k."""
    gap = np.asarray(gap, dtype=np.float64)
    return np.searchsorted(np.asarray(TIME_BUCKET_EDGES), gap, side="right") - 1


def query_key_positions(p: "SeqMaskParams", rows: np.ndarray) -> np.ndarray:
    """Position of each query row in key coordinates: a context row keeps its
    index; UIH and target rows shift by u_kv - u (bottom-right alignment)."""
    rows = np.asarray(rows, dtype=np.int64)
    return np.where(rows < p.context, rows, rows + (p.uih_kv - p.uih_q))


def rab_indices(p: "SeqMaskParams", rows, ts_q, ts_kv, n_pos: int):
    """For the given query rows of one sequence: the time-gap bucket of every
    (row, key) pair (None when ts_q is None) and the clamped distance
    min(|pos_i - j|, n_pos - 1) (None when n_pos is 0)."""
    rows = np.asarray(rows, dtype=np.int64)
    bucket = dist = None
    if ts_q is not None:
        gap = np.abs(np.asarray(ts_q, dtype=np.float64)[rows][:, None] -
                     np.asarray(ts_kv, dtype=np.float64)[None, :])
        bucket = time_gap_bucket(gap)
    if n_pos > 0:
        d = np.abs(query_key_positions(p, rows)[:, None] - np.arange(p.L_kv)[None, :])
        dist = np.minimum(d, n_pos - 1)
    return bucket, dist


def rab_rows(p: "SeqMaskParams", rows, h: int, ts_q, ts_kv, rab_time, rab_pos) -> np.ndarray:
    """rab[i, j] for the given query rows of one sequence and head; ts_q / ts_kv
    are the sequence's timestamps (None: no temporal term)."""
    rows = np.asarray(rows, dtype=np.int64)
    bias = np.zeros((rows.shape[0], p.L_kv), dtype=np.float64)
    n_pos = 0 if rab_pos is None else np.asarray(rab_pos).shape[1]
    bucket, dist = rab_indices(p, rows, ts_q if rab_time is not None else None, ts_kv, n_pos)
    if bucket is not None:
        bias += np.asarray(rab_time, dtype=np.float64)[h][bucket]
    if dist is not None:
        bias += np.asarray(rab_pos, dtype=np.float64)[h][dist]
    return bias


def _head_forward(q, k, v, allowed, alpha, attn_scale, softmax, bias=None):
    """One (sequence, head): q [n, Dqk], k [L_kv, Dqk], v [L_kv, Dv], allowed [n, L_kv],
    bias [n, L_kv] (relative attention bias) or None."""
    s = alpha * (q @ k.T)
    if bias is not None:
        s = s + bias
    if not softmax:
        p = np.where(allowed, silu(s), 0.0)
        return attn_scale * (p @ v), None
    masked = np.where(allowed, s, -np.inf)
    m = masked.max(axis=1) if masked.shape[1] else np.full(masked.shape[0], -np.inf)
    has_key = np.isfinite(m)
    m_safe = np.where(has_key, m, 0.0)
    e = np.where(allowed, np.exp(s - m_safe[:, None]), 0.0)
    l = e.sum(axis=1)
    l_safe = np.where(has_key, l, 1.0)
    o = attn_scale * (e @ v) / l_safe[:, None]
    o[~has_key] = 0.0
    lse = np.where(has_key, m_safe + np.log(l_safe), -np.inf)
    return o, lse


# ----------------------------------------------------------------------------
# Whole forward
# ----------------------------------------------------------------------------
@dataclass
class HstuParams:
    """Host-side description of one forward call (arrays are per group)."""

    num_groups: int = 1
    context_len: Sequence[int] = (0,)
    local_len: Sequence[int] = (0,)
    minfull_len: Sequence[int] = (0,)
    max_uih_len: Sequence[int] = (0,)      # 0 = take the largest Q UIH length of the group
    attn_scale: Sequence[float] = (0.0,)   # 0 = 1/max_uih of the group
    alpha: float = 0.0                     # 0 = 1/sqrt(hdim_qk)
    causal: bool = True
    softmax: bool = False
    kv_targets: bool = False               # cross-attention keys end with the targets' own keys
    # relative attention bias (None: none): per-token timestamps in seconds
    # ([total_q]; [total_kv] for cross-attention), rab_time [H, 11], rab_pos [H, P]
    timestamps_q: Optional[np.ndarray] = None
    timestamps_kv: Optional[np.ndarray] = None
    rab_time: Optional[np.ndarray] = None
    rab_pos: Optional[np.ndarray] = None

    @property
    def has_rab(self) -> bool:
        return (self.rab_time is not None and self.timestamps_q is not None) or self.rab_pos is not None


def _seq_bias(params: HstuParams, sp, q0: int, kv0: int, h: int, rows) -> Optional[np.ndarray]:
    """rab rows of one sequence and head, or None when the call has no bias."""
    if not params.has_rab:
        return None
    ts_q = ts_kv = None
    if params.timestamps_q is not None:
        ts_q = np.asarray(params.timestamps_q)[q0:q0 + sp.L_q]
        tkv = params.timestamps_kv if sp.cross else params.timestamps_q
        ts_kv = np.asarray(tkv)[kv0:kv0 + sp.L_kv]
    return rab_rows(sp, rows, h, ts_q, ts_kv, params.rab_time, params.rab_pos)


def _seq_params(params: HstuParams, b: int, batch: int, off_q, off_kv, targets):
    g = group_of_batch(b, batch, params.num_groups)
    c = int(params.context_len[g])
    t = int(targets[b]) if targets is not None else 0
    L_q = int(off_q[b + 1] - off_q[b])
    cross = off_kv is not None
    L_kv = int(off_kv[b + 1] - off_kv[b]) if cross else L_q
    if L_q < c + t:
        raise ValueError(f"batch {b}: query length {L_q} < context {c} + targets {t}")
    kvt = bool(params.kv_targets) and cross
    if cross and L_kv < c + (t if kvt else 0):
        raise ValueError(f"batch {b}: key length {L_kv} < context {c}" + (f" + targets {t}" if kvt else ""))
    sp = SeqMaskParams(L_q=L_q, L_kv=L_kv, context=c, targets=t, causal=bool(params.causal),
                       local=int(params.local_len[g]), minfull=int(params.minfull_len[g]),
                       cross=cross, kv_targets=kvt)
    return g, sp


def resolved_attn_scales(params: HstuParams, batch: int, off_q, targets) -> np.ndarray:
    """Per-group attn_scale after the zero-means-default rule."""
    scales = np.zeros(params.num_groups, dtype=np.float64)
    for g in range(params.num_groups):
        if params.attn_scale[g] != 0:
            scales[g] = float(params.attn_scale[g])
            continue
        m = int(params.max_uih_len[g])
        if m <= 0:
            for b in range(batch):
                if group_of_batch(b, batch, params.num_groups) == g:
                    _, sp = _seq_params(params, b, batch, off_q, None, targets)
                    m = max(m, sp.uih_q)
        scales[g] = 1.0 / m if m > 0 else 1.0
    return scales


def resolved_alpha(params: HstuParams, hdim_qk: int) -> float:
    return float(params.alpha) if params.alpha != 0 else 1.0 / math.sqrt(hdim_qk)


def hstu_attention_forward(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets,
                           params: HstuParams):
    """Full forward.  q [total_q, H, Dqk], k [total_kv, H, Dqk], v [total_kv, H, Dv]
    (any float dtype; converted to float64).  seq_offsets_kv None = self-attention.

    Returns (o [total_q, H, Dv] float64, lse [H, total_q] float64 or None).
    Rows that belong to no sequence stay zero (o) / -inf (lse).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    off_q = np.asarray(seq_offsets_q, dtype=np.int64)
    off_kv = None if seq_offsets_kv is None else np.asarray(seq_offsets_kv, dtype=np.int64)
    batch = off_q.shape[0] - 1
    H = q.shape[1]
    alpha = resolved_alpha(params, q.shape[2])
    scales = resolved_attn_scales(params, batch, off_q, num_targets)
    o = np.zeros((q.shape[0], H, v.shape[2]), dtype=np.float64)
    lse = np.full((H, q.shape[0]), -np.inf) if params.softmax else None
    for b in range(batch):
        g, sp = _seq_params(params, b, batch, off_q, off_kv, num_targets)
        allowed = dense_mask(sp)
        q0 = off_q[b]
        kv0 = off_kv[b] if off_kv is not None else q0
        for h in range(H):
            bias = _seq_bias(params, sp, q0, kv0, h, np.arange(sp.L_q))
            ob, lb = _head_forward(q[q0:q0 + sp.L_q, h], k[kv0:kv0 + sp.L_kv, h],
                                   v[kv0:kv0 + sp.L_kv, h], allowed, alpha, scales[g],
                                   params.softmax, bias)
            o[q0:q0 + sp.L_q, h] = ob
            if lse is not None:
                lse[h, q0:q0 + sp.L_q] = lb
    return o, lse


def hstu_attention_forward_rows(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets,
                                params: HstuParams, b: int, h: int, rows):
    """Outputs of the chosen in-sequence query rows of one (batch, head) only.

    Same definition as :func:`hstu_attention_forward`, restricted to ``rows``
    (indices inside sequence b).  Returns (o [len(rows), Dv], lse [len(rows)] or None).
    """
    off_q = np.asarray(seq_offsets_q, dtype=np.int64)
    off_kv = None if seq_offsets_kv is None else np.asarray(seq_offsets_kv, dtype=np.int64)
    batch = off_q.shape[0] - 1
    alpha = resolved_alpha(params, q.shape[2])
    scales = resolved_attn_scales(params, batch, off_q, num_targets)
    g, sp = _seq_params(params, b, batch, off_q, off_kv, num_targets)
    rows = np.asarray(rows, dtype=np.int64)
    q0 = int(off_q[b])
    kv0 = int(off_kv[b]) if off_kv is not None else q0
    qb = np.asarray(q[q0 + rows, h], dtype=np.float64)
    kb = np.asarray(k[kv0:kv0 + sp.L_kv, h], dtype=np.float64)
    vb = np.asarray(v[kv0:kv0 + sp.L_kv, h], dtype=np.float64)
    bias = _seq_bias(params, sp, q0, kv0, h, rows)
    return _head_forward(qb, kb, vb, mask_rows(sp, rows), alpha, scales[g], params.softmax, bias)


def allowed_pair_count(seq_offsets_q, seq_offsets_kv, num_targets, params: HstuParams,
                       nhead: int) -> int:
    """Number of allowed (b, h, i, j) entries: the useful work of the two GEMMs."""
    off_q = np.asarray(seq_offsets_q, dtype=np.int64)
    off_kv = None if seq_offsets_kv is None else np.asarray(seq_offsets_kv, dtype=np.int64)
    batch = off_q.shape[0] - 1
    total = 0
    for b in range(batch):
        _, sp = _seq_params(params, b, batch, off_q, off_kv, num_targets)
        total += int(dense_mask(sp).sum())
    return total * nhead


def executed_tile_count(seq_offsets_q, seq_offsets_kv, num_targets, params: HstuParams,
                        nhead: int, block_m: int = 128, block_n: int = 128) -> int:
    """Number of (b, h, q-tile, kv-tile) blocks of the dense mask holding at least one
    allowed entry (the tiles a kernel that skips fully masked tiles must execute)."""
    off_q = np.asarray(seq_offsets_q, dtype=np.int64)
    off_kv = None if seq_offsets_kv is None else np.asarray(seq_offsets_kv, dtype=np.int64)
    batch = off_q.shape[0] - 1
    total = 0
    for b in range(batch):
        _, sp = _seq_params(params, b, batch, off_q, off_kv, num_targets)
        m = dense_mask(sp)
        nq = -(-sp.L_q // block_m)
        nk = -(-sp.L_kv // block_n)
        for a in range(nq):
            blk = m[a * block_m:(a + 1) * block_m]
            for c in range(nk):
                if blk[:, c * block_n:(c + 1) * block_n].any():
                    total += 1
    return total * nhead


# ----------------------------------------------------------------------------
# Backward (the gradients of the forward above; the README's training mode saves
# the softmax LSE for it)
# ----------------------------------------------------------------------------
def silu_grad(s: np.ndarray) -> np.ndarray:
    """d/ds SiLU(s) = sigma(s) * (1 + s * (1 - sigma(s))), elementwise, fp64."""
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-s))
    return sig * (1.0 + s * (1.0 - sig))


def _head_backward(q, k, v, g, allowed, alpha, attn_scale, softmax, bias=None):
    """One (sequence, head): the gradients of _head_forward's o with respect to q,
    k and v for the output gradient g [n, Dv].

    SiLU:    o = c * (M . SiLU(s)) v,            s = alpha q k^T
             dv = c a^T g,  da = c g v^T,  ds = M . da . SiLU'(s)
    softmax: o = c * p v,   p = M . exp(s - lse) (row-normalised over allowed keys)
             dv = c p^T g,  dp = c g v^T,  ds = p . (dp - rowsum(p . dp))
    both:    dq = alpha ds k,  dk = alpha ds^T q.
    A relative attention bias enters s, and through it every derivative; ds
    is also its gradient (s = alpha q k^T + rab).  Returns (dq, dk, dv, ds)."""
    s = alpha * (q @ k.T)
    if bias is not None:
        s = s + bias
    if not softmax:
        a = np.where(allowed, silu(s), 0.0)
        dv = attn_scale * (a.T @ g)
        da = attn_scale * (g @ v.T)
        ds = np.where(allowed, da * silu_grad(s), 0.0)
    else:
        masked = np.where(allowed, s, -np.inf)
        m = masked.max(axis=1) if masked.shape[1] else np.full(masked.shape[0], -np.inf)
        has_key = np.isfinite(m)
        m_safe = np.where(has_key, m, 0.0)
        e = np.where(allowed, np.exp(s - m_safe[:, None]), 0.0)
        l = e.sum(axis=1)
        p = e / np.where(has_key, l, 1.0)[:, None]
        dv = attn_scale * (p.T @ g)
        dp = attn_scale * (g @ v.T)
        ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return alpha * (ds @ k), alpha * (ds.T @ q), dv, ds


def hstu_attention_backward(q, k, v, d_o, seq_offsets_q, seq_offsets_kv, num_targets,
                            params: HstuParams, rab_grads: bool = False):
    """Gradients (dq, dk, dv) of the full forward for the output gradient d_o
    [total_q, H, Dv], in float64.  Rows outside every sequence get zero.

    rab_grads: also return the gradients of the relative attention bias tables,
    (dq, dk, dv, d_rab_time [H, 11] or None, d_rab_pos [H, P] or None): a
    table entry's gradient is the sum of ds over the (row, key) pairs of every
    sequence that read it (masked pairs have ds = 0)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    d_o = np.asarray(d_o, dtype=np.float64)
    off_q = np.asarray(seq_offsets_q, dtype=np.int64)
    off_kv = None if seq_offsets_kv is None else np.asarray(seq_offsets_kv, dtype=np.int64)
    batch = off_q.shape[0] - 1
    H = q.shape[1]
    alpha = resolved_alpha(params, q.shape[2])
    scales = resolved_attn_scales(params, batch, off_q, num_targets)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    use_time = params.rab_time is not None and params.timestamps_q is not None
    n_pos = 0 if params.rab_pos is None else np.asarray(params.rab_pos).shape[1]
    d_rab_time = np.zeros((H, len(TIME_BUCKET_EDGES))) if rab_grads and use_time else None
    d_rab_pos = np.zeros((H, n_pos)) if rab_grads and n_pos > 0 else None
    for b in range(batch):
        g_, sp = _seq_params(params, b, batch, off_q, off_kv, num_targets)
        allowed = dense_mask(sp)
        q0 = off_q[b]
        kv0 = off_kv[b] if off_kv is not None else q0
        if rab_grads and params.has_rab:
            ts_q = ts_kv = None
            if use_time:
                ts_q = np.asarray(params.timestamps_q)[q0:q0 + sp.L_q]
                ts_kv = np.asarray(params.timestamps_kv if sp.cross else params.timestamps_q)[kv0:kv0 + sp.L_kv]
            bucket, dist = rab_indices(sp, np.arange(sp.L_q), ts_q, ts_kv, n_pos)
        for h in range(H):
            bias = _seq_bias(params, sp, q0, kv0, h, np.arange(sp.L_q))
            a, bk, c, ds = _head_backward(q[q0:q0 + sp.L_q, h], k[kv0:kv0 + sp.L_kv, h],
                                          v[kv0:kv0 + sp.L_kv, h], d_o[q0:q0 + sp.L_q, h], allowed,
                                          alpha, scales[g_], params.softmax, bias)
            dq[q0:q0 + sp.L_q, h] += a
            dk[kv0:kv0 + sp.L_kv, h] += bk
            dv[kv0:kv0 + sp.L_kv, h] += c
            if d_rab_time is not None:
                d_rab_time[h] += np.bincount(bucket.ravel(), weights=ds.ravel(), minlength=d_rab_time.shape[1])
            if d_rab_pos is not None:
                d_rab_pos[h] += np.bincount(dist.ravel(), weights=ds.ravel(), minlength=n_pos)
    if rab_grads:
        return dq, dk, dv, d_rab_time, d_rab_pos
    return dq, dk, dv
