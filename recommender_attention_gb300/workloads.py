"""Seeded synthetic inputs for the HSTU attention forward.

This module only lays out inputs: per-batch segment lengths, jagged offsets
and Q/K/V values.  It holds none of the attention arithmetic, so both the
CUDA path's tests/bench and the fp64 oracle can draw from it.

Layout of one sequence (composable_kernel ``18_hstu_attention`` README,
"Masking": physical length = context + UIH + targets): ``[context | UIH |
targets]`` on the query side; the key side is the same sequence for
self-attention and ``[context | UIH_kv]`` for cross-attention, or
``[context | UIH_kv | targets]`` when it carries the targets' own keys (an
M-FALCON microbatch over a cached history: "From transformer parallelism to
HSTU", section 5.3).  Jagged tensors
are flattened ``[total_tokens, nhead, hdim]`` with ``seq_offsets`` of length
``batch + 1`` (README "Batch modes"); batched mode is the special case of equal
lengths.

Random numbers come from numpy's PCG64 generator seeded with the workload's
seed, drawn in a fixed order: UIH lengths (Q, then KV), targets, then q, k, v
(token-major).  uniform means U[-1, 1); normal means N(0, 1).  Values are
rounded once, round-to-nearest-even, to the storage dtype.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    batch: int
    nhead: int
    hdim_qk: int
    hdim_v: int
    dtype: str                       # "fp16" | "bf16"
    uih_q: List[int]                 # per batch
    targets: List[int]               # per batch
    uih_kv: Optional[List[int]] = None   # per batch; None = self-attention
    num_groups: int = 1
    context_len: List[int] = field(default_factory=lambda: [0])   # per group
    local_len: List[int] = field(default_factory=lambda: [0])
    minfull_len: List[int] = field(default_factory=lambda: [0])
    max_uih_len: List[int] = field(default_factory=lambda: [0])   # 0 = automatic
    attn_scale: List[float] = field(default_factory=lambda: [0.0])  # 0 = default
    alpha: float = 0.0               # 0 = default
    causal: bool = True
    softmax: bool = False
    dist: str = "uniform"            # "uniform" | "normal"
    seed: int = 0
    has_targets: bool = True         # False: pass no num_targets array (all zero)
    kv_targets: bool = False         # cross-attention: the key side ends with the targets' keys
    rab_pos_buckets: int = 0         # > 0: a relative attention bias (timestamps, both tables)

    # ----------------------------------------------------------- layout
    @property
    def cross(self) -> bool:
        return self.uih_kv is not None

    def group(self, b: int) -> int:
        return b // (self.batch // self.num_groups)

    def lengths_q(self) -> np.ndarray:
        return np.array([self.context_len[self.group(b)] + self.uih_q[b] + self.targets[b]
                         for b in range(self.batch)], dtype=np.int64)

    def lengths_kv(self) -> np.ndarray:
        if not self.cross:
            return self.lengths_q()
        return np.array([self.context_len[self.group(b)] + self.uih_kv[b] +
                         (self.targets[b] if self.kv_targets else 0)
                         for b in range(self.batch)], dtype=np.int64)

    def seq_offsets_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths_q())]).astype(np.int32)

    def seq_offsets_kv(self) -> Optional[np.ndarray]:
        if not self.cross:
            return None
        return np.concatenate([[0], np.cumsum(self.lengths_kv())]).astype(np.int32)

    def num_targets(self) -> Optional[np.ndarray]:
        if not self.has_targets:
            return None
        return np.asarray(self.targets, dtype=np.int32)

    @property
    def total_q(self) -> int:
        return int(self.lengths_q().sum())

    @property
    def total_kv(self) -> int:
        return int(self.lengths_kv().sum())

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    # ----------------------------------------------------------- values
    def tensors(self):
        """(q, k, v) as CPU torch tensors of the storage dtype, [tokens, nhead, hdim]."""
        # The lengths were drawn by the constructor from the plain seed; the
        # values come from a separate stream so they do not depend on how many
        # length draws were made.
        vrng = np.random.default_rng([self.seed, 1])
        shapes = [(self.total_q, self.nhead, self.hdim_qk),
                  (self.total_kv, self.nhead, self.hdim_qk),
                  (self.total_kv, self.nhead, self.hdim_v)]
        out = []
        for shp in shapes:
            if self.dist == "normal":
                x = vrng.standard_normal(size=shp, dtype=np.float32)
            else:
                x = vrng.uniform(-1.0, 1.0, size=shp).astype(np.float32)
            out.append(torch.from_numpy(x).to(DTYPES[self.dtype]))
        return tuple(out)

    def rab_inputs(self):
        """Relative attention bias inputs (numpy): (timestamps_q int64 [total_q],
        timestamps_kv int64 [total_kv] or None for self-attention, rab_time
        float32 [nhead, 11], rab_pos float32 [nhead, rab_pos_buckets]).

        Per sequence the key timestamps (seconds) start near 1.7e9 and grow by
        gaps that are 0 one time in ten and otherwise log-uniform on [1 s,
        ~37 days], so every time-gap bucket occurs.  Query rows take the
        timestamp of the key at their key-coordinate position (context row i:
        key i; UIH and target rows: key i + u_kv - u); rows past the last key
        continue it by the same gap law.  The tables are N(0, 1)."""
        rng = np.random.default_rng([self.seed, 3])
        okv = self.seq_offsets_kv() if self.cross else self.seq_offsets_q()
        oq = self.seq_offsets_q()
        ts_kv = np.zeros(int(okv[-1]), dtype=np.int64)
        ts_q = np.zeros(int(oq[-1]), dtype=np.int64)

        def gaps(n):
            g = np.floor(10.0 ** rng.uniform(0.0, 6.5, size=n)).astype(np.int64)
            g[rng.uniform(size=n) < 0.1] = 0
            return g

        for b in range(self.batch):
            lkv = int(okv[b + 1] - okv[b])
            lq = int(oq[b + 1] - oq[b])
            start = 1_700_000_000 + int(rng.integers(0, 10 ** 7))
            keys = start + np.concatenate([[0], np.cumsum(gaps(max(lkv - 1, 0)))])[:lkv]
            ts_kv[okv[b]:okv[b] + lkv] = keys
            c = self.context_len[self.group(b)]
            u = self.uih_q[b]
            ukv = self.uih_kv[b] if self.cross else u
            last = int(keys[-1]) if lkv else start
            extra = last + np.cumsum(gaps(lq))
            for i in range(lq):
                pos = i if i < c else i + (ukv - u)
                ts_q[oq[b] + i] = keys[min(max(pos, 0), lkv - 1)] if 0 <= pos < lkv else int(extra[i])
        rab_time = rng.standard_normal((self.nhead, 11)).astype(np.float32)
        rab_pos = rng.standard_normal((self.nhead, max(self.rab_pos_buckets, 1))).astype(np.float32)
        return ts_q, (ts_kv if self.cross else None), rab_time, rab_pos

    def grad_output(self):
        """An output gradient dO [total_q, nhead, hdim_v] (CPU, storage dtype)
        for the backward, from its own stream of the seed, same distribution."""
        grng = np.random.default_rng([self.seed, 2])
        shp = (self.total_q, self.nhead, self.hdim_v)
        if self.dist == "normal":
            x = grng.standard_normal(size=shp, dtype=np.float32)
        else:
            x = grng.uniform(-1.0, 1.0, size=shp).astype(np.float32)
        return torch.from_numpy(x).to(DTYPES[self.dtype])


def _draw_ints(rng, lo, hi, n):
    """n integers uniform on [lo, hi] inclusive."""
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


# ---------------------------------------------------------------- the configs
def tiny_batched() -> Workload:
    """B=2, nhead=2, hdim 64, fp16, UIH 64, 4 targets, context 2, causal,
    local 5, minfull 4, alpha 1/8, attn_scale 1/64, U[-1,1], seed 13579
    (physical length 70)."""
    return Workload(name="tiny_batched_silu", batch=2, nhead=2, hdim_qk=64, hdim_v=64,
                    dtype="fp16", uih_q=[64, 64], targets=[4, 4], context_len=[2],
                    local_len=[5], minfull_len=[4], alpha=1.0 / 8, attn_scale=[1.0 / 64],
                    causal=True, dist="uniform", seed=13579)


def jagged_readme() -> Workload:
    """The README's jagged validation case: B=10, nhead=4, hdim 128, bf16,
    UIH 750..779, targets 5..6, causal, local 5, context 6, minfull 6."""
    return Workload(name="jagged_silu_b10", batch=10, nhead=4, hdim_qk=128, hdim_v=128,
                    dtype="bf16",
                    uih_q=[750, 730, 733, 860, 870, 788, 760, 821, 833, 779],
                    targets=[5, 5, 6, 6, 5, 6, 5, 6, 4, 6], context_len=[6], local_len=[5],
                    minfull_len=[6], causal=True, dist="uniform", seed=13579)


def batched_default() -> Workload:
    """B=12, nhead=4, hdim 64, fp16, UIH 400, 16 targets, causal, local 5,
    context 6, minfull 6, alpha 1/8, attn_scale 1/400, N(0,1), seed 1."""
    return Workload(name="batched_silu_b12", batch=12, nhead=4, hdim_qk=64, hdim_v=64,
                    dtype="fp16", uih_q=[400] * 12, targets=[16] * 12, context_len=[6],
                    local_len=[5], minfull_len=[6], alpha=1.0 / 8, attn_scale=[1.0 / 400],
                    causal=True, dist="normal", seed=1)


def large_jagged(hdim: int = 128, batch: int = 64, seed: int = 7, hdim_v: Optional[int] = None) -> Workload:
    """B=64, nhead=4, bf16, UIH ~ U_int[1024, 4096], targets ~ U_int[1, 32],
    full causal (local 0), context 6, minfull 0, N(0,1), seed 7."""
    rng = np.random.default_rng(seed)
    uih = _draw_ints(rng, 1024, 4096, batch)
    tg = _draw_ints(rng, 1, 32, batch)
    dv = hdim if hdim_v is None else hdim_v
    return Workload(name=f"large_jagged_silu_d{hdim}" + ("" if dv == hdim else f"_{dv}"), batch=batch,
                    nhead=4, hdim_qk=hdim, hdim_v=dv, dtype="bf16", uih_q=uih, targets=tg, context_len=[6],
                    local_len=[0], minfull_len=[0], causal=True, dist="normal", seed=seed)


def group_cross_splitkv(softmax: bool = False, batch: int = 32, seed: int = 11) -> Workload:
    """G=4 group HSTU cross-attention: B=32, nhead=8, hdim 128, bf16,
    UIH_q ~ U[64, 256], UIH_kv ~ U[4096, 8192], targets ~ U[1, 16], per-group
    local {0,32,128,512}, context {0,6,16,32}, minfull {0,8,16,64}, N(0,1), seed 11."""
    rng = np.random.default_rng(seed)
    uq = _draw_ints(rng, 64, 256, batch)
    ukv = _draw_ints(rng, 4096, 8192, batch)
    tg = _draw_ints(rng, 1, 16, batch)
    return Workload(name="group_cross_splitkv_" + ("softmax" if softmax else "silu"),
                    batch=batch, nhead=8, hdim_qk=128, hdim_v=128, dtype="bf16", uih_q=uq,
                    uih_kv=ukv, targets=tg, num_groups=4, context_len=[0, 6, 16, 32],
                    local_len=[0, 32, 128, 512], minfull_len=[0, 8, 16, 64],
                    max_uih_len=[0] * 4, attn_scale=[0.0] * 4, causal=True, softmax=softmax,
                    dist="normal", seed=seed)


def mfalcon(batch: int = 16, candidates: int = 128, seed: int = 21, softmax: bool = False,
            history=(2048, 8192)) -> Workload:
    """M-FALCON microbatch ("From transformer parallelism to HSTU", section 5.3):
    per request a cached history of UIH_kv ~ U_int[history] (default [2048, 8192]) keys/values plus
    the keys of `candidates` candidates; the queries are the 6 context rows and
    the candidates (no history rows).  nhead 4, hdim 128, bf16, causal, N(0,1).
    attn_scale is 1/8192 (the longest history a request may have), since the
    query side has no UIH rows to take the default from."""
    rng = np.random.default_rng(seed)
    ukv = _draw_ints(rng, history[0], history[1], batch)
    return Workload(name="mfalcon", batch=batch, nhead=4, hdim_qk=128, hdim_v=128, dtype="bf16",
                    uih_q=[0] * batch, uih_kv=ukv, targets=[candidates] * batch,
                    context_len=[6], attn_scale=[1.0 / 8192], causal=True, softmax=softmax,
                    dist="normal", seed=seed, kv_targets=True)


CONFIGS = {
    "tiny": tiny_batched,
    "jagged": jagged_readme,
    "batched": batched_default,
    "large": large_jagged,
    "group_cross": group_cross_splitkv,
    "mfalcon": mfalcon,
}


def random_small(seed: int, *, dtype: str = "bf16", hdim: int = 64, softmax: bool = False,
                 cross: Optional[bool] = None, max_uih: int = 300, kv_targets: bool = False,
                 hdim_v: Optional[int] = None) -> Workload:
    """A small random workload for fuzzing: ragged lengths, random mask parameters.
    kv_targets=True makes it a cross-attention call whose keys end with the
    targets' own keys."""
    rng = np.random.default_rng(1000 + seed)
    num_groups = int(rng.choice([1, 1, 2, 3]))
    batch = num_groups * int(rng.integers(1, 4))
    if cross is None:
        cross = bool(rng.integers(0, 2))
    if kv_targets:
        cross = True
    uq = _draw_ints(rng, 0, max_uih, batch)
    ukv = _draw_ints(rng, 0, 2 * max_uih, batch) if cross else None
    tg = _draw_ints(rng, 0, 20, batch)
    ctx = _draw_ints(rng, 0, 9, num_groups)
    loc = [int(rng.choice([0, 1, 5, 33, 200])) for _ in range(num_groups)]
    mf = [int(rng.choice([0, 3, 17, 150])) for _ in range(num_groups)]
    return Workload(name=f"fuzz{seed}", batch=batch, nhead=int(rng.integers(1, 4)),
                    hdim_qk=hdim, hdim_v=hdim if hdim_v is None else hdim_v, dtype=dtype,
                    uih_q=uq, uih_kv=ukv, targets=tg,
                    num_groups=num_groups, context_len=ctx, local_len=loc, minfull_len=mf,
                    max_uih_len=[0] * num_groups,
                    attn_scale=[0.0] * num_groups, alpha=0.0,
                    causal=bool(rng.integers(0, 4) > 0), softmax=softmax,
                    dist="normal" if rng.integers(0, 2) else "uniform", seed=seed,
                    kv_targets=kv_targets)
