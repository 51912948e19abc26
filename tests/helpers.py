"""Glue between the seeded workloads and the fp64 oracle (test side only)."""
from __future__ import annotations

import numpy as np

from oracle.hstu_oracle import HstuParams


def oracle_params(w, rab=None, use_time=True, use_pos=True) -> HstuParams:
    """The oracle's parameters of workload w; rab = w.rab_inputs() adds the
    relative attention bias (use_time / use_pos keep one term only)."""
    p = HstuParams(num_groups=w.num_groups, context_len=list(w.context_len),
                   local_len=list(w.local_len), minfull_len=list(w.minfull_len),
                   max_uih_len=list(w.max_uih_len), attn_scale=list(w.attn_scale),
                   alpha=w.alpha, causal=w.causal, softmax=w.softmax,
                   kv_targets=w.kv_targets)
    if rab is not None:
        ts_q, ts_kv, rab_time, rab_pos = rab
        if use_time:
            p.timestamps_q, p.timestamps_kv, p.rab_time = ts_q, ts_kv, rab_time
        if use_pos:
            p.rab_pos = rab_pos
    return p


def as_f64(t) -> np.ndarray:
    return t.float().numpy().astype(np.float64)


def oracle_forward(w, q, k, v, rab=None, use_time=True, use_pos=True):
    from oracle.hstu_oracle import hstu_attention_forward
    return hstu_attention_forward(as_f64(q), as_f64(k), as_f64(v), w.seq_offsets_q(),
                                  w.seq_offsets_kv(), w.num_targets(),
                                  oracle_params(w, rab, use_time, use_pos))


def read_mask_fixture(path):
    params = {}
    rows = []
    for line in open(path):
        line = line.strip()
        if line.startswith("# params:"):
            for kv in line[len("# params:"):].split():
                key, val = kv.split("=")
                params[key] = int(val)
        elif line and not line.startswith("#"):
            rows.append([ch == "X" for ch in line])
    return params, np.array(rows, dtype=bool)


def kernel_query_tiles(L_q: int, c: int):
    """Rows (within a sequence) of each query tile the forward kernel runs.

    Its layout: tile m holds rows [128 m, 128 m + 128); when there is more than
    one tile and ceil(c/8)*8 lanes are free at the top of the last tile, the c
    context rows (which see every UIH key) move from tile 0 to the last tile."""
    nq = -(-L_q // 128)
    tiles = [list(range(128 * m, min(128 * m + 128, L_q))) for m in range(nq)]
    if c > 0 and nq > 1 and -(-c // 8) * 8 <= 128 - (L_q - 128 * (nq - 1)):
        tiles[0] = [r for r in tiles[0] if r >= c]
        tiles[-1] += list(range(c))
    return tiles


def kernel_executed_tiles(w) -> int:
    """(b, h, query tile, 128-key tile) blocks of the kernel's layout that hold at
    least one allowed entry of the oracle's dense mask."""
    from oracle.hstu_oracle import _seq_params, dense_mask
    p = oracle_params(w)
    off_q, off_kv, tg = w.seq_offsets_q(), w.seq_offsets_kv(), w.num_targets()
    total = 0
    for b in range(w.batch):
        _, sp = _seq_params(p, b, w.batch, off_q, off_kv, tg)
        mask = dense_mask(sp)
        nk = -(-sp.L_kv // 128)
        for rows in kernel_query_tiles(sp.L_q, sp.context):
            blk = mask[rows]
            total += sum(1 for n in range(nk) if blk[:, 128 * n:128 * n + 128].any())
    return total * w.nhead


def _oracle_sequence(task):
    """One sequence of a one-group self-attention workload through the oracle
    (a worker of oracle_forward_parallel)."""
    from oracle.hstu_oracle import hstu_attention_forward
    qs, ks, vs, targets, params = task
    L = qs.shape[0]
    return hstu_attention_forward(qs, ks, vs, np.array([0, L]), None, np.array([targets], dtype=np.int32),
                                  params)


def oracle_forward_parallel(w, q, k, v, processes=None):
    """oracle_forward of a one-group self-attention workload, one sequence per
    task on a pool of spawned processes (one BLAS thread each).  Each task gets
    the attn_scale the whole batch resolves to, so the result equals the
    whole-batch call.  Returns (o, lse) like oracle_forward."""
    import dataclasses
    import multiprocessing as mp
    import os

    from oracle.hstu_oracle import resolved_attn_scales
    assert w.num_groups == 1 and not w.cross
    p = oracle_params(w)
    off, tg = w.seq_offsets_q(), w.num_targets()
    tg = np.zeros(w.batch, dtype=np.int32) if tg is None else tg
    p = dataclasses.replace(p, attn_scale=[float(resolved_attn_scales(p, w.batch, off, tg)[0])])
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    order = list(np.argsort(-w.lengths_q()))   # longest first, for the pool's balance
    tasks = [(qd[off[b]:off[b + 1]], kd[off[b]:off[b + 1]], vd[off[b]:off[b + 1]], int(tg[b]), p) for b in order]
    saved = {x: os.environ.get(x) for x in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for x in saved:
        os.environ[x] = "1"
    try:
        with mp.get_context("spawn").Pool(processes or os.cpu_count()) as pool:
            results = pool.map(_oracle_sequence, tasks, chunksize=1)
    finally:
        for x, val in saved.items():
            if val is None:
                os.environ.pop(x, None)
            else:
                os.environ[x] = val
    o = np.zeros((w.total_q, w.nhead, w.hdim_v))
    lse = np.full((w.nhead, w.total_q), -np.inf) if w.softmax else None
    for b, (ob, lb) in zip(order, results):
        o[off[b]:off[b + 1]] = ob
        if lse is not None:
            lse[:, off[b]:off[b + 1]] = lb
    return o, lse
