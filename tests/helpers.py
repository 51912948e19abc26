"""Glue between the seeded workloads and the fp64 oracle (test side only)."""
from __future__ import annotations

import numpy as np

from oracle.hstu_oracle import HstuParams


def oracle_params(w) -> HstuParams:
    return HstuParams(num_groups=w.num_groups, context_len=list(w.context_len),
                      local_len=list(w.local_len), minfull_len=list(w.minfull_len),
                      max_uih_len=list(w.max_uih_len), attn_scale=list(w.attn_scale),
                      alpha=w.alpha, causal=w.causal, softmax=w.softmax,
                      kv_targets=w.kv_targets)


def as_f64(t) -> np.ndarray:
    return t.float().numpy().astype(np.float64)


def oracle_forward(w, q, k, v):
    from oracle.hstu_oracle import hstu_attention_forward
    return hstu_attention_forward(as_f64(q), as_f64(k), as_f64(v), w.seq_offsets_q(),
                                  w.seq_offsets_kv(), w.num_targets(), oracle_params(w))


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
