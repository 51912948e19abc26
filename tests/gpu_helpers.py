"""Runs a seeded workload through the C-ABI binding and compares with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from recommender_attention_gb300.hstu import HstuCall, hstu_attn_fwd

# Tolerances of the forward: max |err| relative to max |o| per dtype, an
# elementwise rtol, and an absolute bound on LSE (natural log).
TOL = {"fp16": 1e-2, "bf16": 2e-2}
RTOL = 2e-2
LSE_ATOL = 1e-3


def device_inputs(w, q, k, v, device="cuda"):
    off_q = torch.from_numpy(w.seq_offsets_q()).to(device)
    okv = w.seq_offsets_kv()
    off_kv = torch.from_numpy(okv).to(device) if okv is not None else None
    tg = w.num_targets()
    tg = torch.from_numpy(tg).to(device) if tg is not None else None
    return q.to(device), k.to(device), v.to(device), off_q, off_kv, tg


def call_kwargs(w, **over):
    kw = dict(alpha=w.alpha, attn_scale=list(w.attn_scale), causal=w.causal,
              local_len=list(w.local_len), context_len=list(w.context_len),
              minfull_len=list(w.minfull_len), max_uih_len=list(w.max_uih_len),
              num_groups=w.num_groups, softmax=w.softmax,
              max_seqlen_q=int(w.lengths_q().max()), max_seqlen_kv=int(w.lengths_kv().max()),
              kv_targets=w.kv_targets)
    kw.update(over)
    return kw


def rab_kwargs(rab, use_time=True, use_pos=True, device="cuda"):
    """HstuCall keyword arguments of w.rab_inputs() (numpy) as device tensors."""
    ts_q, ts_kv, rab_time, rab_pos = rab
    kw = {}
    if use_time:
        kw["timestamps_q"] = torch.from_numpy(ts_q).to(device)
        kw["timestamps_kv"] = None if ts_kv is None else torch.from_numpy(ts_kv).to(device)
        kw["rab_time"] = torch.from_numpy(rab_time).to(device)
    if use_pos:
        kw["rab_pos"] = torch.from_numpy(rab_pos).to(device)
    return kw


def gpu_forward(w, q, k, v, **over):
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    o, lse = hstu_attn_fwd(dq, dk, dv, off_q, off_kv, tg, check=True, **call_kwargs(w, **over))
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), (None if lse is None else lse.cpu().numpy())


def gpu_call(w, q, k, v, **over) -> HstuCall:
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    return HstuCall(dq, dk, dv, off_q, off_kv, tg, **call_kwargs(w, **over))


def assert_parity(o_gpu, o_ref, dtype, lse_gpu=None, lse_ref=None, what=""):
    tol = TOL[dtype]
    scale = float(np.abs(o_ref).max())
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    err = np.abs(o_gpu - o_ref)
    worst = float(err.max()) if err.size else 0.0
    assert worst <= tol * max(scale, 1e-30), (
        f"{what}: max|err| {worst:.3e} > {tol} * max|o| {scale:.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    np.testing.assert_allclose(o_gpu, o_ref, rtol=RTOL, atol=tol * max(scale, 1e-30), err_msg=what)
    if lse_ref is not None:
        assert lse_gpu is not None
        fin = np.isfinite(lse_ref)
        assert np.array_equal(fin, np.isfinite(lse_gpu)), f"{what}: LSE -inf pattern differs"
        assert np.all(lse_gpu[~fin] == -np.inf)
        if fin.any():
            d = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max())
            assert d <= LSE_ATOL, f"{what}: LSE max err {d:.3e}"
