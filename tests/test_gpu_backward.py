"""Backward parity: dQ, dK, dV of the CUDA path (through the C ABI) against the
fp64 oracle's hstu_attention_backward, element by element, on the same seeded
inputs and output gradient.

Softmax mode feeds the backward the forward's own o and lse (from the CUDA
forward, as a training step would).  Tolerance: the forward's per-dtype bound
on max |err| relative to max |reference| of each gradient, plus the same
elementwise rtol; the kernels round P and dS to the storage type before the
two gradient products, exactly as the forward rounds P before P V."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle.hstu_oracle import hstu_attention_backward, resolved_attn_scales
from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import TOL, assert_parity, call_kwargs, device_inputs, rab_kwargs
from tests.helpers import as_f64, oracle_forward, oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


def gpu_backward(w, q, k, v, d_o, rab_grads=False, **over):
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    kw = call_kwargs(w, **over)
    o = lse = None
    if w.softmax:
        o, lse = hstu.hstu_attn_fwd(dq, dk, dv, off_q, off_kv, tg, check=True, **kw)
    g = hstu.hstu_attn_bwd(dq, dk, dv, d_o.cuda(), off_q, off_kv, tg, o=o, lse=lse, check=True,
                           rab_grads=rab_grads, **kw)
    torch.cuda.synchronize()
    return tuple(None if x is None else _host(x) for x in g)


def check_backward(w, rab=False, use_time=True, use_pos=True, **over):
    """rab: with the workload's relative attention bias (Workload.rab_inputs),
    and then the gradients of its tables as well (use_time / use_pos keep one
    table only)."""
    q, k, v = w.tensors()
    d_o = w.grad_output()
    bias = w.rab_inputs() if rab else None
    if rab:
        over = {**over, **rab_kwargs(bias, use_time, use_pos)}
    got = gpu_backward(w, q, k, v, d_o, rab_grads=rab, **over)
    ref = hstu_attention_backward(as_f64(q), as_f64(k), as_f64(v), as_f64(d_o), w.seq_offsets_q(),
                                  w.seq_offsets_kv(), w.num_targets(), oracle_params(w, bias, use_time, use_pos),
                                  rab_grads=rab)
    names = ("dq", "dk", "dv", "d_rab_time", "d_rab_pos")
    delta_mass = None
    for name, a, b in zip(names, got, ref):
        if name.startswith("d_rab"):
            # the tables a call uses get gradients; the others none
            assert (a is None) == (b is None), f"{w.name} {name}: presence differs"
            if a is None:
                continue
            if w.softmax:
                # ds = p (dp - delta), delta_i = sum_e dO_ie O_ie from the forward's O as
                # stored (fp16 / bf16: each element within 2^-11 / 2^-9 relative).  With
                # sum_j p_ij <= 1 that moves every table entry of head h by at most
                # u sum_i sum_e |dO_ie O_ie|, which the entries' cancellation (a softmax
                # row's ds sums to zero) does not shrink: it bounds the error on top of
                # the usual tolerance.
                if delta_mass is None:
                    o_ref, _ = oracle_forward(w, q, k, v, bias, use_time, use_pos)
                    u = 2.0 ** -9 if w.dtype == "bf16" else 2.0 ** -11
                    delta_mass = u * np.abs(as_f64(d_o) * o_ref).sum(axis=(0, 2))   # [H]
                err = np.abs(a - b)
                lim = TOL[w.dtype] * np.abs(b).max() + delta_mass[:, None]
                assert np.all(err <= lim), (f"{w.name} {name}: max|err| {err.max():.3e}, "
                                            f"bound {lim.ravel()[err.argmax()]:.3e}")
                continue
        assert_parity(a, b, w.dtype, what=f"{w.name} {name}")


# ---------------------------------------------------------------- the small configs
@pytest.mark.parametrize("cfg", ["tiny", "jagged", "batched"])
@pytest.mark.parametrize("softmax", [False, True])
def test_small_configs_backward(cfg, softmax):
    w = W.CONFIGS[cfg]().with_(softmax=softmax)
    check_backward(w)


@pytest.mark.parametrize("softmax", [False, True])
def test_group_cross_backward(softmax):
    check_backward(W.group_cross_splitkv(softmax=softmax, batch=8))


@pytest.mark.parametrize("softmax", [False, True])
def test_mfalcon_backward(softmax):
    check_backward(W.mfalcon(batch=3, candidates=200, softmax=softmax, history=(300, 900)))


# ---------------------------------------------------------------- fuzz
@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("softmax", [False, True])
def test_fuzz_backward(seed, softmax):
    hdim = [64, 128][seed % 2]
    dtype = "bf16" if seed % 3 else "fp16"
    w = W.random_small(seed, dtype=dtype, hdim=hdim, softmax=softmax, kv_targets=seed % 5 == 4)
    check_backward(w)


# ---------------------------------------------------------------- head dimension 96, and 96/64
@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("dv", [96, 64])
def test_hdim96_backward(softmax, dv):
    check_backward(W.jagged_readme().with_(hdim_qk=96, hdim_v=dv, softmax=softmax))


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_hdim96_backward(seed):
    w = W.random_small(200 + seed, hdim=96, hdim_v=[96, 64][seed % 2], softmax=seed % 3 == 2,
                       dtype="bf16" if seed % 2 else "fp16", kv_targets=seed == 5)
    check_backward(w)


# ---------------------------------------------------------------- with a relative attention bias
@pytest.mark.parametrize("cfg", ["tiny", "jagged"])
@pytest.mark.parametrize("softmax", [False, True])
def test_small_configs_backward_rab(cfg, softmax):
    check_backward(W.CONFIGS[cfg]().with_(softmax=softmax, rab_pos_buckets=64), rab=True)


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_backward_rab(seed):
    w = W.random_small(100 + seed, hdim=[64, 128][seed % 2], softmax=seed % 4 >= 2,
                       dtype="bf16" if seed % 3 else "fp16", kv_targets=seed % 4 == 3)
    check_backward(w.with_(rab_pos_buckets=[1, 9, 64, 256][seed % 4]), rab=True)


@pytest.mark.parametrize("dv", [96, 64])
@pytest.mark.parametrize("softmax", [False, True])
def test_hdim96_backward_rab(softmax, dv):
    """The bias at hdim 96 and 96/64: dq, dk, dv and the tables' gradients."""
    check_backward(W.jagged_readme().with_(hdim_qk=96, hdim_v=dv, softmax=softmax, rab_pos_buckets=64), rab=True)
    w = W.random_small(400 + dv, hdim=96, hdim_v=dv, softmax=softmax, dtype="bf16", kv_targets=True)
    check_backward(w.with_(rab_pos_buckets=17), rab=True)


@pytest.mark.parametrize("use_time,use_pos", [(True, False), (False, True)])
@pytest.mark.parametrize("softmax", [False, True])
def test_backward_rab_one_table(softmax, use_time, use_pos):
    """A bias with one table only: its gradient alone (the other output stays
    unset), and dq, dk, dv through it."""
    check_backward(W.jagged_readme().with_(softmax=softmax, rab_pos_buckets=32), rab=True, use_time=use_time,
                   use_pos=use_pos)


@pytest.mark.parametrize("softmax", [False, True])
def test_mfalcon_backward_rab(softmax):
    check_backward(W.mfalcon(batch=2, candidates=150, softmax=softmax, history=(300, 700)).with_(rab_pos_buckets=100),
                   rab=True)


# ---------------------------------------------------------------- edges
def test_backward_edge_empty_sequences_and_rows_without_keys():
    # cross-attention with an empty key sequence: its query rows see nothing
    # (dq = 0), an empty query sequence leaves its keys without a query
    # (dk = dv = 0), plus a sequence with only context rows
    w = W.Workload(name="edges_bwd", batch=4, nhead=2, hdim_qk=64, hdim_v=64, dtype="bf16",
                   uih_q=[0, 130, 0, 300], uih_kv=[0, 0, 260, 129], targets=[0, 3, 0, 5],
                   context_len=[0], local_len=[0], causal=True, seed=5)
    for softmax in (False, True):
        check_backward(w.with_(softmax=softmax))
    w2 = W.Workload(name="ctx_only", batch=2, nhead=1, hdim_qk=128, hdim_v=128, dtype="bf16",
                    uih_q=[0, 200], targets=[0, 1], context_len=[7], causal=True, seed=6,
                    max_uih_len=[64])
    check_backward(w2)


def test_backward_rows_outside_sequences_untouched():
    w = W.random_small(3, hdim=64)
    q, k, v = w.tensors()
    d_o = w.grad_output()
    pad = 37
    qp = torch.cat([q, torch.zeros((pad,) + q.shape[1:], dtype=q.dtype)])
    kp = torch.cat([k, torch.zeros((pad,) + k.shape[1:], dtype=k.dtype)])
    vp = torch.cat([v, torch.zeros((pad,) + v.shape[1:], dtype=v.dtype)])
    dop = torch.cat([d_o, torch.zeros((pad,) + d_o.shape[1:], dtype=d_o.dtype)])
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, qp, kp, vp)
    sentinel = 3.0
    gq, gk, gv = (torch.full_like(x, sentinel) for x in (dq, dk, dv))
    hstu.hstu_attn_bwd(dq, dk, dv, dop.cuda(), off_q, off_kv, tg, dq=gq, dk=gk, dv=gv, check=True,
                       **call_kwargs(w))
    torch.cuda.synchronize()
    nq, nkv = w.total_q, w.total_kv
    assert torch.all(gq[nq:] == sentinel) and torch.all(gk[nkv:] == sentinel) and torch.all(gv[nkv:] == sentinel)
    ref = hstu_attention_backward(as_f64(q), as_f64(k), as_f64(v), as_f64(d_o), w.seq_offsets_q(),
                                  w.seq_offsets_kv(), w.num_targets(), oracle_params(w))
    for name, a, b in zip(("dq", "dk", "dv"), (gq[:nq], gk[:nkv], gv[:nkv]), ref):
        assert_parity(_host(a), b, w.dtype, what=name)


def test_backward_device_error_leaves_gradients_untouched():
    w = W.CONFIGS["tiny"]()
    q, k, v = w.tensors()
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    gq, gk, gv = (torch.full_like(x, 5.0) for x in (dq, dk, dv))
    call = hstu.HstuBwdCall(dq, dk, dv, w.grad_output().cuda(), off_q, off_kv, tg, dq=gq, dk=gk, dv=gv,
                            **call_kwargs(w, max_seqlen_q=10, max_seqlen_kv=10))
    call.launch()
    with pytest.raises(hstu.HstuError) as e:
        call.check()
    assert e.value.device_error & 8   # max_seqlen
    assert torch.all(gq == 5.0) and torch.all(gk == 5.0) and torch.all(gv == 5.0)


def test_backward_repeated_calls_are_identical():
    w = W.random_small(7, hdim=128, softmax=True)
    q, k, v = w.tensors()
    d_o = w.grad_output()
    a = gpu_backward(w, q, k, v, d_o)
    b = gpu_backward(w, q, k, v, d_o)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ---------------------------------------------------------------- full size, sampled sequences
@pytest.mark.parametrize("softmax,rab", [(False, False), (True, False), (False, True)])
def test_large_jagged_backward_sampled(softmax, rab):
    """The large jagged workload at full size through one backward call (with
    rab: plus the relative attention bias); the oracle recomputes a few whole
    sequences (a sequence's gradients depend on that sequence alone), with the
    attn_scale the full batch resolves to."""
    w = W.large_jagged(hdim=128).with_(softmax=softmax, rab_pos_buckets=128 if rab else 0)
    q, k, v = w.tensors()
    d_o = w.grad_output()
    bias = w.rab_inputs() if rab else None
    got = gpu_backward(w, q, k, v, d_o, **(rab_kwargs(bias) if rab else {}))
    off = w.seq_offsets_q()
    p = oracle_params(w)
    scale = float(resolved_attn_scales(p, w.batch, off, w.num_targets())[0])
    lens = w.lengths_q()
    rng = np.random.default_rng(3)
    for b in [int(np.argmin(lens)), int(rng.integers(0, w.batch))]:
        s0, s1 = int(off[b]), int(off[b + 1])
        sub = dataclasses.replace(p, attn_scale=[scale])
        if rab:
            sub = dataclasses.replace(sub, timestamps_q=bias[0][s0:s1], rab_time=bias[2], rab_pos=bias[3])
        ref = hstu_attention_backward(as_f64(q[s0:s1]), as_f64(k[s0:s1]), as_f64(v[s0:s1]),
                                      as_f64(d_o[s0:s1]), np.array([0, s1 - s0]), None,
                                      np.array([w.targets[b]]), sub)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            assert_parity(a[s0:s1], r, w.dtype, what=f"b{b} {name}")
