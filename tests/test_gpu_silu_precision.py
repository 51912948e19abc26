"""The SiLU stage element by element, forward and backward, against the oracle.

composable_kernel 18_hstu_attention README, "Forward computation" and "Data
types": the scores are accumulated in fp32 and the mask and SiLU are computed
in fp32; only P, the A operand of the second product, is rounded to the
16-bit storage type.  A normal parity test sums P over hundreds of keys, so an
error in the small (negative-score) entries of P hides under max|o|.  Here the
key and value matrices are the identity (one sequence of 128 tokens, one head,
hdim 128, alpha = attn_scale = 1), so every output element is one entry:

    K = I, V = I:            s = Q,   o = SiLU(s)                 (forward)
    ... and dO = ones:       dQ = SiLU'(s)                        (dQ kernel)
    Q = I, K = G^T, V = I:   s = G,   dO = ones:  dK = SiLU'(s)^T (dK/dV kernel)
                                      dO = I:     dV = SiLU(s)^T  (dK/dV kernel)

with the scores drawn uniformly over [-12, 6] and rounded once to the storage
type, so the strongly negative tail, where SiLU(s) ~ s e^s is small, is hit.
Each case is checked twice:
  * against the oracle with the parity tolerance (rtol 2e-2, atol 1e-3 max|x|);
  * against a bound derived from the fp32 arithmetic: tanh.approx.f32 has an
    absolute error below 2^-10.9 (PTX ISA, tanh), so SiLU(s) = h + h tanh(h),
    h = s/2, is off by at most |h| 2^-10.9 before its one rounding (2^-9
    relative for bf16, 2^-12 for fp16; 2^-8 and 2^-10 are used), and SiLU'(s)
    = sig + SiLU(s)(1 - sig), sig = (1 + tanh h)/2, by at most
    2^-10.9 (1/2 + |h| + |SiLU(s)|/2) before its rounding.
Masked entries (causal) must be exactly zero.
"""
import numpy as np
import pytest
import torch

from oracle.hstu_oracle import hstu_attention_backward, hstu_attention_forward
from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import RTOL, call_kwargs, device_inputs
from tests.helpers import as_f64, oracle_params

pytestmark = pytest.mark.gpu

N = 128
TANH_ERR = 2.0 ** -10.9
ROUND = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -10}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def _workload(dtype, causal):
    return W.Workload(name=f"silu_exposed_{dtype}_{'causal' if causal else 'full'}", batch=1, nhead=1,
                      hdim_qk=N, hdim_v=N, dtype=dtype, uih_q=[N], targets=[0], context_len=[0],
                      causal=causal, alpha=1.0, attn_scale=[1.0], softmax=False)


def _scores(dtype, seed=3):
    rng = np.random.default_rng([seed, 9])
    g = rng.uniform(-12.0, 6.0, size=(N, N)).astype(np.float32)
    return torch.from_numpy(g).to(W.DTYPES[dtype])


def _eye(dtype):
    return torch.eye(N, dtype=W.DTYPES[dtype])


def _as3(t):
    return t.reshape(N, 1, N).contiguous()


def _host(t):
    return t.float().cpu().numpy().astype(np.float64).reshape(N, N)


def _silu_bound(s, ref, dtype):
    return np.abs(s) / 2 * TANH_ERR + ROUND[dtype] * np.abs(ref) + 1e-30


def _dsilu_bound(s, ref, dtype):
    a = s / (1.0 + np.exp(-s))
    return TANH_ERR * (0.5 + np.abs(s) / 2 + np.abs(a) / 2) + ROUND[dtype] * np.abs(ref) + 1e-30


def _check(got, ref, s, allowed, bound, what):
    scale = float(np.abs(ref).max())
    np.testing.assert_allclose(got, ref, rtol=RTOL, atol=1e-3 * scale, err_msg=what)
    assert np.all(got[~allowed] == 0.0), f"{what}: masked entries are not zero"
    err = np.abs(got - ref)[allowed]
    lim = bound[allowed]
    worst = int(np.argmax(err / lim))
    assert np.all(err <= lim), (f"{what}: |err| {err[worst]:.3e} above the fp32 bound {lim[worst]:.3e} "
                                f"at s = {s[allowed][worst]:.4f}")


def _allowed(causal):
    return np.tril(np.ones((N, N), dtype=bool)) if causal else np.ones((N, N), dtype=bool)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_p_element_by_element(dtype, causal):
    w = _workload(dtype, causal)
    g = _scores(dtype)
    q, k, v = _as3(g), _as3(_eye(dtype)), _as3(_eye(dtype))
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    o, _ = hstu.hstu_attn_fwd(dq, dk, dv, off_q, off_kv, tg, check=True, **call_kwargs(w))
    torch.cuda.synchronize()
    o_ref, _ = hstu_attention_forward(as_f64(q), as_f64(k), as_f64(v), w.seq_offsets_q(), None,
                                      w.num_targets(), oracle_params(w))
    s = as_f64(g)
    ref = o_ref.reshape(N, N)
    _check(_host(o), ref, s, _allowed(causal), _silu_bound(s, ref, dtype), f"{w.name} o = SiLU(s)")


def _backward(w, q, k, v, d_o):
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    got = hstu.hstu_attn_bwd(dq, dk, dv, d_o.cuda(), off_q, off_kv, tg, check=True, **call_kwargs(w))
    torch.cuda.synchronize()
    ref = hstu_attention_backward(as_f64(q), as_f64(k), as_f64(v), as_f64(d_o), w.seq_offsets_q(), None,
                                  w.num_targets(), oracle_params(w))
    return [_host(x) for x in got], [r.reshape(N, N) for r in ref]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_dq_kernel_silu_grad_element_by_element(dtype, causal):
    w = _workload(dtype, causal)
    g = _scores(dtype)
    eye = _as3(_eye(dtype))
    ones = torch.ones((N, 1, N), dtype=W.DTYPES[dtype])
    (gdq, _, _), (rdq, _, _) = _backward(w, _as3(g), eye, eye, ones)
    s = as_f64(g)
    _check(gdq, rdq, s, _allowed(causal), _dsilu_bound(s, rdq, dtype), f"{w.name} dQ = SiLU'(s)")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_dkdv_kernel_silu_and_grad_element_by_element(dtype, causal):
    w = _workload(dtype, causal)
    g = _scores(dtype)
    eye = _as3(_eye(dtype))
    kt = _as3(g.t().contiguous())   # s = alpha Q K^T = G with Q = I
    s = as_f64(g)
    allowed_t = _allowed(causal).T
    ones = torch.ones((N, 1, N), dtype=W.DTYPES[dtype])
    (_, gdk, _), (_, rdk, _) = _backward(w, eye, kt, eye, ones)
    _check(gdk, rdk, s.T, allowed_t, _dsilu_bound(s.T, rdk, dtype), f"{w.name} dK = SiLU'(s)^T")
    (_, _, gdv), (_, _, rdv) = _backward(w, eye, kt, eye, eye)
    _check(gdv, rdv, s.T, allowed_t, _silu_bound(s.T, rdv, dtype), f"{w.name} dV = SiLU(s)^T")
