"""Calls captured as CUDA graphs (``HstuCall.graph`` / ``HstuBwdCall.graph``).

A replay reruns the call's kernels on the same buffers without the host side
of a call.  The forward and the dQ, dK, dV gradients are deterministic (each
output element has one owner, and the split-KV combine adds the splits in a
fixed order), so a replay must reproduce a direct launch bit for bit, and
after an in-place update of the inputs it must match a direct launch on the
updated inputs.  Covered: the in-kernel schedule (batch <= 128) and the
scheduler kernel (larger batches), split-KV with the combine kernel, softmax
with LSE, and the backward.
"""
import pytest
import torch

from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import call_kwargs, device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def _many_short(batch=150):
    """More sequences than the in-kernel schedule takes: the scheduler kernel runs."""
    return W.Workload(name="many_short", batch=batch, nhead=2, hdim_qk=64, hdim_v=64, dtype="bf16",
                      uih_q=[(37 * b) % 200 + 1 for b in range(batch)], targets=[b % 5 for b in range(batch)],
                      context_len=[3], causal=True, seed=13)


def _forward_graph_case(w, **over):
    q, k, v = w.tensors()
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    call = hstu.HstuCall(dq, dk, dv, off_q, off_kv, tg, **call_kwargs(w, **over))
    call.launch()
    call.check()
    o_ref = call.o.clone()
    lse_ref = None if call.lse is None else call.lse.clone()
    g = call.graph()
    call.o.fill_(float("nan"))
    if call.lse is not None:
        call.lse.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert call.check() == 0
    assert torch.equal(call.o, o_ref), f"{w.name}: replay differs from a direct launch"
    if lse_ref is not None:
        assert torch.equal(call.lse, lse_ref), f"{w.name}: replayed LSE differs"
    # the graph reads its input buffers again on every replay
    dq.mul_(0.5)
    dv.mul_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    o_graph = call.o.clone()
    call.launch()
    call.check()
    assert torch.equal(o_graph, call.o), f"{w.name}: replay after an input update differs from a launch"
    assert not torch.equal(o_graph, o_ref)


@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("cfg", ["tiny", "jagged"])
def test_forward_graph_in_kernel_schedule(cfg, softmax):
    _forward_graph_case(W.CONFIGS[cfg]().with_(softmax=softmax))


@pytest.mark.parametrize("softmax", [False, True])
def test_forward_graph_splitkv_combine(softmax):
    _forward_graph_case(W.group_cross_splitkv(softmax=softmax, batch=8), num_splits=3)


def test_forward_graph_scheduler_kernel():
    _forward_graph_case(_many_short())


@pytest.mark.parametrize("softmax", [False, True])
def test_backward_graph(softmax):
    w = W.jagged_readme().with_(softmax=softmax)
    q, k, v = w.tensors()
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, q, k, v)
    kw = call_kwargs(w)
    o = lse = None
    if softmax:
        o, lse = hstu.hstu_attn_fwd(dq, dk, dv, off_q, off_kv, tg, check=True, **kw)
    call = hstu.HstuBwdCall(dq, dk, dv, w.grad_output().cuda(), off_q, off_kv, tg, o=o, lse=lse, **kw)
    call.launch()
    call.check()
    ref = [t.clone() for t in (call.dq, call.dk, call.dv)]
    g = call.graph()
    for t in (call.dq, call.dk, call.dv):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert call.check() == 0
    for name, got, want in zip(("dq", "dk", "dv"), (call.dq, call.dk, call.dv), ref):
        assert torch.equal(got, want), f"{w.name}: replayed {name} differs from a direct launch"
