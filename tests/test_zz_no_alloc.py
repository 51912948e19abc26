"""hstu_attn_fwd_static_ws (the forward on the library's fixed scratch) against
hstu_attn_fwd, both through the C ABI.

Collected last on purpose, so that in a full run it also executes after every
other GPU test has used the library; it passes run alone as well.  Each case
makes two static-scratch calls in a row (the second one finds the first one's
leftovers in the scratch) and checks that both equal the workspace entry
point's output bit for bit.
"""
import os
import re

import numpy as np
import pytest
import torch

from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import assert_parity, call_kwargs, device_inputs

pytestmark = pytest.mark.gpu


def _static_ws_bytes() -> int:
    header = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "hstu_attn.h")
    m = re.search(r"#define HSTU_STATIC_WS_BYTES \((\d+)u << (\d+)\)", open(header).read())
    assert m, "HSTU_STATIC_WS_BYTES not found in include/hstu_attn.h"
    return int(m.group(1)) << int(m.group(2))


STATIC_WS_BYTES = _static_ws_bytes()


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def _host(o):
    return o.float().cpu().numpy().astype(np.float64)


def _compare_two_calls(w, **over):
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, *w.tensors())
    kw = call_kwargs(w, **over)
    o_ws, lse_ws = hstu.hstu_attn_fwd(dq, dk, dv, off_q, off_kv, tg, check=True, **kw)
    torch.cuda.synchronize()
    ref = _host(o_ws)
    ref_lse = None if lse_ws is None else lse_ws.cpu().numpy()
    for n in range(2):
        call = hstu.HstuCall(dq, dk, dv, off_q, off_kv, tg, static_workspace=True, **kw)
        assert call.workspace_bytes <= STATIC_WS_BYTES
        call.launch_static_ws()
        assert call.check() == 0
        assert call.static_ws_ptr
        lse = None if call.lse is None else call.lse.cpu().numpy()
        assert_parity(_host(call.o), ref, w.dtype, lse, ref_lse, what=f"{w.name} static call {n + 1}")
        # The forward is deterministic (each unit has one owner, the combine
        # adds splits in a fixed order), so stale scratch from an earlier call
        # would show up as any difference at all.
        assert torch.equal(call.o, o_ws), f"{w.name} static call {n + 1}: o differs from the workspace call"
        if lse_ws is not None:
            assert torch.equal(call.lse, lse_ws), f"{w.name} static call {n + 1}: lse differs"


@pytest.mark.parametrize("cfg", ["tiny", "jagged"])
def test_static_ws_matches_workspace_entry(cfg):
    _compare_two_calls(W.CONFIGS[cfg]())


def test_static_ws_split_kv_softmax():
    w = W.random_small(3, softmax=True, cross=True, hdim=128)
    _compare_two_calls(w, num_splits=2)


def test_static_ws_large_jagged():
    _compare_two_calls(W.large_jagged(hdim=128))


def test_static_ws_rejects_oversize_before_launch():
    w = W.group_cross_splitkv(softmax=True)
    dq, dk, dv, off_q, off_kv, tg = device_inputs(w, *w.tensors())
    call = hstu.HstuCall(dq, dk, dv, off_q, off_kv, tg, static_workspace=True,
                         **call_kwargs(w, num_splits=3))
    assert call.workspace_bytes > STATIC_WS_BYTES
    sentinel = torch.full_like(call.o, 7.0)
    call.o.copy_(sentinel)
    with pytest.raises(hstu.HstuError) as e:
        call.launch_static_ws()
    assert e.value.status == 3   # HSTU_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.equal(call.o, sentinel)
