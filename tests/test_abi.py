"""The C-ABI library: it loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU.  No GPU needed."""
import ctypes
import os
import re

import pytest
import torch

from recommender_attention_gb300 import build as B
from recommender_attention_gb300 import hstu

HEADER = os.path.join(B.INCLUDE, "hstu_attn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return hstu.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hstu_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "hstu_attn_fwd" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(hstu.EXPORTS)


def test_version_strings_and_struct_layout(lib):
    assert lib.hstu_abi_version() == 6
    for s in range(6):
        assert lib.hstu_status_string(s)
    assert lib.hstu_status_string(99) == b"unknown status"
    assert lib.hstu_fwd_args_size() == ctypes.sizeof(hstu.FwdArgs)
    assert lib.hstu_bwd_args_size() == ctypes.sizeof(hstu.BwdArgs)


def _args(**kw):
    a = hstu.FwdArgs()
    a.dtype, a.batch, a.nhead, a.hdim_qk, a.hdim_v = 1, 4, 2, 128, 128
    a.total_q = a.total_kv = 1000
    a.max_seqlen_q = a.max_seqlen_kv = 300
    a.causal, a.num_groups = 1, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _ws(lib, a):
    n = ctypes.c_size_t(0)
    st = lib.hstu_attn_fwd_workspace_size(ctypes.byref(a), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("field,value,status", [
    ("hdim_qk", 96, 2), ("hdim_v", 64, 2), ("dtype", 7, 2), ("batch", 0, 1), ("nhead", 0, 1),
    ("num_groups", 3, 1), ("num_groups", 0, 1), ("num_splits", 17, 2), ("num_splits", -1, 1),
    ("q_row_stride", 100, 1), ("q_row_stride", 3, 1), ("total_kv", 999, 1), ("alpha", -1.0, 1),
    ("causal", 2, 1), ("max_seqlen_q", -5, 1),
    ("kv_targets", 2, 1), ("kv_targets", 1, 1),    # target keys on the key side need cross-attention
    ("cta_pairs", 2, 1), ("cta_pairs", -2, 1), ("cta_pairs", 1, 0), ("cta_pairs", -1, 0)])
def test_host_validation(lib, field, value, status):
    st, _ = _ws(lib, _args(**{field: value}))
    assert st == status


@pytest.mark.parametrize("dqk,dv,status", [(96, 96, 0), (96, 64, 0), (64, 64, 0), (256, 256, 0),
                                            (96, 128, 2), (128, 64, 2), (64, 96, 2), (32, 32, 2)])
def test_head_dimension_pairs(lib, dqk, dv, status):
    st, _ = _ws(lib, _args(hdim_qk=dqk, hdim_v=dv))
    assert st == status


def test_group_array_validation(lib):
    g = (ctypes.c_int32 * 2)(5, -1)
    a = _args(num_groups=2, local_len=ctypes.cast(g, ctypes.c_void_p))
    assert _ws(lib, a)[0] == 1
    big = _args(batch=512, num_groups=512)
    assert _ws(lib, big)[0] == 2


def test_workspace_grows_with_splits(lib):
    st1, n1 = _ws(lib, _args(num_splits=1))
    st4, n4 = _ws(lib, _args(num_splits=4))
    assert st1 == st4 == 0
    # fp32 partials: 4 splits x 1000 rows x 2 heads x 128 + row stats
    assert n4 - n1 >= 4 * 1000 * 2 * 128 * 4


def test_forward_rejects_before_launch(lib):
    a = _args()
    # missing pointers / workspace are host-side errors: nothing is launched
    assert lib.hstu_attn_fwd(ctypes.byref(a), None) == 1
    a.q = a.k = a.v = a.o = a.seq_offsets_q = 4096
    assert lib.hstu_attn_fwd(ctypes.byref(a), None) == 3
    a.workspace = 4096 + 8
    assert lib.hstu_attn_fwd(ctypes.byref(a), None) == 3
    a.q = 4096 + 2
    a.workspace = 8192
    assert lib.hstu_attn_fwd(ctypes.byref(a), None) == 1


def test_rab_host_validation(lib):
    t = (ctypes.c_float * 8)()
    ok = _args(rab_pos=ctypes.cast(t, ctypes.c_void_p), rab_pos_buckets=4)
    assert _ws(lib, ok)[0] == 0
    assert _ws(lib, _args(rab_pos=ctypes.cast(t, ctypes.c_void_p), rab_pos_buckets=0))[0] == 1
    assert _ws(lib, _args(rab_pos=ctypes.cast(t, ctypes.c_void_p), rab_pos_buckets=257))[0] == 1
    # the time term needs timestamps (and key timestamps for cross-attention)
    assert _ws(lib, _args(rab_time=ctypes.cast(t, ctypes.c_void_p)))[0] == 1
    assert _ws(lib, _args(rab_time=ctypes.cast(t, ctypes.c_void_p), timestamps_q=4096))[0] == 0
    assert _ws(lib, _args(rab_time=ctypes.cast(t, ctypes.c_void_p), timestamps_q=4096,
                          seq_offsets_kv=4096))[0] == 1
    # the bias works at every head-dimension pair the forward supports, and no other
    for dqk, dv, st in ((64, 64, 0), (96, 96, 0), (96, 64, 0), (128, 128, 0), (256, 256, 0), (128, 64, 2)):
        assert _ws(lib, _args(hdim_qk=dqk, hdim_v=dv, rab_pos=ctypes.cast(t, ctypes.c_void_p),
                              rab_pos_buckets=4))[0] == st
    # the backward takes the same bias fields and checks
    b = _bwd()
    b.fwd.rab_pos = ctypes.cast(t, ctypes.c_void_p)
    b.fwd.rab_pos_buckets = 4
    assert _bwd_ws(lib, b)[0] == 0
    b.fwd.rab_pos_buckets = 300
    assert _bwd_ws(lib, b)[0] == 1
    # ... at the backward's head dimensions (no 256)
    b.fwd.rab_pos_buckets = 4
    for dqk, dv, st in ((96, 96, 0), (96, 64, 0), (256, 256, 2)):
        b.fwd.hdim_qk, b.fwd.hdim_v = dqk, dv
        assert _bwd_ws(lib, b)[0] == st


def _bwd(**kw):
    b = hstu.BwdArgs()
    b.fwd = _args(**{k: v for k, v in kw.items() if k in dict(hstu.FwdArgs._fields_)})
    for k, v in kw.items():
        if k in dict(hstu.BwdArgs._fields_):
            setattr(b, k, v)
    return b


def _bwd_ws(lib, b):
    n = ctypes.c_size_t(0)
    st = lib.hstu_attn_bwd_workspace_size(ctypes.byref(b), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("kw,status", [
    ({}, 0), ({"hdim_qk": 64, "hdim_v": 64}, 0), ({"num_splits": 5}, 0),   # splits are ignored
    ({"hdim_qk": 96, "hdim_v": 96}, 0), ({"hdim_qk": 256, "hdim_v": 256}, 2),
    ({"hdim_qk": 96, "hdim_v": 64}, 0), ({"dtype": 7}, 2), ({"batch": 0}, 1),
    # dv / dO strides are checked against nhead * hdim_v (128 here), dq / dk against nhead * hdim_qk (192)
    ({"hdim_qk": 96, "hdim_v": 64, "dv_row_stride": 136}, 0), ({"hdim_qk": 96, "hdim_v": 64, "do_row_stride": 120}, 1),
    ({"hdim_qk": 96, "hdim_v": 64, "dq_row_stride": 136}, 1),
    ({"do_row_stride": 100}, 1), ({"dk_row_stride": 258}, 1), ({"dv_row_stride": 260}, 1)])
def test_backward_host_validation(lib, kw, status):
    assert _bwd_ws(lib, _bwd(**kw))[0] == status


def test_backward_workspace_holds_row_sums_in_softmax_mode(lib):
    st0, n0 = _bwd_ws(lib, _bwd(softmax=0))
    st1, n1 = _bwd_ws(lib, _bwd(softmax=1))
    assert st0 == st1 == 0
    assert n1 - n0 >= 2 * 1000 * 4            # delta: [H, total_q] fp32
    stf, nf = _ws(lib, _args(num_splits=1))
    assert n0 > nf                            # plus query-tile records and key-tile units


def test_backward_rejects_before_launch(lib):
    b = _bwd()
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1
    b.fwd.q = b.fwd.k = b.fwd.v = b.fwd.seq_offsets_q = 4096
    b.d_o = b.dq = b.dk = b.dv = 8192
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 3     # no workspace
    b.fwd.workspace = 4096 + 16
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 3     # misaligned workspace
    b.fwd.workspace = 1 << 20
    b.dk = 8192 + 4
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1     # misaligned gradient
    b.dk = 8192
    b.fwd.softmax = 1
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1     # softmax needs o and lse


def test_backward_rab_gradients_need_their_table(lib):
    """A bias-table gradient is only computed for a table the call uses (the
    time table with its timestamps); otherwise the call returns
    HSTU_ERR_INVALID_ARG before anything else is checked or launched."""
    b = _bwd()
    b.fwd.q = b.fwd.k = b.fwd.v = b.fwd.seq_offsets_q = 4096
    b.d_o = b.dq = b.dk = b.dv = 8192
    b.d_rab_time = 1 << 16
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1          # no time table
    b.fwd.rab_time = 1 << 17
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1          # no timestamps
    b.fwd.timestamps_q = 1 << 18
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 3          # accepted; then: no workspace
    b.d_rab_pos = 1 << 19
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1          # no positional table
    b.fwd.rab_pos, b.fwd.rab_pos_buckets = 1 << 20, 16
    b.d_rab_pos = (1 << 19) + 2
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 1          # misaligned
    b.d_rab_pos = 1 << 19
    assert lib.hstu_attn_bwd(ctypes.byref(b), None) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(hstu, "_LIB", None)
    monkeypatch.setattr(hstu, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        hstu.load_library()
