"""The seeded input generators (recommender_attention_gb300/workloads.py)
against the recipe they state: independent streams per input, the jagged
layout, the large workload's shape, and the relative attention bias inputs
(sorted key timestamps whose gaps reach every time bucket of "From transformer
parallelism to HSTU", section 3.5; query rows at their key-coordinate
position).  CPU only."""
import numpy as np
import torch

from oracle.hstu_oracle import time_gap_bucket
from recommender_attention_gb300 import workloads as W


def test_values_are_deterministic_and_streams_independent():
    w = W.random_small(3, hdim=64, softmax=True)
    a, b = w.tensors(), w.tensors()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert torch.equal(w.grad_output(), w.grad_output())
    # the bias draws come from their own stream: q, k, v do not move with them
    for x, y in zip(a, w.with_(rab_pos_buckets=16).tensors()):
        assert torch.equal(x, y)
    q, k, v = a
    assert not torch.equal(q[:, :, : w.hdim_v], w.grad_output())
    assert q.dtype == W.DTYPES[w.dtype] and q.shape == (w.total_q, w.nhead, w.hdim_qk)
    assert v.shape == (w.total_kv, w.nhead, w.hdim_v)


def test_uniform_values_lie_in_the_stated_range():
    w = W.tiny_batched()
    for x in w.tensors():
        xf = x.float()
        assert float(xf.min()) >= -1.0 and float(xf.max()) <= 1.0
        assert x.dtype == torch.float16


def test_jagged_layout():
    w = W.group_cross_splitkv()
    oq, okv = w.seq_offsets_q(), w.seq_offsets_kv()
    assert oq[0] == 0 and okv[0] == 0
    np.testing.assert_array_equal(np.diff(oq), w.lengths_q())
    np.testing.assert_array_equal(np.diff(okv), w.lengths_kv())
    for b in range(w.batch):
        g = w.group(b)
        assert w.lengths_q()[b] == w.context_len[g] + w.uih_q[b] + w.targets[b]
        assert w.lengths_kv()[b] == w.context_len[g] + w.uih_kv[b]
    assert [w.group(b) for b in range(w.batch)] == [b // 8 for b in range(32)]


def test_large_workload_shape():
    w = W.large_jagged(hdim=128)
    assert (w.batch, w.nhead, w.hdim_qk, w.hdim_v, w.dtype) == (64, 4, 128, 128, "bf16")
    assert all(1024 <= u <= 4096 for u in w.uih_q) and all(1 <= t <= 32 for t in w.targets)
    assert w.total_q == 172291          # the token count every measurement quotes
    assert w.context_len == [6] and w.local_len == [0] and w.minfull_len == [0] and w.causal
    # hdim 256 repeats the same sequences
    assert W.large_jagged(hdim=256).uih_q == w.uih_q


def test_bias_inputs_recipe():
    w = W.large_jagged(hdim=128, batch=8).with_(rab_pos_buckets=128)
    ts_q, ts_kv, rab_time, rab_pos = w.rab_inputs()
    assert ts_kv is None                         # self-attention reuses the query side's
    assert ts_q.dtype == np.int64 and ts_q.shape == (w.total_q,)
    assert rab_time.shape == (w.nhead, 11) and rab_pos.shape == (w.nhead, 128)
    off = w.seq_offsets_q()
    buckets = set()
    for b in range(w.batch):
        t = ts_q[off[b]:off[b + 1]]
        assert 1_700_000_000 <= t[0] < 1_710_000_000
        gaps = np.diff(t)
        assert (gaps >= 0).all()                 # keys in time order
        buckets |= {time_gap_bucket(int(g)) for g in gaps}
    assert buckets == set(range(11))             # every time bucket occurs


def test_bias_inputs_cross_attention_rows_follow_their_key_position():
    w = W.random_small(4, cross=True).with_(rab_pos_buckets=8)
    ts_q, ts_kv, _, _ = w.rab_inputs()
    assert ts_kv is not None and ts_kv.shape == (w.total_kv,)
    oq, okv = w.seq_offsets_q(), w.seq_offsets_kv()
    for b in range(w.batch):
        c = w.context_len[w.group(b)]
        u, ukv = w.uih_q[b], w.uih_kv[b]
        lkv = int(okv[b + 1] - okv[b])
        for i in range(int(oq[b + 1] - oq[b])):
            pos = i if i < c else i + (ukv - u)
            if 0 <= pos < lkv:
                assert ts_q[oq[b] + i] == ts_kv[okv[b] + pos]
