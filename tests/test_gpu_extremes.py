"""Size extremes through the C ABI against the fp64 oracle:
- more sequences than the scheduler keeps in shared memory (its scratch
  moves to the workspace, and sequences keep their input order), forward and
  backward;
- one long sequence: 32 000 tokens forward on sampled rows (250+ query tiles
  per head), and 8 100 tokens through the backward with the whole-sequence
  oracle."""
import numpy as np
import pytest
import torch

from oracle.hstu_oracle import hstu_attention_backward, hstu_attention_forward_rows
from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import assert_parity, gpu_forward
from tests.helpers import as_f64, oracle_forward, oracle_params
from tests.test_gpu_backward import check_backward

pytestmark = pytest.mark.gpu

SCHEDULER_SMEM_BATCH = 2048   # batches above this use the workspace scratch


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def many_short(softmax: bool) -> W.Workload:
    rng = np.random.default_rng(77)
    batch = SCHEDULER_SMEM_BATCH + 952
    uih = [int(x) for x in rng.integers(0, 50, size=batch)]
    tg = [int(x) for x in rng.integers(0, 4, size=batch)]
    return W.Workload(name="many_short", batch=batch, nhead=2, hdim_qk=64, hdim_v=64, dtype="bf16",
                      uih_q=uih, targets=tg, context_len=[2], local_len=[7], minfull_len=[3], causal=True,
                      softmax=softmax, dist="normal", seed=77)


@pytest.mark.parametrize("softmax", [False, True])
def test_many_short_sequences_forward(softmax):
    w = many_short(softmax)
    q, k, v = w.tensors()
    o, lse = gpu_forward(w, q, k, v)
    o_ref, lse_ref = oracle_forward(w, q, k, v)
    assert_parity(o, o_ref, w.dtype, lse, lse_ref, what=w.name)


def test_many_short_sequences_backward():
    check_backward(many_short(False))


@pytest.mark.parametrize("softmax", [False, True])
def test_one_long_sequence_forward_sampled(softmax):
    w = W.Workload(name="long_one", batch=1, nhead=2, hdim_qk=128, hdim_v=128, dtype="bf16",
                   uih_q=[31_954], targets=[40], context_len=[6], causal=True, softmax=softmax,
                   dist="normal", seed=31)
    q, k, v = w.tensors()
    o, lse = gpu_forward(w, q, k, v)
    off = w.seq_offsets_q()
    L = int(off[1])
    p = oracle_params(w)
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    rng = np.random.default_rng(3)
    rows = sorted(set([0, 5, 6, 127, 128, 16_383, 16_384, L - 41, L - 40, L - 1] +
                      rng.integers(0, L, size=24).tolist()))
    for h in range(w.nhead):
        ob, lb = hstu_attention_forward_rows(qd, kd, vd, off, None, w.num_targets(), p, 0, h, rows)
        assert_parity(o[np.array(rows), h], ob, w.dtype, None if lse is None else lse[h, np.array(rows)], lb,
                      what=f"long h{h}")


def test_long_sequence_backward():
    w = W.Workload(name="long_bwd", batch=1, nhead=1, hdim_qk=128, hdim_v=128, dtype="bf16",
                   uih_q=[8_064], targets=[30], context_len=[6], causal=True, dist="normal", seed=32)
    check_backward(w)
