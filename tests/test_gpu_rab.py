"""Forward with the relative attention bias ("From transformer parallelism to
HSTU", sections 2.4 and 3.5) through the C ABI, against the fp64 oracle on the
same seeded timestamps and tables (``Workload.rab_inputs``), element by
element, with the forward's tolerances.  The kernel keeps the bias weights in
fp32 and adds them to alpha * <q, k> in fp32 before the SiLU / softmax
arithmetic it shares with the unbiased path."""
import numpy as np
import pytest
import torch

from oracle.hstu_oracle import hstu_attention_forward_rows
from recommender_attention_gb300 import hstu
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import assert_parity, gpu_forward, rab_kwargs
from tests.helpers import as_f64, oracle_forward, oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    hstu.load_library()


def check_rab(w, use_time=True, use_pos=True, **over):
    q, k, v = w.tensors()
    rab = w.rab_inputs()
    o, lse = gpu_forward(w, q, k, v, **rab_kwargs(rab, use_time, use_pos), **over)
    o_ref, lse_ref = oracle_forward(w, q, k, v, rab, use_time, use_pos)
    assert_parity(o, o_ref, w.dtype, lse, lse_ref, what=f"{w.name} rab")


@pytest.mark.parametrize("cfg", ["tiny", "jagged", "batched"])
@pytest.mark.parametrize("softmax", [False, True])
def test_small_configs_rab(cfg, softmax):
    check_rab(W.CONFIGS[cfg]().with_(softmax=softmax, rab_pos_buckets=64))


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_rab(seed):
    softmax = seed % 2 == 1
    hdim = [64, 128][(seed // 2) % 2]
    w = W.random_small(seed, hdim=hdim, softmax=softmax, dtype="bf16" if seed % 3 else "fp16",
                       kv_targets=seed % 6 == 5)
    w = w.with_(rab_pos_buckets=[1, 7, 64, 256][seed % 4])
    check_rab(w, num_splits=[1, 2, 0][seed % 3])


@pytest.mark.parametrize("dqk,dv", [(96, 96), (96, 64), (256, 256)])
@pytest.mark.parametrize("softmax", [False, True])
def test_rab_other_head_dims(dqk, dv, softmax):
    """The bias at hdim 96, 96/64 and 256: the jagged validation case, and a
    random case with a cross-attention key side and split-KV."""
    check_rab(W.jagged_readme().with_(hdim_qk=dqk, hdim_v=dv, softmax=softmax, rab_pos_buckets=64))
    w = W.random_small(300 + dqk + dv, hdim=dqk, hdim_v=dv, softmax=softmax, dtype="fp16", cross=True)
    check_rab(w.with_(rab_pos_buckets=9), num_splits=2)


@pytest.mark.parametrize("use_time,use_pos", [(True, False), (False, True)])
@pytest.mark.parametrize("softmax", [False, True])
def test_rab_one_term(use_time, use_pos, softmax):
    check_rab(W.jagged_readme().with_(softmax=softmax, rab_pos_buckets=32), use_time, use_pos)


@pytest.mark.parametrize("softmax", [False, True])
def test_mfalcon_rab(softmax):
    check_rab(W.mfalcon(batch=3, candidates=200, softmax=softmax, history=(300, 900)).with_(rab_pos_buckets=128))


@pytest.mark.parametrize("softmax", [False, True])
def test_group_cross_rab_splitkv(softmax):
    check_rab(W.group_cross_splitkv(softmax=softmax, batch=8).with_(rab_pos_buckets=64), num_splits=3)


@pytest.mark.parametrize("softmax", [False, True])
def test_large_jagged_rab_sampled(softmax):
    """The large jagged workload at full size with a bias; the oracle on sampled rows."""
    w = W.large_jagged(hdim=128).with_(softmax=softmax, rab_pos_buckets=128)
    q, k, v = w.tensors()
    rab = w.rab_inputs()
    o, lse = gpu_forward(w, q, k, v, **rab_kwargs(rab))
    off = w.seq_offsets_q()
    p = oracle_params(w, rab)
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    rng = np.random.default_rng(4)
    for b in rng.choice(w.batch, size=3, replace=False).tolist():
        L = int(off[b + 1] - off[b])
        rows = sorted(set([0, 5, 6, 127, 128, L - 1] + rng.integers(0, L, size=16).tolist()))
        for h in range(w.nhead):
            ob, lb = hstu_attention_forward_rows(qd, kd, vd, off, None, w.num_targets(), p, b, h, rows)
            assert_parity(o[off[b] + np.array(rows), h], ob, w.dtype,
                          None if lse is None else lse[h, off[b] + np.array(rows)], lb, what=f"b{b} h{h}")
