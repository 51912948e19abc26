"""The two hdim-128 forward kernels, each against the fp64 oracle on the same inputs.

At hdim 128 without a bias the library has two forward kernels: CTA pairs
(two query tiles of one sequence and head on the two SMs of a TPC, one
256-row tcgen05 product of cta_group::2, each SM loading half of every key and
value tile) and single CTAs (one query tile per SM, the automatic choice).
Every case here runs through both (``cta_pairs`` 1 and -1), the pair kernel
also on workloads whose sequences hold a single query tile.  The cases cover
what is particular to a pair: sequences of an odd number of tiles (the first
tile runs with an empty partner), the context rows moved onto the last tile,
a pair whose two tiles see different key tiles (the union runs, and the tiles
outside one tile's own set must contribute nothing), split-KV partials,
M-FALCON and random mask parameters.
"""
import pytest
import torch

from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import assert_parity, gpu_forward
from tests.helpers import oracle_forward

pytestmark = pytest.mark.gpu

KERNELS = {"pairs": 1, "single": -1}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from recommender_attention_gb300 import hstu
    hstu.load_library()


def check(w, kernel, **over):
    q, k, v = w.tensors()
    o_ref, lse_ref = oracle_forward(w, q, k, v)
    o, lse = gpu_forward(w, q, k, v, cta_pairs=KERNELS[kernel], **over)
    assert_parity(o, o_ref, w.dtype, lse, lse_ref, what=f"{w.name} ({kernel})")


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("softmax", [False, True])
def test_jagged(kernel, softmax):
    check(W.jagged_readme().with_(softmax=softmax), kernel)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_odd_and_even_tile_counts(kernel, softmax, dtype):
    """Sequences of 1 .. 4 query tiles, ragged and whole, with context rows
    (moved onto the last tile where they fit) and targets."""
    w = W.Workload(name=f"tiles_{dtype}", batch=9, nhead=2, hdim_qk=128, hdim_v=128, dtype=dtype,
                   uih_q=[1, 100, 115, 116, 240, 243, 360, 370, 490], targets=[0, 3, 7, 6, 9, 4, 2, 10, 12],
                   context_len=[6], causal=True, softmax=softmax, dist="normal", seed=41)
    check(w, kernel)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("softmax", [False, True])
def test_local_window_and_minfull(kernel, softmax):
    """A local window narrower than a tile and a min-full tail: the two tiles
    of a pair see different, partly disjoint key tiles."""
    w = W.Workload(name="window", batch=4, nhead=2, hdim_qk=128, hdim_v=128, dtype="bf16",
                   uih_q=[700, 515, 389, 260], targets=[5, 16, 1, 0], context_len=[3], local_len=[40],
                   minfull_len=[70], causal=True, softmax=softmax, seed=43)
    check(w, kernel)
    check(w.with_(causal=False), kernel)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_group_cross_splitkv(kernel, softmax, splits):
    check(W.group_cross_splitkv(softmax=softmax, batch=8), kernel, num_splits=splits)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("softmax", [False, True])
def test_mfalcon(kernel, softmax):
    check(W.mfalcon(batch=4, candidates=200, softmax=softmax, history=(300, 1500)), kernel, num_splits=2)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_window_wider_than_sequence_and_single_row(kernel):
    w = W.Workload(name="edge_wide", batch=3, nhead=2, hdim_qk=128, hdim_v=128, dtype="bf16",
                   uih_q=[1, 129, 257], targets=[0, 1, 2], context_len=[1], local_len=[10000],
                   minfull_len=[2], causal=True, seed=7)
    check(w, kernel)
    check(w.with_(causal=False, softmax=True), kernel)


@pytest.mark.parametrize("kernel", list(KERNELS))
def test_empty_sequences(kernel):
    w = W.Workload(name="edge_empty", batch=4, nhead=2, hdim_qk=128, hdim_v=128, dtype="fp16",
                   uih_q=[0, 300, 0, 3], targets=[0, 0, 0, 0], context_len=[0], causal=True, seed=3,
                   has_targets=False)
    check(w, kernel)


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("kernel", list(KERNELS))
def test_fuzz(seed, kernel):
    w = W.random_small(200 + seed, dtype="bf16" if seed % 2 else "fp16", hdim=128, softmax=bool(seed % 3 == 1),
                       max_uih=500, kv_targets=seed % 4 == 3)
    check(w, kernel, num_splits=[1, 2, 0][seed % 3])
