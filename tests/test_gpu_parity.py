"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every test here needs a GB300 and the built library (``-m gpu``).
"""
import numpy as np
import pytest
import torch

from oracle.hstu_oracle import (allowed_pair_count,
                                hstu_attention_forward_rows)
from recommender_attention_gb300 import workloads as W
from tests.gpu_helpers import assert_parity, gpu_call, gpu_forward
from tests.helpers import as_f64, kernel_executed_tiles, oracle_forward, oracle_forward_parallel, oracle_params

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from recommender_attention_gb300 import hstu
    hstu.load_library()


def check_full(w, **over):
    q, k, v = w.tensors()
    o_ref, lse_ref = oracle_forward(w, q, k, v)
    o, lse = gpu_forward(w, q, k, v, **over)
    assert_parity(o, o_ref, w.dtype, lse, lse_ref, what=w.name)


# ---------------------------------------------------------------- the configs
@pytest.mark.parametrize("cfg", ["tiny", "jagged", "batched"])
def test_small_configs_full_parity(cfg):
    check_full(W.CONFIGS[cfg]())


@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_group_cross_splitkv_parity(softmax, splits):
    w = W.group_cross_splitkv(softmax=softmax)
    check_full(w, num_splits=splits)


def test_softmax_rescale_in_some_rows_of_a_warp():
    """Softmax rows whose running max jumps by far more than 2^8 on the second
    key tile next to rows whose max stays put, in every warp: the kernel's O
    rescale is needed by some rows of a warp and not by the others.  Keys of
    tile 0 are zero (every score 0); keys of tile 1 are large; odd query rows
    are large, even rows zero."""
    w = W.Workload(name="rescale_mix", batch=1, nhead=2, hdim_qk=64, hdim_v=64, dtype="bf16",
                   uih_q=[256], targets=[0], context_len=[0], causal=False, softmax=True,
                   alpha=1.0 / 8, seed=17)
    rng = np.random.default_rng([17, 5])
    q = rng.standard_normal((256, 2, 64)).astype(np.float32) * 4
    q[0::2] = 0.0
    k = rng.standard_normal((256, 2, 64)).astype(np.float32) * 4
    k[:128] = 0.0
    v = rng.standard_normal((256, 2, 64)).astype(np.float32)
    q, k, v = (torch.from_numpy(x).to(torch.bfloat16) for x in (q, k, v))
    o, lse = gpu_forward(w, q, k, v)
    o_ref, lse_ref = oracle_forward(w, q, k, v)
    assert_parity(o, o_ref, w.dtype, lse, lse_ref, what=w.name)


@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("splits", [0, 5, 16])
def test_splitkv_runs_of_empty_split_units(softmax, splits):
    """Local-window groups give query tiles of 2-3 key tiles: with 5 or 16
    splits (and the automatic choice on 8 sequences) most of their split
    units are empty, several in a row, between non-empty ones."""
    w = W.group_cross_splitkv(softmax=softmax, batch=8)
    check_full(w, num_splits=splits)


@pytest.mark.parametrize("hdim", [128, 256])
def test_large_jagged_sampled_parity(hdim):
    """Full-size large jagged workload, same launch as the bench; oracle on sampled rows."""
    w = W.large_jagged(hdim=hdim)
    q, k, v = w.tensors()
    o, _ = gpu_forward(w, q, k, v)
    off = w.seq_offsets_q()
    rng = np.random.default_rng(0)
    p = oracle_params(w)
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    for b in rng.choice(w.batch, size=4, replace=False).tolist() + [int(np.argmax(w.lengths_q()))]:
        L = int(off[b + 1] - off[b])
        # first rows (context), a ragged last tile, tile edges and random rows
        rows = sorted(set([0, 5, 6, 127, 128, L - 1, L - 2, (L // 128) * 128 - 1] +
                          rng.integers(0, L, size=24).tolist()))
        rows = [r for r in rows if 0 <= r < L]
        for h in range(w.nhead):
            ob, _ = hstu_attention_forward_rows(qd, kd, vd, off, None, w.num_targets(), p, b, h, rows)
            assert_parity(o[off[b] + np.array(rows), h], ob, w.dtype, what=f"b{b} h{h}")


def test_large_jagged_whole_output_parity():
    """The headline workload (hdim 128, SiLU) exactly as the bench launches it,
    every row of every head against the oracle (composable_kernel README,
    "Test / Verify": -v=1 checks the whole output against the host reference).
    The oracle runs after the GPU call, on a pool of spawned processes."""
    w = W.large_jagged(hdim=128)
    q, k, v = w.tensors()
    o, _ = gpu_forward(w, q, k, v)
    o_ref, _ = oracle_forward_parallel(w, q, k, v)
    assert_parity(o, o_ref, w.dtype, what=f"{w.name}: all {w.total_q} rows x {w.nhead} heads")


# ---------------------------------------------------------------- fuzz
@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("softmax", [False, True])
def test_fuzz_small_parity(seed, softmax):
    hdim = [64, 128, 256][seed % 3]
    dtype = "bf16" if seed % 2 else "fp16"
    w = W.random_small(seed, dtype=dtype, hdim=hdim, softmax=softmax)
    splits = [1, 2, 0][seed % 3]
    check_full(w, num_splits=splits)


# ---------------------------------------------------------------- head dimension 96, and 96/64
@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("dv", [96, 64])
def test_hdim96_jagged_parity(softmax, dv):
    w = W.jagged_readme().with_(hdim_qk=96, hdim_v=dv, softmax=softmax)
    check_full(w)


@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("dv", [96, 64])
def test_hdim96_group_cross_splitkv_parity(softmax, dv):
    w = W.group_cross_splitkv(softmax=softmax, batch=8).with_(hdim_qk=96, hdim_v=dv)
    check_full(w, num_splits=3)


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_hdim96_parity(seed):
    w = W.random_small(200 + seed, dtype="bf16" if seed % 2 else "fp16", hdim=96,
                       hdim_v=[96, 64][seed % 2], softmax=seed % 3 == 1, kv_targets=seed == 5)
    check_full(w, num_splits=[1, 2, 0][seed % 3])


def test_large_jagged_hdim96_sampled_parity():
    w = W.large_jagged(hdim=96, batch=16)
    q, k, v = w.tensors()
    o, _ = gpu_forward(w, q, k, v)
    off = w.seq_offsets_q()
    p = oracle_params(w)
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    rng = np.random.default_rng(1)
    for b in rng.choice(w.batch, size=3, replace=False).tolist():
        L = int(off[b + 1] - off[b])
        rows = sorted(set([0, 5, 6, 127, 128, L - 1] + rng.integers(0, L, size=16).tolist()))
        for h in range(w.nhead):
            ob, _ = hstu_attention_forward_rows(qd, kd, vd, off, None, w.num_targets(), p, b, h, rows)
            assert_parity(o[off[b] + np.array(rows), h], ob, w.dtype, what=f"b{b} h{h}")


# ---------------------------------------------------------------- M-FALCON (keys end with the targets')
@pytest.mark.parametrize("softmax", [False, True])
@pytest.mark.parametrize("splits", [1, 3])
def test_mfalcon_parity(softmax, splits):
    w = W.mfalcon(batch=4, candidates=130, softmax=softmax, history=(300, 1500))
    check_full(w, num_splits=splits)


def test_mfalcon_equals_full_sequence_target_rows_on_gpu():
    """Through the kernel: the candidates scored against the cached history keys
    equal the context and target rows of the whole-sequence self-attention."""
    full = W.Workload(name="mf_full", batch=2, nhead=2, hdim_qk=128, hdim_v=128, dtype="bf16",
                      uih_q=[700, 333], targets=[64, 129], context_len=[6], attn_scale=[0.001],
                      causal=True, dist="normal", seed=31)
    q, k, v = full.tensors()
    o_full, _ = gpu_forward(full, q, k, v)
    off = full.seq_offsets_q()
    rows = np.concatenate([np.r_[off[b]:off[b] + 6, off[b] + 6 + full.uih_q[b]:off[b + 1]]
                           for b in range(full.batch)])
    mf = full.with_(name="mf", uih_q=[0, 0], uih_kv=list(full.uih_q), kv_targets=True)
    q_mf = q[torch.from_numpy(rows)]
    o_mf, _ = gpu_forward(mf, q_mf, k, v)
    np.testing.assert_allclose(o_mf, o_full[rows], rtol=2e-2, atol=2e-2 * np.abs(o_full).max())


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_kv_targets_parity(seed):
    w = W.random_small(100 + seed, dtype="bf16" if seed % 2 else "fp16", hdim=[64, 128, 256][seed % 3],
                       softmax=bool(seed % 2), kv_targets=True)
    check_full(w, num_splits=[1, 2, 0][seed % 3])


# ---------------------------------------------------------------- edge cases
def test_edge_empty_sequences_and_no_targets_array():
    w = W.Workload(name="edge_empty", batch=4, nhead=2, hdim_qk=64, hdim_v=64, dtype="bf16",
                   uih_q=[0, 200, 0, 3], targets=[0, 0, 0, 0], context_len=[0], local_len=[0],
                   minfull_len=[0], causal=True, seed=3, has_targets=False)
    check_full(w)


def test_edge_rows_without_keys():
    # cross-attention, no context, far fewer key UIH than query UIH: early rows see nothing
    w = W.Workload(name="edge_nokeys", batch=2, nhead=1, hdim_qk=64, hdim_v=64, dtype="fp16",
                   uih_q=[300, 50], uih_kv=[40, 0], targets=[3, 2], context_len=[0],
                   local_len=[0], minfull_len=[0], causal=True, seed=5)
    check_full(w)
    check_full(w.with_(softmax=True))


def test_edge_window_wider_than_sequence_and_single_row():
    w = W.Workload(name="edge_wide", batch=3, nhead=2, hdim_qk=128, hdim_v=128, dtype="bf16",
                   uih_q=[1, 129, 257], targets=[0, 1, 2], context_len=[1], local_len=[10000],
                   minfull_len=[2], causal=True, seed=7)
    check_full(w)
    check_full(w.with_(causal=False, softmax=True))


def test_output_rows_outside_sequences_untouched():
    w = W.jagged_readme().with_(batch=3, uih_q=[100, 300, 5], targets=[1, 2, 3])
    q, k, v = w.tensors()
    total = w.total_q
    pad = 40
    qd = torch.cat([q, torch.zeros(pad, *q.shape[1:], dtype=q.dtype)]).cuda()
    kd = torch.cat([k, torch.zeros(pad, *k.shape[1:], dtype=k.dtype)]).cuda()
    vd = torch.cat([v, torch.zeros(pad, *v.shape[1:], dtype=v.dtype)]).cuda()
    out = torch.full((total + pad, w.nhead, w.hdim_v), 7.0, dtype=q.dtype, device="cuda")
    from recommender_attention_gb300.hstu import hstu_attn_fwd
    from tests.gpu_helpers import call_kwargs
    off_q = torch.from_numpy(w.seq_offsets_q()).cuda()
    tg = torch.from_numpy(w.num_targets()).cuda()
    hstu_attn_fwd(qd, kd, vd, off_q, None, tg, out=out, check=True, **call_kwargs(w))
    o_ref, _ = oracle_forward(w, q, k, v)
    assert torch.all(out[total:] == 7.0)
    assert_parity(out[:total].float().cpu().numpy().astype(np.float64), o_ref, w.dtype)


# ---------------------------------------------------------------- schedule accounting
@pytest.mark.parametrize("cfg", ["tiny", "jagged", "batched", "group_cross", "mfalcon"])
def test_tile_skip_and_pair_accounting(cfg):
    w = W.CONFIGS[cfg]()
    q, k, v = w.tensors()
    stats = gpu_call(w, q, k, v).stats()
    p = oracle_params(w)
    args = (w.seq_offsets_q(), w.seq_offsets_kv(), w.num_targets(), p, w.nhead)
    assert stats["executed_tiles"] == kernel_executed_tiles(w)
    assert stats["allowed_pairs"] == allowed_pair_count(*args)
    assert stats["device_error"] == 0


@pytest.mark.parametrize("seed", range(12))
def test_tile_skip_accounting_fuzz(seed):
    w = W.random_small(seed, hdim=64, kv_targets=seed >= 8)
    q, k, v = w.tensors()
    stats = gpu_call(w, q, k, v, num_splits=1).stats()
    p = oracle_params(w)
    args = (w.seq_offsets_q(), w.seq_offsets_kv(), w.num_targets(), p, w.nhead)
    assert stats["executed_tiles"] == kernel_executed_tiles(w)
    assert stats["allowed_pairs"] == allowed_pair_count(*args)


# ---------------------------------------------------------------- device-side errors
def test_device_error_bad_offsets_and_layout():
    from recommender_attention_gb300.hstu import HstuError
    w = W.tiny_batched()
    # non-monotone offsets
    offs = torch.tensor([0, 80, 70], dtype=torch.int32, device="cuda")
    q, k, v = w.tensors()
    call = gpu_call(w, q, k, v)
    call._keep.append(offs)
    call.args.seq_offsets_q = offs.data_ptr()
    call.launch()
    with pytest.raises(HstuError) as ei:
        call.check()
    assert ei.value.device_error & 1
    # a sequence shorter than context + targets
    offs2 = torch.tensor([0, 3, 140], dtype=torch.int32, device="cuda")
    call2 = gpu_call(w, q, k, v)
    call2._keep.append(offs2)
    call2.args.seq_offsets_q = offs2.data_ptr()
    call2.launch()
    with pytest.raises(HstuError) as ei:
        call2.check()
    assert ei.value.device_error & 2
    # a length beyond the max_seqlen hint
    call3 = gpu_call(w, q, k, v, max_seqlen_q=50, max_seqlen_kv=50)
    call3.launch()
    with pytest.raises(HstuError) as ei:
        call3.check()
    assert ei.value.device_error & 8
    # the context stays usable afterwards
    o, _ = gpu_forward(w, q, k, v)
    assert np.isfinite(o).all()


def test_bounded_wait_gives_up_and_reports():
    from recommender_attention_gb300.hstu import selftest_wait_timeout
    assert selftest_wait_timeout(20_000_000) is True
    # and a forward right after still runs
    check_full(W.tiny_batched())


def test_repeated_calls_reuse_workspace():
    w = W.jagged_readme()
    q, k, v = w.tensors()
    call = gpu_call(w, q, k, v)
    call.launch()
    first = call.o.clone()
    for _ in range(3):
        call.launch()
    call.check()
    assert torch.equal(first, call.o)
