"""Thin ctypes binding over ``libhstu_attn.so`` (see ``include/hstu_attn.h``).

Argument marshalling only: every step of the forward and the backward runs in
the library's CUDA kernels.  PyTorch provides device memory and streams.  There is no CPU or
framework fallback: when the library is missing every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Union

import torch

from . import build as _build

_LIB = None

HSTU_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
                3: "workspace missing, misaligned or too small", 4: "CUDA error",
                5: "device-side check failed"}
DEVERR_BITS = {1: "offsets", 2: "query layout", 4: "key layout", 8: "max_seqlen", 16: "timeout"}
DTYPE_CODES = {torch.float16: 0, torch.bfloat16: 1}


class HstuError(RuntimeError):
    def __init__(self, status: int, what: str, device_error: int = 0):
        self.status = status
        self.device_error = device_error
        msg = f"{what}: {STATUS_NAMES.get(status, status)}"
        if device_error:
            bits = [n for b, n in DEVERR_BITS.items() if device_error & b]
            msg += f" (device error {device_error}: {', '.join(bits)})"
        super().__init__(msg)


class FwdArgs(ctypes.Structure):
    """Mirror of ``hstu_fwd_args``."""
    _fields_ = [
        ("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("nhead", ctypes.c_int32),
        ("hdim_qk", ctypes.c_int32), ("hdim_v", ctypes.c_int32), ("total_q", ctypes.c_int32),
        ("total_kv", ctypes.c_int32), ("max_seqlen_q", ctypes.c_int32),
        ("max_seqlen_kv", ctypes.c_int32), ("causal", ctypes.c_int32), ("softmax", ctypes.c_int32),
        ("num_groups", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("alpha", ctypes.c_float),
        ("q_row_stride", ctypes.c_int64), ("k_row_stride", ctypes.c_int64),
        ("v_row_stride", ctypes.c_int64), ("o_row_stride", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("seq_offsets_q", ctypes.c_void_p), ("seq_offsets_kv", ctypes.c_void_p),
        ("num_targets", ctypes.c_void_p), ("local_len", ctypes.c_void_p),
        ("context_len", ctypes.c_void_p), ("minfull_len", ctypes.c_void_p),
        ("max_uih_len", ctypes.c_void_p), ("attn_scale", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("event_fwd_begin", ctypes.c_void_p), ("event_fwd_end", ctypes.c_void_p),
        ("kv_targets", ctypes.c_int32),
        ("timestamps_q", ctypes.c_void_p), ("timestamps_kv", ctypes.c_void_p),
        ("rab_time", ctypes.c_void_p), ("rab_pos", ctypes.c_void_p), ("rab_pos_buckets", ctypes.c_int32),
        ("cta_pairs", ctypes.c_int32),
    ]


class BwdArgs(ctypes.Structure):
    """Mirror of ``hstu_bwd_args``."""
    _fields_ = [
        ("fwd", FwdArgs), ("d_o", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p), ("do_row_stride", ctypes.c_int64), ("dq_row_stride", ctypes.c_int64),
        ("dk_row_stride", ctypes.c_int64), ("dv_row_stride", ctypes.c_int64),
        ("d_rab_time", ctypes.c_void_p), ("d_rab_pos", ctypes.c_void_p),
    ]


class FwdStats(ctypes.Structure):
    """Mirror of ``hstu_fwd_stats``."""
    _fields_ = [("executed_tiles", ctypes.c_int64), ("allowed_pairs", ctypes.c_int64),
                ("work_units", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("device_error", ctypes.c_int32), ("reserved", ctypes.c_int32)]


EXPORTS = {
    "hstu_abi_version": (ctypes.c_int32, []),
    "hstu_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "hstu_attn_fwd_workspace_size": (ctypes.c_int, [ctypes.POINTER(FwdArgs), ctypes.POINTER(ctypes.c_size_t)]),
    "hstu_attn_fwd": (ctypes.c_int, [ctypes.POINTER(FwdArgs), ctypes.c_void_p]),
    "hstu_attn_fwd_check": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "hstu_attn_fwd_stats": (ctypes.c_int, [ctypes.POINTER(FwdArgs), ctypes.c_void_p, ctypes.POINTER(FwdStats)]),
    "hstu_device_sm_count": (ctypes.c_int32, []),
    "hstu_fwd_args_size": (ctypes.c_size_t, []),
    "hstu_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p,
                                                  ctypes.POINTER(ctypes.c_int32)]),
    "hstu_attn_fwd_static_ws": (ctypes.c_int, [ctypes.POINTER(FwdArgs), ctypes.c_void_p,
                                               ctypes.POINTER(ctypes.c_void_p)]),
    "hstu_bwd_args_size": (ctypes.c_size_t, []),
    "hstu_attn_bwd_workspace_size": (ctypes.c_int, [ctypes.POINTER(BwdArgs), ctypes.POINTER(ctypes.c_size_t)]),
    "hstu_attn_bwd": (ctypes.c_int, [ctypes.POINTER(BwdArgs), ctypes.c_void_p]),
}


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = False):
    """Loads the C-ABI library (once).  Raises when it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing: build it with recommender_attention_gb300.build.build()")
        _build.build()
    lib = ctypes.CDLL(path)
    for name, (res, args) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _per_group(x, g: int, ctype):
    vals = list(x) if isinstance(x, (list, tuple)) else [x] * g
    if len(vals) != g:
        raise ValueError(f"expected {g} per-group values, got {len(vals)}")
    return (ctype * g)(*vals)


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _capture(launch) -> "torch.cuda.CUDAGraph":
    """A CUDA graph of one call: `launch(stream)` enqueues the call's kernels
    (the header reset or scheduler, the forward or the two gradient kernels,
    the combine) on a capture stream; replaying the graph repeats them on the
    same buffers without the host work of a call (argument checks, tensor-map
    encoding, launches).  The library's kernels are launched with plain stream
    semantics and programmatic dependencies, which capture keeps."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=side):
        launch(side)
    torch.cuda.current_stream().wait_stream(side)
    return g


class HstuCall:
    """One marshalled call: keeps the ctypes arrays alive alongside the args."""

    def __init__(self, q, k, v, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                 alpha: float = 0.0, attn_scale: Union[float, Sequence[float]] = 0.0,
                 causal: bool = True, local_len=0, context_len=0, minfull_len=0, max_uih_len=0,
                 num_groups: int = 1, softmax: bool = False, max_seqlen_q: int = 0,
                 max_seqlen_kv: int = 0, num_splits: int = 0,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 save_lse: bool = True, workspace: Optional[torch.Tensor] = None,
                 static_workspace: bool = False, kv_targets: bool = False,
                 timestamps_q: Optional[torch.Tensor] = None, timestamps_kv: Optional[torch.Tensor] = None,
                 rab_time: Optional[torch.Tensor] = None, rab_pos: Optional[torch.Tensor] = None,
                 cta_pairs: int = 0):
        self.lib = load_library()
        if q.dtype not in DTYPE_CODES or k.dtype != q.dtype or v.dtype != q.dtype:
            raise TypeError("q, k, v must share a dtype, fp16 or bf16")
        total_q, nhead, dqk = q.shape
        total_kv = k.shape[0]
        dv = v.shape[2]
        batch = seq_offsets_q.numel() - 1
        if out is None:
            out = torch.empty((total_q, nhead, dv), dtype=q.dtype, device=q.device)
        if softmax and save_lse and lse is None:
            lse = torch.empty((nhead, total_q), dtype=torch.float32, device=q.device)
        self.o, self.lse = out, (lse if softmax else None)
        g = num_groups
        self._groups = [_per_group(local_len, g, ctypes.c_int32), _per_group(context_len, g, ctypes.c_int32),
                        _per_group(minfull_len, g, ctypes.c_int32), _per_group(max_uih_len, g, ctypes.c_int32),
                        _per_group(attn_scale, g, ctypes.c_float)]
        self._keep = [q, k, v, seq_offsets_q, seq_offsets_kv, num_targets,
                      timestamps_q, timestamps_kv, rab_time, rab_pos]
        for t, dt in ((timestamps_q, torch.int64), (timestamps_kv, torch.int64),
                      (rab_time, torch.float32), (rab_pos, torch.float32)):
            if t is not None and (t.dtype != dt or not t.is_contiguous()):
                raise TypeError("timestamps must be contiguous int64, rab tables contiguous float32")
        a = FwdArgs()
        a.dtype = DTYPE_CODES[q.dtype]
        a.batch, a.nhead, a.hdim_qk, a.hdim_v = batch, nhead, dqk, dv
        a.total_q, a.total_kv = total_q, total_kv
        a.max_seqlen_q, a.max_seqlen_kv = max_seqlen_q, max_seqlen_kv
        a.causal, a.softmax = int(bool(causal)), int(bool(softmax))
        a.num_groups, a.num_splits, a.alpha = g, num_splits, alpha
        a.kv_targets = int(bool(kv_targets))
        a.timestamps_q, a.timestamps_kv = _ptr(timestamps_q), _ptr(timestamps_kv)
        a.rab_time, a.rab_pos = _ptr(rab_time), _ptr(rab_pos)
        a.rab_pos_buckets = 0 if rab_pos is None else rab_pos.shape[-1]
        a.cta_pairs = int(cta_pairs)
        a.q_row_stride, a.k_row_stride = q.stride(0), k.stride(0)
        a.v_row_stride, a.o_row_stride = v.stride(0), out.stride(0)
        for t in (q, k, v, out):
            if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
                raise ValueError("q/k/v/o must be [tokens, nhead, hdim] with packed heads")
        a.q, a.k, a.v, a.o = _ptr(q), _ptr(k), _ptr(v), _ptr(out)
        a.lse = _ptr(self.lse)
        a.seq_offsets_q = _ptr(seq_offsets_q)
        a.seq_offsets_kv = _ptr(seq_offsets_kv)
        a.num_targets = _ptr(num_targets)
        a.local_len, a.context_len, a.minfull_len, a.max_uih_len, a.attn_scale = [
            ctypes.cast(x, ctypes.c_void_p) for x in self._groups]
        self.args = a
        self.static_workspace = static_workspace
        self.static_ws_ptr = None
        size = ctypes.c_size_t(0)
        st = self.lib.hstu_attn_fwd_workspace_size(ctypes.byref(a), ctypes.byref(size))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_fwd_workspace_size")
        self.workspace_bytes = size.value
        if static_workspace:   # the library's own scratch; nothing to allocate here
            self.workspace = None
            return
        if workspace is None or workspace.numel() < self.workspace_bytes:
            workspace = torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=q.device)
        self.workspace = workspace
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel()

    def launch(self, stream: Optional[torch.cuda.Stream] = None,
               events: Optional[tuple] = None) -> None:
        """Enqueues the forward on `stream`.  `events` = (begin, end) torch.cuda.Event
        pair recorded around the forward kernel alone (both recorded once before)."""
        if events is not None:
            self.args.event_fwd_begin = events[0].cuda_event
            self.args.event_fwd_end = events[1].cuda_event
        st = self.lib.hstu_attn_fwd(ctypes.byref(self.args), ctypes.c_void_p(_stream_handle(stream)))
        if events is not None:
            self.args.event_fwd_begin = self.args.event_fwd_end = None
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_fwd")

    def graph(self) -> "torch.cuda.CUDAGraph":
        """This call captured as a CUDA graph (``graph.replay()`` reruns it on
        the same buffers: inputs updated in place are read again)."""
        return _capture(self.launch)

    def launch_static_ws(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Enqueues the forward through ``hstu_attn_fwd_static_ws`` (library scratch)."""
        used = ctypes.c_void_p(0)
        st = self.lib.hstu_attn_fwd_static_ws(ctypes.byref(self.args),
                                              ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(used))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_fwd_static_ws")
        self.static_ws_ptr = used.value

    def check(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        err = ctypes.c_int32(0)
        ws = self.static_ws_ptr if self.static_workspace else self.workspace.data_ptr()
        st = self.lib.hstu_attn_fwd_check(ctypes.c_void_p(ws),
                                          ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(err))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_fwd_check", err.value)
        return err.value

    def stats(self, stream: Optional[torch.cuda.Stream] = None) -> dict:
        s = FwdStats()
        st = self.lib.hstu_attn_fwd_stats(ctypes.byref(self.args),
                                          ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(s))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_fwd_stats", s.device_error)
        return {"executed_tiles": s.executed_tiles, "allowed_pairs": s.allowed_pairs,
                "work_units": s.work_units, "num_splits": s.num_splits,
                "device_error": s.device_error}


class HstuBwdCall:
    """One marshalled backward call.  ``o`` and ``lse`` are the forward's outputs
    (read in softmax mode only); the keyword arguments are the forward's."""

    def __init__(self, q, k, v, d_o, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                 o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                 dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 rab_grads: bool = False, **kw):
        kw.pop("num_splits", None)
        kw.pop("save_lse", None)
        self.fwd = HstuCall(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets, out=o, lse=lse,
                            save_lse=False, static_workspace=True, **kw)
        self.lib = self.fwd.lib
        if d_o.dtype != q.dtype or d_o.shape != self.fwd.o.shape:
            raise ValueError("d_o must match o in shape and dtype")
        self.dq = torch.empty_like(q) if dq is None else dq
        self.dk = torch.empty_like(k) if dk is None else dk
        self.dv = torch.empty_like(v) if dv is None else dv
        for t in (d_o, self.dq, self.dk, self.dv):
            if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
                raise ValueError("d_o/dq/dk/dv must be [tokens, nhead, hdim] with packed heads")
        self._keep = [d_o]
        b = BwdArgs()
        b.fwd = self.fwd.args
        b.d_o, b.dq, b.dk, b.dv = _ptr(d_o), _ptr(self.dq), _ptr(self.dk), _ptr(self.dv)
        b.do_row_stride, b.dq_row_stride = d_o.stride(0), self.dq.stride(0)
        b.dk_row_stride, b.dv_row_stride = self.dk.stride(0), self.dv.stride(0)
        # gradients of the bias tables the call uses (rab_grads=True)
        self.d_rab_time = self.d_rab_pos = None
        if rab_grads:
            nh = q.shape[1]
            if kw.get("rab_time") is not None and kw.get("timestamps_q") is not None:
                self.d_rab_time = torch.empty((nh, 11), dtype=torch.float32, device=q.device)
            if kw.get("rab_pos") is not None:
                self.d_rab_pos = torch.empty((nh, kw["rab_pos"].shape[1]), dtype=torch.float32, device=q.device)
        b.d_rab_time, b.d_rab_pos = _ptr(self.d_rab_time), _ptr(self.d_rab_pos)
        size = ctypes.c_size_t(0)
        st = self.lib.hstu_attn_bwd_workspace_size(ctypes.byref(b), ctypes.byref(size))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_bwd_workspace_size")
        self.workspace_bytes = size.value
        if workspace is None or workspace.numel() < self.workspace_bytes:
            workspace = torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=q.device)
        self.workspace = workspace
        b.fwd.workspace = workspace.data_ptr()
        b.fwd.workspace_bytes = workspace.numel()
        self.args = b

    def launch(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        st = self.lib.hstu_attn_bwd(ctypes.byref(self.args), ctypes.c_void_p(_stream_handle(stream)))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_bwd")

    def graph(self) -> "torch.cuda.CUDAGraph":
        """This call captured as a CUDA graph (see HstuCall.graph)."""
        return _capture(self.launch)

    def check(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        err = ctypes.c_int32(0)
        st = self.lib.hstu_attn_fwd_check(ctypes.c_void_p(self.workspace.data_ptr()),
                                          ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(err))
        if st != HSTU_OK:
            raise HstuError(st, "hstu_attn_bwd (device check)", err.value)
        return err.value


def hstu_attn_bwd(q, k, v, d_o, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                  stream: Optional[torch.cuda.Stream] = None, check: bool = False, **kw):
    """HSTU attention backward (``hstu_attn_bwd`` in ``include/hstu_attn.h``):
    the gradients of the forward with the same keyword arguments for the output
    gradient ``d_o``.  Softmax mode needs the forward's ``o=`` and ``lse=``.
    Returns ``(dq, dk, dv)``, or with ``rab_grads=True``
    ``(dq, dk, dv, d_rab_time, d_rab_pos)`` (None for a table the call has no
    use of)."""
    call = HstuBwdCall(q, k, v, d_o, seq_offsets_q, seq_offsets_kv, num_targets, **kw)
    call.launch(stream)
    if check:
        call.check(stream)
    if kw.get("rab_grads"):
        return call.dq, call.dk, call.dv, call.d_rab_time, call.d_rab_pos
    return call.dq, call.dk, call.dv


def hstu_attn_fwd(q, k, v, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                  stream: Optional[torch.cuda.Stream] = None, check: bool = False, **kw):
    """HSTU attention forward (same names and meaning as ``hstu_attn_fwd`` in
    ``include/hstu_attn.h``).  Returns ``(o, lse)``; lse is None in SiLU mode."""
    call = HstuCall(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets, **kw)
    call.launch(stream)
    if check:
        call.check(stream)
    return call.o, call.lse


def hstu_attn_fwd_static_ws(q, k, v, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                            stream: Optional[torch.cuda.Stream] = None, check: bool = False, **kw):
    """The forward on the library's fixed scratch (``hstu_attn_fwd_static_ws`` in
    ``include/hstu_attn.h``): same arguments and results as ``hstu_attn_fwd``,
    no workspace.  Returns ``(o, lse)``."""
    call = HstuCall(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets, static_workspace=True, **kw)
    call.launch_static_ws(stream)
    if check:
        call.check(stream)
    return call.o, call.lse


def hstu_attn_fwd_stats(q, k, v, seq_offsets_q, seq_offsets_kv=None, num_targets=None, *,
                        stream: Optional[torch.cuda.Stream] = None, **kw) -> dict:
    """Schedule counters of a call (executed tiles, allowed pairs, units, splits)."""
    return HstuCall(q, k, v, seq_offsets_q, seq_offsets_kv, num_targets, **kw).stats(stream)


def device_sm_count() -> int:
    return int(load_library().hstu_device_sm_count())


def selftest_wait_timeout(timeout_ns: int = 50_000_000,
                          stream: Optional[torch.cuda.Stream] = None) -> bool:
    """Runs the bounded-wait self-test; True when the wait gave up as designed."""
    lib = load_library()
    flag = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    out = ctypes.c_int32(-1)
    st = lib.hstu_selftest_wait_timeout(ctypes.c_void_p(flag.data_ptr()), timeout_ns,
                                        ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(out))
    if st != HSTU_OK:
        raise HstuError(st, "hstu_selftest_wait_timeout")
    return out.value == 1
