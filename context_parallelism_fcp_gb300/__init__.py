"""Block-wise variable-length attention for FCP (flexible context parallelism) on GB300.

A thin binding of the C ABI in ``include/fcp.h`` (``libfcp.so``, built in-tree for
sm_103a). Every step of the hot path runs in the library: the host plan (sharding G,
Zig-Zag, LPT assignment M, work list, coalesced runs) in C++, and the forward, merge and
backward in hand-written tcgen05/TMA kernels. This module only marshals arguments:
torch supplies device memory and streams. There is no fallback: if the library is
missing or fails to load, every call raises.

Pages: "Unleashing Scalable Context Parallelism for Foundation Models Pre-Training via
FCP" -- Section 3.3 (G, M, loads), Section 4.1 (block distributor), Section 3.2 / Figure 4
(Zig-Zag), Section 2.2 (attention), Section 2.3 (associative reduction), Section 4.2
(coalescer).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "FcpError",
    "Plan",
    "lib",
    "library_path",
    "block_attn_fwd",
    "block_attn_fwd_stage",
    "block_attn_merge",
    "block_attn_bwd",
    "block_attn_bwd_prologue",
    "block_attn_bwd_tiles",
    "block_attn_bwd_dq_convert",
    "block_attn_bwd_tiles_banded",
    "reshuffle",
    "FcpAttention",
    "MASK_FULL",
    "MASK_CAUSAL_DIAG",
    "EXPORTED_SYMBOLS",
]

MASK_FULL = 0
MASK_CAUSAL_DIAG = 1

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_PKG_DIR, "libfcp.so")


class FcpError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: fcp status {status}"
        if _LIB is not None:
            msg += f" ({_LIB.fcp_status_string(status).decode()})"
        if detail:
            msg += f": {detail}"
        super().__init__(msg)


class _Block(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("first_seg", "n_segs", "tokens", "seq", "seq_block_idx",
                                              "seq_nblocks", "zz_partner", "worker")] + [("cost", ctypes.c_int64)]


class _Segment(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("seq", "start_in_seq", "len", "tok0")]


class _Item(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("worker", "q_block", "kv_block", "q_tok0", "q_len", "kv_tok0",
                                              "kv_len", "mask", "run", "reserved")]


class _Run(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("worker", "q_block", "q_tok0", "q_len", "item_begin", "item_end",
                                              "part_row0", "stage")]


class _Transfer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("kv_block", "src", "dst", "stage", "tokens", "reserved")]


class _View(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_seqs", "n_blocks", "n_segs", "n_items", "n_runs", "n_workers",
                                              "block_size", "causal", "coalesce", "distributed",
                                              "n_exec_stages")] + [
        (n, ctypes.c_int64) for n in ("total_tokens", "token_cap", "total_pairs", "partial_rows")] + [
        ("seqlens", ctypes.POINTER(ctypes.c_int32)),
        ("blocks", ctypes.POINTER(_Block)),
        ("segs", ctypes.POINTER(_Segment)),
        ("items", ctypes.POINTER(_Item)),
        ("runs", ctypes.POINTER(_Run)),
        ("worker_load", ctypes.POINTER(ctypes.c_int64)),
        ("worker_tokens", ctypes.POINTER(ctypes.c_int64)),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

# symbol -> (restype, argtypes); every function declared in include/fcp.h
_SIGNATURES = {
    "fcp_partition": (_ST, [ctypes.POINTER(_I32), _I32, _I32, _I32, ctypes.POINTER(_P)]),
    "fcp_distribute": (_ST, [_P, _I32, _I64]),
    "fcp_partition_ring": (_ST, [ctypes.POINTER(_I32), _I32, _I32, _I32, ctypes.POINTER(_P)]),
    "fcp_coalesce": (_ST, [_P, _I32]),
    "fcp_schedule": (_ST, [_P, _I32, ctypes.POINTER(_I32)]),
    "fcp_plan_query": (_ST, [_P, ctypes.POINTER(_View)]),
    "fcp_plan_validate": (_ST, [_P]),
    "fcp_solve_stages": (_ST, [_P]),
    "fcp_set_stages": (_ST, [_P, ctypes.POINTER(_I32), _I32]),
    "fcp_plan_transfers": (_ST, [_P, ctypes.POINTER(ctypes.POINTER(_Transfer)), ctypes.POINTER(_I32),
                                 ctypes.POINTER(_I32)]),
    "fcp_plan_device_bytes": (_SZ, [_P]),
    "fcp_plan_upload": (_ST, [_P, _P, _SZ, _P]),
    "fcp_partial_sizes": (_ST, [_P, _I32, _I32, ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    "fcp_block_attn_fwd": (_ST, [_P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "fcp_block_attn_fwd_stage": (_ST, [_P, _P, _I32, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "fcp_block_attn_merge": (_ST, [_P, _P, _P, _P, _I32, _I32, _P, _P, _P]),
    "fcp_block_attn_bwd_prologue": (_ST, [_P, _P, _P, _I32, _I32, _P, _P, _P]),
    "fcp_bwd_workspace_bytes": (_SZ, [_P, _I32, _I32]),
    "fcp_plan_set_bwd_band": (_ST, [_P, _I32]),
    "fcp_plan_bwd_bands": (_ST, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "fcp_bwd_band_workspace_bytes": (_SZ, [_P, _I32, _I32]),
    "fcp_block_attn_bwd_tiles_banded": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "fcp_block_attn_bwd": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]),
    "fcp_block_attn_bwd_tiles": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P]),
    "fcp_block_attn_bwd_dq_convert": (_ST, [_P, _P, _I32, _I32, _P, _P]),
    "fcp_bwd_static_scratch_bytes": (_SZ, []),
    "fcp_block_attn_bwd_static_scratch": (_ST, [_P, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P]),
    "fcp_reshuffle": (_ST, [_P, _P, _P, _P, _I32, _I32, _I32, _P]),
    "fcp_selftest_bounded_wait": (_ST, [_P, _P]),
    "fcp_device_error": (_ST, [_P, ctypes.POINTER(_I32), _P]),
    "fcp_plan_free": (None, [_P]),
    "fcp_status_string": (ctypes.c_char_p, [_ST]),
    "fcp_last_error": (ctypes.c_char_p, []),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded libfcp.so. Raises if it has not been built (run ``__graft_entry__.build()``
    or ``python -m context_parallelism_fcp_gb300._build``)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with python -m context_parallelism_fcp_gb300._build")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def _check(status: int, where: str) -> None:
    if status != 0:
        detail = lib().fcp_last_error().decode() if status == 4 else ""
        raise FcpError(status, where, detail)


def _arr(ptr, n: int, dtype, cols: Optional[Sequence[str]] = None) -> np.ndarray:
    if n == 0:
        return np.zeros((0, len(cols)) if cols else (0,), dtype=np.int64)
    if cols is None:
        return np.ctypeslib.as_array(ptr, shape=(n,)).astype(np.int64)
    raw = np.ctypeslib.as_array(ptr, shape=(n,))
    return np.stack([raw[c].astype(np.int64) for c in cols], axis=1)


class Plan:
    """Host plan: sharding G with packing and Zig-Zag partners (fcp_partition), LPT
    assignment under a token cap and the work list (fcp_distribute), coalesced runs
    (fcp_coalesce)."""

    BLOCK_COLS = ("first_seg", "n_segs", "tokens", "seq", "seq_block_idx", "seq_nblocks", "zz_partner", "cost")
    SEG_COLS = ("seq", "start_in_seq", "len", "tok0")
    ITEM_COLS = ("worker", "q_block", "kv_block", "q_tok0", "q_len", "kv_tok0", "kv_len", "mask")
    RUN_COLS = ("worker", "q_block", "q_tok0", "q_len", "item_begin", "item_end", "part_row0", "stage")

    def __init__(self, seqlens: Sequence[int], block_size: int, causal: bool):
        L = lib()
        arr = (_I32 * len(seqlens))(*[int(x) for x in seqlens])
        h = _P()
        _check(L.fcp_partition(arr, len(seqlens), int(block_size), 1 if causal else 0, ctypes.byref(h)),
               "fcp_partition")
        self._h = h
        self.seqlens = [int(x) for x in seqlens]
        self.block_size = int(block_size)
        self.causal = bool(causal)

    @classmethod
    def ring(cls, seqlens: Sequence[int], n_workers: int, causal: bool) -> "Plan":
        """The ring-attention baseline plan: 2N equal blocks per sequence, worker w holding
        blocks w and 2N-1-w (fcp_partition_ring); already distributed."""
        self = cls.__new__(cls)
        L = lib()
        arr = (_I32 * len(seqlens))(*[int(x) for x in seqlens])
        h = _P()
        _check(L.fcp_partition_ring(arr, len(seqlens), int(n_workers), 1 if causal else 0, ctypes.byref(h)),
               "fcp_partition_ring")
        self._h = h
        self.seqlens = [int(x) for x in seqlens]
        self.block_size = None
        self.causal = bool(causal)
        return self

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _LIB is not None:
            _LIB.fcp_plan_free(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def distribute(self, n_workers: int, token_cap: Optional[int] = None) -> "Plan":
        _check(lib().fcp_distribute(self._h, int(n_workers), int(token_cap or 0)), "fcp_distribute")
        return self

    def coalesce(self, degree: int) -> "Plan":
        _check(lib().fcp_coalesce(self._h, int(degree)), "fcp_coalesce")
        return self

    def schedule(self, degree: int) -> int:
        """Block-level pipeline with the bottom-up coalescer (fcp_schedule): items ordered by
        the execution stage of their KV block, `degree` congestion-free sub-stages per stage.
        Returns the number of execution stages."""
        n = _I32()
        _check(lib().fcp_schedule(self._h, int(degree), ctypes.byref(n)), "fcp_schedule")
        return int(n.value)

    def solve(self) -> dict:
        """Congestion-free sub-stages (fcp_solve_stages): transfers as rows (kv_block, src, dst,
        stage, tokens) and the number of stages."""
        _check(lib().fcp_solve_stages(self._h), "fcp_solve_stages")
        return self.transfers()

    def set_stages(self, stages: Sequence[int]) -> None:
        """Install a caller-supplied congestion-free plan: one sub-stage per data-flow edge,
        edges in the order solve() lists them (fcp_set_stages)."""
        arr = (_I32 * max(1, len(stages)))(*[int(x) for x in stages])
        _check(lib().fcp_set_stages(self._h, arr, len(stages)), "fcp_set_stages")

    def transfers(self) -> dict:
        """The current congestion-free plan (fcp_plan_transfers), as solve() returns it."""
        ptr = ctypes.POINTER(_Transfer)()
        n, st = _I32(), _I32()
        _check(lib().fcp_plan_transfers(self._h, ctypes.byref(ptr), ctypes.byref(n), ctypes.byref(st)),
               "fcp_plan_transfers")
        rows = _arr(ptr, n.value, None, ("kv_block", "src", "dst", "stage", "tokens"))
        return {"transfers": rows, "n_stages": int(st.value)}

    def view(self) -> dict:
        v = _View()
        _check(lib().fcp_plan_query(self._h, ctypes.byref(v)), "fcp_plan_query")
        out = {k: getattr(v, k) for k in ("n_seqs", "n_blocks", "n_segs", "n_items", "n_runs", "n_workers",
                                           "block_size", "causal", "coalesce", "distributed", "n_exec_stages",
                                           "total_tokens",
                                           "token_cap", "total_pairs", "partial_rows")}
        out["blocks"] = _arr(v.blocks, v.n_blocks, None, self.BLOCK_COLS)
        out["worker_of_block"] = _arr(v.blocks, v.n_blocks, None, ("worker",))[:, 0] if v.n_blocks else \
            np.zeros(0, np.int64)
        out["segs"] = _arr(v.segs, v.n_segs, None, self.SEG_COLS)
        if v.distributed:
            out["items"] = _arr(v.items, v.n_items, None, self.ITEM_COLS)
            out["item_run"] = _arr(v.items, v.n_items, None, ("run",))[:, 0] if v.n_items else np.zeros(0, np.int64)
            out["runs"] = _arr(v.runs, v.n_runs, None, self.RUN_COLS)
            out["load"] = _arr(v.worker_load, v.n_workers, None)
            out["tokens"] = _arr(v.worker_tokens, v.n_workers, None)
        return out

    def validate(self) -> "Plan":
        """Check every index of the plan and its device image (fcp_plan_validate); raises
        FcpError naming the first violation."""
        _check(lib().fcp_plan_validate(self._h), "fcp_plan_validate")
        return self

    def device_bytes(self) -> int:
        return int(lib().fcp_plan_device_bytes(self._h))

    def partial_sizes(self, hq: int, head_dim: int) -> Tuple[int, int]:
        o, l = _SZ(), _SZ()
        _check(lib().fcp_partial_sizes(self._h, hq, head_dim, ctypes.byref(o), ctypes.byref(l)), "fcp_partial_sizes")
        return int(o.value), int(l.value)

    def workspace_bytes(self, hq: int, head_dim: int) -> int:
        return int(lib().fcp_bwd_workspace_bytes(self._h, hq, head_dim))

    def set_bwd_band(self, band_rows: int) -> "Plan":
        """Query bands of the backward (fcp_plan_set_bwd_band): -1 lets the plan choose, 0 none,
        > 0 rows per band (a multiple of 64). Upload the plan again afterwards."""
        _check(lib().fcp_plan_set_bwd_band(self._h, int(band_rows)), "fcp_plan_set_bwd_band")
        return self

    def bwd_bands(self) -> Tuple[int, int]:
        """(number of backward query bands, rows per band) of the distributed plan."""
        n, r = _I32(), _I32()
        _check(lib().fcp_plan_bwd_bands(self._h, ctypes.byref(n), ctypes.byref(r)), "fcp_plan_bwd_bands")
        return int(n.value), int(r.value)

    def band_workspace_bytes(self, hkv: int, head_dim: int) -> int:
        """Float32 dK/dV scratch of the banded backward (0 without bands)."""
        return int(lib().fcp_bwd_band_workspace_bytes(self._h, hkv, head_dim))

    def upload(self, d_plan, stream=None) -> None:
        """Copy the device image into ``d_plan`` (a CUDA uint8 tensor of >= device_bytes())."""
        _check(lib().fcp_plan_upload(self._h, _ptr(d_plan), d_plan.numel() * d_plan.element_size(),
                                     _stream(stream)), "fcp_plan_upload")


# ---------------------------------------------------------------- device calls
def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t, dtype, shape, name):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def block_attn_fwd(plan: Plan, d_plan, q, k, v, part_o, part_lse, stream=None) -> None:
    """Partial (O, LSE) of every run over the work list (fcp_block_attn_fwd)."""
    import torch

    hq, T, D = q.shape
    hkv = k.shape[0]
    _need(q, torch.bfloat16, None, "q")
    _need(k, torch.bfloat16, (hkv, T, D), "k")
    _need(v, torch.bfloat16, (hkv, T, D), "v")
    _need(part_o, torch.float32, None, "part_o")
    _need(part_lse, torch.float32, None, "part_lse")
    _check(lib().fcp_block_attn_fwd(plan.handle, _ptr(d_plan), _ptr(q), _ptr(k), _ptr(v), hq, hkv, D, _ptr(part_o),
                                    _ptr(part_lse), _stream(stream)), "fcp_block_attn_fwd")


def block_attn_fwd_stage(plan: Plan, d_plan, stage: int, q, k, v, part_o, part_lse, stream=None) -> None:
    """Partial (O, LSE) of the runs of one execution stage (fcp_block_attn_fwd_stage)."""
    import torch

    hq, T, D = q.shape
    hkv = k.shape[0]
    _need(q, torch.bfloat16, None, "q")
    _need(k, torch.bfloat16, (hkv, T, D), "k")
    _need(v, torch.bfloat16, (hkv, T, D), "v")
    _need(part_o, torch.float32, None, "part_o")
    _need(part_lse, torch.float32, None, "part_lse")
    _check(lib().fcp_block_attn_fwd_stage(plan.handle, _ptr(d_plan), int(stage), _ptr(q), _ptr(k), _ptr(v), hq, hkv,
                                          D, _ptr(part_o), _ptr(part_lse), _stream(stream)),
           "fcp_block_attn_fwd_stage")


def block_attn_merge(plan: Plan, d_plan, part_o, part_lse, o, lse, stream=None) -> None:
    """Log-sum-exp merge of the partials into O (bf16) and LSE (fp32) (fcp_block_attn_merge)."""
    import torch

    hq, T, D = o.shape
    _need(o, torch.bfloat16, None, "o")
    _need(lse, torch.float32, (hq, T), "lse")
    _check(lib().fcp_block_attn_merge(plan.handle, _ptr(d_plan), _ptr(part_o), _ptr(part_lse), hq, D, _ptr(o),
                                      _ptr(lse), _stream(stream)), "fcp_block_attn_merge")


def block_attn_bwd_prologue(plan: Plan, o, dout, di, dq_acc, stream=None) -> None:
    """Di = rowsum(dO * O) and a zeroed dQ accumulator (fcp_block_attn_bwd_prologue)."""
    import torch

    hq, T, D = o.shape
    _need(o, torch.bfloat16, None, "o")
    _need(dout, torch.bfloat16, (hq, T, D), "dout")
    _need(di, torch.float32, (hq, T), "di")
    _need(dq_acc, torch.float32, (hq, T, D), "dq_acc")
    _check(lib().fcp_block_attn_bwd_prologue(plan.handle, _ptr(o), _ptr(dout), hq, D, _ptr(di), _ptr(dq_acc),
                                             _stream(stream)), "fcp_block_attn_bwd_prologue")


def block_attn_bwd(plan: Plan, d_plan, q, k, v, o, dout, lse, dq, dk, dv, workspace, stream=None) -> None:
    """dQ, dK, dV over the work list (fcp_block_attn_bwd)."""
    import torch

    hq, T, D = q.shape
    hkv = k.shape[0]
    for name, t, shp in (("q", q, (hq, T, D)), ("k", k, (hkv, T, D)), ("v", v, (hkv, T, D)), ("o", o, (hq, T, D)),
                         ("dout", dout, (hq, T, D)), ("dq", dq, (hq, T, D)), ("dk", dk, (hkv, T, D)),
                         ("dv", dv, (hkv, T, D))):
        _need(t, torch.bfloat16, shp, name)
    _need(lse, torch.float32, (hq, T), "lse")
    _check(lib().fcp_block_attn_bwd(plan.handle, _ptr(d_plan), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                                    _ptr(lse), hq, hkv, D, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "fcp_block_attn_bwd")


def block_attn_bwd_tiles(plan: Plan, d_plan, q, k, v, dout, lse, di, dq_acc, dk, dv, stream=None) -> None:
    """The backward tile kernel alone (fcp_block_attn_bwd_tiles); dq_acc/di from the prologue."""
    import torch

    hq, T, D = q.shape
    hkv = k.shape[0]
    _need(dq_acc, torch.float32, (hq, T, D), "dq_acc")
    _need(di, torch.float32, (hq, T), "di")
    _check(lib().fcp_block_attn_bwd_tiles(plan.handle, _ptr(d_plan), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                          _ptr(lse), _ptr(di), hq, hkv, D, _ptr(dq_acc), _ptr(dk), _ptr(dv),
                                          _stream(stream)), "fcp_block_attn_bwd_tiles")


def block_attn_bwd_tiles_banded(plan: Plan, d_plan, q, k, v, dout, lse, di, dq_acc, dkv_acc, dk, dv,
                                stream=None) -> None:
    """The banded tile kernels (fcp_block_attn_bwd_tiles_banded): one launch per query band,
    dK/dV summed in dkv_acc (uint8 or float32 scratch of Plan.band_workspace_bytes)."""
    import torch

    hq, T, D = q.shape
    hkv = k.shape[0]
    _need(dq_acc, torch.float32, (hq, T, D), "dq_acc")
    _need(di, torch.float32, (hq, T), "di")
    if dkv_acc.numel() * dkv_acc.element_size() < plan.band_workspace_bytes(hkv, D):
        raise ValueError("dkv_acc is smaller than Plan.band_workspace_bytes")
    _check(lib().fcp_block_attn_bwd_tiles_banded(plan.handle, _ptr(d_plan), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                                 _ptr(lse), _ptr(di), hq, hkv, D, _ptr(dq_acc), _ptr(dkv_acc),
                                                 _ptr(dk), _ptr(dv), _stream(stream)),
           "fcp_block_attn_bwd_tiles_banded")


def block_attn_bwd_dq_convert(plan: Plan, dq_acc, dq, stream=None) -> None:
    """dq = bf16(dq_acc / sqrt(D)) (fcp_block_attn_bwd_dq_convert)."""
    import torch

    hq, T, D = dq.shape
    _need(dq_acc, torch.float32, (hq, T, D), "dq_acc")
    _need(dq, torch.bfloat16, (hq, T, D), "dq")
    _check(lib().fcp_block_attn_bwd_dq_convert(plan.handle, _ptr(dq_acc), hq, D, _ptr(dq), _stream(stream)),
           "fcp_block_attn_bwd_dq_convert")


def reshuffle(plan: Plan, d_plan, src, dst, to_workers: bool = True, stream=None) -> None:
    """Permute the token rows of src [H, T, ...] between the user's and the workers' layout
    into dst (fcp_reshuffle)."""
    if src.shape != dst.shape or src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same shape and dtype")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    heads = src.shape[0]
    row_bytes = src[0, 0].numel() * src.element_size() if src.shape[1] else 16
    _check(lib().fcp_reshuffle(plan.handle, _ptr(d_plan), _ptr(src), _ptr(dst), heads, row_bytes,
                               0 if to_workers else 1, _stream(stream)), "fcp_reshuffle")


def selftest_bounded_wait(d_plan, stream=None) -> None:
    """Launch the bounded-wait self-test into d_plan's error word (fcp_selftest_bounded_wait)."""
    _check(lib().fcp_selftest_bounded_wait(_ptr(d_plan), _stream(stream)), "fcp_selftest_bounded_wait")


def device_error(d_plan, stream=None) -> int:
    """Read and clear the device plan's error word (0 = none)."""
    code = _I32(0)
    st = lib().fcp_device_error(_ptr(d_plan), ctypes.byref(code), _stream(stream))
    if st not in (0, 6):
        _check(st, "fcp_device_error")
    return int(code.value)


class FcpAttention:
    """A planned batch: the plan, its device image and the partial/workspace buffers, with
    forward (fwd + merge) and backward over the same work list. With ``pipeline=c`` the
    plan is scheduled as the block-level pipeline with coalesce degree c (Plan.schedule) and
    the forward launches one execution stage at a time before the merge. ``bwd_band`` sets the
    backward's query bands (Plan.set_bwd_band; None keeps the plan's own choice); the
    workspace holds their dK/dV sums, so a plan with bands runs its backward banded."""

    def __init__(self, seqlens: Sequence[int], block_size: int, causal: bool, n_workers: int, hq: int, hkv: int,
                 head_dim: int, token_cap: Optional[int] = None, coalesce: int = 1, device="cuda",
                 backward: bool = True, pipeline: Optional[int] = None, bwd_band: Optional[int] = None):
        self._recipe = (int(block_size), bool(causal), int(n_workers), token_cap, int(coalesce), pipeline, bwd_band)
        self._setup(self._make_plan(seqlens), hq, hkv, head_dim, device, backward)

    def _make_plan(self, seqlens) -> "Plan":
        block_size, causal, n_workers, token_cap, coalesce, pipeline, bwd_band = self._recipe
        plan = Plan(seqlens, block_size, causal)
        if bwd_band is not None:
            plan.set_bwd_band(bwd_band)
        plan.distribute(n_workers, token_cap)
        if pipeline is not None:
            plan.schedule(pipeline)
        elif coalesce != 1:
            plan.coalesce(coalesce)
        return plan

    def replan(self, seqlens: Optional[Sequence[int]] = None, stream=None) -> None:
        """Plan a new batch (by default the same lengths again) with the same block size,
        mask, workers, cap and coalescing, as a training loop does for every batch: partition,
        distribute and coalesce run on the host, and the new device image is uploaded in
        ``stream`` order, so kernels enqueued earlier on that stream still see the old plan.
        The batch must fit the buffers allocated at construction (same total tokens, no more
        partial rows or device-image bytes)."""
        if getattr(self, "_recipe", None) is None:
            raise RuntimeError("replan needs an FcpAttention built from a batch description, not from_plan")
        plan = self._make_plan(self.plan.seqlens if seqlens is None else seqlens)
        v = plan.view()
        if (int(v["total_tokens"]) != self.T or int(v["partial_rows"]) > self.part_o.shape[1]
                or plan.device_bytes() > self.d_plan.numel()):
            raise ValueError("the new batch does not fit the buffers of this FcpAttention")
        if int(v["n_exec_stages"]) != self.n_stages:
            raise ValueError("the new batch has a different number of pipeline stages")
        plan.upload(self.d_plan, stream)
        self.plan = plan

    @classmethod
    def from_plan(cls, plan: "Plan", hq: int, hkv: int, head_dim: int, device="cuda",
                  backward: bool = True) -> "FcpAttention":
        """Wrap an already distributed plan (e.g. Plan.ring(...))."""
        self = cls.__new__(cls)
        self._recipe = None
        self._setup(plan, hq, hkv, head_dim, device, backward)
        return self

    def _setup(self, plan, hq, hkv, head_dim, device, backward):
        import torch

        self.plan = plan
        self.n_stages = int(plan.view()["n_exec_stages"])
        self.hq, self.hkv, self.head_dim = hq, hkv, head_dim
        self.T = sum(int(x) for x in plan.seqlens)
        self.device = torch.device(device)
        nbytes = self.plan.device_bytes()
        # room for the device images of later batches of the same size (replan), whose
        # work lists differ in length
        self.d_plan = torch.empty(max(2 * nbytes, 65536), dtype=torch.uint8, device=self.device)
        self.plan.upload(self.d_plan)
        ob, lb = self.plan.partial_sizes(hq, head_dim)
        rows = self.plan.view()["partial_rows"]
        self.part_o = torch.empty((hq, max(rows, 1), head_dim), dtype=torch.float32, device=self.device)
        self.part_lse = torch.empty((hq, max(rows, 1)), dtype=torch.float32, device=self.device)
        assert self.part_o.numel() * 4 >= ob and self.part_lse.numel() * 4 >= lb
        self.workspace = None
        if backward:
            # with query bands, room for their float32 dK/dV sums, so that the backward runs banded
            ws = self.plan.workspace_bytes(hq, head_dim) + self.plan.band_workspace_bytes(hkv, head_dim)
            self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)

    def forward(self, q, k, v, o=None, lse=None, stream=None):
        import torch

        if o is None:
            o = torch.empty((self.hq, self.T, self.head_dim), dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty((self.hq, self.T), dtype=torch.float32, device=self.device)
        if self.n_stages > 1:
            for st in range(self.n_stages):
                block_attn_fwd_stage(self.plan, self.d_plan, st, q, k, v, self.part_o, self.part_lse, stream)
        else:
            block_attn_fwd(self.plan, self.d_plan, q, k, v, self.part_o, self.part_lse, stream)
        block_attn_merge(self.plan, self.d_plan, self.part_o, self.part_lse, o, lse, stream)
        return o, lse

    def backward(self, q, k, v, o, lse, dout, dq=None, dk=None, dv=None, stream=None):
        import torch

        if self.workspace is None:
            raise RuntimeError("constructed with backward=False")
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(k) if dk is None else dk
        dv = torch.empty_like(v) if dv is None else dv
        block_attn_bwd(self.plan, self.d_plan, q, k, v, o, dout, lse, dq, dk, dv, self.workspace, stream)
        return dq, dk, dv

    def check_device_error(self, stream=None) -> None:
        code = device_error(self.d_plan, stream)
        if code:
            raise FcpError(6, "device", f"error word 0x{code:x}")
