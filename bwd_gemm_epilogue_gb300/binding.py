"""ctypes binding of the C ABI in ``include/swiglu_mlp.h`` and ``include/swiglu_moe.h``
-- argument marshalling only.

Each function has the name of the C entry point it calls and takes torch CUDA
tensors (bf16, contiguous) for the pointer arguments; torch supplies device
memory and the current stream, every step of the computation runs in the
library's kernels.  Outputs and workspaces the caller does not pass are
allocated with torch.  A non-OK status raises ``SwigluError``; a missing
library raises ``RuntimeError`` (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libswiglu_mlp.so")

STATUS_NAMES = {
    0: "SWIGLU_OK",
    1: "SWIGLU_ERR_INVALID_ARG",
    2: "SWIGLU_ERR_UNSUPPORTED_SHAPE",
    3: "SWIGLU_ERR_MISALIGNED",
    4: "SWIGLU_ERR_WORKSPACE_TOO_SMALL",
    5: "SWIGLU_ERR_LAUNCH",
    6: "SWIGLU_ERR_TIMEOUT",
    7: "SWIGLU_ERR_CUDA",
}

# Every symbol include/swiglu_mlp.h and include/swiglu_moe.h declare: name -> (restype, argtypes)
_vp, _i64, _i32, _u64, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
SIGNATURES = {
    "swiglu_mlp_fwd_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "swiglu_mlp_bwd_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "swiglu_mlp_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_mlp_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_mlp_fwd_residual": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_mlp_bwd_residual": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_mlp_fwd_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp]),
    "swiglu_mlp_fwd_fp8_workspace_size": (_sz, [_i64, _i64, _i64, _i64]),
    "swiglu_mlp_fwd_fp8": (_i32, [_vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_mlp_fused_grad_preact": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "swiglu_mlp_gemm_bf16": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp]),
    "swiglu_mlp_device_status": (_i32, [_vp]),
    "swiglu_mlp_strerror": (ctypes.c_char_p, [_i32]),
    "swiglu_mlp_last_error_detail": (ctypes.c_char_p, []),
    "swiglu_mlp_set_wait_timeout_ns": (None, [_u64]),
    "swiglu_mlp_set_debug_flags": (None, [_i32]),
    "swiglu_mlp_set_raster_band": (None, [_i32]),
    "swiglu_mlp_split_plan": (_i32, [_i64, _i64, _i64, _i32, _vp, _i32]),
    "swiglu_mlp_trace_begin": (None, [_vp, _vp, _i32]),
    "swiglu_mlp_trace_end": (_i32, []),
    "swiglu_mlp_abi_version": (_i32, []),
    "swiglu_mlp_tp_shard_pack": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp]),
    "swiglu_mlp_tp_shard_unpack_grads": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _vp]),
    "swiglu_mlp_tp_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp, _vp, _sz, _vp]),
    "swiglu_mlp_tp_chunk_rows": (_i64, [_i64, _i32]),
    "swiglu_mlp_tp_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _sz,
                                 _vp]),
    "swiglu_moe_fwd_workspace_size": (_sz, [_vp, _i64, _i64, _i64, _i64]),
    "swiglu_moe_bwd_workspace_size": (_sz, [_vp, _i64, _i64, _i64, _i64]),
    "swiglu_moe_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "swiglu_moe_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _sz,
                              _vp]),
}

KERNEL_KINDS = {1: "fwd_preact", 2: "fwd_down", 3: "bwd_grad_h", 4: "bwd_dW2", 5: "bwd_dx", 6: "bwd_dW1", 7: "gemm",
                8: "bwd_gemms", 9: "elementwise"}


class SwigluError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        self.detail = detail
        msg = f"{where}: {STATUS_NAMES.get(status, status)}"
        super().__init__(f"{msg} ({detail})" if detail else msg)


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise SwigluError(status, where, lib().swiglu_mlp_last_error_detail().decode(errors="replace"))


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if t.dtype not in (torch.bfloat16, torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"expected bf16, FP8 E4M3 (or a uint8 workspace), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    """The current stream of `device`, which must be the current CUDA device: the
    library launches on the current device (and keeps its per-device state there),
    so tensors on another GPU would be addressed from the wrong one."""
    if device is not None:
        device = torch.device(device)
        if device.type == "cuda" and device.index is not None and device.index != torch.cuda.current_device():
            raise ValueError(f"tensors are on {device} but the current CUDA device is cuda:"
                             f"{torch.cuda.current_device()}; call inside torch.cuda.device({device.index})")
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _empty(shape, like: torch.Tensor) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.bfloat16, device=like.device)


# The kernels' tensor maps are built from the sizes, not from the tensors: a buffer of the
# wrong shape would be read or written past its end.  So every tensor a call receives is
# checked against the shape, dtype and device the sizes imply, before anything is launched.

def _expect(t: torch.Tensor, name: str, shape, dtype, device) -> torch.Tensor:
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: {t.dtype}, expected {dtype}")
    if t.device != device:
        raise ValueError(f"{name}: on {t.device}, the call's other tensors are on {device}")
    return t


def _out(t, name: str, shape, like: torch.Tensor, dtype=torch.bfloat16) -> torch.Tensor:
    """A caller's output buffer, checked, or a new one."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    return _expect(t, name, shape, dtype, like.device)


def _same_device(like: torch.Tensor, **tensors) -> None:
    for name, t in tensors.items():
        if t is not None and t.device != like.device:
            raise ValueError(f"{name}: on {t.device}, the call's other tensors are on {like.device}")


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


# ---------------------------------------------------------------------------- sizes / status

def swiglu_mlp_fwd_workspace_size(M: int, D: int, H: int, Dout: int) -> int:
    return int(lib().swiglu_mlp_fwd_workspace_size(M, D, H, Dout))


def swiglu_mlp_bwd_workspace_size(M: int, D: int, H: int, Dout: int) -> int:
    return int(lib().swiglu_mlp_bwd_workspace_size(M, D, H, Dout))


def swiglu_mlp_strerror(status: int) -> str:
    return lib().swiglu_mlp_strerror(status).decode()


def swiglu_mlp_device_status(device=None) -> int:
    """Synchronise the current stream and return the device status code (0 = OK)."""
    return int(lib().swiglu_mlp_device_status(_stream(device)))


def swiglu_mlp_set_wait_timeout_ns(ns: int) -> None:
    lib().swiglu_mlp_set_wait_timeout_ns(int(ns))


def swiglu_mlp_set_debug_flags(flags: int) -> None:
    lib().swiglu_mlp_set_debug_flags(int(flags))


def swiglu_mlp_set_raster_band(n_tiles: int) -> None:
    lib().swiglu_mlp_set_raster_band(int(n_tiles))


def swiglu_mlp_split_plan(M: int, N: int, K: int, units: int):
    """Tile lists of the down projection with split tiles (host only): a list of
    (pair, tile, first k-block, end k-block, split index or -1), or None where the
    forward splits no tiles for this shape."""
    n = int(lib().swiglu_mlp_split_plan(int(M), int(N), int(K), int(units), None, 0))
    if n < 0:
        return None
    buf = (ctypes.c_int32 * (5 * max(n, 1)))()
    lib().swiglu_mlp_split_plan(int(M), int(N), int(K), int(units), ctypes.cast(buf, ctypes.c_void_p), n)
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(n)]


def swiglu_mlp_abi_version() -> int:
    return int(lib().swiglu_mlp_abi_version())


class LaunchTrace:
    """Brackets every kernel launch of the library (from this thread) with CUDA
    events, for per-kernel timing inside larger calls:

        with LaunchTrace(capacity) as tr:
            ...calls...
        tr.records()  ->  [(kind_name, milliseconds), ...] in launch order
    """

    def __init__(self, capacity: int):
        self.capacity = int(capacity)
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * self.capacity)]
        for e in self.events:          # torch creates the CUDA event lazily, on first record
            e.record()
        torch.cuda.synchronize()
        self._handles = (ctypes.c_void_p * len(self.events))(*[e.cuda_event for e in self.events])
        self._kinds = (ctypes.c_int * self.capacity)()
        self.count = 0

    def __enter__(self):
        lib().swiglu_mlp_trace_begin(ctypes.cast(self._handles, ctypes.c_void_p),
                                     ctypes.cast(self._kinds, ctypes.c_void_p), self.capacity)
        return self

    def __exit__(self, *exc):
        self.count = int(lib().swiglu_mlp_trace_end())
        return False

    def records(self):
        torch.cuda.synchronize()
        n = min(self.count, self.capacity)
        return [(KERNEL_KINDS.get(self._kinds[i], str(self._kinds[i])),
                 self.events[2 * i].elapsed_time(self.events[2 * i + 1])) for i in range(n)]


# ---------------------------------------------------------------------------- compute

def _dims(x, W1, W2, dtype=torch.bfloat16):
    M, D = x.shape
    H2, D1 = W1.shape
    Dout, H = W2.shape
    if D1 != D or H2 != 2 * H:
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, W1 {tuple(W1.shape)}, W2 {tuple(W2.shape)}")
    for name, t in (("x", x), ("W1", W1), ("W2", W2)):
        _expect(t, name, t.shape, dtype, x.device)
    return M, D, H, Dout


def swiglu_mlp_fwd(x, W1, W2, preact=None, y=None, workspace=None, residual: bool = False):
    """Forward; returns (preact [M,2H], y [M,Dout]).  residual: y = x + MLP(x)
    (swiglu_mlp_fwd_residual; D == Dout)."""
    M, D, H, Dout = _dims(x, W1, W2)
    preact = _out(preact, "preact", (M, 2 * H), x)
    y = _out(y, "y", (M, Dout), x)
    _same_device(x, workspace=workspace)
    need = swiglu_mlp_fwd_workspace_size(M, D, H, Dout)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    fn = lib().swiglu_mlp_fwd_residual if residual else lib().swiglu_mlp_fwd
    st = fn(_ptr(x), _ptr(W1), _ptr(W2), _ptr(preact), _ptr(y), M, D, H, Dout,
            _ptr(workspace), _nbytes(workspace), _stream(x.device))
    _check(st, "swiglu_mlp_fwd_residual" if residual else "swiglu_mlp_fwd")
    return preact, y


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def swiglu_mlp_fwd_noalloc(x, W1, W2, preact=None, y=None):
    """Forward whose transient h lives in the library's built-in 64 MiB device array
    instead of a caller workspace (for callers that cannot allocate; M*H <= 2^25).
    Calls share that array: calls that overlap on the GPU race.  Returns (preact, y)."""
    M, D, H, Dout = _dims(x, W1, W2)
    preact = _out(preact, "preact", (M, 2 * H), x)
    y = _out(y, "y", (M, Dout), x)
    st = lib().swiglu_mlp_fwd_noalloc(_ptr(x), _ptr(W1), _ptr(W2), _ptr(preact), _ptr(y), M, D, H, Dout,
                                      _stream(x.device))
    _check(st, "swiglu_mlp_fwd_noalloc")
    return preact, y


def swiglu_mlp_bwd(x, W1, W2, preact, dy, dx=None, dW1=None, dW2=None, workspace=None, residual: bool = False):
    """Backward; returns (dx [M,D], dW1 [2H,D], dW2 [Dout,H]).  residual: dx += dy
    (swiglu_mlp_bwd_residual; D == Dout)."""
    M, D, H, Dout = _dims(x, W1, W2)
    _expect(preact, "preact", (M, 2 * H), torch.bfloat16, x.device)
    _expect(dy, "dy", (M, Dout), torch.bfloat16, x.device)
    dx = _out(dx, "dx", (M, D), x)
    dW1 = _out(dW1, "dW1", (2 * H, D), x)
    dW2 = _out(dW2, "dW2", (Dout, H), x)
    _same_device(x, workspace=workspace)
    need = swiglu_mlp_bwd_workspace_size(M, D, H, Dout)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    fn = lib().swiglu_mlp_bwd_residual if residual else lib().swiglu_mlp_bwd
    st = fn(_ptr(x), _ptr(W1), _ptr(W2), _ptr(preact), _ptr(dy), _ptr(dx), _ptr(dW1), _ptr(dW2),
            M, D, H, Dout, _ptr(workspace), _nbytes(workspace), _stream(x.device))
    _check(st, "swiglu_mlp_bwd_residual" if residual else "swiglu_mlp_bwd")
    return dx, dW1, dW2


# ---------------------------------------------------------------------------- tensor-parallel shards

def swiglu_mlp_tp_shard_pack(W1, W2, j0: int, Hs: int, W1_shard=None, W2_shard=None):
    """Rank shard of the full weights: W1_shard [2*Hs, D] (rows j0.. and H + j0..),
    W2_shard [Dout, Hs] (columns j0..)."""
    H2, D = W1.shape
    Dout, H = W2.shape
    if H2 != 2 * H:
        raise ValueError(f"shape mismatch: W1 {tuple(W1.shape)}, W2 {tuple(W2.shape)}")
    _expect(W1, "W1", (2 * H, D), torch.bfloat16, W1.device)
    _expect(W2, "W2", (Dout, H), torch.bfloat16, W1.device)
    W1_shard = _out(W1_shard, "W1_shard", (2 * Hs, D), W1)
    W2_shard = _out(W2_shard, "W2_shard", (Dout, Hs), W1)
    st = lib().swiglu_mlp_tp_shard_pack(_ptr(W1), _ptr(W2), _ptr(W1_shard), _ptr(W2_shard), D, H, Dout, j0, Hs,
                                        _stream(W1.device))
    _check(st, "swiglu_mlp_tp_shard_pack")
    return W1_shard, W2_shard


def swiglu_mlp_tp_shard_unpack_grads(dW1_shard, dW2_shard, dW1, dW2, j0: int):
    """Write a shard's weight gradients into rows j0.., H + j0.. of dW1 and columns j0.. of dW2."""
    H2, D = dW1.shape
    Dout, H = dW2.shape
    Hs = dW2_shard.shape[1]
    _expect(dW1, "dW1", (2 * H, D), torch.bfloat16, dW1.device)
    _expect(dW2, "dW2", (Dout, H), torch.bfloat16, dW1.device)
    _expect(dW1_shard, "dW1_shard", (2 * Hs, D), torch.bfloat16, dW1.device)
    _expect(dW2_shard, "dW2_shard", (Dout, Hs), torch.bfloat16, dW1.device)
    st = lib().swiglu_mlp_tp_shard_unpack_grads(_ptr(dW1_shard), _ptr(dW2_shard), _ptr(dW1), _ptr(dW2), D, H, Dout,
                                                j0, Hs, _stream(dW1.device))
    _check(st, "swiglu_mlp_tp_shard_unpack_grads")
    return dW1, dW2


def swiglu_mlp_tp_chunk_rows(M: int, n_chunks: int) -> int:
    return int(lib().swiglu_mlp_tp_chunk_rows(M, n_chunks))


def _events(events):
    if not events:
        return None, None
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return arr, len(events)


def swiglu_mlp_tp_fwd(x, W1_shard, W2_shard, preact=None, y=None, workspace=None, n_chunks: int = 1,
                      chunk_events=None):
    """Shard forward: (preact_shard [M, 2*Hs], partial y [M, Dout]).  chunk_events: n_chunks
    torch.cuda.Event objects, recorded when the rows of chunk c of y are final."""
    M, D, Hs, Dout = _dims(x, W1_shard, W2_shard)
    preact = _out(preact, "preact", (M, 2 * Hs), x)
    y = _out(y, "y", (M, Dout), x)
    _same_device(x, workspace=workspace)
    if workspace is None:
        workspace = torch.empty(max(16, swiglu_mlp_fwd_workspace_size(M, D, Hs, Dout)), dtype=torch.uint8,
                                device=x.device)
    if chunk_events is not None and len(chunk_events) != n_chunks:
        raise ValueError(f"chunk_events: {len(chunk_events)} events for {n_chunks} chunks")
    for e in chunk_events or ():
        if e.cuda_event == 0:   # a torch event is created on its first record
            e.record(torch.cuda.current_stream(x.device))
    arr, _ = _events(chunk_events)
    st = lib().swiglu_mlp_tp_fwd(_ptr(x), _ptr(W1_shard), _ptr(W2_shard), _ptr(preact), _ptr(y), M, D, Hs, Dout,
                                 n_chunks, arr, _ptr(workspace), _nbytes(workspace), _stream(x.device))
    _check(st, "swiglu_mlp_tp_fwd")
    return preact, y


def swiglu_mlp_tp_bwd(x, W1_shard, W2_shard, preact, dy, dx=None, dW1=None, dW2=None, workspace=None,
                      dx_event=None):
    """Shard backward: (partial dx [M, D], dW1_shard [2*Hs, D], dW2_shard [Dout, Hs]).
    dx_event: a torch.cuda.Event recorded when dx is final, before the weight gradients."""
    M, D, Hs, Dout = _dims(x, W1_shard, W2_shard)
    _expect(preact, "preact", (M, 2 * Hs), torch.bfloat16, x.device)
    _expect(dy, "dy", (M, Dout), torch.bfloat16, x.device)
    dx = _out(dx, "dx", (M, D), x)
    dW1 = _out(dW1, "dW1", (2 * Hs, D), x)
    dW2 = _out(dW2, "dW2", (Dout, Hs), x)
    _same_device(x, workspace=workspace)
    if workspace is None:
        workspace = torch.empty(max(16, swiglu_mlp_bwd_workspace_size(M, D, Hs, Dout)), dtype=torch.uint8,
                                device=x.device)
    ev = None
    if dx_event is not None:
        if dx_event.cuda_event == 0:
            dx_event.record(torch.cuda.current_stream(x.device))
        ev = ctypes.c_void_p(dx_event.cuda_event)
    st = lib().swiglu_mlp_tp_bwd(_ptr(x), _ptr(W1_shard), _ptr(W2_shard), _ptr(preact), _ptr(dy), _ptr(dx),
                                 _ptr(dW1), _ptr(dW2), M, D, Hs, Dout, ev, _ptr(workspace), _nbytes(workspace),
                                 _stream(x.device))
    _check(st, "swiglu_mlp_tp_bwd")
    return dx, dW1, dW2


def bwd_workspace_views(workspace: torch.Tensor, M: int, H: int):
    """(h [M,H], grad_preact [M,2H]) views of a backward workspace."""
    off = ((M * H * 2) + 255) // 256 * 256
    h = workspace[: M * H * 2].view(torch.bfloat16).view(M, H)
    gp = workspace[off: off + M * 2 * H * 2].view(torch.bfloat16).view(M, 2 * H)
    return h, gp


def swiglu_mlp_fwd_fp8_workspace_size(M: int, D: int, H: int, Dout: int) -> int:
    return int(lib().swiglu_mlp_fwd_fp8_workspace_size(M, D, H, Dout))


def swiglu_mlp_fwd_fp8(x8, W1_8, W2_8, s_x: float, s_w1: float, s_w2: float, s_h: float,
                       preact=None, h8=None, y=None, store_preact: bool = True, workspace=None):
    """FP8 forward (E4M3 operands, per-tensor scales); returns (preact [M,2H] bf16 or
    None, h8 [M,H] E4M3, y [M,Dout] bf16)."""
    M, D, H, Dout = _dims(x8, W1_8, W2_8, dtype=torch.float8_e4m3fn)
    if store_preact:
        preact = _out(preact, "preact", (M, 2 * H), x8)
    h8 = _out(h8, "h8", (M, H), x8, dtype=torch.float8_e4m3fn)
    y = _out(y, "y", (M, Dout), x8)
    _same_device(x8, workspace=workspace)
    if workspace is None:
        n = swiglu_mlp_fwd_fp8_workspace_size(M, D, H, Dout)
        workspace = torch.empty(n, dtype=torch.uint8, device=x8.device) if n else None
    st = lib().swiglu_mlp_fwd_fp8(_ptr(x8), _ptr(W1_8), _ptr(W2_8), s_x, s_w1, s_w2, s_h,
                                  _ptr(preact) if store_preact else None, _ptr(h8), _ptr(y), M, D, H, Dout,
                                  _ptr(workspace), _nbytes(workspace), _stream(x8.device))
    _check(st, "swiglu_mlp_fwd_fp8")
    return (preact if store_preact else None), h8, y


def swiglu_mlp_fused_grad_preact(dy, W2, preact, grad_preact=None, h=None):
    """The fused grad_h GEMM + SwiGLU backward alone; returns (grad_preact [M,2H], h [M,H])."""
    M, Dout = dy.shape
    Dout2, H = W2.shape
    if Dout2 != Dout or tuple(preact.shape) != (M, 2 * H):
        raise ValueError("shape mismatch")
    for name, t in (("dy", dy), ("W2", W2), ("preact", preact)):
        _expect(t, name, t.shape, torch.bfloat16, dy.device)
    grad_preact = _out(grad_preact, "grad_preact", (M, 2 * H), dy)
    h = _out(h, "h", (M, H), dy)
    st = lib().swiglu_mlp_fused_grad_preact(_ptr(dy), _ptr(W2), _ptr(preact), _ptr(grad_preact), _ptr(h),
                                            M, H, Dout, _stream(dy.device))
    _check(st, "swiglu_mlp_fused_grad_preact")
    return grad_preact, h


def swiglu_mlp_gemm_bf16(A, B, M: int, N: int, K: int, a_mn_major: bool, b_mn_major: bool, C=None):
    """C [M,N] = A * B^T; A is [M,K] (or [K,M] if a_mn_major), B is [N,K] (or [K,N] if b_mn_major)."""
    _expect(A, "A", (K, M) if a_mn_major else (M, K), torch.bfloat16, A.device)
    _expect(B, "B", (K, N) if b_mn_major else (N, K), torch.bfloat16, A.device)
    C = _out(C, "C", (M, N), A)
    st = lib().swiglu_mlp_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(a_mn_major), int(b_mn_major),
                                    _stream(A.device))
    _check(st, "swiglu_mlp_gemm_bf16")
    return C


class SwiGLUMLP(torch.autograd.Function):
    """autograd wrapper: forward saves (x, W1, W2, preact) and drops h; backward
    calls swiglu_mlp_bwd.  Leading dimensions of x are flattened.  With residual
    set it is the block y = x + MLP(x) (the residual entry points)."""

    @staticmethod
    def forward(ctx, x, W1, W2, residual=False):
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        preact, y = swiglu_mlp_fwd(x2, W1.contiguous(), W2.contiguous(), residual=residual)
        ctx.save_for_backward(x2, W1, W2, preact)
        ctx.residual = residual
        return y.reshape(*x.shape[:-1], y.shape[-1])

    @staticmethod
    def backward(ctx, grad_y):
        x2, W1, W2, preact = ctx.saved_tensors
        dy = grad_y.reshape(-1, grad_y.shape[-1]).contiguous()
        dx, dW1, dW2 = swiglu_mlp_bwd(x2, W1.contiguous(), W2.contiguous(), preact, dy, residual=ctx.residual)
        return dx.reshape(*grad_y.shape[:-1], dx.shape[-1]), dW1, dW2, None


def swiglu_mlp(x, W1, W2, residual: bool = False):
    return SwiGLUMLP.apply(x, W1, W2, residual)


# ---------------------------------------------------------------------------- mixture of experts

def _counts(counts):
    """Host int64 array of the per-expert row counts (kept alive by the caller's frame)."""
    vals = [int(v) for v in (counts.tolist() if hasattr(counts, "tolist") else counts)]
    return (ctypes.c_int64 * len(vals))(*vals), len(vals), sum(vals)


def _moe_dims(x, W1, W2):
    T, D = x.shape
    E, H2, D1 = W1.shape
    E2, Dout, H = W2.shape
    if D1 != D or H2 != 2 * H or E2 != E:
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, W1 {tuple(W1.shape)}, W2 {tuple(W2.shape)}")
    for name, t in (("x", x), ("W1", W1), ("W2", W2)):
        _expect(t, name, t.shape, torch.bfloat16, x.device)
    return T, E, D, H, Dout


def swiglu_moe_fwd_workspace_size(counts, D: int, H: int, Dout: int) -> int:
    arr, E, _ = _counts(counts)
    return int(lib().swiglu_moe_fwd_workspace_size(ctypes.cast(arr, _vp), E, D, H, Dout))


def swiglu_moe_bwd_workspace_size(counts, D: int, H: int, Dout: int) -> int:
    arr, E, _ = _counts(counts)
    return int(lib().swiglu_moe_bwd_workspace_size(ctypes.cast(arr, _vp), E, D, H, Dout))


def swiglu_moe_fwd(x, W1, W2, counts, preact=None, y=None, workspace=None):
    """Forward of every expert on its rows (x grouped by expert, counts per expert);
    returns (preact [T,2H], y [T,Dout])."""
    T, E, D, H, Dout = _moe_dims(x, W1, W2)
    arr, En, total = _counts(counts)
    if En != E or total != T:
        raise ValueError(f"counts: {En} experts summing to {total}, expected {E} and {T}")
    preact = _out(preact, "preact", (T, 2 * H), x)
    y = _out(y, "y", (T, Dout), x)
    _same_device(x, workspace=workspace)
    if workspace is None:
        workspace = torch.empty(max(16, swiglu_moe_fwd_workspace_size(counts, D, H, Dout)), dtype=torch.uint8,
                                device=x.device)
    st = lib().swiglu_moe_fwd(_ptr(x), _ptr(W1), _ptr(W2), _ptr(preact), _ptr(y), ctypes.cast(arr, _vp), E, D, H,
                              Dout, _ptr(workspace), _nbytes(workspace), _stream(x.device))
    _check(st, "swiglu_moe_fwd")
    return preact, y


def swiglu_moe_bwd(x, W1, W2, preact, dy, counts, dx=None, dW1=None, dW2=None, workspace=None):
    """Backward of every expert on its rows; returns (dx [T,D], dW1 [E,2H,D], dW2 [E,Dout,H])."""
    T, E, D, H, Dout = _moe_dims(x, W1, W2)
    arr, En, total = _counts(counts)
    if En != E or total != T:
        raise ValueError(f"counts: {En} experts summing to {total}, expected {E} and {T}")
    _expect(preact, "preact", (T, 2 * H), torch.bfloat16, x.device)
    _expect(dy, "dy", (T, Dout), torch.bfloat16, x.device)
    dx = _out(dx, "dx", (T, D), x)
    dW1 = _out(dW1, "dW1", (E, 2 * H, D), x)
    dW2 = _out(dW2, "dW2", (E, Dout, H), x)
    _same_device(x, workspace=workspace)
    if workspace is None:
        workspace = torch.empty(max(16, swiglu_moe_bwd_workspace_size(counts, D, H, Dout)), dtype=torch.uint8,
                                device=x.device)
    st = lib().swiglu_moe_bwd(_ptr(x), _ptr(W1), _ptr(W2), _ptr(preact), _ptr(dy), _ptr(dx), _ptr(dW1),
                              _ptr(dW2), ctypes.cast(arr, _vp), E, D, H, Dout, _ptr(workspace),
                              _nbytes(workspace), _stream(x.device))
    _check(st, "swiglu_moe_bwd")
    return dx, dW1, dW2
