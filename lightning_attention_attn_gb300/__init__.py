"""GB300-native lightning attention: chunkwise decayed causal linear attention.

Python binding over the C ABI of ``liblightning_attn.so`` (declared in
``include/lightning_attn.h``).  This module only marshals arguments -- torch
tensors become device pointers and sizes, the current CUDA stream becomes a
``cudaStream_t`` -- every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if the library is not built, or a call is not
supported, an exception is raised.

    o_t = sum_{u <= t} lambda_h^(t-u) (q_t . k_u) v_u     (per sequence, head)

(MiniMax-01 technical report, §2.2.1 Lightning Attention, eqs. 4-5 with the
per-head diagonal decay of Fig. 12; §3.3 inference kernels.)
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
import weakref

import torch

from . import workloads  # noqa: F401  (seeded input recipes)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "liblightning_attn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "lightning_attn.h")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT = range(5)
LA_DTYPE_BF16, LA_DTYPE_FP32 = 0, 1

_lock = threading.Lock()
_lib = None


class LightningAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


# Decay tensors already found inside (0, 1]: id -> (weak reference, version).
# Reading the values back costs a device synchronisation, so each tensor is
# checked once per in-place version rather than on every call.
_decay_checked: dict = {}


def check_decay_range(decay: torch.Tensor) -> None:
    """Raise ValueError unless every lambda in ``decay`` lies in (0, 1] (the
    range the method's decay factors assume).  Checked once per tensor and
    in-place version; skipped while a CUDA stream is being captured, where no
    value can be read back."""
    key = id(decay)
    hit = _decay_checked.get(key)
    if hit is not None and hit[0]() is decay and hit[1] == decay._version:
        return
    if decay.is_cuda and torch.cuda.is_current_stream_capturing():
        return
    if not bool(((decay > 0) & (decay <= 1)).all()):
        raise ValueError("decay values must lie in (0, 1]")
    if len(_decay_checked) > 256:
        _decay_checked.clear()
    _decay_checked[key] = (weakref.ref(decay), decay._version)


def header_functions(path: str = HEADER) -> list[str]:
    """Names of the functions the public header declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(lightning_attn_\w+)\s*\(", text, flags=re.M)


def load(path: str = LIB_PATH):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"lightning-attention CUDA library not found at {path}; build it with "
                    "`python -m lightning_attention_attn_gb300.build`")
            lib = ctypes.CDLL(path)
            vp, i32 = ctypes.c_void_p, ctypes.c_int32
            lib.lightning_attn_prefill.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                   i32, ctypes.c_int, vp, vp, vp]
            lib.lightning_attn_prefill.restype = ctypes.c_int
            lib.lightning_attn_prefill_with_state.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32,
                                                              i32, i32, ctypes.c_int, vp, vp,
                                                              vp, vp]
            lib.lightning_attn_prefill_with_state.restype = ctypes.c_int
            lib.lightning_attn_backward.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                    ctypes.c_int, vp, vp, vp, vp, vp,
                                                    ctypes.c_int64, vp]
            lib.lightning_attn_backward.restype = ctypes.c_int
            lib.lightning_attn_backward_workspace_bytes.argtypes = [i32, i32, i32, ctypes.c_int]
            lib.lightning_attn_backward_workspace_bytes.restype = ctypes.c_int64
            lib.lightning_attn_mixed_step.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                      ctypes.c_int, vp, vp, vp, vp, vp]
            lib.lightning_attn_mixed_step.restype = ctypes.c_int
            lib.lightning_attn_prefill_channel_decay.argtypes = [vp, vp, vp, vp, vp, i32, i32,
                                                                 i32, i32, i32, ctypes.c_int, vp,
                                                                 vp, vp, vp]
            lib.lightning_attn_prefill_channel_decay.restype = ctypes.c_int
            lib.lightning_attn_decode_channel_decay.argtypes = [vp, vp, vp, vp, vp, i32, i32,
                                                                i32, ctypes.c_int, vp, vp]
            lib.lightning_attn_decode_channel_decay.restype = ctypes.c_int
            lib.lightning_attn_prefill_snapshots.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32,
                                                             i32, i32, ctypes.c_int, vp, vp, vp,
                                                             i32, vp, vp]
            lib.lightning_attn_prefill_snapshots.restype = ctypes.c_int
            lib.lightning_attn_snapshot_count.argtypes = [vp, i32, i32]
            lib.lightning_attn_snapshot_count.restype = ctypes.c_int64
            lib.lightning_attn_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32,
                                                  ctypes.c_int, vp, vp]
            lib.lightning_attn_decode.restype = ctypes.c_int
            lib.lightning_attn_status_string.argtypes = [ctypes.c_int]
            lib.lightning_attn_status_string.restype = ctypes.c_char_p
            lib.lightning_attn_last_error.argtypes = []
            lib.lightning_attn_last_error.restype = ctypes.c_char_p
            lib.lightning_attn_version.argtypes = []
            lib.lightning_attn_version.restype = ctypes.c_int32
            lib.lightning_attn_device_status.argtypes = [vp]
            lib.lightning_attn_device_status.restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != LA_OK:
        lib = load()
        name = lib.lightning_attn_status_string(status).decode()
        msg = lib.lightning_attn_last_error().decode()
        raise LightningAttnError(status, f"{what}: {name}: {msg}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LA_DTYPE_BF16
    if t.dtype == torch.float32:
        return LA_DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def prefill(q, k, v, decay, cu_seqlens=None, *, chunk: int = 0, out=None,
            final_state=None, return_state: bool = True, stream=None,
            initial_state=None):
    """Chunkwise lightning-attention prefill.

    q, k, v: [T, H, d] (bf16 or fp32, same dtype, CUDA, contiguous), packed
    token-major; cu_seqlens: int32 [nseq + 1] on the device (None = one
    sequence of length T); decay: fp32 [H].  Returns ``(out, final_state)``
    with out [T, H, d] in the input dtype and final_state fp32
    [nseq, H, d, d] (None if ``return_state`` is False).

    initial_state: optional fp32 [nseq, H, d, d] cached state each sequence
    continues from (prefix KV cache); it may be passed as ``final_state``
    too, to update the cache in place.
    """
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor")
    if decay.dtype != torch.float32 or decay.numel() != H:
        raise ValueError("decay must be fp32 [H]")
    check_decay_range(decay)
    nseq = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if final_state is None and return_state:
        final_state = torch.empty((nseq, H, d, d), dtype=torch.float32, device=q.device)
    if initial_state is not None and (initial_state.dtype != torch.float32 or
                                      tuple(initial_state.shape) != (nseq, H, d, d)):
        raise ValueError("initial_state must be fp32 [nseq, H, d, d]")
    lib = load()
    fs = None if final_state is None else _dev(final_state, "final_state")
    if initial_state is None:
        st = lib.lightning_attn_prefill(
            _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
            _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, int(chunk), _dtype_code(q),
            _dev(out, "out"), fs, _stream_handle(stream))
        _check(st, "lightning_attn_prefill")
    else:
        st = lib.lightning_attn_prefill_with_state(
            _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
            _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, int(chunk), _dtype_code(q),
            _dev(initial_state, "initial_state"), _dev(out, "out"), fs,
            _stream_handle(stream))
        _check(st, "lightning_attn_prefill_with_state")
    return out, final_state


def backward_workspace_bytes(total_tokens: int, num_heads: int, head_dim: int,
                             dtype=torch.bfloat16) -> int:
    """Bytes of device workspace :func:`backward` needs."""
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_FP32
    n = int(load().lightning_attn_backward_workspace_bytes(total_tokens, num_heads, head_dim,
                                                             code))
    if n < 0:
        raise ValueError("invalid sizes for the backward workspace")
    return n


def backward(q, k, v, decay, cu_seqlens, dout, *, chunk: int = 0, dq=None, dk=None,
             dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of sum_t dout_t . o_t for o = prefill(q, k, v,
    decay, cu_seqlens) (zero initial states).  Shapes and dtypes as in
    :func:`prefill`; ``workspace`` is a uint8 CUDA tensor of at least
    :func:`backward_workspace_bytes` bytes, needed on the CUDA-core path
    only (allocated here when None); the tensor-core path (bf16, d = 128,
    chunk 0, 16, 32, 64, 128 or 256) runs without one.
    """
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor")
    if decay.dtype != torch.float32 or decay.numel() != H:
        raise ValueError("decay must be fp32 [H]")
    check_decay_range(decay)
    nseq = cu_seqlens.numel() - 1
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    tensor_cores = q.dtype == torch.bfloat16 and d == 128 and int(chunk) in (0, 16, 32, 64, 128, 256)
    if workspace is None and not tensor_cores:
        need = backward_workspace_bytes(T, H, d, q.dtype)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    ws_ptr = None if workspace is None else _dev(workspace, "workspace")
    ws_bytes = 0 if workspace is None else int(workspace.numel() * workspace.element_size())
    st = load().lightning_attn_backward(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
        _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, int(chunk), _dtype_code(q),
        _dev(dout, "dout"), _dev(dq, "dq"), _dev(dk, "dk"), _dev(dv, "dv"),
        ws_ptr, ws_bytes, _stream_handle(stream))
    _check(st, "lightning_attn_backward")
    return dq, dk, dv


def mixed_step(q, k, v, decay, cu_seqlens, state, *, out=None, prefill_stream=None,
               decode_stream=None, cu_seqlens_host=None):
    """One serving step over a packed batch continuing from cached states:
    sequences with one new token take the decode kernel on ``decode_stream``,
    longer ones the chunkwise prefill on ``prefill_stream``; ``state`` fp32
    [nseq, H, d, d] is updated in place.  Returns out [T, H, d]; the step is
    ordered on ``prefill_stream`` (the current stream when None).
    ``cu_seqlens_host`` (a host sequence of ints, optional) lets the prefill
    launch cover only the sequences with two or more new tokens.  A decode
    stream of higher priority than the prefill stream (e.g.
    ``torch.cuda.Stream(priority=-1)``) lets the small decode blocks start
    before the prefill's large ones fill the SMs."""
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor")
    if decay.dtype != torch.float32 or decay.numel() != H:
        raise ValueError("decay must be fp32 [H]")
    check_decay_range(decay)
    nseq = cu_seqlens.numel() - 1
    if state.dtype != torch.float32 or tuple(state.shape) != (nseq, H, d, d):
        raise ValueError("state must be fp32 [nseq, H, d, d]")
    if out is None:
        out = torch.empty_like(q)
    ps = _stream_handle(prefill_stream)
    ds = ps if decode_stream is None else int(decode_stream.cuda_stream)
    host_cu = None
    if cu_seqlens_host is not None:
        host_cu = (ctypes.c_int32 * (nseq + 1))(*[int(x) for x in cu_seqlens_host])
    st = load().lightning_attn_mixed_step(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
        _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, _dtype_code(q), _dev(state, "state"),
        _dev(out, "out"), None if host_cu is None else ctypes.addressof(host_cu), ps, ds)
    _check(st, "lightning_attn_mixed_step")
    return out


def snapshot_count(cu_seqlens, snapshot_interval: int) -> int:
    """Number of per-block state snapshots :func:`prefill_snapshots` writes:
    sum over sequences of floor(L_s / snapshot_interval).  ``cu_seqlens`` may
    live on either device (a host copy is made)."""
    cu = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
    n = int(load().lightning_attn_snapshot_count(cu.data_ptr(), cu.numel() - 1,
                                                 int(snapshot_interval)))
    if n < 0:
        raise ValueError("invalid cu_seqlens or snapshot_interval")
    return n


def prefill_snapshots(q, k, v, decay, cu_seqlens, snapshot_interval: int, *, chunk: int = 0,
                      out=None, final_state=None, snapshots=None, initial_state=None,
                      stream=None):
    """Prefill that also returns the state after every ``snapshot_interval``
    tokens of each sequence (a per-block prefix cache).  Returns ``(out,
    final_state, snapshots)`` with snapshots fp32 [N, H, d, d] in sequence
    order (see :func:`snapshot_count`); the interval is a multiple of the
    block the call computes with (128 on the tensor-core path)."""
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor")
    if decay.dtype != torch.float32 or decay.numel() != H:
        raise ValueError("decay must be fp32 [H]")
    check_decay_range(decay)
    nseq = cu_seqlens.numel() - 1
    if snapshots is None:
        # sizing needs the lengths on the host (one synchronising copy); pass
        # `snapshots` of snapshot_count() entries to avoid it
        n = snapshot_count(cu_seqlens, snapshot_interval)
        snapshots = torch.empty((max(n, 1), H, d, d), dtype=torch.float32,
                                device=q.device)[:n]
    elif snapshots.dtype != torch.float32 or snapshots.dim() != 4 or \
            tuple(snapshots.shape[1:]) != (H, d, d):
        raise ValueError("snapshots must be fp32 [N, H, d, d] with N = snapshot_count()")
    if out is None:
        out = torch.empty_like(q)
    if final_state is None:
        final_state = torch.empty((nseq, H, d, d), dtype=torch.float32, device=q.device)
    st = load().lightning_attn_prefill_snapshots(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
        _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, int(chunk), _dtype_code(q),
        None if initial_state is None else _dev(initial_state, "initial_state"),
        _dev(out, "out"), _dev(final_state, "final_state"), int(snapshot_interval),
        _dev(snapshots, "snapshots"), _stream_handle(stream))
    _check(st, "lightning_attn_prefill_snapshots")
    return out, final_state, snapshots


def prefill_channel_decay(q, k, v, decay, cu_seqlens=None, *, chunk: int = 0, out=None,
                          final_state=None, return_state: bool = True, stream=None,
                          initial_state=None):
    """Prefill with one decay per head and key channel: ``decay`` fp32
    [H, d].  Otherwise as :func:`prefill`, with chunk 0, 16, 32 or 64: bf16
    with d = 128 and chunk 0 or 64 runs the tensor-core kernel, the rest the
    CUDA-core kernel."""
    if q.dim() != 3:
        raise ValueError("q must be [T, H, d]")
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=q.device)
    if decay.dtype != torch.float32 or tuple(decay.shape) != (H, d):
        raise ValueError("decay must be fp32 [H, d]")
    check_decay_range(decay)
    nseq = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    if final_state is None and return_state:
        final_state = torch.empty((nseq, H, d, d), dtype=torch.float32, device=q.device)
    st = load().lightning_attn_prefill_channel_decay(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
        _dev(cu_seqlens, "cu_seqlens"), nseq, T, H, d, int(chunk), _dtype_code(q),
        None if initial_state is None else _dev(initial_state, "initial_state"),
        _dev(out, "out"), None if final_state is None else _dev(final_state, "final_state"),
        _stream_handle(stream))
    _check(st, "lightning_attn_prefill_channel_decay")
    return out, final_state


def decode_channel_decay(q, k, v, decay, state, *, out=None, stream=None):
    """Decode step with one decay per head and key channel (decay fp32 [H, d])."""
    Bn, H, d = q.shape
    if decay.dtype != torch.float32 or tuple(decay.shape) != (H, d):
        raise ValueError("decay must be fp32 [H, d]")
    check_decay_range(decay)
    if out is None:
        out = torch.empty_like(q)
    st = load().lightning_attn_decode_channel_decay(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"), _dev(state, "state"),
        Bn, H, d, _dtype_code(q), _dev(out, "out"), _stream_handle(stream))
    _check(st, "lightning_attn_decode_channel_decay")
    return out


def decode(q, k, v, decay, state, *, out=None, stream=None):
    """One decode step: state <- lambda state + k^T v (in place), out = q state.

    q, k, v: [B, H, d]; state: fp32 [B, H, d, d] (updated in place);
    decay: fp32 [H].  Returns out [B, H, d] in the input dtype.
    """
    if q.dim() != 3:
        raise ValueError("q must be [B, H, d]")
    Bn, H, d = q.shape
    for name, t in (("k", k), ("v", v)):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise ValueError(f"{name} must match q in shape and dtype")
    if state.dtype != torch.float32 or tuple(state.shape) != (Bn, H, d, d):
        raise ValueError("state must be fp32 [B, H, d, d]")
    if decay.dtype != torch.float32 or decay.numel() != H:
        raise ValueError("decay must be fp32 [H]")
    check_decay_range(decay)
    if out is None:
        out = torch.empty_like(q)
    lib = load()
    st = lib.lightning_attn_decode(
        _dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(decay, "decay"),
        _dev(state, "state"), Bn, H, d, _dtype_code(q), _dev(out, "out"),
        _stream_handle(stream))
    _check(st, "lightning_attn_decode")
    return out


def device_status(stream=None) -> None:
    """Synchronises ``stream`` and raises if a kernel reported a device-side
    error (a bounded wait that gave up)."""
    _check(load().lightning_attn_device_status(_stream_handle(stream)),
           "lightning_attn_device_status")


def version() -> tuple[int, int]:
    v = int(load().lightning_attn_version())
    return v >> 16, v & 0xFFFF
