"""CPU fp64 oracle for lightning attention -- test infrastructure only.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never loads it, and it never loads the product path.

The arithmetic lives in ``lightning_oracle.c`` (plain C, fp64, OpenMP over
(sequence, head)); this module compiles it with gcc and marshals numpy arrays.
Sources followed (MiniMax-01 technical report, CSDN full translation):
  * §2.2.1, eq. 4 -- left product  O = [(Q K^T) (.) M] V, M_ts = [t >= s]
  * §2.2.1, eq. 5 -- right-product recursion kv_t = kv_{t-1} + k_t^T v_t
  * Fig. 12 caption -- the diagonal decay matrix: weight lambda_h^(t-u)
  * §3.2 "data packing" -- packed sequences are independent
  * §3.3.1 prefix KV cache -- a sequence may continue from a cached state
  * gradients of the left product for training (§2.2.1, §2.2.2)
  * channel-wise (per key channel) decay -- K3 report reading notes
Parity pins: tests/test_oracle.py (golden hand examples, closed forms,
two-form agreement, exact rational brute force, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lightning_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblightning_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_up = ctypes.POINTER(ctypes.c_uint8)


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (-O2 -fopenmp, no -ffast-math, no FMA
    contraction) into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def _declare(lib):
    lib.la_oracle_quadratic.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, _up, _dp, _dp,
                                        ctypes.c_int]
    lib.la_oracle_recurrent.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, _up, _dp, _dp,
                                        _dp, ctypes.c_int]
    lib.la_oracle_decode.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, _dp, ctypes.c_int]
    lib.la_oracle_max_threads.argtypes = [ctypes.c_int]
    lib.la_oracle_backward.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _dp, _dp, _dp, _dp, ctypes.c_int]
    lib.la_oracle_quadratic_cw.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, _dp, _dp, ctypes.c_int]
    lib.la_oracle_recurrent_cw.argtypes = [_dp, _dp, _dp, _dp, _ip, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, _dp, _dp, _dp, ctypes.c_int]
    lib.la_oracle_decode_cw.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, _dp, ctypes.c_int]
    for f in (lib.la_oracle_quadratic, lib.la_oracle_recurrent,
              lib.la_oracle_decode, lib.la_oracle_max_threads, lib.la_oracle_backward,
              lib.la_oracle_quadratic_cw, lib.la_oracle_recurrent_cw, lib.la_oracle_decode_cw):
        f.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library.  With ``path``
    given, load that library instead (used to test planted mutants)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _f64(a) -> np.ndarray:
    """fp64 C-contiguous copy of an array-like (torch tensors included:
    bf16/fp32 values are upcast exactly)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def decay_as_seen(decay) -> np.ndarray:
    """The per-head decay the kernels see: fp32-rounded, promoted to fp64."""
    if hasattr(decay, "detach"):
        decay = decay.detach().to("cpu").numpy()
    return np.asarray(decay, dtype=np.float32).astype(np.float64)


def _shape(q):
    T, H, d = q.shape
    return T, H, d


def _sel(head_sel, H):
    if head_sel is None:
        return None
    m = np.zeros(H, dtype=np.uint8)
    m[np.asarray(list(head_sel), dtype=np.int64)] = 1
    return m


def _init(initial_state, nseq, H, d):
    if initial_state is None:
        return None
    s0 = _f64(initial_state)
    assert s0.shape == (nseq, H, d, d), s0.shape
    return s0


def quadratic(q, k, v, decay, cu_seqlens, heads=None, nthreads=0, lib=None,
              initial_state=None):
    """Left-product form.  q, k, v: [T, H, d]; decay: [H]; cu_seqlens:
    [nseq+1]; initial_state: cached state per sequence [nseq, H, d, d] or
    None.  Returns out [T, H, d] fp64 (rows of unselected heads are 0)."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    lam = _f64(decay_as_seen(decay))
    cu = _i32(cu_seqlens)
    T, H, d = _shape(q)
    assert cu[-1] == T
    s0 = _init(initial_state, len(cu) - 1, H, d)
    out = np.zeros((T, H, d), dtype=np.float64)
    sel = _sel(heads, H)
    rc = lib.la_oracle_quadratic(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                                 _ptr(lam, _dp), _ptr(cu, _ip), len(cu) - 1, H,
                                 d, None if sel is None else _ptr(sel, _up),
                                 None if s0 is None else _ptr(s0, _dp),
                                 _ptr(out, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_quadratic failed ({rc})")
    return out


def recurrent(q, k, v, decay, cu_seqlens, heads=None, want_out=True,
              nthreads=0, lib=None, initial_state=None):
    """Right-product recursion, from zero or from ``initial_state``
    [nseq, H, d, d].  Returns (out [T,H,d] or None, final_state [nseq,H,d,d]),
    both fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    lam = _f64(decay_as_seen(decay))
    cu = _i32(cu_seqlens)
    T, H, d = _shape(q)
    assert cu[-1] == T
    nseq = len(cu) - 1
    out = np.zeros((T, H, d), dtype=np.float64) if want_out else None
    st = np.zeros((nseq, H, d, d), dtype=np.float64)
    s0 = _init(initial_state, nseq, H, d)
    sel = _sel(heads, H)
    rc = lib.la_oracle_recurrent(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                                 _ptr(lam, _dp), _ptr(cu, _ip), nseq, H, d,
                                 None if sel is None else _ptr(sel, _up),
                                 None if s0 is None else _ptr(s0, _dp),
                                 None if out is None else _ptr(out, _dp),
                                 _ptr(st, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_recurrent failed ({rc})")
    return out, st


def decode(q, k, v, decay, state, nthreads=0, lib=None):
    """One recurrent step per (sequence, head).  q, k, v: [B, H, d];
    state: [B, H, d, d].  Returns (out [B,H,d], new_state), fp64; the input
    state is not modified."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    lam = _f64(decay_as_seen(decay))
    st = _f64(state).copy()
    B, H, d = q.shape
    out = np.zeros((B, H, d), dtype=np.float64)
    rc = lib.la_oracle_decode(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                              _ptr(lam, _dp), _ptr(st, _dp), B, H, d,
                              _ptr(out, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_decode failed ({rc})")
    return out, st


def backward(q, k, v, decay, cu_seqlens, dout, nthreads=0, lib=None):
    """Gradients (dq, dk, dv) [T, H, d] fp64 of sum_t dout_t . o_t, with o
    the left-product form (zero state at each sequence start)."""
    lib = lib or load()
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    lam = _f64(decay_as_seen(decay))
    cu = _i32(cu_seqlens)
    T, H, d = _shape(q)
    assert cu[-1] == T and g.shape == q.shape
    dq, dk, dv = (np.zeros((T, H, d), dtype=np.float64) for _ in range(3))
    rc = lib.la_oracle_backward(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(lam, _dp),
                                _ptr(cu, _ip), len(cu) - 1, H, d, _ptr(g, _dp),
                                _ptr(dq, _dp), _ptr(dk, _dp), _ptr(dv, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_backward failed ({rc})")
    return dq, dk, dv


def _decay_cw(decay, H, d):
    lam = _f64(decay_as_seen(decay)).reshape(-1)
    assert lam.size == H * d, "channel-wise decay must be [H, d]"
    return np.ascontiguousarray(lam)


def quadratic_cw(q, k, v, decay, cu_seqlens, nthreads=0, lib=None, initial_state=None):
    """Left-product form with channel-wise decay (decay [H, d]: lambda of
    each key channel).  Returns out [T, H, d] fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = _i32(cu_seqlens)
    T, H, d = _shape(q)
    assert cu[-1] == T
    lam = _decay_cw(decay, H, d)
    s0 = _init(initial_state, len(cu) - 1, H, d)
    out = np.zeros((T, H, d), dtype=np.float64)
    rc = lib.la_oracle_quadratic_cw(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(lam, _dp),
                                    _ptr(cu, _ip), len(cu) - 1, H, d,
                                    None if s0 is None else _ptr(s0, _dp), _ptr(out, _dp),
                                    nthreads)
    if rc:
        raise ValueError(f"la_oracle_quadratic_cw failed ({rc})")
    return out


def recurrent_cw(q, k, v, decay, cu_seqlens, nthreads=0, lib=None, initial_state=None):
    """Recursion with channel-wise decay.  Returns (out, final_state) fp64."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu = _i32(cu_seqlens)
    T, H, d = _shape(q)
    assert cu[-1] == T
    nseq = len(cu) - 1
    lam = _decay_cw(decay, H, d)
    s0 = _init(initial_state, nseq, H, d)
    out = np.zeros((T, H, d), dtype=np.float64)
    st = np.zeros((nseq, H, d, d), dtype=np.float64)
    rc = lib.la_oracle_recurrent_cw(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(lam, _dp),
                                    _ptr(cu, _ip), nseq, H, d,
                                    None if s0 is None else _ptr(s0, _dp), _ptr(out, _dp),
                                    _ptr(st, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_recurrent_cw failed ({rc})")
    return out, st


def decode_cw(q, k, v, decay, state, nthreads=0, lib=None):
    """One decode step with channel-wise decay; returns (out, new_state)."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    st = _f64(state).copy()
    B, H, d = q.shape
    lam = _decay_cw(decay, H, d)
    out = np.zeros((B, H, d), dtype=np.float64)
    rc = lib.la_oracle_decode_cw(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(lam, _dp),
                                 _ptr(st, _dp), B, H, d, _ptr(out, _dp), nthreads)
    if rc:
        raise ValueError(f"la_oracle_decode_cw failed ({rc})")
    return out, st


def max_threads(nthreads: int = 0) -> int:
    """Threads the oracle's OpenMP regions use (after an optional request)."""
    return int(load().la_oracle_max_threads(nthreads))


def source_path() -> str:
    return _SRC
