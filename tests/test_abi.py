"""C-ABI checks that need no GPU: the library loads, exports every function
the public header declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import subprocess

import pytest

import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild


@pytest.fixture(scope="module")
def lib():
    path = labuild.build()
    return la.load(path)


def test_header_declares_expected_calls():
    names = la.header_functions()
    for n in ("lightning_attn_prefill", "lightning_attn_prefill_with_state",
              "lightning_attn_backward", "lightning_attn_backward_workspace_bytes",
              "lightning_attn_mixed_step", "lightning_attn_prefill_channel_decay",
              "lightning_attn_decode_channel_decay",
              "lightning_attn_prefill_snapshots", "lightning_attn_snapshot_count",
              "lightning_attn_decode",
              "lightning_attn_status_string", "lightning_attn_last_error",
              "lightning_attn_version", "lightning_attn_device_status",
              "lightning_attn_selftest_wait_timeout"):
        assert n in names, n


def test_library_exports_every_header_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", la.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in la.header_functions():
        assert name in exported, f"{name} declared in the header but not exported"
        assert hasattr(lib, name)


def test_version(lib):
    assert la.version() == (1, 5)


def test_status_strings(lib):
    for code, name in enumerate(["LA_OK", "LA_ERR_INVALID_ARG", "LA_ERR_UNSUPPORTED",
                                 "LA_ERR_CUDA", "LA_ERR_TIMEOUT"]):
        assert lib.lightning_attn_status_string(code).decode() == name
    assert lib.lightning_attn_status_string(99).decode() == "LA_ERR_UNKNOWN"


A = 0x10000  # a 16-byte aligned fake address: validation must fail before any use


def _prefill(lib, **kw):
    args = dict(q=A, k=A, v=A, decay=A, cu=A, nseq=1, T=8, H=2, d=128, chunk=0,
                dtype=la.LA_DTYPE_BF16, out=A, fs=A, stream=None)
    args.update(kw)
    return lib.lightning_attn_prefill(args["q"], args["k"], args["v"], args["decay"],
                                      args["cu"], args["nseq"], args["T"], args["H"],
                                      args["d"], args["chunk"], args["dtype"], args["out"],
                                      args["fs"], args["stream"])


@pytest.mark.parametrize("kw, status", [
    (dict(nseq=-1), la.LA_ERR_INVALID_ARG),
    (dict(T=-5), la.LA_ERR_INVALID_ARG),
    (dict(H=0), la.LA_ERR_INVALID_ARG),
    (dict(d=96), la.LA_ERR_INVALID_ARG),
    (dict(dtype=7), la.LA_ERR_INVALID_ARG),
    (dict(chunk=48), la.LA_ERR_INVALID_ARG),
    (dict(q=None), la.LA_ERR_INVALID_ARG),
    (dict(out=None), la.LA_ERR_INVALID_ARG),
    (dict(cu=None), la.LA_ERR_INVALID_ARG),
    (dict(decay=None), la.LA_ERR_INVALID_ARG),
    (dict(q=A + 4), la.LA_ERR_INVALID_ARG),
    (dict(fs=A + 8), la.LA_ERR_INVALID_ARG),
    (dict(dtype=la.LA_DTYPE_FP32, chunk=128), la.LA_ERR_UNSUPPORTED),
    (dict(d=64, chunk=256), la.LA_ERR_UNSUPPORTED),
    (dict(nseq=0), la.LA_OK),  # nothing to do: returns before any CUDA call
])
def test_prefill_host_validation(lib, kw, status):
    assert _prefill(lib, **kw) == status


def _prefill_state(lib, init, **kw):
    args = dict(q=A, k=A, v=A, decay=A, cu=A, nseq=1, T=8, H=2, d=128, chunk=0,
                dtype=la.LA_DTYPE_BF16, out=A, fs=A + 0x100000, stream=None)
    args.update(kw)
    return lib.lightning_attn_prefill_with_state(
        args["q"], args["k"], args["v"], args["decay"], args["cu"], args["nseq"], args["T"],
        args["H"], args["d"], args["chunk"], args["dtype"], init, args["out"], args["fs"],
        args["stream"])


@pytest.mark.parametrize("init, kw, status", [
    (A + 4, {}, la.LA_ERR_INVALID_ARG),                      # misaligned cached state
    (A + 0x100000 + 16, {}, la.LA_ERR_INVALID_ARG),          # overlaps final_state partly
    (A + 0x100000 - 16, {}, la.LA_ERR_INVALID_ARG),          # overlaps final_state partly
    (A, dict(H=0), la.LA_ERR_INVALID_ARG),
    (A, dict(nseq=0), la.LA_OK),
])
def test_prefill_with_state_host_validation(lib, init, kw, status):
    assert _prefill_state(lib, init, **kw) == status
    if status != la.LA_OK:
        assert lib.lightning_attn_last_error().decode() != ""


def _decode(lib, **kw):
    args = dict(q=A, k=A, v=A, decay=A, state=A, B=4, H=2, d=128,
                dtype=la.LA_DTYPE_BF16, out=A, stream=None)
    args.update(kw)
    return lib.lightning_attn_decode(args["q"], args["k"], args["v"], args["decay"],
                                     args["state"], args["B"], args["H"], args["d"],
                                     args["dtype"], args["out"], args["stream"])


@pytest.mark.parametrize("kw, status", [
    (dict(B=-1), la.LA_ERR_INVALID_ARG),
    (dict(H=0), la.LA_ERR_INVALID_ARG),
    (dict(d=32), la.LA_ERR_INVALID_ARG),
    (dict(dtype=3), la.LA_ERR_INVALID_ARG),
    (dict(state=None), la.LA_ERR_INVALID_ARG),
    (dict(out=A + 2), la.LA_ERR_INVALID_ARG),
    (dict(B=0), la.LA_OK),
])
def test_decode_host_validation(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_binding_fails_loudly_without_library(tmp_path):
    import importlib
    mod = importlib.import_module("lightning_attention_attn_gb300")
    with pytest.raises(RuntimeError, match="not found"):
        # a fresh loader pointed at a missing file must raise, never fall back
        saved = mod._lib
        mod._lib = None
        try:
            mod.load(str(tmp_path / "missing.so"))
        finally:
            mod._lib = saved


def test_product_path_does_not_import_oracle():
    pkg = os.path.dirname(la.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "lightning_oracle" not in text, f


def test_backward_workspace_bytes(lib):
    f = lib.lightning_attn_backward_workspace_bytes
    assert f(8192, 64, 128, la.LA_DTYPE_BF16) == 3 * 8192 * 64 * 128 * 2
    assert f(3, 1, 64, la.LA_DTYPE_FP32) == 3 * 768          # 768 B per array, 256-aligned
    assert f(0, 4, 128, la.LA_DTYPE_BF16) == 0
    assert f(-1, 4, 128, la.LA_DTYPE_BF16) == -1
    assert f(8, 4, 96, la.LA_DTYPE_BF16) == -1


W = 0x200000  # 256-byte aligned fake workspace address


def _backward(lib, **kw):
    args = dict(q=A, k=A + 0x10, v=A + 0x20, decay=A, cu=A, nseq=1, T=8, H=2, d=128, chunk=0,
                dtype=la.LA_DTYPE_BF16, g=A + 0x30, dq=A + 0x40000, dk=A + 0x50000,
                dv=A + 0x60000, ws=W, wsb=1 << 20, stream=None)
    args.update(kw)
    return lib.lightning_attn_backward(
        args["q"], args["k"], args["v"], args["decay"], args["cu"], args["nseq"], args["T"],
        args["H"], args["d"], args["chunk"], args["dtype"], args["g"], args["dq"], args["dk"],
        args["dv"], args["ws"], args["wsb"], args["stream"])


@pytest.mark.parametrize("kw, status", [
    # the workspace is checked on the CUDA-core path (fp32), which uses it
    (dict(ws=None, dtype=la.LA_DTYPE_FP32), la.LA_ERR_INVALID_ARG),
    (dict(wsb=100, dtype=la.LA_DTYPE_FP32), la.LA_ERR_INVALID_ARG),    # workspace too small
    (dict(ws=W + 16, dtype=la.LA_DTYPE_FP32), la.LA_ERR_INVALID_ARG),  # not 256-aligned
    (dict(ws=None, dq=A), la.LA_ERR_INVALID_ARG),           # tensor-core path, no workspace:
                                                            # the other checks still apply
    (dict(dq=A), la.LA_ERR_INVALID_ARG),                    # gradient aliases q
    (dict(dk=A + 0x40000), la.LA_ERR_INVALID_ARG),          # dk is dq
    (dict(g=A + 8), la.LA_ERR_INVALID_ARG),                 # misaligned
    (dict(d=96), la.LA_ERR_INVALID_ARG),
    (dict(nseq=0), la.LA_OK),
    (dict(T=0), la.LA_OK),
])
def test_backward_host_validation(lib, kw, status):
    assert _backward(lib, **kw) == status


def test_backward_noalloc_rejects_sizes_beyond_its_array(lib):
    f = lib.lightning_attn_backward_noalloc
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int32] * 5 + [ctypes.c_int] + \
        [ctypes.c_void_p] * 5
    f.restype = ctypes.c_int
    lib.lightning_attn_backward_noalloc_max_bytes.restype = ctypes.c_int64
    cap = lib.lightning_attn_backward_noalloc_max_bytes()
    assert cap == 64 << 20
    # fp32: the CUDA-core path, whose time reversals need the scratch
    T = cap // (3 * 64 * 128 * 4) + 1  # one token more than the array holds (fp32)
    st = f(A, A, A, A, A, 1, T, 64, 128, 64, la.LA_DTYPE_FP32, A, A + 0x40000, A + 0x50000,
           A + 0x60000, None)
    assert st == la.LA_ERR_INVALID_ARG
    assert "scratch" in lib.lightning_attn_last_error().decode()


@pytest.mark.parametrize("kw, status", [
    (dict(state=None), la.LA_ERR_INVALID_ARG),
    (dict(state=A + 4), la.LA_ERR_INVALID_ARG),
    (dict(d=80), la.LA_ERR_INVALID_ARG),
    (dict(nseq=0), la.LA_OK),
])
def test_mixed_step_host_validation(lib, kw, status):
    args = dict(q=A, k=A, v=A, decay=A, cu=A, nseq=4, T=9, H=2, d=128,
                dtype=la.LA_DTYPE_BF16, state=A + 0x100000, out=A + 0x200000)
    args.update(kw)
    st = lib.lightning_attn_mixed_step(args["q"], args["k"], args["v"], args["decay"], args["cu"],
                                       args["nseq"], args["T"], args["H"], args["d"],
                                       args["dtype"], args["state"], args["out"], None, None,
                                       None)
    assert st == status


def test_channel_decay_host_validation(lib):
    f = lib.lightning_attn_prefill_channel_decay
    common = (A, A, A, A, A, 1, 8, 2, 128)
    # chunk 128 is the tensor-core block, which has no channel-wise variant
    assert f(*common, 128, la.LA_DTYPE_BF16, None, A, A, None) == la.LA_ERR_UNSUPPORTED
    assert f(*common, 48, la.LA_DTYPE_BF16, None, A, A, None) == la.LA_ERR_INVALID_ARG
    assert f(A, A, A, A + 4, A, 1, 8, 2, 128, 0, la.LA_DTYPE_BF16, None, A, A, None) == \
        la.LA_ERR_INVALID_ARG
    assert f(A, A, A, A, A, 0, 8, 2, 128, 0, la.LA_DTYPE_BF16, None, A, A, None) == la.LA_OK
    g = lib.lightning_attn_decode_channel_decay
    assert g(A, A, A, A, A, 4, 2, 96, la.LA_DTYPE_BF16, A, None) == la.LA_ERR_INVALID_ARG
    assert g(A, A, A, A, A, 0, 2, 128, la.LA_DTYPE_BF16, A, None) == la.LA_OK


def test_snapshot_host_validation(lib):
    f = lib.lightning_attn_prefill_snapshots
    common = (A, A, A, A, A, 1, 8, 2, 128)
    # interval <= 0, or not a multiple of the block the call computes with
    assert f(*common, 0, la.LA_DTYPE_BF16, None, A, A, 0, A, None) == la.LA_ERR_INVALID_ARG
    assert f(*common, 0, la.LA_DTYPE_BF16, None, A, A, 192, A, None) == la.LA_ERR_INVALID_ARG
    assert f(*common, 0, la.LA_DTYPE_FP32, None, A, A, 96, A, None) == la.LA_ERR_INVALID_ARG
    assert f(*common, 32, la.LA_DTYPE_FP32, None, A, A, 48, A, None) == la.LA_ERR_INVALID_ARG
    # missing or misaligned snapshot array
    assert f(*common, 0, la.LA_DTYPE_BF16, None, A, A, 256, None, None) == la.LA_ERR_INVALID_ARG
    assert f(*common, 0, la.LA_DTYPE_BF16, None, A, A, 256, A + 8, None) == la.LA_ERR_INVALID_ARG
    # chunk 256 has no kernel; no sequences: nothing to do
    assert f(*common, 256, la.LA_DTYPE_FP32, None, A, A, 256, A, None) == la.LA_ERR_UNSUPPORTED
    assert f(A, A, A, A, A, 0, 8, 2, 128, 0, la.LA_DTYPE_BF16, None, A, A, 128, A, None) == \
        la.LA_OK


def test_snapshot_count(lib):
    import torch
    cu = (ctypes.c_int32 * 5)(0, 100, 356, 356, 1000)
    g = lib.lightning_attn_snapshot_count
    assert g(cu, 4, 128) == 0 + 2 + 0 + 5
    assert g(cu, 4, 64) == 1 + 4 + 0 + 10
    assert g(cu, 4, 0) == -1
    assert g(None, 4, 64) == -1
    bad = (ctypes.c_int32 * 3)(0, 10, 5)
    assert g(bad, 2, 64) == -1
    assert la.snapshot_count(torch.tensor([0, 100, 356, 356, 1000], dtype=torch.int32), 128) == 7


def test_binding_checks_the_decay_range():
    """The binding rejects lambda outside (0, 1] (0, above 1, NaN) before any
    launch, checks a tensor once per in-place version, and re-checks after an
    in-place change."""
    import torch
    good = torch.tensor([0.5, 1.0, 1e-30], dtype=torch.float32)
    la.check_decay_range(good)
    la.check_decay_range(good)  # cached
    for bad in ([0.5, 0.0], [1.5, 0.5], [float("nan"), 0.5], [-0.1, 0.5]):
        with pytest.raises(ValueError, match="decay"):
            la.check_decay_range(torch.tensor(bad, dtype=torch.float32))
    good[0] = 2.0  # in place: a new version, checked again
    with pytest.raises(ValueError, match="decay"):
        la.check_decay_range(good)
    cw = torch.full((2, 4), 0.9, dtype=torch.float32)
    la.check_decay_range(cw)
    cw[1, 3] = 0.0
    with pytest.raises(ValueError, match="decay"):
        la.check_decay_range(cw)


def test_entry_points_reject_decay_out_of_range():
    """prefill, decode and the channel-wise calls refuse lambda outside (0, 1]
    before the library is called (CPU tensors: the check needs no device)."""
    import torch
    T, H, d = 8, 2, 64
    q = torch.zeros((T, H, d), dtype=torch.float32)
    cu = torch.tensor([0, T], dtype=torch.int32)
    with pytest.raises(ValueError, match="decay"):
        la.prefill(q, q, q, torch.tensor([0.5, 1.5]), cu)
    with pytest.raises(ValueError, match="decay"):
        la.prefill_channel_decay(q, q, q, torch.full((H, d), 0.0), cu)
    state = torch.zeros((1, H, d, d), dtype=torch.float32)
    with pytest.raises(ValueError, match="decay"):
        la.decode(q[:1], q[:1], q[:1], torch.tensor([float("nan"), 0.5]), state)
