"""The backward entry point that allocates nothing (its scratch is a fixed
array inside the library), for callers that cannot allocate device memory
when they call it.  Called through the C ABI and compared with the regular
lightning_attn_backward on the same inputs, twice in a row (the shared array
keeps the previous call's contents, which must not leak into the next
result).  The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = la.load(labuild.build())
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.lightning_attn_backward_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                    ctypes.c_int, vp, vp, vp, vp, vp]
    lib.lightning_attn_backward_noalloc.restype = ctypes.c_int
    lib.lightning_attn_backward_noalloc_max_bytes.restype = ctypes.c_int64
    return lib


def noalloc_backward(lib, inp, dout, chunk):
    T, H, d = inp.q.shape
    dq, dk, dv = (torch.full_like(inp.q, float("nan")) for _ in range(3))
    code = la.LA_DTYPE_BF16 if inp.q.dtype == torch.bfloat16 else la.LA_DTYPE_FP32
    st = lib.lightning_attn_backward_noalloc(
        inp.q.data_ptr(), inp.k.data_ptr(), inp.v.data_ptr(), inp.decay.data_ptr(),
        inp.cu_seqlens.data_ptr(), inp.cu_seqlens.numel() - 1, T, H, d, chunk, code,
        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == la.LA_OK, lib.lightning_attn_last_error().decode()
    return dq, dk, dv


@pytest.mark.parametrize("dtype, chunk, tol", [(torch.bfloat16, 128, TOL_BF16),
                                               (torch.float32, 64, TOL_FP32)])
def test_noalloc_backward_matches_workspace_backward(lib, dtype, chunk, tol):
    for call, (lengths, seed) in enumerate([([300, 0, 129, 17], 31), ([513, 64], 32)]):
        inp = wl.prefill_inputs(lengths, 4, 128, dtype=dtype, seed=seed, device="cuda")
        g = torch.Generator(device="cuda")
        g.manual_seed(seed + 1)
        dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(dtype)
        got = noalloc_backward(lib, inp, dout, chunk)
        want = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, chunk=chunk)
        torch.cuda.synchronize()
        for x, w, name in zip(got, want, ("dq", "dk", "dv")):
            assert_close(x, w, tol, f"no-alloc call {call + 1} {name}")


def test_noalloc_tensor_core_path_has_no_size_limit(lib):
    """bf16, d = 128: the anti-causal launches need no scratch, so a problem
    whose workspace would exceed the built-in array is still accepted."""
    lengths = [1500, 700]
    inp = wl.prefill_inputs(lengths, 64, 128, dtype=torch.bfloat16, seed=33, device="cuda")
    T, H, d = inp.q.shape
    assert la.backward_workspace_bytes(T, H, d) > lib.lightning_attn_backward_noalloc_max_bytes()
    g = torch.Generator(device="cuda")
    g.manual_seed(34)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    got = noalloc_backward(lib, inp, dout, 0)
    want = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout)
    torch.cuda.synchronize()
    for x, w, name in zip(got, want, ("dq", "dk", "dv")):
        assert torch.equal(x, w), name
