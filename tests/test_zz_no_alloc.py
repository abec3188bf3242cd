"""The backward entry point that allocates nothing (its scratch is a fixed
array inside the library), for callers that cannot allocate device memory
when they call it.  Called through the C ABI and compared with the regular
lightning_attn_backward on the same inputs, twice in a row (the shared array
keeps the previous call's contents, which must not leak into the next
result).  Both entry points run the same deterministic kernels, so the
gradients must agree bit for bit.  The file name makes pytest collect it
last.
"""
import ctypes

import pytest
import torch

import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl

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


def noalloc_call(lib, inp, dout, chunk, grads=None):
    T, H, d = inp.q.shape
    dq, dk, dv = grads if grads is not None else (torch.full_like(inp.q, float("nan"))
                                                  for _ in range(3))
    code = la.LA_DTYPE_BF16 if inp.q.dtype == torch.bfloat16 else la.LA_DTYPE_FP32
    st = lib.lightning_attn_backward_noalloc(
        inp.q.data_ptr(), inp.k.data_ptr(), inp.v.data_ptr(), inp.decay.data_ptr(),
        inp.cu_seqlens.data_ptr(), inp.cu_seqlens.numel() - 1, T, H, d, chunk, code,
        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    return st, (dq, dk, dv)


def noalloc_backward(lib, inp, dout, chunk):
    st, grads = noalloc_call(lib, inp, dout, chunk)
    assert st == la.LA_OK, lib.lightning_attn_last_error().decode()
    return grads


def make_case(lengths, H, d, dtype, seed):
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=seed, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(dtype)
    return inp, dout


def uses_scratch(lib, inp):
    """Whether the case runs on the CUDA-core path and fits the fixed array
    (so the no-allocation call really works through it)."""
    T, H, d = inp.q.shape
    need = la.backward_workspace_bytes(T, H, d, dtype=inp.q.dtype)
    return 0 < need <= lib.lightning_attn_backward_noalloc_max_bytes()


# bf16 with head_dim 64 and fp32 both run on the CUDA-core path, whose
# time-reversed copies live in the fixed array
@pytest.mark.parametrize("dtype, d, chunk", [(torch.bfloat16, 64, 64), (torch.float32, 128, 64),
                                             (torch.float32, 64, 32)])
def test_noalloc_backward_matches_workspace_backward(lib, dtype, d, chunk):
    for call, (lengths, seed) in enumerate([([300, 0, 129, 17], 31), ([513, 64], 32)]):
        inp, dout = make_case(lengths, 4, d, dtype, seed)
        assert uses_scratch(lib, inp)
        got = noalloc_backward(lib, inp, dout, chunk)
        want = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, chunk=chunk)
        torch.cuda.synchronize()
        for x, w, name in zip(got, want, ("dq", "dk", "dv")):
            assert torch.equal(x, w), f"no-alloc call {call + 1} {name} differs"


def test_noalloc_backward_at_the_size_limit(lib):
    """fp32, 4 heads, d = 128: the largest token count whose scratch fits the
    array, then one token more (rejected before any launch)."""
    H, d = 4, 128
    limit = lib.lightning_attn_backward_noalloc_max_bytes()
    T = limit // (3 * H * d * 4)
    inp, dout = make_case([T - 1000, 1000], H, d, torch.float32, 35)
    assert la.backward_workspace_bytes(T, H, d, dtype=torch.float32) <= limit
    got = noalloc_backward(lib, inp, dout, 64)
    want = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, chunk=64)
    torch.cuda.synchronize()
    for x, w, name in zip(got, want, ("dq", "dk", "dv")):
        assert torch.equal(x, w), name
    over, dout2 = make_case([T + 1], H, d, torch.float32, 36)
    assert la.backward_workspace_bytes(T + 1, H, d, dtype=torch.float32) > limit
    sentinel = tuple(torch.full_like(over.q, -5.0) for _ in range(3))
    st, grads = noalloc_call(lib, over, dout2, 64, grads=sentinel)
    assert st == la.LA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert all(bool((g == -5.0).all()) for g in grads)  # nothing written


def test_noalloc_edge_statuses_match_workspace_entry_point(lib):
    """Empty calls succeed and unsupported block sizes report UNSUPPORTED,
    as the workspace entry point does, whatever the size."""
    inp, dout = make_case([0, 0], 4, 128, torch.float32, 37)
    st, _ = noalloc_call(lib, inp, dout, 64)
    assert st == la.LA_OK
    inp, dout = make_case([20000], 4, 128, torch.float32, 38)
    st, _ = noalloc_call(lib, inp, dout, 128)  # no CUDA-core kernel for 128-token blocks
    assert st == la.LA_ERR_UNSUPPORTED


def test_noalloc_tensor_core_path_has_no_size_limit(lib):
    """bf16, d = 128: the anti-causal launches need no scratch, so a problem
    whose workspace would exceed the built-in array is still accepted."""
    inp, dout = make_case([1500, 700], 64, 128, torch.bfloat16, 33)
    T, H, d = inp.q.shape
    assert la.backward_workspace_bytes(T, H, d) > lib.lightning_attn_backward_noalloc_max_bytes()
    got = noalloc_backward(lib, inp, dout, 0)
    want = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout)
    torch.cuda.synchronize()
    for x, w, name in zip(got, want, ("dq", "dk", "dv")):
        assert torch.equal(x, w), name
