"""GPU parity of the backward pass (dq, dk, dv) against the fp64 CPU oracle.

The C-ABI call runs the prefill kernels on permuted and time-reversed
operands; its results are compared element by element with the oracle's
direct sums (oracle.backward, pinned by exact central differences of the
forward form) on the same seeded inputs, with the tolerances of parity.py.
"""
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close

pytestmark = pytest.mark.gpu

RAGGED = [1, 0, 15, 16, 17, 127, 128, 129, 255, 256, 300, 0, 513]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def run(lengths, H, d, dtype, chunk, seed):
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=seed, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 1000)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda", dtype=torch.float32).to(dtype)
    dq, dk, dv = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, chunk=chunk)
    torch.cuda.synchronize()
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(), dout)
    return (dq, dk, dv), ref


def test_tensor_core_backward_ragged_varlen():
    got, ref = run(RAGGED, 4, 128, torch.bfloat16, 128, 21)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"bf16 tc {name}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("chunk", [16, 64])
def test_cuda_core_fp32_backward(d, chunk):
    got, ref = run(RAGGED, 3, d, torch.float32, chunk, 22)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_FP32, f"fp32 d={d} B={chunk} {name}")


def test_backward_layer_sized_sampled_heads():
    """2 sequences of 2048 + 1000 tokens, 64 heads (the decay schedule of the
    64-head layer); the oracle checks heads 0, 31 and 63 in full."""
    inp = wl.prefill_inputs([2048, 1000], 64, 128, dtype=torch.bfloat16, seed=23, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(1023)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    dq, dk, dv = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout)
    torch.cuda.synchronize()
    heads = [0, 31, 63]
    sub = lambda t: t[:, heads].contiguous()
    ref = oracle.backward(sub(inp.q), sub(inp.k), sub(inp.v), inp.decay[heads],
                          inp.cu_seqlens.cpu(), sub(dout))
    for x, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert_close(sub(x), r, TOL_BF16, f"layer-sized {name}")


@pytest.mark.parametrize("lam", [1.0, 1e-30, 0.5])
def test_tensor_core_backward_special_decays(lam):
    """lambda = 1 (prefix and suffix sums), lambda -> 0 (only the diagonal
    term) and 1/2 through the causal and anti-causal tensor-core launches."""
    lengths, H, d = [300, 5, 129], 2, 128
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=24, device="cuda")
    decay = torch.full((H,), lam, dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(1024)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    got = la.backward(inp.q, inp.k, inp.v, decay, inp.cu_seqlens, dout)
    torch.cuda.synchronize()
    ref = oracle.backward(inp.q, inp.k, inp.v, decay.cpu(), inp.cu_seqlens.cpu(), dout)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"lambda={lam} {name}")


def test_tensor_core_backward_many_sequences():
    """More sequences than the in-kernel length sort handles (natural order)
    in the anti-causal launches."""
    g = torch.Generator().manual_seed(25)
    lengths = torch.randint(0, 260, (150,), generator=g).tolist()
    got, ref = run(lengths, 2, 128, torch.bfloat16, 0, 26)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"150 sequences {name}")


def test_backward_writes_stay_inside_gradients():
    """Sentinel guard regions around dq, dk and dv stay untouched."""
    lengths, H, d = [5, 200, 129], 2, 128
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=27, device="cuda")
    T, G = inp.total_tokens, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(1027)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    bigs = [torch.full((T * H * d + 2 * G,), 321.0, dtype=torch.bfloat16, device="cuda")
            for _ in range(3)]
    dq, dk, dv = (b[G:G + T * H * d].view(T, H, d) for b in bigs)
    la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for b in bigs:
        assert (b[:G] == 321.0).all() and (b[-G:] == 321.0).all()
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(), dout)
    for x, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"guarded {name}")


@pytest.mark.parametrize("chunk", [32, 64, 256])
def test_tensor_core_backward_block_sizes(chunk):
    """The anti-causal launches with 32- and 64-token blocks (128-row tiles
    advancing one block at a time, walked last to first) and 256-token blocks
    (two tiles each)."""
    got, ref = run([1, 0, 31, 33, 64, 65, 200, 129], 3, 128, torch.bfloat16, chunk, 28)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"tc B={chunk} {name}")
