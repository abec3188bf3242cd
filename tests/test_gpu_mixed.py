"""GPU parity of the mixed serving step (MiniMax-01 report §3.3.2: length-1
and longer inputs on separate kernels and streams, every sequence continuing
from its cached state) against the fp64 CPU oracle, which runs the plain
recursion from each cached state over all new tokens."""
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close

pytestmark = pytest.mark.gpu

# the report's example: a batch of 20 with prefix caches, one or two inputs
# of ~50 tokens, the rest one token (plus an empty entry and a longer one)
LENGTHS = [1, 50, 1, 1, 1, 0, 1, 1, 1, 1, 1, 47, 1, 1, 1, 1, 1, 1, 300, 1]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def run(dtype, d, H, two_streams, seed, host_cu=True):
    inp = wl.prefill_inputs(LENGTHS, H, d, dtype=dtype, seed=seed, device="cuda")
    s0 = wl.cached_states(len(LENGTHS), H, d, seed=seed + 100, device="cuda")
    state = s0.clone()
    ps = torch.cuda.current_stream()
    ds = torch.cuda.Stream() if two_streams else None
    out = la.mixed_step(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, state,
                        prefill_stream=ps, decode_stream=ds,
                        cu_seqlens_host=inp.cu_seqlens.cpu().tolist() if host_cu else None)
    ps.synchronize()
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(),
                                   initial_state=s0.cpu())
    return out, state, ref, ref_st, s0


@pytest.mark.parametrize("two_streams", [True, False])
def test_mixed_step_bf16_tensor_core(two_streams):
    out, state, ref, ref_st, s0 = run(torch.bfloat16, 128, 8, two_streams, 41)
    assert_close(out, ref, TOL_BF16, f"mixed bf16 out (two streams: {two_streams})")
    assert_close(state, ref_st, TOL_BF16, "mixed bf16 state")
    assert torch.equal(state[LENGTHS.index(0)], s0[LENGTHS.index(0)])


def test_mixed_step_fp32_cuda_core():
    out, state, ref, ref_st, _ = run(torch.float32, 64, 4, True, 42)
    assert_close(out, ref, TOL_FP32, "mixed fp32 out")
    assert_close(state, ref_st, TOL_FP32, "mixed fp32 state")


def test_two_streams_match_one_stream():
    a = run(torch.bfloat16, 128, 4, True, 43)
    b = run(torch.bfloat16, 128, 4, False, 43)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_without_host_lengths_same_result():
    """Without the host copy of the lengths every sequence gets prefill CTAs
    that leave the short ones alone: same numbers."""
    a = run(torch.bfloat16, 128, 4, True, 44, host_cu=True)
    b = run(torch.bfloat16, 128, 4, True, 44, host_cu=False)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
