"""GPU parity of prefill continuing from a cached state (prefix KV cache,
MiniMax-01 report §3.3.1) against the fp64 CPU oracle: kv_{-1} = S0, so
o_t gains lambda^(t+1) q_t S0 and the final state lambda^L S0.

The cached states are seeded synthetic inputs; the oracle never sees a value
the GPU produced.  Continuation cases chain two GPU calls and compare with
the oracle's single pass over both segments.  Tolerances as in parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close, to64

pytestmark = pytest.mark.gpu

RAGGED = [1, 0, 15, 16, 17, 127, 128, 129, 255, 256, 300, 0, 513]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def run_with_state(lengths, H, d, dtype, chunk, seed):
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=seed, device="cuda")
    s0 = wl.cached_states(len(lengths), H, d, seed=seed + 100, device="cuda")
    out, st = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk,
                         initial_state=s0)
    torch.cuda.synchronize()
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(),
                                   initial_state=s0.cpu())
    return inp, s0, out, st, ref, ref_st


def test_tensor_core_ragged_varlen_with_state():
    inp, s0, out, st, ref, ref_st = run_with_state(RAGGED, 4, 128, torch.bfloat16, 128, 11)
    assert_close(out, ref, TOL_BF16, "bf16 tc + S0 out")
    assert_close(st, ref_st, TOL_BF16, "bf16 tc + S0 final state")
    # empty sequences hand their cached state through unchanged
    for sidx, L in enumerate(RAGGED):
        if L == 0:
            assert torch.equal(st[sidx], s0[sidx])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("chunk", [16, 64])
def test_cuda_core_fp32_with_state(d, chunk):
    inp, s0, out, st, ref, ref_st = run_with_state(RAGGED, 3, d, torch.float32, chunk, 12)
    assert_close(out, ref, TOL_FP32, f"fp32 d={d} B={chunk} + S0 out")
    assert_close(st, ref_st, TOL_FP32, f"fp32 d={d} B={chunk} + S0 final state")


def test_quadratic_form_agrees_with_state():
    """The left-product form with the lambda^(t+1) q_t S0 term, independently."""
    inp, s0, out, st, ref, ref_st = run_with_state([300, 129], 2, 64, torch.float32, 64, 13)
    refq = oracle.quadratic(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(),
                            initial_state=s0.cpu())
    assert_close(out, refq, TOL_FP32, "fp32 + S0 vs quadratic")


@pytest.mark.parametrize("dtype, chunk, tol", [(torch.bfloat16, 128, TOL_BF16),
                                               (torch.bfloat16, 256, TOL_BF16),
                                               (torch.float32, 64, TOL_FP32)])
def test_two_segment_continuation(dtype, chunk, tol):
    """prefill(A) then prefill(B | final state of A) == one pass over A + B."""
    H, d = 8, 128
    La, Lb = [700, 0, 1536], [300, 77, 1]
    full_len = [a + b for a, b in zip(La, Lb)]
    inp = wl.prefill_inputs(full_len, H, d, dtype=dtype, seed=14, device="cuda")
    cu = inp.cu_seqlens.cpu().numpy()
    ia = np.concatenate([np.arange(cu[s], cu[s] + La[s]) for s in range(len(La))])
    ib = np.concatenate([np.arange(cu[s] + La[s], cu[s + 1]) for s in range(len(La))])
    cua = wl.cu_from_lengths(La).cuda()
    cub = wl.cu_from_lengths(Lb).cuda()
    ta, tb = torch.as_tensor(ia, device="cuda"), torch.as_tensor(ib, device="cuda")
    oa, sa = la.prefill(inp.q[ta].contiguous(), inp.k[ta].contiguous(), inp.v[ta].contiguous(),
                        inp.decay, cua, chunk=chunk)
    ob, sb = la.prefill(inp.q[tb].contiguous(), inp.k[tb].contiguous(), inp.v[tb].contiguous(),
                        inp.decay, cub, chunk=chunk, initial_state=sa)
    torch.cuda.synchronize()
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu())
    assert_close(ob, ref[ib], tol, "second segment out")
    assert_close(oa, ref[ia], tol, "first segment out")
    assert_close(sb, ref_st, tol, "final state after both segments")


@pytest.mark.parametrize("dtype, chunk", [(torch.bfloat16, 128), (torch.float32, 32)])
def test_in_place_cache_update(dtype, chunk):
    """initial_state may be the final_state array: same result as out of place."""
    inp = wl.prefill_inputs([200, 0, 513], 4, 128, dtype=dtype, seed=15, device="cuda")
    s0 = wl.cached_states(3, 4, 128, seed=115, device="cuda")
    out1, st1 = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk,
                           initial_state=s0)
    cache = s0.clone()
    out2, st2 = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk,
                           initial_state=cache, final_state=cache)
    torch.cuda.synchronize()
    assert st2.data_ptr() == cache.data_ptr()
    assert torch.equal(out1, out2)
    assert torch.equal(st1, cache)
