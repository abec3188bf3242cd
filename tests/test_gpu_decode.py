"""GPU parity of the decode step against the fp64 CPU oracle, and the
prefill -> decode continuation (the prefix-cache use of the final state)."""
import numpy as np
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_small(d, dtype):
    inp = wl.decode_inputs(5, 3, d, steps=1, dtype=dtype, seed=1, device="cuda")
    st0 = inp.state.clone()
    out = la.decode(inp.q[0], inp.k[0], inp.v[0], inp.decay, inp.state)
    torch.cuda.synchronize()
    ref, ref_st = oracle.decode(inp.q[0], inp.k[0], inp.v[0], inp.decay, st0)
    tol = TOL_FP32 if dtype == torch.float32 else TOL_BF16
    assert_close(out, ref, tol, "decode out")
    # the state is fp32 on both sides; only the k^T v term saw bf16 inputs
    assert_close(inp.state, ref_st, TOL_FP32, "decode state")


def test_decode_batched_config_first_step():
    """128 sequences x 64 heads x d=128, fp32 state ~ N(0, 0.02^2), bf16
    tokens: the first step, every sequence and head."""
    cfg = wl.DECODE_128
    inp = wl.decode_inputs(cfg["batch"], cfg["num_heads"], cfg["head_dim"], steps=1,
                           dtype=torch.bfloat16, seed=0, device="cuda")
    st0 = inp.state.cpu()
    out = la.decode(inp.q[0], inp.k[0], inp.v[0], inp.decay, inp.state)
    torch.cuda.synchronize()
    ref, ref_st = oracle.decode(inp.q[0], inp.k[0], inp.v[0], inp.decay, st0)
    assert_close(out, ref, TOL_BF16, "decode out")
    assert_close(inp.state, ref_st, TOL_FP32, "decode state")


def test_decode_many_steps_subset():
    """50 consecutive steps on the full batch; the oracle replays every step
    for sequences 0, 77 and 127 (all heads)."""
    cfg = wl.DECODE_128
    steps, sel = 50, [0, 77, 127]
    inp = wl.decode_inputs(cfg["batch"], cfg["num_heads"], cfg["head_dim"], steps=steps,
                           dtype=torch.bfloat16, seed=2, device="cuda")
    ref_st = to64(inp.state[sel])
    outs = []
    for t in range(steps):
        outs.append(la.decode(inp.q[t], inp.k[t], inp.v[t], inp.decay, inp.state))
    torch.cuda.synchronize()
    for t in range(steps):
        ref, ref_st = oracle.decode(inp.q[t][sel], inp.k[t][sel], inp.v[t][sel], inp.decay, ref_st)
        assert_close(outs[t][sel], ref, TOL_BF16, f"step {t}")
    assert_close(inp.state[sel], ref_st, TOL_FP32, "state after 50 steps")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prefill_then_decode_continues(dtype):
    """prefill(L) -> final state -> decode(token L) equals prefill(L + 1)'s
    row L and final state (prefix-cache continuation)."""
    L, H, d = 389, 4, 128
    inp = wl.prefill_inputs([L + 1], H, d, dtype=dtype, seed=3, device="cuda")
    chunk = 64 if dtype == torch.float32 else 0
    full, st_full = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk)
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    _, st = la.prefill(inp.q[:L].contiguous(), inp.k[:L].contiguous(), inp.v[:L].contiguous(),
                       inp.decay, cu, chunk=chunk)
    o = la.decode(inp.q[L:], inp.k[L:], inp.v[L:], inp.decay, st[:, :, :, :].view(1, H, d, d))
    torch.cuda.synchronize()
    tol = TOL_FP32 if dtype == torch.float32 else TOL_BF16
    assert_close(o[0], full[L], tol, "decode row vs prefill row")
    assert_close(st[0], st_full[0], tol, "state vs prefill state")
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu())
    assert_close(o[0], ref[L], tol, "decode row vs oracle")


def test_decode_zero_batch_is_noop():
    q = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((0, 2, 128, 128), device="cuda")
    out = la.decode(q, q, q, wl.decay_schedule(2).cuda(), st)
    assert out.shape == (0, 2, 128)
