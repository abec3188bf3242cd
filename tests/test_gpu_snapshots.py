"""GPU parity of the per-block state snapshots (prefix cache kept once per
block of tokens, K3 report notes on the inference engine) against the fp64
CPU oracle: snapshot j of sequence s must be the final state of the oracle's
recurrence over the first (j + 1) * interval tokens of s, from the same
cached initial state.  Tolerances as in parity.py."""
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def prefix_states(inp, lengths, interval, s0):
    """Oracle final states of every whole-block prefix, in snapshot order."""
    qs, ks, vs, cu, init = [], [], [], [0], []
    starts = [0]
    for L in lengths:
        starts.append(starts[-1] + L)
    for s, L in enumerate(lengths):
        for j in range(L // interval):
            P = (j + 1) * interval
            a = starts[s]
            qs.append(inp.q[a:a + P].cpu())
            ks.append(inp.k[a:a + P].cpu())
            vs.append(inp.v[a:a + P].cpu())
            cu.append(cu[-1] + P)
            if s0 is not None:
                init.append(s0[s:s + 1].cpu())
    if not qs:
        return None
    cat = lambda xs: torch.cat(xs, 0)
    _, st = oracle.recurrent(cat(qs), cat(ks), cat(vs), inp.decay.cpu(),
                             torch.tensor(cu, dtype=torch.int32),
                             initial_state=None if s0 is None else cat(init))
    return st


@pytest.mark.parametrize("dtype, d, chunk, interval, with_state, tol", [
    (torch.bfloat16, 128, 0, 128, True, TOL_BF16),    # tensor cores, every block
    (torch.bfloat16, 128, 128, 256, False, TOL_BF16),  # tensor cores, every second block
    (torch.bfloat16, 128, 256, 256, True, TOL_BF16),   # tensor cores, 256-token blocks
    (torch.bfloat16, 128, 64, 64, True, TOL_BF16),     # tensor cores, 64-token blocks
    (torch.float32, 128, 64, 128, True, TOL_FP32),     # CUDA cores
    (torch.float32, 64, 32, 64, False, TOL_FP32),
])
def test_snapshots_match_prefix_states(dtype, d, chunk, interval, with_state, tol):
    lengths = [1, 0, 127, 128, 129, 256, 300, 0, 513, 1024]
    H = 3
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=61, device="cuda")
    s0 = wl.cached_states(len(lengths), H, d, seed=62, device="cuda") if with_state else None
    out, fs, snaps = la.prefill_snapshots(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens,
                                          interval, chunk=chunk, initial_state=s0)
    torch.cuda.synchronize()
    assert snaps.shape[0] == sum(L // interval for L in lengths)
    ref_snaps = prefix_states(inp, lengths, interval, s0)
    assert_close(snaps, ref_snaps, tol, f"snapshots {dtype} d={d} interval={interval}")
    # the outputs and final states are those of the plain prefill
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(),
                                   initial_state=None if s0 is None else s0.cpu())
    assert_close(out, ref, tol, "out")
    assert_close(fs, ref_st, tol, "final state")


def test_snapshots_layer_sized():
    """8K-token layer (64 heads), a snapshot every 1024 tokens; the oracle
    checks heads 0 and 63 of snapshots 0, 3 and 7 (the last one is the final
    state)."""
    inp = wl.prefill_inputs([8192], 64, 128, dtype=torch.bfloat16, seed=63, device="cuda")
    out, fs, snaps = la.prefill_snapshots(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, 1024)
    torch.cuda.synchronize()
    assert snaps.shape[0] == 8
    assert torch.equal(snaps[7], fs[0])
    heads = [0, 63]
    for j in (0, 3):
        P = (j + 1) * 1024
        sub = lambda t: t[:P, heads].contiguous()
        _, st = oracle.recurrent(sub(inp.q), sub(inp.k), sub(inp.v), inp.decay[heads],
                                 torch.tensor([0, P], dtype=torch.int32))
        assert_close(snaps[j, heads], st[0], TOL_BF16, f"layer snapshot {j}")


def test_snapshots_many_sequences():
    """150 sequences (more than the in-kernel length sort handles): every
    CTA finds its sequence's first snapshot by counting those before it."""
    g = torch.Generator().manual_seed(64)
    lengths = torch.randint(0, 700, (150,), generator=g).tolist()
    H, d, interval = 2, 128, 256
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=65, device="cuda")
    out, fs, snaps = la.prefill_snapshots(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens,
                                          interval)
    torch.cuda.synchronize()
    assert snaps.shape[0] == sum(L // interval for L in lengths)
    assert_close(snaps, prefix_states(inp, lengths, interval, None), TOL_BF16,
                 "150 sequences snapshots")
