"""Seeded random configurations against the fp64 CPU oracle: dtype, head_dim,
block size, ragged lengths (including empty and one-token sequences), per-head
decays anywhere in (0, 1], cached states on or off, the backward pass on
the tensor-core path, and the channel-wise decay on both of its kernels.  Each
case is small enough for the oracle to finish at
once; together they cover combinations the hand-picked cases do not."""
import random

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


def random_case(seed):
    rng = random.Random(seed)
    dtype = rng.choice([torch.bfloat16, torch.bfloat16, torch.float32])
    d = rng.choice([64, 128]) if dtype == torch.float32 else rng.choice([64, 128, 128])
    if dtype == torch.bfloat16 and d == 128:
        chunk = rng.choice([0, 16, 32, 64, 128])
    else:
        chunk = rng.choice([0, 16, 32, 64])
    nseq = rng.randint(1, 6)
    lengths = [rng.choice([0, 1, rng.randint(2, 40), rng.randint(41, 400)]) for _ in range(nseq)]
    if sum(lengths) == 0:
        lengths[0] = 5
    H = rng.randint(1, 3)
    decay = torch.tensor([rng.choice([1.0, rng.uniform(0.3, 1.0), rng.uniform(1e-3, 0.3)])
                          for _ in range(H)], dtype=torch.float32)
    with_state = rng.random() < 0.5
    return dtype, d, chunk, lengths, H, decay, with_state


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_matches_oracle(seed):
    dtype, d, chunk, lengths, H, decay, with_state = random_case(1000 + seed)
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=seed, device="cuda",
                            decay=decay)
    s0 = wl.cached_states(len(lengths), H, d, seed=seed + 77, device="cuda") \
        if with_state else None
    out, st = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk,
                         initial_state=s0)
    torch.cuda.synchronize()
    ref, ref_st = oracle.recurrent(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(),
                                   initial_state=None if s0 is None else s0.cpu())
    tol = TOL_FP32 if dtype == torch.float32 else TOL_BF16
    what = f"seed {seed}: {dtype} d={d} B={chunk} lengths={lengths} lambda={decay.tolist()}"
    assert_close(out, ref, tol, what + " out")
    assert_close(st, ref_st, tol, what + " state")


@pytest.mark.parametrize("seed", range(8))
def test_random_backward_matches_oracle(seed):
    rng = random.Random(2000 + seed)
    chunk = rng.choice([0, 32, 64, 128])
    lengths = [rng.choice([0, 1, rng.randint(2, 60), rng.randint(61, 300)])
               for _ in range(rng.randint(1, 5))]
    if sum(lengths) == 0:
        lengths[0] = 9
    H = rng.randint(1, 2)
    decay = torch.tensor([rng.uniform(0.3, 1.0) for _ in range(H)], dtype=torch.float32)
    inp = wl.prefill_inputs(lengths, H, 128, dtype=torch.bfloat16, seed=seed, device="cuda",
                            decay=decay)
    g = torch.Generator(device="cuda")
    g.manual_seed(3000 + seed)
    dout = torch.randn(inp.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    got = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout, chunk=chunk)
    torch.cuda.synchronize()
    ref = oracle.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens.cpu(), dout)
    for x, r, name in zip(got, ref, ("dq", "dk", "dv")):
        assert_close(x, r, TOL_BF16, f"seed {seed}: B={chunk} lengths={lengths} {name}")


def random_cw_case(seed):
    """A channel-wise case: per (head, key channel) decays drawn from 1, a
    moderate range, a small range and 1e-20 (every power above the first
    underflows), mixed within each head."""
    rng = random.Random(seed)
    dtype = rng.choice([torch.bfloat16, torch.bfloat16, torch.bfloat16, torch.float32])
    d = rng.choice([64, 128, 128, 128])
    chunk = rng.choice([0, 64, 64, 32, 16])
    nseq = rng.randint(1, 5)
    lengths = [rng.choice([0, 1, rng.randint(2, 70), rng.randint(71, 500)]) for _ in range(nseq)]
    if sum(lengths) == 0:
        lengths[0] = 9
    H = rng.randint(1, 3)
    lam = torch.empty((H, d), dtype=torch.float64)
    for h in range(H):
        for i in range(d):
            lam[h, i] = rng.choice([1.0, rng.uniform(0.3, 1.0), rng.uniform(0.3, 1.0),
                                    rng.uniform(1e-3, 0.3), 1e-20])
    with_state = rng.random() < 0.5
    return dtype, d, chunk, lengths, H, lam.to(torch.float32), with_state


@pytest.mark.parametrize("seed", range(16))
def test_random_channel_decay_prefill_matches_oracle(seed):
    dtype, d, chunk, lengths, H, lam, with_state = random_cw_case(3000 + seed)
    inp = wl.prefill_inputs(lengths, H, d, dtype=dtype, seed=seed + 300, device="cuda")
    s0 = wl.cached_states(len(lengths), H, d, seed=seed + 377, device="cuda") \
        if with_state else None
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens,
                                       chunk=chunk, initial_state=s0)
    torch.cuda.synchronize()
    la.device_status()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu(),
                                      initial_state=None if s0 is None else s0.cpu())
    tol = TOL_FP32 if dtype == torch.float32 else TOL_BF16
    what = f"cw fuzz {seed}: {dtype} d={d} B={chunk} L={lengths} state={with_state}"
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all(), what
    assert_close(out, ref, tol, what + " out")
    assert_close(st, ref_st, tol, what + " state")
