"""GPU parity of the channel-wise (per key channel) decay variant against the
fp64 CPU oracle (K3 report reading notes: the scalar decay generalised to one
decay per channel; kv_t[i][j] = lambda_i kv_{t-1}[i][j] + k_t[i] v_t[j]).
Tolerances as in parity.py."""
import pytest
import torch

import oracle
import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl
from parity import TOL_BF16, TOL_FP32, assert_close

pytestmark = pytest.mark.gpu

RAGGED = [1, 0, 15, 16, 17, 63, 64, 65, 129, 300, 0, 257]


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def channel_decays(H, d, seed):
    """lambda_{h,i} spread over [0.3, 1.0] (seeded), fp32 [H, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (0.3 + 0.7 * torch.rand((H, d), generator=g)).to(torch.float32)


@pytest.mark.parametrize("dtype, d, chunk, tol", [
    (torch.float32, 64, 16, TOL_FP32), (torch.float32, 128, 64, TOL_FP32),
    (torch.float32, 128, 32, TOL_FP32), (torch.float32, 128, 16, TOL_FP32),
    (torch.bfloat16, 128, 64, TOL_BF16), (torch.bfloat16, 64, 32, TOL_BF16)])
def test_channel_decay_prefill(dtype, d, chunk, tol):
    H = 3
    inp = wl.prefill_inputs(RAGGED, H, d, dtype=dtype, seed=51, device="cuda")
    lam = channel_decays(H, d, 52)
    s0 = wl.cached_states(len(RAGGED), H, d, seed=53, device="cuda")
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens,
                                       chunk=chunk, initial_state=s0)
    torch.cuda.synchronize()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu(),
                                      initial_state=s0.cpu())
    assert_close(out, ref, tol, f"channel decay {dtype} d={d} B={chunk} out")
    assert_close(st, ref_st, tol, f"channel decay {dtype} d={d} B={chunk} state")


@pytest.mark.parametrize("chunk", [16, 64])
def test_channel_decay_extreme_decays(chunk):
    """Channels with lambda = 1 (no decay) next to lambda = 1e-30 (every power
    above the first underflows in fp32): the per-channel tables hold only
    non-negative exponents, so nothing overflows and no NaN appears."""
    H, d = 2, 128
    inp = wl.prefill_inputs([200, 3, 64], H, d, dtype=torch.float32, seed=55, device="cuda")
    lam = channel_decays(H, d, 56)
    lam[:, 0::3] = 1.0
    lam[:, 1::3] = 1e-30
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens,
                                       chunk=chunk)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(st).all()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu())
    assert_close(out, ref, TOL_FP32, f"extreme channel decays B={chunk} out")
    assert_close(st, ref_st, TOL_FP32, f"extreme channel decays B={chunk} state")


# ---------------------------------------- the tensor-core kernel (bf16, d=128, B=64)
RAGGED_TC = [1, 0, 15, 16, 17, 31, 33, 63, 64, 65, 127, 129, 200, 0, 513]


@pytest.mark.parametrize("with_state", [False, True])
def test_channel_decay_tensor_core_ragged(with_state):
    """Ragged packed sequences (empty, shorter than a sub-block, across
    sub-block and block edges) through the tcgen05 kernel, with and without
    cached states."""
    H, d = 4, 128
    inp = wl.prefill_inputs(RAGGED_TC, H, d, dtype=torch.bfloat16, seed=57, device="cuda")
    lam = channel_decays(H, d, 58)
    s0 = wl.cached_states(len(RAGGED_TC), H, d, seed=59, device="cuda") if with_state else None
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens,
                                       initial_state=s0)
    torch.cuda.synchronize()
    la.device_status()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu(),
                                      initial_state=None if s0 is None else s0.cpu())
    assert_close(out, ref, TOL_BF16, f"tc channel decay state={with_state} out")
    assert_close(st, ref_st, TOL_BF16, f"tc channel decay state={with_state} state")


@pytest.mark.parametrize("pattern", ["one_and_tiny", "near_one", "spread_small"])
def test_channel_decay_tensor_core_extreme_decays(pattern):
    """Channel decays at the extremes on the tcgen05 kernel: lambda = 1 next to
    lambda = 1e-30 (every power above the first underflows), all near 1 (long
    memory, the largest state), and spread down to 1e-3.  Only non-negative
    exponents are formed, so nothing overflows and no NaN appears."""
    H, d = 2, 128
    inp = wl.prefill_inputs([300, 3, 64, 129], H, d, dtype=torch.bfloat16, seed=60, device="cuda")
    lam = channel_decays(H, d, 61)
    if pattern == "one_and_tiny":
        lam[:, 0::3] = 1.0
        lam[:, 1::3] = 1e-30
    elif pattern == "near_one":
        lam = 1.0 - 1e-3 * torch.rand((H, d), generator=torch.Generator().manual_seed(62))
    else:
        lam = 10.0 ** (-3.0 * torch.rand((H, d), generator=torch.Generator().manual_seed(63)))
    lam = lam.to(torch.float32)
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens)
    torch.cuda.synchronize()
    la.device_status()
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu())
    assert_close(out, ref, TOL_BF16, f"tc extreme channel decays ({pattern}) out")
    assert_close(st, ref_st, TOL_BF16, f"tc extreme channel decays ({pattern}) state")


def test_channel_decay_tensor_core_layer_heads():
    """A 64-head, 4096-token layer (the measured layer's shape, shorter): every
    head, every token and the final states."""
    H, d = 64, 128
    inp = wl.prefill_inputs([4096], H, d, dtype=torch.bfloat16, seed=64, device="cuda")
    lam = inp.decay.cpu()[:, None].repeat(1, d)
    lam = (lam * (1.0 - 0.01 * torch.linspace(0, 1, d))[None, :]).to(torch.float32)
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens)
    torch.cuda.synchronize()
    la.device_status()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu())
    assert_close(out, ref, TOL_BF16, "tc channel decay 64 heads out")
    assert_close(st, ref_st, TOL_BF16, "tc channel decay 64 heads state")


def test_channel_decay_tensor_core_long_varlen_with_states():
    """Long packed sequences (about 31 K tokens, 8 heads) with cached states:
    hundreds of blocks per CTA carry the state through the TMEM accumulator
    and its hi/lo copy; every head, every token and the final states."""
    H, d = 8, 128
    lengths = [20000, 7000, 1, 4129]
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=67, device="cuda")
    lam = inp.decay.cpu()[:, None].repeat(1, d)
    lam = (lam * (1.0 - 0.05 * torch.rand((H, d), generator=torch.Generator().manual_seed(68))))
    lam = lam.to(torch.float32)
    s0 = wl.cached_states(len(lengths), H, d, seed=69, device="cuda")
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens,
                                       initial_state=s0)
    torch.cuda.synchronize()
    la.device_status()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu(),
                                      initial_state=s0.cpu())
    assert_close(out, ref, TOL_BF16, "tc channel decay long varlen out")
    assert_close(st, ref_st, TOL_BF16, "tc channel decay long varlen state")


def test_channel_decay_tensor_core_many_sequences():
    """More CTAs than SMs (300 short sequences x 2 heads x 2 value slices):
    sequences are taken longest first across several waves."""
    H, d = 2, 128
    g = torch.Generator().manual_seed(70)
    lengths = torch.randint(0, 300, (300,), generator=g).tolist()
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=71, device="cuda")
    lam = channel_decays(H, d, 72)
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam.cuda(), inp.cu_seqlens)
    torch.cuda.synchronize()
    la.device_status()
    ref, ref_st = oracle.recurrent_cw(inp.q, inp.k, inp.v, lam, inp.cu_seqlens.cpu())
    assert_close(out, ref, TOL_BF16, "tc channel decay 300 sequences out")
    assert_close(st, ref_st, TOL_BF16, "tc channel decay 300 sequences state")


def test_channel_decay_tensor_core_matches_cuda_cores():
    """The tcgen05 kernel (chunk 64) and the CUDA-core kernel (chunk 32) agree
    to the bf16 bound on the same inputs."""
    H, d = 3, 128
    inp = wl.prefill_inputs([700, 129], H, d, dtype=torch.bfloat16, seed=65, device="cuda")
    lam = channel_decays(H, d, 66).cuda()
    a, sa = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens, chunk=64)
    b, sb = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens, chunk=32)
    torch.cuda.synchronize()
    assert_close(a, b.double(), TOL_BF16, "tc vs cuda-core channel decay out", u=2.0 ** -7)
    assert_close(sa, sb.double(), TOL_BF16, "tc vs cuda-core channel decay state")


def test_channel_decay_uniform_equals_scalar_kernel():
    """Equal channel decays give the scalar-decay result (CUDA-core path)."""
    H, d = 4, 128
    inp = wl.prefill_inputs([300, 65], H, d, dtype=torch.float32, seed=54, device="cuda")
    lam_cw = inp.decay[:, None].repeat(1, d).contiguous()
    a, sa = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam_cw, inp.cu_seqlens, chunk=64)
    b, sb = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=64)
    torch.cuda.synchronize()
    assert_close(a, b.double(), TOL_FP32, "uniform channel decay vs scalar out")
    assert_close(sa, sb.double(), TOL_FP32, "uniform channel decay vs scalar state")


@pytest.mark.parametrize("dtype, tol", [(torch.float32, TOL_FP32), (torch.bfloat16, TOL_BF16)])
def test_channel_decay_decode(dtype, tol):
    B, H, d = 6, 4, 128
    dinp = wl.decode_inputs(B, H, d, steps=1, dtype=dtype, seed=55, device="cuda")
    lam = channel_decays(H, d, 56)
    st0 = dinp.state.cpu()
    out = la.decode_channel_decay(dinp.q[0], dinp.k[0], dinp.v[0], lam.cuda(), dinp.state)
    torch.cuda.synchronize()
    ref, ref_st = oracle.decode_cw(dinp.q[0], dinp.k[0], dinp.v[0], lam, st0)
    assert_close(out, ref, tol, f"channel decay decode {dtype} out")
    assert_close(dinp.state, ref_st, TOL_FP32, f"channel decay decode {dtype} state")


def test_channel_decay_tensor_core_repeatable():
    """Ten launches on the 8K-token 64-head layer: every output and final
    state equal to the first bit for bit, and no bounded wait gives up."""
    H, d = 64, 128
    inp = wl.prefill_inputs([8192], H, d, dtype=torch.bfloat16, seed=81, device="cuda")
    lam = (inp.decay[:, None] * (1.0 - 0.01 * torch.linspace(0, 1, d, device="cuda"))[None, :])
    lam = lam.to(torch.float32).contiguous()
    first, first_st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens)
    out = torch.empty_like(first)
    st = torch.empty_like(first_st)
    for _ in range(10):
        la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens, out=out,
                                 final_state=st)
        torch.cuda.synchronize()
        assert torch.equal(out, first) and torch.equal(st, first_st)
    la.device_status()


def test_channel_decay_tensor_core_state_in_place():
    """initial_state may be final_state itself (the prefix cache updated in
    place): the same result as with separate buffers."""
    H, d = 4, 128
    lengths = [300, 0, 129, 65]
    inp = wl.prefill_inputs(lengths, H, d, dtype=torch.bfloat16, seed=82, device="cuda")
    lam = channel_decays(H, d, 83).cuda()
    s0 = wl.cached_states(len(lengths), H, d, seed=84, device="cuda")
    ref, ref_st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens,
                                           initial_state=s0)
    cache = s0.clone()
    out = torch.empty_like(inp.q)
    la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens, out=out,
                             final_state=cache, initial_state=cache)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(cache, ref_st)


def test_channel_decay_tensor_core_128k_context():
    """One 131072-token sequence x 64 heads (2048 blocks per CTA): heads 0,
    31 and 63 (the fastest, a middle and the slowest decay) against the
    oracle, all tokens and final states; every head finite."""
    H, d = 64, 128
    inp = wl.prefill_inputs([131072], H, d, dtype=torch.bfloat16, seed=85, device="cuda")
    lam = (inp.decay[:, None] * (1.0 - 0.01 * torch.linspace(0, 1, d, device="cuda"))[None, :])
    lam = lam.to(torch.float32).contiguous()
    out, st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens)
    torch.cuda.synchronize()
    la.device_status()
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()
    heads = [0, 31, 63]
    sel = lambda t: t[:, heads].contiguous()
    ref, ref_st = oracle.recurrent_cw(sel(inp.q), sel(inp.k), sel(inp.v), lam[heads].cpu(),
                                      inp.cu_seqlens.cpu())
    assert_close(out[:, heads], ref, TOL_BF16, "tc channel decay 128k out (heads 0, 31, 63)")
    assert_close(st[:, heads], ref_st, TOL_BF16, "tc channel decay 128k state (heads 0, 31, 63)")
