"""The library's calls inside CUDA graphs: captured once and replayed, each
gives the same bits as the same call issued directly (no call allocates,
synchronises or reads host state that capture would freeze wrongly).  The
capture runs on a side stream; the mixed step's second stream joins the
capture through its fork/join events."""
import pytest
import torch

import lightning_attention_attn_gb300 as la
from lightning_attention_attn_gb300 import build as labuild
from lightning_attention_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.load(labuild.build())
    yield
    la.device_status()


def capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    return g, s


def replay(g, s):
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()


@pytest.mark.parametrize("chunk", [0, 64])
def test_prefill_in_a_graph(chunk):
    inp = wl.prefill_inputs([300, 0, 129, 700], 4, 128, dtype=torch.bfloat16, seed=71,
                            device="cuda")
    s0 = wl.cached_states(4, 4, 128, seed=72, device="cuda")
    ref, ref_st = la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, chunk=chunk,
                             initial_state=s0)
    out = torch.empty_like(inp.q)
    st = torch.empty_like(ref_st)
    g, s = capture(lambda s: la.prefill(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens,
                                        chunk=chunk, out=out, final_state=st,
                                        initial_state=s0, stream=s))
    replay(g, s)
    assert torch.equal(out, ref) and torch.equal(st, ref_st)


def test_decode_steps_in_a_graph():
    d = wl.decode_inputs(16, 4, 128, steps=5, dtype=torch.bfloat16, seed=73, device="cuda")
    state0 = d.state.clone()
    outs_ref = [la.decode(d.q[t], d.k[t], d.v[t], d.decay, d.state).clone() for t in range(5)]
    state_ref = d.state.clone()
    d.state.copy_(state0)
    outs = [torch.empty_like(d.q[0]) for _ in range(5)]

    def steps(s):
        for t in range(5):
            la.decode(d.q[t], d.k[t], d.v[t], d.decay, d.state, out=outs[t], stream=s)
    g, s = capture(steps)
    torch.cuda.synchronize()
    d.state.copy_(state0)  # capture launches nothing; start from the same state
    replay(g, s)
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a, b)
    assert torch.equal(d.state, state_ref)


def test_backward_in_a_graph():
    inp = wl.prefill_inputs([200, 77], 2, 128, dtype=torch.bfloat16, seed=74, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(75)
    dout = torch.randn(inp.q.shape, generator=gen, device="cuda").to(torch.bfloat16)
    ref = la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout)
    got = [torch.empty_like(inp.q) for _ in range(3)]
    g, s = capture(lambda s: la.backward(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, dout,
                                         dq=got[0], dk=got[1], dv=got[2], stream=s))
    replay(g, s)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_mixed_step_in_a_graph():
    lengths = [1, 40, 1, 0, 1, 130]
    inp = wl.prefill_inputs(lengths, 2, 128, dtype=torch.bfloat16, seed=76, device="cuda")
    cu_host = inp.cu_seqlens.cpu().tolist()
    st0 = wl.cached_states(len(lengths), 2, 128, seed=77, device="cuda")
    st_ref = st0.clone()
    out_ref = la.mixed_step(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, st_ref,
                            cu_seqlens_host=cu_host)
    torch.cuda.synchronize()
    st = st0.clone()
    out = torch.empty_like(inp.q)
    dstream = torch.cuda.Stream(priority=-1)
    g, s = capture(lambda s: la.mixed_step(inp.q, inp.k, inp.v, inp.decay, inp.cu_seqlens, st,
                                           out=out, prefill_stream=s, decode_stream=dstream,
                                           cu_seqlens_host=cu_host))
    torch.cuda.synchronize()
    st.copy_(st0)
    replay(g, s)
    assert torch.equal(out, out_ref) and torch.equal(st, st_ref)


def test_channel_decay_prefill_in_a_graph():
    """The channel-wise tensor-core kernel replayed from a graph gives the
    eager result bit for bit (cached states, an empty sequence)."""
    inp = wl.prefill_inputs([300, 0, 129, 700], 4, 128, dtype=torch.bfloat16, seed=78,
                            device="cuda")
    jitter = torch.rand((4, 128), generator=torch.Generator().manual_seed(79))
    lam = (inp.decay.cpu()[:, None] * (1.0 - 0.3 * jitter)).to(torch.float32).cuda()
    s0 = wl.cached_states(4, 4, 128, seed=80, device="cuda")
    ref, ref_st = la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens,
                                           initial_state=s0)
    out = torch.empty_like(inp.q)
    st = torch.empty_like(ref_st)
    g, s = capture(lambda s: la.prefill_channel_decay(inp.q, inp.k, inp.v, lam, inp.cu_seqlens,
                                                      out=out, final_state=st,
                                                      initial_state=s0, stream=s))
    replay(g, s)
    assert torch.equal(out, ref) and torch.equal(st, ref_st)
