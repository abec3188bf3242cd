"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle itself.

Sources (MiniMax-01 technical report, CSDN full translation, §2.2.1):
eq. 4 (left product with causal mask), eq. 5 (right-product recursion from
kv_0 = 0), Fig. 12 caption (diagonal decay matrix); §3.2 (data packing);
§3.3.1/§3.3.2 (decode continues a cached state one token at a time).

Every pin is a function of the oracle library so the planted-mistake test at
the bottom can run the same pins on deliberately broken builds of the oracle.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        g = json.load(f)
    return {k: (np.array(v, dtype=np.float64) if isinstance(v, list) else v)
            for k, v in g.items()}


def rnd(rng, T, H, d):
    return [rng.standard_normal((T, H, d)) for _ in range(3)]


# --------------------------------------------------------------- pins
def pin_golden_prefill(lib, name):
    g = golden(name)
    s0 = g.get("initial_state")
    for form in ("quadratic", "recurrent"):
        if form == "quadratic":
            out = oracle.quadratic(g["q"], g["k"], g["v"], g["lambda"],
                                   g["cu_seqlens"], lib=lib, initial_state=s0)
        else:
            out, st = oracle.recurrent(g["q"], g["k"], g["v"], g["lambda"],
                                       g["cu_seqlens"], lib=lib, initial_state=s0)
            np.testing.assert_allclose(st, g["final_state"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(out, g["out"], rtol=0, atol=1e-15,
                                   err_msg=f"{name} {form}")


def pin_golden_backward(lib):
    g = golden("hand_example_backward.json")
    dq, dk, dv = oracle.backward(g["q"], g["k"], g["v"], g["lambda"], g["cu_seqlens"],
                                 g["dout"], lib=lib)
    for got, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        np.testing.assert_allclose(got, g[name], rtol=0, atol=1e-15, err_msg=name)


def pin_backward_finite_differences(lib):
    """The loss sum_t dout_t . o_t is linear in each of q, k and v, so a
    central difference of the (separately pinned) forward form with step 1
    is that argument's exact gradient, up to rounding."""
    rng = np.random.default_rng(10)
    lengths, H, d = [5, 0, 7], 2, 3
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v = rnd(rng, T, H, d)
    g = rng.standard_normal((T, H, d))
    lam = [0.6, 0.95]

    def loss(q_, k_, v_):
        return float(np.sum(oracle.quadratic(q_, k_, v_, lam, cu, lib=lib) * g))

    grads = oracle.backward(q, k, v, lam, cu, g, lib=lib)
    for which, grad in enumerate(grads):
        num = np.zeros_like(grad)
        for idx in np.ndindex(T, H, d):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += 1.0
            args_m[which][idx] -= 1.0
            num[idx] = 0.5 * (loss(*args_p) - loss(*args_m))
        np.testing.assert_allclose(grad, num, rtol=1e-10, atol=1e-10,
                                   err_msg="dq dk dv"[3 * which:3 * which + 2])


def pin_backward_lambda_one(lib):
    """lambda = 1: dq_t = dout_t (prefix sum of v k^T), dk_u = (suffix sum
    of q dout^T) v_u, dv_u = (suffix sum of dout q^T) k_u (numpy cumsum)."""
    rng = np.random.default_rng(11)
    T, H, d = 19, 2, 4
    q, k, v = rnd(rng, T, H, d)
    g = rng.standard_normal((T, H, d))
    pre_vk = np.cumsum(np.einsum("thi,thj->thij", v, k), axis=0)
    suf_qg = np.cumsum(np.einsum("thi,thj->thij", q, g)[::-1], axis=0)[::-1]
    want_dq = np.einsum("thi,thij->thj", g, pre_vk)
    want_dk = np.einsum("thij,thj->thi", suf_qg, v)
    want_dv = np.einsum("thij,thi->thj", suf_qg, k)
    dq, dk, dv = oracle.backward(q, k, v, [1.0, 1.0], [0, T], g, lib=lib)
    for got, want in ((dq, want_dq), (dk, want_dk), (dv, want_dv)):
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def pin_golden_channel_decay(lib):
    g = golden("hand_example_channel_decay.json")
    outq = oracle.quadratic_cw(g["q"], g["k"], g["v"], g["lambda_cw"], g["cu_seqlens"], lib=lib)
    outr, st = oracle.recurrent_cw(g["q"], g["k"], g["v"], g["lambda_cw"], g["cu_seqlens"],
                                   lib=lib)
    for got in (outq, outr):
        np.testing.assert_allclose(got, g["out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(st, g["final_state"], rtol=0, atol=1e-15)


def pin_channel_decay_uniform_reduces(lib):
    """Equal channel decays reduce to the (separately pinned) scalar forms,
    with and without a cached state; the decode step likewise."""
    rng = np.random.default_rng(12)
    lengths, H, d = [7, 0, 19], 3, 5
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = rnd(rng, int(cu[-1]), H, d)
    lam = np.array([0.4, 0.9, 1.0])
    lam_cw = np.repeat(lam[:, None], d, axis=1)
    s0 = rng.standard_normal((len(lengths), H, d, d))
    for init in (None, s0):
        want_q = oracle.quadratic(q, k, v, lam, cu, lib=lib, initial_state=init)
        want_r, want_st = oracle.recurrent(q, k, v, lam, cu, lib=lib, initial_state=init)
        got_q = oracle.quadratic_cw(q, k, v, lam_cw, cu, lib=lib, initial_state=init)
        got_r, got_st = oracle.recurrent_cw(q, k, v, lam_cw, cu, lib=lib, initial_state=init)
        np.testing.assert_allclose(got_q, want_q, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got_r, want_r, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(got_st, want_st, rtol=1e-12, atol=1e-12)
    qd, kd, vd = (rng.standard_normal((4, H, d)) for _ in range(3))
    st = rng.standard_normal((4, H, d, d))
    o1, n1 = oracle.decode(qd, kd, vd, lam, st, lib=lib)
    o2, n2 = oracle.decode_cw(qd, kd, vd, lam_cw, st, lib=lib)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(n2, n1, rtol=1e-12, atol=1e-12)


def pin_channel_decay_two_forms(lib):
    """With distinct channel decays the left product and the recursion
    (independent formulations) agree, from zero and from a cached state;
    the decode step continues the recursion."""
    rng = np.random.default_rng(13)
    lengths, H, d = [40, 1, 0, 23], 2, 6
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = rnd(rng, int(cu[-1]), H, d)
    lam_cw = rng.uniform(0.3, 1.0, size=(H, d))
    s0 = rng.standard_normal((len(lengths), H, d, d))
    for init in (None, s0):
        oq = oracle.quadratic_cw(q, k, v, lam_cw, cu, lib=lib, initial_state=init)
        orr, _ = oracle.recurrent_cw(q, k, v, lam_cw, cu, lib=lib, initial_state=init)
        assert np.max(np.abs(oq - orr)) <= 1e-10 * max(1.0, float(np.sqrt(np.mean(orr ** 2))))
    L = 12
    full, st_full = oracle.recurrent_cw(q[:L + 1], k[:L + 1], v[:L + 1], lam_cw, [0, L + 1], lib=lib)
    _, st = oracle.recurrent_cw(q[:L], k[:L], v[:L], lam_cw, [0, L], lib=lib)
    o, st2 = oracle.decode_cw(q[L:L + 1], k[L:L + 1], v[L:L + 1], lam_cw, st, lib=lib)
    np.testing.assert_allclose(o[0], full[L], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(st2, st_full, rtol=1e-12, atol=1e-13)


def pin_golden_decode(lib):
    g = golden("hand_example_decode.json")
    out, st = oracle.decode(g["q"], g["k"], g["v"], g["lambda"], g["state"], lib=lib)
    np.testing.assert_allclose(out, g["out"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(st, g["new_state"], rtol=0, atol=1e-15)


def pin_geometric_d1(lib):
    """q = k = v = 1, d = 1: o_t = sum_{u<=t} lambda^(t-u) = (1-lambda^(t+1))/(1-lambda)."""
    L = 50
    for lam in (0.5, 0.9, 0.3997):
        ones = np.ones((L, 1, 1))
        want = np.array([(1 - lam ** (t + 1)) / (1 - lam) for t in range(L)])
        want_state = want[-1]
        for form in ("quadratic", "recurrent"):
            if form == "quadratic":
                out = oracle.quadratic(ones, ones, ones, [lam], [0, L], lib=lib)
            else:
                out, st = oracle.recurrent(ones, ones, ones, [lam], [0, L], lib=lib)
                lam32 = float(np.float32(lam))
                want_state = (1 - lam32 ** L) / (1 - lam32)
                np.testing.assert_allclose(st.ravel(), [want_state], rtol=1e-12)
            lam32 = float(np.float32(lam))
            want = np.array([(1 - lam32 ** (t + 1)) / (1 - lam32) for t in range(L)])
            np.testing.assert_allclose(out.ravel(), want, rtol=1e-12)


def pin_geometric_d1_with_state(lib):
    """q = k = v = 1, d = 1, cached state S0:
    kv_t = lambda^(t+1) S0 + (1 - lambda^(t+1)) / (1 - lambda) = o_t."""
    L = 40
    for lam, s0 in ((0.5, 3.0), (0.9, -2.0), (0.3997, 0.25)):
        ones = np.ones((L, 1, 1))
        lam32 = float(np.float32(lam))
        want = np.array([lam32 ** (t + 1) * s0 + (1 - lam32 ** (t + 1)) / (1 - lam32)
                         for t in range(L)])
        init = np.full((1, 1, 1, 1), s0)
        outq = oracle.quadratic(ones, ones, ones, [lam], [0, L], lib=lib, initial_state=init)
        outr, st = oracle.recurrent(ones, ones, ones, [lam], [0, L], lib=lib, initial_state=init)
        np.testing.assert_allclose(outq.ravel(), want, rtol=1e-12)
        np.testing.assert_allclose(outr.ravel(), want, rtol=1e-12)
        np.testing.assert_allclose(st.ravel(), [want[-1]], rtol=1e-12)


def pin_prefix_cache_equivalence(lib):
    """A segment run from the state of its prefix equals the tail of one run
    over prefix + segment; the prefix state is taken from the closed form
    sum_u lambda^(P-1-u) k_u^T v_u (numpy), not from the oracle."""
    rng = np.random.default_rng(9)
    P, L, H, d = 23, 17, 3, 5
    q, k, v = rnd(rng, P + L, H, d)
    lam = np.array([0.3997, 0.8, 0.99])
    lam32 = np.float32(lam).astype(np.float64)
    w = lam32[None, :] ** (P - 1 - np.arange(P))[:, None]
    s_prefix = np.einsum("uh,uhi,uhj->hij", w, k[:P], v[:P])[None]
    full_q = oracle.quadratic(q, k, v, lam, [0, P + L], lib=lib)
    full_r, st_full = oracle.recurrent(q, k, v, lam, [0, P + L], lib=lib)
    seg = slice(P, P + L)
    seg_q = oracle.quadratic(q[seg], k[seg], v[seg], lam, [0, L], lib=lib,
                             initial_state=s_prefix)
    seg_r, st_seg = oracle.recurrent(q[seg], k[seg], v[seg], lam, [0, L], lib=lib,
                                     initial_state=s_prefix)
    for got, full in ((seg_q, full_q), (seg_r, full_r)):
        np.testing.assert_allclose(got, full[seg], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(st_seg, st_full, rtol=1e-11, atol=1e-12)
    # an empty segment hands the cached state straight through
    _, st_empty = oracle.recurrent(q[:0], k[:0], v[:0], lam, [0, 0], lib=lib,
                                   initial_state=s_prefix)
    np.testing.assert_array_equal(st_empty, s_prefix)


def pin_lambda_one_prefix_sums(lib):
    """lambda = 1: o_t = q_t . (prefix sum over u <= t of outer(k_u, v_u))."""
    rng = np.random.default_rng(1)
    T, H, d = 37, 2, 5
    q, k, v = rnd(rng, T, H, d)
    outer = np.einsum("thi,thj->thij", k, v)
    C = np.cumsum(outer, axis=0)
    want = np.einsum("thi,thij->thj", q, C)
    for form in ("quadratic", "recurrent"):
        if form == "quadratic":
            out = oracle.quadratic(q, k, v, [1.0, 1.0], [0, T], lib=lib)
        else:
            out, st = oracle.recurrent(q, k, v, [1.0, 1.0], [0, T], lib=lib)
            np.testing.assert_allclose(st[0], C[-1], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def pin_lambda_tiny(lib):
    """lambda -> 0: only the diagonal term survives, o_t = (q_t . k_t) v_t."""
    rng = np.random.default_rng(2)
    T, H, d = 20, 1, 4
    q, k, v = rnd(rng, T, H, d)
    want = np.einsum("thi,thi->th", q, k)[..., None] * v
    for form in ("quadratic", "recurrent"):
        if form == "quadratic":
            out = oracle.quadratic(q, k, v, [1e-30], [0, T], lib=lib)
        else:
            out, _ = oracle.recurrent(q, k, v, [1e-30], [0, T], lib=lib)
        np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-25)


def exact_brute(q, k, v, lam, L):
    """Exact rationals: O = (Q K^T (.) W) V with W_tu = lam^(t-u) for t >= u."""
    d = q.shape[1]
    out = [[Fraction(0)] * d for _ in range(L)]
    for t in range(L):
        for u in range(t + 1):
            s = sum(Fraction(int(q[t, i])) * Fraction(int(k[u, i])) for i in range(d))
            w = lam ** (t - u)
            for j in range(d):
                out[t][j] += s * w * Fraction(int(v[u, j]))
    st = [[sum(lam ** (L - 1 - u) * int(k[u, i]) * int(v[u, j]) for u in range(L))
           for j in range(d)] for i in range(d)]
    return out, st


def pin_brute_force_exact(lib, Ls=range(1, 9), ds=range(1, 5), reps=2):
    """Small integer inputs, lambda = 1/2: every fp64 operation is exact, so
    both forms must reproduce the exact rational result bit for bit."""
    rng = np.random.default_rng(3)
    lam = Fraction(1, 2)
    for L, d, _ in itertools.product(Ls, ds, range(reps)):
        q, k, v = (rng.integers(-3, 4, size=(L, d)).astype(np.float64) for _ in range(3))
        want, want_st = exact_brute(q, k, v, lam, L)
        want = np.array([[float(x) for x in r] for r in want])
        want_st = np.array([[float(x) for x in r] for r in want_st])
        args = (q[:, None, :], k[:, None, :], v[:, None, :], [0.5], [0, L])
        oq = oracle.quadratic(*args, lib=lib)[:, 0, :]
        orr, st = oracle.recurrent(*args, lib=lib)
        assert np.array_equal(oq, want), (L, d)
        assert np.array_equal(orr[:, 0, :], want), (L, d)
        assert np.array_equal(st[0, 0], want_st), (L, d)


def pin_two_forms_agree(lib, cases=None):
    """eq. 4 (left product) and eq. 5 (recursion) are the same function."""
    rng = np.random.default_rng(4)
    cases = cases or [([300], 1, 64), ([1, 7, 64, 129, 0, 33], 3, 16), ([256], 1, 64)]
    for lengths, H, d in cases:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        T = int(cu[-1])
        q, k, v = rnd(rng, T, H, d)
        q *= d ** -0.5
        k *= d ** -0.5
        lam = np.exp(-2.0 ** (-8.0 * (np.arange(H) + 1) / H))
        oq = oracle.quadratic(q, k, v, lam, cu, lib=lib)
        orr, _ = oracle.recurrent(q, k, v, lam, cu, lib=lib)
        scale = max(1.0, float(np.sqrt(np.mean(orr ** 2))))
        assert np.max(np.abs(oq - orr)) <= 1e-10 * scale


def pin_final_state_closed_form(lib):
    """final state = sum_u lambda^(L-1-u) k_u^T v_u (per sequence, per head)."""
    rng = np.random.default_rng(5)
    lengths, H, d = [5, 0, 40, 17], 3, 6
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = rnd(rng, int(cu[-1]), H, d)
    lam = np.array([0.3997, 0.9, 1.0])
    _, st = oracle.recurrent(q, k, v, lam, cu, lib=lib)
    lam32 = np.float32(lam).astype(np.float64)
    for s, L in enumerate(lengths):
        seg = slice(cu[s], cu[s + 1])
        w = lam32[None, :] ** (L - 1 - np.arange(L))[:, None]  # [L, H]
        want = np.einsum("uh,uhi,uhj->hij", w, k[seg], v[seg])
        np.testing.assert_allclose(st[s], want, rtol=1e-12, atol=1e-13)


def pin_packing(lib):
    """Packed sequences equal separate runs (state restarts at each start)."""
    rng = np.random.default_rng(6)
    lengths, H, d = [9, 1, 0, 30], 2, 8
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    q, k, v = rnd(rng, int(cu[-1]), H, d)
    lam = [0.7, 0.95]
    for form in (oracle.quadratic, oracle.recurrent):
        packed = form(q, k, v, lam, cu, lib=lib)
        packed = packed[0] if isinstance(packed, tuple) else packed
        for s in range(len(lengths)):
            seg = slice(cu[s], cu[s + 1])
            L = lengths[s]
            one = form(q[seg], k[seg], v[seg], lam, [0, L], lib=lib)
            one = one[0] if isinstance(one, tuple) else one
            np.testing.assert_array_equal(packed[seg], one)


def pin_decode_continuation(lib):
    """Prefill of L tokens then one decode step equals prefill of L + 1."""
    rng = np.random.default_rng(7)
    L, H, d = 12, 2, 4
    q, k, v = rnd(rng, L + 1, H, d)
    lam = [0.5, 0.99]
    full, st_full = oracle.recurrent(q, k, v, lam, [0, L + 1], lib=lib)
    _, st = oracle.recurrent(q[:L], k[:L], v[:L], lam, [0, L], lib=lib)
    o, st2 = oracle.decode(q[L:], k[L:], v[L:], lam, st, lib=lib)
    np.testing.assert_allclose(o[0], full[L], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(st2, st_full, rtol=1e-13, atol=1e-14)
    quad = oracle.quadratic(q, k, v, lam, [0, L + 1], lib=lib)
    np.testing.assert_allclose(o[0], quad[L], rtol=1e-11, atol=1e-12)


ALL_PINS = {
    "golden_a": lambda lib: pin_golden_prefill(lib, "hand_example_a.json"),
    "golden_b": lambda lib: pin_golden_prefill(lib, "hand_example_b.json"),
    "golden_packed": lambda lib: pin_golden_prefill(lib, "hand_example_packed.json"),
    "golden_state": lambda lib: pin_golden_prefill(lib, "hand_example_state.json"),
    "golden_decode": pin_golden_decode,
    "golden_backward": pin_golden_backward,
    "golden_channel_decay": pin_golden_channel_decay,
    "cw_uniform": pin_channel_decay_uniform_reduces,
    "cw_two_forms": pin_channel_decay_two_forms,
    "backward_fd": pin_backward_finite_differences,
    "backward_lambda_one": pin_backward_lambda_one,
    "geometric_d1_state": pin_geometric_d1_with_state,
    "prefix_cache": pin_prefix_cache_equivalence,
    "geometric_d1": pin_geometric_d1,
    "lambda_one": pin_lambda_one_prefix_sums,
    "lambda_tiny": pin_lambda_tiny,
    "brute_force": lambda lib: pin_brute_force_exact(lib, Ls=range(1, 6), ds=range(1, 4), reps=1),
    "two_forms": lambda lib: pin_two_forms_agree(lib, cases=[([40, 0, 9], 2, 6)]),
    "final_state": pin_final_state_closed_form,
    "packing": pin_packing,
    "decode_continuation": pin_decode_continuation,
}


# --------------------------------------------------------------- tests
@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("name", ["hand_example_a.json", "hand_example_b.json",
                                  "hand_example_packed.json", "hand_example_state.json"])
def test_golden_prefill(lib, name):
    pin_golden_prefill(lib, name)


def test_golden_backward(lib):
    pin_golden_backward(lib)


def test_backward_finite_differences(lib):
    pin_backward_finite_differences(lib)


def test_backward_lambda_one(lib):
    pin_backward_lambda_one(lib)


def test_golden_channel_decay(lib):
    pin_golden_channel_decay(lib)


def test_channel_decay_uniform_reduces(lib):
    pin_channel_decay_uniform_reduces(lib)


def test_channel_decay_two_forms(lib):
    pin_channel_decay_two_forms(lib)


def test_golden_decode(lib):
    pin_golden_decode(lib)


def test_geometric_d1(lib):
    pin_geometric_d1(lib)


def test_geometric_d1_with_state(lib):
    pin_geometric_d1_with_state(lib)


def test_prefix_cache_equivalence(lib):
    pin_prefix_cache_equivalence(lib)


def test_lambda_one_prefix_sums(lib):
    pin_lambda_one_prefix_sums(lib)


def test_lambda_tiny(lib):
    pin_lambda_tiny(lib)


def test_brute_force_exact(lib):
    pin_brute_force_exact(lib)


def test_two_forms_agree(lib):
    pin_two_forms_agree(lib)


def test_final_state_closed_form(lib):
    pin_final_state_closed_form(lib)


def test_packing(lib):
    pin_packing(lib)


def test_decode_continuation(lib):
    pin_decode_continuation(lib)


def test_head_selection(lib):
    rng = np.random.default_rng(8)
    q, k, v = rnd(rng, 10, 4, 3)
    lam = [0.5, 0.6, 0.7, 0.8]
    full, st = oracle.recurrent(q, k, v, lam, [0, 10], lib=lib)
    part, stp = oracle.recurrent(q, k, v, lam, [0, 10], heads=[1, 3], lib=lib)
    np.testing.assert_array_equal(part[:, [1, 3]], full[:, [1, 3]])
    assert not part[:, [0, 2]].any()
    np.testing.assert_array_equal(stp[:, [1, 3]], st[:, [1, 3]])
    qd = oracle.quadratic(q, k, v, lam, [0, 10], heads=[2], lib=lib)
    assert not qd[:, [0, 1, 3]].any()


def test_bad_cu_seqlens_rejected(lib):
    q = np.zeros((4, 1, 2))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, [0.5], np.array([0, 3, 2, 4]), lib=lib)
    with pytest.raises(ValueError):
        oracle.quadratic(q, q, q, [0.5], np.array([1, 4]), lib=lib)


def test_decay_rounded_to_fp32():
    lam = oracle.decay_as_seen([0.1])
    assert lam[0] == float(np.float32(0.1)) and lam[0] != 0.1


# ------------------------------------------------ planted mistakes
# Each mutant changes one plausible thing in the oracle's C source; at least
# one pin must fail on it.  (Mistakes are planted in the oracle, on the CPU.)
MUTANTS = {
    "quad_exponent_off_by_one": ("pow(la, (double)(t - u))", "pow(la, (double)(t - u + 1))"),
    "quad_drop_diagonal": ("for (long u = 0; u <= t; ++u)", "for (long u = 0; u < t; ++u)"),
    "quad_wrong_sign_exponent": ("pow(la, (double)(t - u))", "pow(la, (double)(u - t))"),
    "rec_transposed_outer": ("la * kv[(long)i * d + j] + kt[i] * vt[j]",
                             "la * kv[(long)i * d + j] + kt[j] * vt[i]"),
    "rec_no_decay": ("la * kv[(long)i * d + j] + kt[i] * vt[j]",
                     "kv[(long)i * d + j] + kt[i] * vt[j]"),
    "rec_transposed_read": ("acc += qt[i] * kv[(long)i * d + j]",
                            "acc += qt[i] * kv[(long)j * d + i]"),
    "rec_no_reset_between_sequences": ("double *kv = (double *)calloc((size_t)d * d, sizeof(double));",
                                       "static __thread double *kvp = 0; if (!kvp) kvp = (double *)calloc(4096, sizeof(double)); double *kv = kvp; int keep = 1;"),
    "init_state_ignored": ("        if (initial_state)\n            memcpy(kv,",
                           "        if (0)\n            memcpy(kv,"),
    "quad_init_exponent_t": ("pow(la, (double)(t + 1))", "pow(la, (double)(t))"),
    "quad_init_transposed": ("acc += qt[i] * s0[(long)i * d + j]",
                             "acc += qt[i] * s0[(long)j * d + i]"),
    "bwd_dk_uses_k": ("dku[i] += w * g_v * qt[i]", "dku[i] += w * g_v * ku[i]"),
    "bwd_dv_wrong_dot": ("dvu[i] += w * q_k * gt[i]", "dvu[i] += w * g_v * gt[i]"),
    "bwd_dq_no_decay": ("dqt[i] += w * g_v * ku[i]", "dqt[i] += g_v * ku[i]"),
    "cw_decay_on_value_columns": ("la[i] * kv[(long)i * d + j] + kt[i] * vt[j]",
                                  "la[j] * kv[(long)i * d + j] + kt[i] * vt[j]"),
    "cw_quad_uniform_decay": ("qt[i] * ku[i] * pow(la[i], (double)(t - u))",
                              "qt[i] * ku[i] * pow(la[0], (double)(t - u))"),
    "cw_dec_decay_on_value_columns": ("la[i] * kv[(long)i * d + j] + kb[i] * vb[j]",
                                      "la[j] * kv[(long)i * d + j] + kb[i] * vb[j]"),
    "dec_read_before_update": (
        "                kv[(long)i * d + j] = la * kv[(long)i * d + j] + kb[i] * vb[j];\n"
        "        for (int j = 0; j < d; ++j) {\n"
        "            double acc = 0.0;\n"
        "            for (int i = 0; i < d; ++i) acc += qb[i] * kv[(long)i * d + j];\n"
        "            out[p * d + j] = acc;\n"
        "        }",
        "                ;\n"
        "        for (int j = 0; j < d; ++j) {\n"
        "            double acc = 0.0;\n"
        "            for (int i = 0; i < d; ++i) acc += qb[i] * kv[(long)i * d + j];\n"
        "            out[p * d + j] = acc;\n"
        "        }\n"
        "        for (int i = 0; i < d; ++i) for (int j = 0; j < d; ++j)"
        " kv[(long)i * d + j] = la * kv[(long)i * d + j] + kb[i] * vb[j];"),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant, tmp_path):
    src = open(oracle.source_path()).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation site for {mutant} not found"
    if mutant == "rec_no_reset_between_sequences":
        # keep the state across (sequence, head) pairs: never free, never clear
        src = src.replace(old, new).replace("        free(kv);\n", "")
    else:
        src = src.replace(old, new)
    path = tmp_path / "mut.c"
    path.write_text(src)
    so = oracle.build(str(path), str(tmp_path / "libmut.so"))
    mlib = oracle.load(so)
    # single thread: the no-reset mutant's state then really carries over
    mlib.la_oracle_max_threads(1)
    failed = []
    try:
        for name, pin in ALL_PINS.items():
            try:
                pin(mlib)
            except AssertionError:
                failed.append(name)
    finally:
        mlib.la_oracle_max_threads(os.cpu_count() or 1)
    assert failed, f"no pin caught planted mistake {mutant}"
