"""Pins of the FP64 oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to something independent of its own code: finite
differences of its forward, closed forms at special inputs, a chunked
(WY / UT transform) restatement, or structural invariants of the recurrence
(causality, value-first orientation, GQA = repeated heads, packed = fixed).
A plausible slip in the oracle (a dropped term, a wrong sign, a transposed
state, the output read before the update, the decay on rows instead of columns,
a wrong GQA map) fails at least one of them.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CONTRACT = json.load(open(os.path.join(GOLDEN, "contract.json")))


def rand_problem(seed, lengths, hqk, hv, dk, dv, gate_scale=1.0):
    """Random float64 problem in packed layout (B = 1)."""
    rng = np.random.default_rng(seed)
    T = sum(lengths)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    N = len(lengths)
    return dict(
        q=rng.standard_normal((1, T, hqk, dk)),
        k=rng.standard_normal((1, T, hqk, dk)),
        v=rng.standard_normal((1, T, hv, dv)),
        g=gate_scale * rng.standard_normal((1, T, hv, dk)),
        beta=rng.standard_normal((1, T, hv)),
        A_log=rng.uniform(0, math.log(16), hv),
        dt_bias=0.1 * rng.standard_normal((hv, dk)),
        h0=0.5 * rng.standard_normal((N, hv, dv, dk)),
        do=rng.standard_normal((1, T, hv, dv)),
        dfinal_state=0.5 * rng.standard_normal((N, hv, dv, dk)),
        cu_seqlens=cu,
    )


FWD_KEYS = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0"]


def fwd(p, **kw):
    return oracle.forward(*[p[x] for x in FWD_KEYS], cu_seqlens=p.get("cu_seqlens"), **kw)


def bwd(p, **kw):
    return oracle.backward(*[p[x] for x in FWD_KEYS], p["do"], p["dfinal_state"],
                           cu_seqlens=p.get("cu_seqlens"), **kw)


def loss(p, **kw):
    o, hT = fwd(p, **kw)
    return float(np.sum(o * p["do"]) + np.sum(hT * p["dfinal_state"]))


def rel(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-300))


# ---------------------------------------------------------------- backward pins

GRAD_INPUTS = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0"]


@pytest.mark.parametrize("dims", [(1, 2, 4, 4, [3, 5]), (2, 2, 4, 6, [6]), (1, 3, 5, 3, [2, 1, 4])])
def test_backward_matches_finite_differences_small(dims):
    """Central differences of the oracle's forward along a random direction,
    separately for each of the eight differentiated inputs (any K, V)."""
    hqk, hv, dk, dv, lengths = dims
    p = rand_problem(11, lengths, hqk, hv, dk, dv)
    grads = dict(zip(GRAD_INPUTS, bwd(p, scale=0.7)))
    rng = np.random.default_rng(5)
    h = 1e-6
    for name in GRAD_INPUTS:
        delta = rng.standard_normal(p[name].shape)
        pp = dict(p); pp[name] = p[name] + h * delta
        pm = dict(p); pm[name] = p[name] - h * delta
        fd = (loss(pp, scale=0.7) - loss(pm, scale=0.7)) / (2 * h)
        an = float(np.sum(grads[name] * delta))
        assert abs(fd - an) <= 2e-7 * max(1.0, abs(an)), (name, fd, an)


def test_backward_matches_finite_differences_full_dim_gqa_packed():
    """Same check at the documented head dimension 128, with GQA (2 value heads
    per query/key head) and two packed sequences."""
    p = rand_problem(3, [3, 2], 1, 2, 128, 128)
    grads = dict(zip(GRAD_INPUTS, bwd(p)))
    rng = np.random.default_rng(7)
    h = 1e-6
    for name in GRAD_INPUTS:
        delta = rng.standard_normal(p[name].shape)
        pp = dict(p); pp[name] = p[name] + h * delta
        pm = dict(p); pm[name] = p[name] - h * delta
        fd = (loss(pp) - loss(pm)) / (2 * h)
        an = float(np.sum(grads[name] * delta))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def _torch_sequential_forward(x, cu, r, scale):
    """The token-by-token recurrence in float64 torch ops (flashinfer.kda_training, module
    description: L2-normalised q and k with eps 1e-6, per-key log decay -5 sigmoid(exp(A_log)
    (g + dt_bias)), sigmoid beta, value-first state; update order decay, delta correction,
    rank-1 write, output from the updated state), written apart from the oracle so that
    autograd can differentiate it mechanically."""
    import torch
    T, Hv = x["v"].shape[1], x["v"].shape[2]
    rows = [[None] * Hv for _ in range(T)]  # rows[t][h] = o_t of value head h
    finals = []
    for n in range(len(cu) - 1):
        per_head = []
        for h in range(x["v"].shape[2]):
            S = x["h0"][n, h]
            for t in range(int(cu[n]), int(cu[n + 1])):
                qv, kv = x["q"][0, t, h // r], x["k"][0, t, h // r]
                qn = qv / torch.sqrt((qv * qv).sum() + 1e-6)
                kn = kv / torch.sqrt((kv * kv).sum() + 1e-6)
                d = torch.exp(-5.0 * torch.sigmoid(torch.exp(x["A_log"][h]) * (x["g"][0, t, h] + x["dt_bias"][h])))
                S = S * d[None, :]
                u = x["v"][0, t, h] - S @ kn
                S = S + torch.sigmoid(x["beta"][0, t, h]) * torch.outer(u, kn)
                rows[t][h] = scale * (S @ qn)
            per_head.append(S)
        finals.append(torch.stack(per_head))
    o = torch.stack([torch.stack(r) for r in rows])[None]
    return o, torch.stack(finals)


def test_backward_matches_autograd_of_sequential_forward():
    """All eight gradients equal, to float64 rounding, those that autograd takes through a
    separately written token-by-token forward (head dimension 128, GQA 1:2, two packed
    sequences); finite differences only hold them to ~1e-7."""
    torch = pytest.importorskip("torch")
    p = rand_problem(31, [4, 3], 1, 2, 128, 128)
    scale = 1.0 / math.sqrt(128.0)
    x = {k: torch.tensor(p[k], dtype=torch.float64, requires_grad=True) for k in GRAD_INPUTS}
    o, hT = _torch_sequential_forward(x, p["cu_seqlens"], 2, scale)
    o_ref, hT_ref = fwd(p)
    assert rel(o.detach().numpy(), o_ref) < 1e-12 and rel(hT.detach().numpy(), hT_ref) < 1e-12
    L = (o * torch.tensor(p["do"])).sum() + (hT * torch.tensor(p["dfinal_state"])).sum()
    auto = torch.autograd.grad(L, [x[k] for k in GRAD_INPUTS])
    for name, a_, b_ in zip(GRAD_INPUTS, auto, bwd(p)):
        assert rel(b_, a_.numpy()) < 1e-10, (name, rel(b_, a_.numpy()))


def test_dinitial_state_independent_of_h0_and_v():
    """The adjoint chain of the state never reads the state itself, so
    dinitial_state must not change when h0 and v change."""
    p = rand_problem(21, [7, 4], 1, 2, 8, 8)
    d1 = bwd(p)[7]
    rng = np.random.default_rng(1)
    p2 = dict(p, h0=rng.standard_normal(p["h0"].shape), v=rng.standard_normal(p["v"].shape))
    d2 = bwd(p2)[7]
    assert np.array_equal(d1, d2)


def test_parameter_gradient_identities():
    """ddt_bias[h] = sum_t dg[t, h]; dA_log[h] = sum_t,k dg (g + dt_bias)."""
    p = rand_problem(4, [9, 5], 2, 4, 6, 5)
    dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dh0 = bwd(p)
    np.testing.assert_allclose(ddt_bias, dg[0].sum(axis=0), rtol=1e-12, atol=1e-14)
    z_over_ea = p["g"][0] + p["dt_bias"][None]
    np.testing.assert_allclose(dA_log, (dg[0] * z_over_ea).sum(axis=(0, 2)), rtol=1e-11, atol=1e-14)


# ----------------------------------------------------------------- forward pins

def basis_queries(T, dk, rng):
    """Rows c * e_j so that the L2-normalised query is known in closed form."""
    idx = rng.integers(0, dk, T)
    c = rng.uniform(0.5, 3.0, T)
    q = np.zeros((1, T, 1, dk))
    q[0, np.arange(T), 0, idx] = c
    qhat = q.copy()
    qhat[0, np.arange(T), 0, idx] = c / np.sqrt(c * c + CONTRACT["norm_eps"]["value"])
    return q, qhat


def test_beta_zero_is_pure_per_dim_decay():
    """beta = sigmoid(-inf) = 0 removes every write: with g + dt_bias = 0 the
    gate is sigmoid(0) = 1/2 in every dimension, d = exp(-2.5), so
    S_T = h0 exp(-2.5 T) and o_t = scale exp(-2.5 (t+1)) h0 q^_t."""
    T, dk, dv = 6, 8, 5
    rng = np.random.default_rng(0)
    q, qhat = basis_queries(T, dk, rng)
    p = dict(q=q, k=rng.standard_normal((1, T, 1, dk)), v=rng.standard_normal((1, T, 1, dv)),
             g=np.zeros((1, T, 1, dk)), beta=np.full((1, T, 1), -np.inf),
             A_log=np.array([0.3]), dt_bias=np.zeros((1, dk)),
             h0=rng.standard_normal((1, 1, dv, dk)))
    o, hT = fwd(p, scale=0.25)
    np.testing.assert_allclose(hT, p["h0"] * math.exp(-2.5 * T), rtol=1e-13)
    for t in range(T):
        want = 0.25 * math.exp(-2.5 * (t + 1)) * p["h0"][0, 0] @ qhat[0, t, 0]
        np.testing.assert_allclose(o[0, t, 0], want, rtol=1e-12, atol=1e-300)


def test_gate_formula_per_key_dimension():
    """With A_log = ln 2 and g + dt_bias = ln(m) per key dim m, the gate is
    sigmoid(2 ln m) = m^2 / (1 + m^2); decay exp(-5 m^2/(1+m^2)) must scale the
    key columns of the value-first state (beta = 0, one token)."""
    dk, dv = 6, 3
    m = np.arange(1, dk + 1, dtype=np.float64)
    rng = np.random.default_rng(2)
    h0 = rng.standard_normal((1, 1, dv, dk))
    g = np.zeros((1, 1, 1, dk)); g[0, 0, 0] = 0.5 * np.log(m)
    dt = (0.5 * np.log(m))[None]
    p = dict(q=rng.standard_normal((1, 1, 1, dk)), k=rng.standard_normal((1, 1, 1, dk)),
             v=rng.standard_normal((1, 1, 1, dv)), g=g, beta=np.full((1, 1, 1), -np.inf),
             A_log=np.array([math.log(2.0)]), dt_bias=dt, h0=h0)
    _, hT = fwd(p)
    d = np.exp(-5.0 * m * m / (1.0 + m * m))
    np.testing.assert_allclose(hT[0, 0], h0[0, 0] * d[None, :], rtol=1e-13)
    # a different lower bound rescales the exponent
    _, hT3 = fwd(p, lower_bound=-3.0)
    np.testing.assert_allclose(hT3[0, 0], h0[0, 0] * np.exp(-3.0 * m * m / (1 + m * m))[None, :],
                               rtol=1e-13)


def test_decay_bounds():
    """exp(-5) <= d <= 1 for any gate input; A_log -> -inf gives d = exp(-2.5)."""
    dk, dv = 16, 2
    rng = np.random.default_rng(3)
    h0 = np.ones((1, 1, dv, dk))
    for A_log, g in [(2.0, 30 * rng.standard_normal(dk)), (0.0, rng.standard_normal(dk)),
                     (-np.inf, 100 * rng.standard_normal(dk))]:
        p = dict(q=rng.standard_normal((1, 1, 1, dk)), k=rng.standard_normal((1, 1, 1, dk)),
                 v=rng.standard_normal((1, 1, 1, dv)), g=g.reshape(1, 1, 1, dk),
                 beta=np.full((1, 1, 1), -np.inf), A_log=np.array([A_log]),
                 dt_bias=np.zeros((1, dk)), h0=h0)
        _, hT = fwd(p)
        d = hT[0, 0, 0]
        assert np.all(d >= math.exp(-5.0) * (1 - 1e-15)) and np.all(d <= 1.0)
        if A_log == -np.inf:
            np.testing.assert_allclose(d, math.exp(-2.5), rtol=1e-15)


def test_beta_one_with_query_equal_key_returns_value():
    """The delta rule with beta = 1 overwrites the memory at the key:
    S_t k^_t = v_t (up to |k^|^2 = 1 - eps/|k|^2). Reading the output from the
    post-update state with q = k then gives o_t = scale v_t for any history."""
    lengths, dk, dv = [5, 9], 128, 128
    p = rand_problem(8, lengths, 2, 4, dk, dv)
    p["q"] = p["k"].copy()
    p["beta"] = np.full_like(p["beta"], np.inf)
    o, _ = fwd(p)
    s = CONTRACT["scale"]["value"]
    np.testing.assert_allclose(o, s * p["v"], rtol=0, atol=1e-7 * s * np.abs(p["v"]).max())


def test_beta_half_first_token_closed_form():
    """First token, beta = sigmoid(0) = 1/2, q = k, gate 1/2 (d = exp(-2.5)):
    o = scale (S' k^ (1 - |k^|^2 / 2) + v |k^|^2 / 2) with S' = h0 exp(-2.5)."""
    dk, dv = 8, 4
    rng = np.random.default_rng(9)
    k = rng.standard_normal((1, 1, 1, dk))
    nk2 = float(np.sum(k * k))
    khat = k[0, 0, 0] / math.sqrt(nk2 + 1e-6)
    kk = float(khat @ khat)
    p = dict(q=k.copy(), k=k, v=rng.standard_normal((1, 1, 1, dv)), g=np.zeros((1, 1, 1, dk)),
             beta=np.zeros((1, 1, 1)), A_log=np.array([1.0]), dt_bias=np.zeros((1, dk)),
             h0=rng.standard_normal((1, 1, dv, dk)))
    o, _ = fwd(p, scale=1.0)
    Sp_k = math.exp(-2.5) * p["h0"][0, 0] @ khat
    want = Sp_k * (1 - 0.5 * kk) + 0.5 * kk * p["v"][0, 0, 0]
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-13)


def test_state_is_value_first():
    """h0 = e_a e_b^T (value row a, key column b), no writes, query along key
    b: only output element a is non-zero. A key-first reading puts it at b."""
    dk, dv, a, b = 8, 8, 2, 5
    h0 = np.zeros((1, 1, dv, dk)); h0[0, 0, a, b] = 1.0
    q = np.zeros((1, 1, 1, dk)); q[0, 0, 0, b] = 2.0
    p = dict(q=q, k=np.ones((1, 1, 1, dk)), v=np.zeros((1, 1, 1, dv)), g=np.zeros((1, 1, 1, dk)),
             beta=np.full((1, 1, 1), -np.inf), A_log=np.array([0.0]), dt_bias=np.zeros((1, dk)),
             h0=h0)
    o, hT = fwd(p, scale=1.0)
    want = np.zeros(dv); want[a] = math.exp(-2.5) * 2.0 / math.sqrt(4.0 + 1e-6)
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-14, atol=1e-300)
    assert hT[0, 0, a, b] == pytest.approx(math.exp(-2.5), rel=1e-15)


def test_worked_example_two_by_two():
    """A hand-worked example with K = V = 2 and two tokens (scale 1, A_log 0,
    dt_bias 0, gate inputs 0 so d = exp(-2.5); beta logits 0 so beta = 1/2)."""
    c = 1.0 / math.sqrt(1.0 + 1e-6)       # |x| = 1 rows normalise to c x
    e = math.exp(-2.5)
    h0 = np.array([[1.0, 2.0], [3.0, 4.0]])
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    k = np.array([[1.0, 0.0], [0.0, 1.0]])
    v = np.array([[1.0, 1.0], [2.0, -1.0]])
    # token 1: S' = e h0; u = v1 - S' k^1 = v1 - c e h0[:,0]; S1 = S' + 1/2 u k^1^T
    u1 = v[0] - c * e * h0[:, 0]
    S1 = e * h0.copy(); S1[:, 0] += 0.5 * c * u1
    o1 = c * S1[:, 0]
    # token 2: S' = e S1; k^2 = c e_2
    Sp = e * S1
    u2 = v[1] - c * Sp[:, 1]
    S2 = Sp.copy(); S2[:, 1] += 0.5 * c * u2
    o2 = c * S2[:, 1]
    p = dict(q=q.reshape(1, 2, 1, 2), k=k.reshape(1, 2, 1, 2), v=v.reshape(1, 2, 1, 2),
             g=np.zeros((1, 2, 1, 2)), beta=np.zeros((1, 2, 1)), A_log=np.array([0.0]),
             dt_bias=np.zeros((1, 2)), h0=h0.reshape(1, 1, 2, 2))
    o, hT = fwd(p, scale=1.0)
    np.testing.assert_allclose(o[0, :, 0], np.stack([o1, o2]), rtol=1e-14)
    np.testing.assert_allclose(hT[0, 0], S2, rtol=1e-14)


@pytest.mark.parametrize("chunk", [1, 16, 32, 64])
def test_chunked_restatement_equals_sequential(chunk):
    """The WY / UT-transform chunked form equals the token-by-token form,
    including ragged (non-multiple-of-chunk) sequence tails."""
    p = rand_problem(5, [17, 64, 3, 45], 2, 4, 128, 128)
    o, hT = fwd(p)
    oc, hTc = oracle.forward_chunked(*[p[x] for x in FWD_KEYS], cu_seqlens=p["cu_seqlens"],
                                     chunk=chunk)
    assert rel(oc, o) < 1e-12 and rel(hTc, hT) < 1e-12


def test_causality():
    """Changing the last token's inputs leaves earlier outputs bit-identical."""
    p = rand_problem(6, [12], 1, 1, 16, 16)
    o1, _ = fwd(p)
    p2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in p.items()}
    for name in ["q", "k", "v", "g"]:
        p2[name][0, -1] += 1.0
    p2["beta"][0, -1] += 1.0
    o2, _ = fwd(p2)
    assert np.array_equal(o1[0, :-1], o2[0, :-1])
    assert not np.array_equal(o1[0, -1], o2[0, -1])


def test_gqa_equals_repeated_heads():
    """Value head h reads query/key head h // r: the GQA run equals an
    equal-head run on repeat-interleaved q, k; dq and dk are the group sums."""
    r = 3
    p = rand_problem(12, [6, 4], 2, 2 * r, 16, 12)
    rep = dict(p, q=np.repeat(p["q"], r, axis=2), k=np.repeat(p["k"], r, axis=2))
    o1, h1 = fwd(p)
    o2, h2 = fwd(rep)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(h1, h2, rtol=1e-13, atol=1e-15)
    g1 = bwd(p)
    g2 = bwd(rep)
    sum_r = lambda x: x.reshape(x.shape[0], x.shape[1], -1, r, x.shape[3]).sum(axis=3)
    np.testing.assert_allclose(g1[0], sum_r(g2[0]), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g1[1], sum_r(g2[1]), rtol=1e-12, atol=1e-14)
    for a, b in zip(g1[2:], g2[2:]):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_packed_equals_fixed():
    """Packed [0, T, 2T] equals fixed B = 2 (each batch row one sequence)."""
    p = rand_problem(13, [7, 7], 1, 2, 8, 8)
    fixed = {k: v for k, v in p.items() if k != "cu_seqlens"}
    for name in ["q", "k", "v", "g", "do"]:
        x = p[name]
        fixed[name] = x.reshape(2, 7, x.shape[2], x.shape[3])
    fixed["beta"] = p["beta"].reshape(2, 7, -1)
    o1, h1 = fwd(p)
    o2, h2 = oracle.forward(*[fixed[x] for x in FWD_KEYS])
    assert np.array_equal(o1.reshape(o2.shape), o2) and np.array_equal(h1, h2)
    g1 = bwd(p)
    g2 = oracle.backward(*[fixed[x] for x in FWD_KEYS], fixed["do"], fixed["dfinal_state"])
    for a, b in zip(g1, g2):
        assert np.array_equal(a.reshape(b.shape), b)


def test_output_linear_in_scale_and_state_independent_of_it():
    p = rand_problem(14, [5], 1, 1, 8, 8)
    o1, h1 = fwd(p, scale=0.5)
    o2, h2 = fwd(p, scale=1.5)
    np.testing.assert_allclose(o2, 3.0 * o1, rtol=1e-14)
    assert np.array_equal(h1, h2)


def test_l2_norm_invariance():
    """Rescaling q or k by a positive factor changes q^, k^ only through eps."""
    p = rand_problem(15, [8], 1, 2, 128, 128)
    o1, h1 = fwd(p)
    o2, h2 = fwd(dict(p, q=4.0 * p["q"], k=0.25 * p["k"]))
    assert rel(o2, o1) < 1e-6 and rel(h2, h1) < 1e-6


def test_default_scale_is_one_over_sqrt_dim():
    p = rand_problem(16, [4], 1, 1, 128, 128)
    o1, _ = fwd(p)
    o2, _ = fwd(p, scale=CONTRACT["scale"]["value"])
    np.testing.assert_allclose(o1, o2, rtol=1e-15, atol=0)


def test_head_subset_matches_full_run():
    """Computing only some query/key heads gives the same numbers for them."""
    p = rand_problem(17, [5, 3], 3, 6, 8, 8)
    full = bwd(p)
    part = bwd(p, heads=[1])
    np.testing.assert_array_equal(part[0][:, :, 1], full[0][:, :, 1])
    np.testing.assert_array_equal(part[2][:, :, 2:4], full[2][:, :, 2:4])
    np.testing.assert_array_equal(part[5][2:4], full[5][2:4])
    np.testing.assert_array_equal(part[7][:, 2:4], full[7][:, 2:4])
    assert np.all(np.isnan(part[2][:, :, 0:2]))


# ------------------------------------------------- inference gate modes
# "flashinfer.kda.recurrent_kda", parameters g ("log-space if pre-computed") and
# beta ("pre-sigmoided unless beta_is_logit"): with the gate precomputed the
# decay is exp(g) per key dimension; with beta presigmoided it is the learning
# rate itself.

def test_log_space_gate_scales_key_columns_and_ignores_gate_parameters():
    """log_space_g with g = ln(m / (m + 1)) per key dim m and presigmoided beta
    = 0 (no write): S_T = h0 diag(prod_t m/(m+1)). A_log and dt_bias are NaN,
    so reading either would poison the result."""
    T, dk, dv = 3, 6, 4
    m = np.arange(1, dk + 1, dtype=np.float64)
    rng = np.random.default_rng(40)
    p = dict(q=rng.standard_normal((1, T, 1, dk)), k=rng.standard_normal((1, T, 1, dk)),
             v=rng.standard_normal((1, T, 1, dv)),
             g=np.broadcast_to(np.log(m / (m + 1)), (1, T, 1, dk)).copy(),
             beta=np.zeros((1, T, 1)), A_log=np.array([np.nan]), dt_bias=np.full((1, dk), np.nan),
             h0=rng.standard_normal((1, 1, dv, dk)))
    o, hT = fwd(p, log_space_g=True, presigmoid_beta=True, lower_bound=np.nan)
    np.testing.assert_allclose(hT[0, 0], p["h0"][0, 0] * ((m / (m + 1)) ** T)[None, :], rtol=1e-13)
    assert np.isfinite(o).all()


def test_presigmoid_beta_first_token_closed_form():
    """First token, no decay (log-space g = 0), presigmoided beta b, q = k:
    o = scale (h0 k^ (1 - b |k^|^2) + b |k^|^2 v)."""
    dk, dv, b = 8, 5, 0.3
    rng = np.random.default_rng(41)
    k = rng.standard_normal((1, 1, 1, dk))
    khat = k[0, 0, 0] / math.sqrt(float(np.sum(k * k)) + 1e-6)
    kk = float(khat @ khat)
    p = dict(q=k.copy(), k=k, v=rng.standard_normal((1, 1, 1, dv)), g=np.zeros((1, 1, 1, dk)),
             beta=np.full((1, 1, 1), b), A_log=np.array([0.0]), dt_bias=np.zeros((1, dk)),
             h0=rng.standard_normal((1, 1, dv, dk)))
    o, _ = fwd(p, scale=1.0, log_space_g=True, presigmoid_beta=True)
    want = p["h0"][0, 0] @ khat * (1 - b * kk) + b * kk * p["v"][0, 0, 0]
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-13)
    # beta = 1 presigmoided overwrites the memory at the key: o = scale v |k^|^2 + h0 k^ (1 - |k^|^2)
    p["beta"][:] = 1.0
    o1, _ = fwd(p, scale=1.0, log_space_g=True, presigmoid_beta=True)
    np.testing.assert_allclose(o1[0, 0, 0], p["v"][0, 0, 0], rtol=0, atol=1e-6 * np.abs(p["v"]).max()
                               + 1e-6 * np.abs(p["h0"]).max())


def test_gate_modes_agree_with_in_kernel_gate_on_transformed_inputs():
    """Feeding the precomputed log decay lb sigmoid(exp(A_log)(g + dt_bias))
    and the presigmoided beta to the modes reproduces the default forward, one
    mode at a time and both together (packed, GQA)."""
    p = rand_problem(42, [7, 12, 3], 2, 4, 16, 12)
    o_ref, s_ref = fwd(p)
    lb = -5.0
    z = np.exp(p["A_log"])[None, None, :, None] * (p["g"] + p["dt_bias"][None, None])
    g_log = lb / (1.0 + np.exp(-z))
    b_sig = 1.0 / (1.0 + np.exp(-p["beta"]))
    for lg, pb in [(True, False), (False, True), (True, True)]:
        x = dict(p)
        if lg:
            x["g"] = g_log
        if pb:
            x["beta"] = b_sig
        o, s = fwd(x, log_space_g=lg, presigmoid_beta=pb)
        assert rel(o, o_ref) < 1e-13 and rel(s, s_ref) < 1e-13, (lg, pb)
