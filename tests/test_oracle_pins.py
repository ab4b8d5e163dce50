"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes the oracle to something independent of its own code: finite
differences of its forward, closed forms written from the recurrence's
definition (flashinfer "kda_backward" page, supported contract), exact
reductions to plain linear attention and to the ungated delta rule, the
split/carry property of a recurrence, Euler's identity for a function
homogeneous of degree one, invariances of the L2 norm, the per-key decay
orientation (the kda-neuron-kernels log, fix T-KDA-02), and a second,
independently derived formulation (the chunk-wise WY/UT form).
"""
import numpy as np
import pytest

import oracle
import chunk_model
from kimi_delta_attention_15_gb300 import inputs as I

SCALE = 1.0 / np.sqrt(128.0)
K = V = 128


def _rand_inputs(lengths, H, seed, h0=True, dhT=True, g_std=1.0, dtype=np.float64):
    """fp64 random inputs (not bf16-rounded) for derivative checks."""
    rng = np.random.default_rng(seed)
    T, N = sum(lengths), len(lengths)
    inp = dict(
        q=rng.standard_normal((T, H, K)), k=rng.standard_normal((T, H, K)),
        v=rng.standard_normal((T, H, V)), g_raw=rng.standard_normal((T, H, K)) * g_std,
        beta_raw=rng.standard_normal((T, H)), A_log=np.log(rng.uniform(1, 16, H)),
        dt_bias=0.1 * rng.standard_normal((H, K)),
        h0=0.1 * rng.standard_normal((N, H, V, K)) if h0 else None,
        do=rng.standard_normal((T, H, V)),
        dhT=0.1 * rng.standard_normal((N, H, V, K)) if dhT else None,
        cu_seqlens=np.cumsum([0] + list(lengths)).astype(np.int64),
    )
    return inp


def _loss(inp, mode="raw"):
    f = oracle.forward(inp, mode=mode)
    L = float((f["o"] * inp["do"]).sum())
    if inp.get("dhT") is not None:
        L += float((f["hT"] * inp["dhT"]).sum())
    return L


GRAD_OF = dict(q="dq", k="dk", v="dv", g_raw="dg_raw", beta_raw="dbeta_raw",
               A_log="dA_log", dt_bias="ddt_bias", h0="dh0")


@pytest.mark.parametrize("lengths,H", [((4,), 1), ((2, 3), 2)])
def test_backward_matches_central_differences(lengths, H):
    """Every gradient against central differences of the forward (h = 1e-6):
    one random direction over the whole tensor, plus single elements."""
    inp = _rand_inputs(lengths, H, seed=11)
    g = oracle.backward(inp)
    rng = np.random.default_rng(3)
    h = 1e-6
    for name, gname in GRAD_OF.items():
        x0 = inp[name]
        d = rng.standard_normal(x0.shape)
        plus = dict(inp); plus[name] = x0 + h * d
        minus = dict(inp); minus[name] = x0 - h * d
        fd = (_loss(plus) - _loss(minus)) / (2 * h)
        an = float((g[gname] * d).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)
        for _ in range(3):
            idx = tuple(int(rng.integers(0, s)) for s in x0.shape)
            e = np.zeros_like(x0); e[idx] = 1.0
            plus[name] = x0 + h * e
            minus[name] = x0 - h * e
            fd = (_loss(plus) - _loss(minus)) / (2 * h)
            an = float(g[gname][idx])
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, idx, fd, an)


def test_core_backward_matches_central_differences():
    """The same in core mode: gradients w.r.t. q^, k^, v, the log-decay g,
    beta and h0, with negative log-decays and beta in (0, 1)."""
    rng = np.random.default_rng(5)
    inp = _rand_inputs((5,), 1, seed=12)
    inp["g_raw"] = -rng.uniform(0, 3, inp["g_raw"].shape)
    inp["beta_raw"] = rng.uniform(0.05, 0.95, inp["beta_raw"].shape)
    inp["q"] = inp["q"] / np.linalg.norm(inp["q"], axis=-1, keepdims=True)
    inp["k"] = inp["k"] / np.linalg.norm(inp["k"], axis=-1, keepdims=True)
    g = oracle.backward(inp, mode="core")
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g_raw", "dg_raw"),
                        ("beta_raw", "dbeta_raw"), ("h0", "dh0")):
        d = rng.standard_normal(inp[name].shape)
        plus = dict(inp); plus[name] = inp[name] + h * d
        minus = dict(inp); minus[name] = inp[name] - h * d
        fd = (_loss(plus, "core") - _loss(minus, "core")) / (2 * h)
        an = float((g[gname] * d).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def _sig(x):
    return 1.0 / (1.0 + np.exp(-x))


def test_single_token_closed_form():
    """T = 1 from the definition: S1 = h0 diag(a) + b (v - h0 diag(a) k^) k^T,
    o = scale S1 q^, with a = exp(lb sigmoid(exp(A_log)(g_raw + dt_bias)))
    per key channel, b = sigmoid(beta_raw), x^ = x / sqrt(|x|^2 + 1e-6).
    A small-norm q makes the epsilon matter."""
    inp = _rand_inputs((1,), 3, seed=21, dhT=False)
    inp["q"][0, 1] *= 1e-3
    f = oracle.forward(inp)
    for h in range(3):
        q, k, v = inp["q"][0, h], inp["k"][0, h], inp["v"][0, h]
        qh = q / np.sqrt(q @ q + 1e-6)
        kh = k / np.sqrt(k @ k + 1e-6)
        a = np.exp(-5.0 * _sig(np.exp(inp["A_log"][h]) * (inp["g_raw"][0, h] + inp["dt_bias"][h])))
        b = _sig(inp["beta_raw"][0, h])
        H0 = inp["h0"][0, h]
        Sd = H0 * a[None, :]
        S1 = Sd + b * np.outer(v - Sd @ kh, kh)
        np.testing.assert_allclose(f["hT"][0, h], S1, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(f["o"][0, h], SCALE * S1 @ qh, rtol=1e-12, atol=1e-15)


def test_single_token_zero_state_gradients():
    """T = 1, h0 = 0: o = scale b (k^.q^) v, so dv = scale b (k^.q^) dO + b dhT k^
    and dbeta = scale (k^.q^)(v.dO) + (v - 0)^T dhT k^ (core mode, exact)."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal(K); q /= np.linalg.norm(q)
    k = rng.standard_normal(K); k /= np.linalg.norm(k)
    v, dO = rng.standard_normal(V), rng.standard_normal(V)
    dhT = rng.standard_normal((V, K))
    b = 0.37
    inp = dict(q=q[None, None], k=k[None, None], v=v[None, None],
               g_raw=-rng.uniform(0, 2, (1, 1, K)), beta_raw=np.array([[b]]), h0=None,
               do=dO[None, None], dhT=dhT[None, None], cu_seqlens=np.array([0, 1]))
    f = oracle.forward(inp, mode="core")
    g = oracle.backward(inp, mode="core")
    np.testing.assert_allclose(f["o"][0, 0], SCALE * b * (k @ q) * v, rtol=1e-13)
    np.testing.assert_allclose(g["dv"][0, 0], SCALE * b * (k @ q) * dO + b * dhT @ k, rtol=1e-12)
    np.testing.assert_allclose(g["dbeta_raw"][0, 0], SCALE * (k @ q) * (v @ dO) + v @ dhT @ k,
                               rtol=1e-12)
    # with zero state the decay has no effect: dg = 0 exactly
    assert np.all(g["dg_raw"] == 0.0)


def test_reduces_to_linear_attention():
    """g = 0, h0 = 0 and mutually orthonormal keys remove the erase term, so
    o_t = scale sum_{j<=t} beta_j v_j (k^_j . q^_t): causal linear attention."""
    rng = np.random.default_rng(9)
    T = 40
    perm = rng.permutation(K)[:T]
    kk = np.eye(K)[perm]                           # orthonormal keys
    q = rng.standard_normal((T, K))
    v = rng.standard_normal((T, V))
    beta = rng.uniform(0.1, 1.0, T)
    inp = dict(q=q[:, None], k=kk[:, None], v=v[:, None], g_raw=np.zeros((T, 1, K)),
               beta_raw=beta[:, None], h0=None, cu_seqlens=np.array([0, T]))
    o = oracle.forward(inp, mode="core")["o"][:, 0]
    att = np.tril(q @ kk.T) * beta[None, :]        # [t, j]
    np.testing.assert_allclose(o, SCALE * att @ v, rtol=1e-12, atol=1e-14)


def test_beta_zero_is_pure_decay():
    """beta = 0 leaves only the decay: S_t = h0 diag(exp(G_t)), G_t = sum_{j<=t} g_j,
    so o_t = scale h0 (exp(G_t) * q^_t), decaying KEY columns of h0."""
    rng = np.random.default_rng(10)
    T = 7
    g = -rng.uniform(0, 1, (T, 1, K))
    h0 = rng.standard_normal((1, 1, V, K))
    q = rng.standard_normal((T, 1, K))
    inp = dict(q=q, k=rng.standard_normal((T, 1, K)), v=rng.standard_normal((T, 1, V)),
               g_raw=g, beta_raw=np.zeros((T, 1)), h0=h0, cu_seqlens=np.array([0, T]))
    f = oracle.forward(inp, mode="core")
    G = np.cumsum(g[:, 0], axis=0)
    for t in range(T):
        np.testing.assert_allclose(f["o"][t, 0], SCALE * h0[0, 0] @ (np.exp(G[t]) * q[t, 0]),
                                   rtol=1e-12)
    np.testing.assert_allclose(f["hT"][0, 0], h0[0, 0] * np.exp(G[-1])[None, :], rtol=1e-12)


def test_decay_acts_on_key_channels():
    """One token, beta = 0, a gate that differs across key channels: the state
    must be scaled per column (key channel), not per row (value channel)."""
    rng = np.random.default_rng(12)
    g = -np.linspace(0.0, 4.0, K)[None, None, :]
    h0 = rng.standard_normal((1, 1, V, K))
    inp = dict(q=np.ones((1, 1, K)), k=np.ones((1, 1, K)), v=np.ones((1, 1, V)), g_raw=g,
               beta_raw=np.zeros((1, 1)), h0=h0, cu_seqlens=np.array([0, 1]))
    hT = oracle.forward(inp, mode="core")["hT"][0, 0]
    np.testing.assert_allclose(hT, h0[0, 0] * np.exp(g[0, 0])[None, :], rtol=1e-14)
    assert not np.allclose(hT, h0[0, 0] * np.exp(g[0, 0])[:, None])


def test_delta_rule_exact_association():
    """Ungated delta rule (g = 0) with beta = 1 and unit keys writes v_t exactly:
    S_t k^_t = v_t, so querying with q^_t = k^_t returns scale v_t. With a gate
    S_t k^_t = (1 - beta) S' k^_t + beta v_t for any beta (|k^| = 1)."""
    rng = np.random.default_rng(13)
    T = 9
    k = rng.standard_normal((T, 1, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, 1, V))
    inp = dict(q=k.copy(), k=k, v=v, g_raw=np.zeros((T, 1, K)), beta_raw=np.ones((T, 1)),
               h0=rng.standard_normal((1, 1, V, K)), cu_seqlens=np.array([0, T]))
    o = oracle.forward(inp, mode="core")["o"]
    np.testing.assert_allclose(o, SCALE * v, rtol=1e-11, atol=1e-12)
    # general beta and gate, one step from a known state
    g = -rng.uniform(0, 2, (1, 1, K)); b = 0.3
    S0 = rng.standard_normal((1, 1, V, K))
    one = dict(q=k[:1], k=k[:1], v=v[:1], g_raw=g, beta_raw=np.array([[b]]), h0=S0,
               cu_seqlens=np.array([0, 1]))
    S1 = oracle.forward(one, mode="core")["hT"][0, 0]
    Sp = S0[0, 0] * np.exp(g[0, 0])[None, :]
    np.testing.assert_allclose(S1 @ k[0, 0], (1 - b) * Sp @ k[0, 0] + b * v[0, 0], rtol=1e-12)


def test_split_and_carry():
    """Running [0, t) then [t, L) from the carried state equals the whole run,
    forward and backward (dh0 of the second part is dhT of the first)."""
    L = 37
    inp = _rand_inputs((L,), 2, seed=30)
    whole_f = oracle.forward(inp)
    whole_b = oracle.backward(inp)
    for t in (1, 16, 30):
        a = {k: (v[:t] if k in ("q", "k", "v", "g_raw", "beta_raw", "do") else v) for k, v in inp.items()}
        b = {k: (v[t:] if k in ("q", "k", "v", "g_raw", "beta_raw", "do") else v) for k, v in inp.items()}
        a["cu_seqlens"] = np.array([0, t]); b["cu_seqlens"] = np.array([0, L - t])
        fa = oracle.forward(a)
        b["h0"] = fa["hT"]
        fb = oracle.forward(b)
        np.testing.assert_allclose(np.concatenate([fa["o"], fb["o"]]), whole_f["o"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(fb["hT"], whole_f["hT"], rtol=1e-12, atol=1e-14)
        gb = oracle.backward(b)
        a["dhT"] = gb["dh0"]
        ga = oracle.backward(a)
        for key in ("dq", "dk", "dv", "dg_raw", "dbeta_raw"):
            np.testing.assert_allclose(np.concatenate([ga[key], gb[key]]), whole_b[key],
                                       rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(ga["dh0"], whole_b["dh0"], rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(ga["ddt_bias"] + gb["ddt_bias"], whole_b["ddt_bias"],
                                   rtol=1e-10, atol=1e-13)


def test_packed_equals_separate_runs_with_empty_sequence():
    """Packed varlen equals separate runs; an empty sequence gives hT = h0 and dh0 = dhT."""
    lengths = (5, 0, 9)
    inp = _rand_inputs(lengths, 2, seed=31)
    f = oracle.forward(inp)
    g = oracle.backward(inp)
    cu = inp["cu_seqlens"]
    tok = ("q", "k", "v", "g_raw", "beta_raw", "do")
    dA, ddt = 0.0, 0.0
    for n in range(3):
        s = {k: (v[cu[n]:cu[n + 1]] if k in tok else v) for k, v in inp.items()}
        s["cu_seqlens"] = np.array([0, lengths[n]])
        s["h0"] = inp["h0"][n:n + 1]; s["dhT"] = inp["dhT"][n:n + 1]
        fs, gs = oracle.forward(s), oracle.backward(s)
        np.testing.assert_array_equal(fs["hT"][0], f["hT"][n])
        np.testing.assert_array_equal(fs["o"], f["o"][cu[n]:cu[n + 1]])
        np.testing.assert_array_equal(gs["dh0"][0], g["dh0"][n])
        np.testing.assert_array_equal(gs["dq"], g["dq"][cu[n]:cu[n + 1]])
        dA = dA + gs["dA_log"]; ddt = ddt + gs["ddt_bias"]
    np.testing.assert_array_equal(f["hT"][1], inp["h0"][1])
    np.testing.assert_array_equal(g["dh0"][1], inp["dhT"][1])
    np.testing.assert_allclose(g["dA_log"], dA, rtol=1e-13)
    np.testing.assert_allclose(g["ddt_bias"], ddt, rtol=1e-13)


def test_euler_identity_in_v_and_h0():
    """(o, hT) are jointly linear in (v, h0), so sum<v, dv> + <h0, dh0> = L."""
    inp = _rand_inputs((23, 41), 2, seed=32)
    g = oracle.backward(inp)
    lhs = float((inp["v"] * g["dv"]).sum() + (inp["h0"] * g["dh0"]).sum())
    assert abs(lhs - _loss(inp)) <= 1e-10 * abs(_loss(inp))


def test_parameter_gradient_identities():
    """ddt_bias[h,c] = sum_t dg_raw[t,h,c];
    dA_log[h] = sum_{t,c} dg_raw[t,h,c] (g_raw + dt_bias)[t,h,c]  (the gate's chain rule)."""
    inp = _rand_inputs((13, 20), 3, seed=33)
    g = oracle.backward(inp)
    np.testing.assert_allclose(g["ddt_bias"], g["dg_raw"].sum(0), rtol=1e-12, atol=1e-15)
    dA = (g["dg_raw"] * (inp["g_raw"] + inp["dt_bias"][None])).sum((0, 2))
    np.testing.assert_allclose(g["dA_log"], dA, rtol=1e-12, atol=1e-15)


def test_l2_norm_invariances():
    """Scaling raw q or k by c > 0 leaves o unchanged (up to the epsilon), and the
    norm's Jacobian annihilates the input direction: <q, dq> ~ 0, <k, dk> ~ 0."""
    inp = _rand_inputs((11,), 2, seed=34)
    f = oracle.forward(inp)
    s = dict(inp); s["q"] = inp["q"] * 3.0; s["k"] = inp["k"] * 0.5
    np.testing.assert_allclose(oracle.forward(s)["o"], f["o"], rtol=1e-5, atol=1e-8)
    g = oracle.backward(inp)
    for x, dx in (("q", "dq"), ("k", "dk")):
        dots = (inp[x] * g[dx]).sum(-1)
        scale = np.abs(inp[x]).sum(-1) * np.abs(g[dx]).sum(-1)
        assert np.all(np.abs(dots) <= 1e-6 * scale + 1e-300)


@pytest.mark.parametrize("C", [4, 16, 32, 64])
def test_chunk_form_equals_recurrence(C):
    """The independently derived chunk-wise WY/UT form (forward and its hand-derived
    adjoints) equals the token recurrence to rounding, with ragged lengths, at every
    chunk size (32 and 64 are the two a chunked implementation is allowed to use): the
    chunk size blocks the computation and does not change the function."""
    w = I.custom([5, 17, 0, 70], 2, h0=True, dhT=True)
    inp = I.make_inputs(w, seed=1)
    fo, bo = oracle.forward(inp), oracle.backward(inp)
    fc, bc = chunk_model.forward(inp, C), chunk_model.backward(inp, C)
    for key in ("o", "hT"):
        np.testing.assert_allclose(fc[key], fo[key], rtol=0, atol=1e-12 * np.abs(fo[key]).max())
    for key in ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias"):
        np.testing.assert_allclose(bc[key], bo[key], rtol=0, atol=1e-12 * np.abs(bo[key]).max())


def test_strong_decay_chunk_is_finite():
    """Large gate pre-activations (G down to -320 over a chunk at lb = -5) stay
    finite in the oracle and agree with the chunk form."""
    w = I.custom([130], 2, g_std=4.0)
    inp = I.make_inputs(w, seed=2)
    inp["A_log"] = np.log(np.full(2, 16.0))
    fo, bo = oracle.forward(inp), oracle.backward(inp)
    for v in list(fo.values()) + list(bo.values()):
        assert np.all(np.isfinite(v))
    fc = chunk_model.forward(inp, 64)
    np.testing.assert_allclose(fc["o"], fo["o"], rtol=0, atol=1e-11 * np.abs(fo["o"]).max())


def _grouped_inputs(lengths, Hk, G, seed):
    """fp64 inputs with G value heads per query/key head (q, k: Hk heads; the rest Hk G)."""
    inp = _rand_inputs(lengths, Hk * G, seed)
    rng = np.random.default_rng(seed + 100)
    T = sum(lengths)
    inp["q"] = rng.standard_normal((T, Hk, K))
    inp["k"] = rng.standard_normal((T, Hk, K))
    return inp


def test_grouped_heads_central_differences():
    """Grouped value heads: the gradients of the shared q, k (summed over each group) and of
    the per-value-head tensors against central differences of the forward."""
    inp = _grouped_inputs((3, 2), Hk=2, G=2, seed=21)
    g = oracle.backward(inp)
    assert g["dq"].shape == inp["q"].shape and g["dv"].shape == inp["v"].shape
    rng = np.random.default_rng(7)
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g_raw", "dg_raw"), ("A_log", "dA_log")):
        x0 = inp[name]
        d = rng.standard_normal(x0.shape)
        plus = dict(inp); plus[name] = x0 + h * d
        minus = dict(inp); minus[name] = x0 - h * d
        fd = (_loss(plus) - _loss(minus)) / (2 * h)
        an = float((g[gname] * d).sum())
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (name, fd, an)


def test_grouped_heads_equal_repeated_query_key_heads():
    """Value head h reading query/key head h // G is the plain layout with q, k repeated G
    times along the head axis (numpy), and dq, dk are the group sums of that run's."""
    Hk, G = 2, 3
    inp = _grouped_inputs((5, 3), Hk=Hk, G=G, seed=22)
    rep = dict(inp)
    rep["q"] = np.repeat(inp["q"], G, axis=1)
    rep["k"] = np.repeat(inp["k"], G, axis=1)
    fg, fr = oracle.forward(inp), oracle.forward(rep)
    assert np.array_equal(fg["o"], fr["o"]) and np.array_equal(fg["hT"], fr["hT"])
    bg, br = oracle.backward(inp), oracle.backward(rep)
    for key in ("dv", "dg_raw", "dbeta_raw", "dA_log", "ddt_bias", "dh0"):
        assert np.array_equal(bg[key], br[key]), key
    T = inp["q"].shape[0]
    for key in ("dq", "dk"):
        summed = br[key].reshape(T, Hk, G, K).sum(axis=2)
        np.testing.assert_allclose(bg[key], summed, rtol=1e-13, atol=1e-13)


def test_grouped_heads_identical_members_scale_the_shared_gradient():
    """A group of G identical value heads (same v, gates, beta, parameters, states and
    adjoints) gives G copies of the single-head outputs and G times its dq, dk."""
    G = 4
    one = _rand_inputs((6,), 1, seed=23)
    grp = dict(one)
    for name in ("v", "g_raw", "beta_raw", "do"):
        grp[name] = np.repeat(one[name], G, axis=1)
    for name in ("A_log", "dt_bias", "h0", "dhT"):
        grp[name] = np.repeat(one[name], G, axis=0 if name in ("A_log", "dt_bias") else 1)
    f1, fg = oracle.forward(one), oracle.forward(grp)
    for j in range(G):
        assert np.array_equal(fg["o"][:, j], f1["o"][:, 0])
    b1, bg = oracle.backward(one), oracle.backward(grp)
    np.testing.assert_allclose(bg["dq"], G * b1["dq"], rtol=1e-14, atol=0)
    np.testing.assert_allclose(bg["dk"], G * b1["dk"], rtol=1e-14, atol=0)
    for j in range(G):
        assert np.array_equal(bg["dv"][:, j], b1["dv"][:, 0])
        assert bg["dA_log"][j] == b1["dA_log"][0]
