"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test pins the oracle to something other than itself: values printed in
a worked example on the pages (fixtures under tests/golden/, each with its
citation), closed forms, special cases that reduce to a library routine,
invariants that follow from the definition, and agreement between two
independently written formulations (recurrent vs masked-parallel vs block).
"""
import math

import numpy as np
import pytest

import oracle

ID = oracle.FMAP_IDENTITY


def arr(x):
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# feature map: elu(x) + 1 with alpha = 1


def test_phi_closed_form_and_library_exp():
    # x > 0: phi(x) = x + 1 (the page's worked example uses exactly this).
    for x in [1e-12, 0.25, 1.0, 2.0, 37.5]:
        assert oracle.phi_scalar(x) == x + 1.0
    # x <= 0: elu(x) + 1 = (exp(x) - 1) + 1 = exp(x); compare with libm.
    for x in [0.0, -1e-9, -0.5, -1.0, -7.25, -700.0]:
        assert oracle.phi_scalar(x) == pytest.approx(math.exp(x), rel=1e-15)
    assert oracle.phi_scalar(0.0) == 1.0
    # continuous at 0 and strictly positive
    assert abs(oracle.phi_scalar(1e-9) - oracle.phi_scalar(-1e-9)) < 3e-9
    xs = np.linspace(-30, 30, 1001)
    assert np.all(oracle.phi(xs) > 0)
    # elementwise version agrees with the scalar one
    ys = oracle.phi(xs)
    assert all(ys[i] == oracle.phi_scalar(xs[i]) for i in range(0, 1001, 50))


def test_phi_matches_elu_definition_via_expm1():
    # elu(x) = expm1(x) for x <= 0 (library routine); phi = elu + 1
    xs = np.linspace(-5, 0, 101)
    np.testing.assert_allclose(oracle.phi(xs), np.expm1(xs) + 1.0, rtol=1e-14)


# --------------------------------------------------------------------------
# worked example of kernel linear attention (non-causal)


def test_worked_example_state_printed(golden):
    g = golden("kernel_la_worked_example.json")
    S, z = oracle.noncausal_state(arr(g["K"]), arr(g["V"]))
    np.testing.assert_array_equal(S, arr(g["phiK_T_V"]))
    # phi(q_1) as printed
    np.testing.assert_array_equal(oracle.phi(arr(g["Q"])[0]), arr(g["phi_q1"]))
    # numerator as printed: phi(q_1)^T [phi(K)^T V]
    num = oracle.state_read(S, z, arr(g["Q"])[:1], normalise=False)
    np.testing.assert_array_equal(num[0], arr(g["num_1"]))
    # denominator as printed: phi(q_1)^T [phi(K)^T 1]
    assert float(oracle.phi(arr(g["Q"])[0]) @ z) == g["denom_1"]


def test_worked_example_output_row1_printed(golden):
    g = golden("kernel_la_worked_example.json")
    y = oracle.noncausal(arr(g["Q"]), arr(g["K"]), arr(g["V"]))
    exact = arr(g["num_1"]) / g["denom_1"]
    np.testing.assert_allclose(y[0], exact, rtol=1e-15)
    np.testing.assert_array_equal(np.round(y[0], 2), arr(g["output_1_2dp"]))


def test_worked_example_causal_special_rows(golden):
    g = golden("kernel_la_worked_example.json")
    Q, K, V = arr(g["Q"]), arr(g["K"]), arr(g["V"])
    yc = oracle.causal(Q, K, V)
    yn = oracle.noncausal(Q, K, V)
    # a single visible key has weight exactly 1: y_1 = v_1
    np.testing.assert_allclose(yc[0], V[0], rtol=0, atol=1e-15)
    # the last causal row sees every key: equals the non-causal last row
    np.testing.assert_allclose(yc[-1], yn[-1], rtol=1e-15)
    # and the non-causal form is not the causal one elsewhere
    assert not np.allclose(yc[1], yn[1])


# --------------------------------------------------------------------------
# RetNet worked example: decayed recurrence and decayed masked-parallel form


def test_retnet_recurrent_states_printed(golden):
    g = golden("retnet_worked_example.json")
    Q, K, V = arr(g["Q"]), arr(g["K"]), arr(g["V"])
    S = np.zeros((4, 4))
    z = np.zeros(4)
    outs = []
    for t in range(4):
        outs.append(oracle.recurrent_step(S, z, Q[t], K[t], V[t], g["gamma"],
                                          fmap=ID, normalise=False))
        if t < 3:
            np.testing.assert_array_equal(S, arr(g[f"S_{t + 1}"]))
    # update first, then read: Output_3 = q_3 S_3
    np.testing.assert_array_equal(outs[2], arr(g["output_3"]))
    np.testing.assert_array_equal(np.stack(outs), arr(g["output_parallel"]))


def test_retnet_parallel_form_printed(golden):
    g = golden("retnet_worked_example.json")
    Q, K, V = arr(g["Q"]), arr(g["K"]), arr(g["V"])
    # the printed D and QK^T multiply to the printed A_ret (fixture sanity)
    np.testing.assert_array_equal(arr(g["QK_T"]) * arr(g["D"]), arr(g["A_ret"]))
    y, W = oracle.quadratic(Q, K, V, [g["gamma"]], fmap=ID, normalise=False,
                            return_weights=True)
    np.testing.assert_array_equal(W, arr(g["A_ret"]))
    np.testing.assert_array_equal(y, arr(g["output_parallel"]))
    # the causal routine, same mode, gives the same (exact in binary)
    yc = oracle.causal(Q, K, V, [g["gamma"]], fmap=ID, normalise=False)
    np.testing.assert_array_equal(yc, arr(g["output_parallel"]))


# --------------------------------------------------------------------------
# Infini-attention worked example: read of a given state


def test_infini_state_read_printed(golden):
    g = golden("infini_read_worked_example.json")
    M, z, Q = arr(g["M_prev"]), arr(g["z_prev"]), arr(g["Q"])
    np.testing.assert_array_equal(oracle.phi(Q), arr(g["sigma_Q"]))
    num = oracle.state_read(M, z, Q, normalise=False)
    np.testing.assert_array_equal(num, arr(g["numerator"]))
    y = oracle.state_read(M, z, Q)
    np.testing.assert_allclose(
        y, arr(g["numerator"]) / arr(g["denominator"])[:, None], rtol=1e-15)
    np.testing.assert_array_equal(np.round(y, 3), arr(g["A_global_3dp"]))


# --------------------------------------------------------------------------
# independent formulations agree; special cases; invariants


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * scale


@pytest.mark.parametrize("decay", [None, [0.9, 0.5, 1.0]])
def test_recurrent_equals_masked_parallel(decay):
    q, k, v = (_rand((2, 3, 13, 5), s) for s in (1, 2, 3))
    yc = oracle.causal(q, k, v, decay)
    yq = oracle.quadratic(q, k, v, decay)
    np.testing.assert_allclose(yc, yq, rtol=1e-12, atol=1e-12)


def test_masked_parallel_weights_nonnegative_and_causal():
    q, k, v = (_rand((1, 2, 17, 6), s, 2.0) for s in (4, 5, 6))
    _, W = oracle.quadratic(q, k, v, [0.8, 1.0], return_weights=True)
    assert np.all(W >= 0)
    iu = np.triu_indices(17, 1)
    assert np.all(W[..., iu[0], iu[1]] == 0)
    assert np.all(np.diagonal(W, axis1=-2, axis2=-1) > 0)


@pytest.mark.parametrize("decay", [None, [0.96875, 0.5]])
def test_decode_steps_equal_causal(decay):
    B, H, N, d = 2, 2, 9, 7
    q, k, v = (_rand((B, H, N, d), s) for s in (7, 8, 9))
    yc = oracle.causal(q, k, v, decay)
    S = np.zeros((B, H, d, d))
    z = np.zeros((B, H, d))
    g = None if decay is None else np.tile(np.asarray(decay), B)
    for t in range(N):
        y = oracle.decode_step(S, z, q[:, :, t], k[:, :, t], v[:, :, t], g)
        np.testing.assert_allclose(y, yc[:, :, t], rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# delta rule (DeltaNet / Gated DeltaNet decode step)


def test_delta_rule_worked_example_printed(golden):
    g = golden("deltanet_worked_example.json")
    # the library's layout is the page's S transposed
    S = np.ascontiguousarray(arr(g["S_prev"]).T)
    k, v = arr(g["k"]), arr(g["v"])
    assert np.array_equal(S.T @ k, arr(g["prediction"]))
    out = oracle.delta_step(S, k, k, v, [g["beta"]])
    np.testing.assert_array_equal(S, arr(g["S_next"]).T)
    # querying with the same key returns exactly v_t (the printed S_t k_t)
    np.testing.assert_array_equal(out, arr(g["S_next_k"]))


def test_delta_rule_properties():
    rng = np.random.default_rng(60)
    d = 6
    S0 = rng.standard_normal((d, d))
    k = rng.standard_normal(d)
    k /= np.linalg.norm(k)
    v, q = rng.standard_normal(d), rng.standard_normal(d)
    # beta = 1 with a unit key stores v exactly: S^T k = v afterwards
    S = S0.copy()
    oracle.delta_step(S, q, k, v, [1.0])
    np.testing.assert_allclose(S.T @ k, v, rtol=1e-12, atol=1e-12)
    # directions orthogonal to k are untouched (without a gate)
    x = rng.standard_normal(d)
    x -= (x @ k) * k
    np.testing.assert_allclose(S.T @ x, S0.T @ x, rtol=1e-12, atol=1e-12)
    # beta = 0 leaves the state alone; the output reads it
    S = S0.copy()
    o = oracle.delta_step(S, q, k, v, [0.0])
    np.testing.assert_array_equal(S, S0)
    np.testing.assert_allclose(o, S0.T @ q, rtol=1e-13)
    # alpha = 0 forgets everything: S = beta k v^T
    S = S0.copy()
    oracle.delta_step(S, q, k, v, [0.5], alpha=[0.0])
    np.testing.assert_allclose(S, 0.5 * np.outer(k, v), rtol=1e-14, atol=1e-14)


def test_gated_delta_rule_closed_form():
    # S_t = alpha S + beta (v - alpha S k) k^T in the page's orientation,
    # written with numpy on the transposed state
    rng = np.random.default_rng(61)
    d = 5
    S0 = rng.standard_normal((d, d))
    k, v, q = (rng.standard_normal(d) for _ in range(3))
    a, b = 0.8, 0.3
    P = S0.T                      # page's orientation
    P1 = a * P + b * np.outer(v - a * P @ k, k)
    S = S0.copy()
    o = oracle.delta_step(S, q, k, v, [b], alpha=[a])
    np.testing.assert_allclose(S, P1.T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(o, P1 @ q, rtol=1e-13, atol=1e-13)


def test_delta_forward_worked_example_as_a_sequence(golden):
    # the page's single write, as a one-token sequence from the printed state
    g = golden("deltanet_worked_example.json")
    k, v = arr(g["k"])[None], arr(g["v"])[None]
    out, S = oracle.delta_forward(k, k, v, [g["beta"]], S0=arr(g["S_prev"]).T)
    np.testing.assert_array_equal(S, arr(g["S_next"]).T)
    np.testing.assert_array_equal(out[0], arr(g["S_next_k"]))


def test_delta_forward_stores_orthonormal_keys():
    # beta = 1, orthonormal keys: each write stores its value without
    # disturbing the others, so reading with the first key returns its value
    # at every step (update, then read), and every key reads back its value
    # at the end
    rng = np.random.default_rng(62)
    d = 6
    K, _ = np.linalg.qr(rng.standard_normal((d, d)))
    V = rng.standard_normal((d, d))
    q = np.repeat(K[:1], d, axis=0)
    out, S = oracle.delta_forward(q, K, V, np.ones(d))
    np.testing.assert_allclose(out, np.repeat(V[:1], d, axis=0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(K @ S, V, rtol=1e-12, atol=1e-12)
    # writing key 0 again with beta = 1 replaces its value
    w = rng.standard_normal(d)
    out2, S2 = oracle.delta_forward(K[:1], K[:1], w[None], [1.0], S0=S)
    np.testing.assert_allclose(out2[0], w, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(K[1:] @ S2, V[1:], rtol=1e-12, atol=1e-12)


def test_delta_forward_gate_zero_restarts_and_beta_zero_keeps():
    rng = np.random.default_rng(63)
    N, d = 9, 5
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    beta = rng.uniform(0.1, 1.0, N)
    alpha = rng.uniform(0.5, 1.0, N)
    alpha[4] = 0.0
    out, S = oracle.delta_forward(q, k, v, beta, alpha)
    # from a zero gate on, the earlier tokens are forgotten
    out_tail, S_tail = oracle.delta_forward(q[4:], k[4:], v[4:], beta[4:], alpha[4:])
    np.testing.assert_allclose(out[4:], out_tail, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, S_tail, rtol=1e-13, atol=1e-13)
    # beta = 0 (no gate) never writes: the start state is read as it is
    S0 = rng.standard_normal((d, d))
    out0, S1 = oracle.delta_forward(q, k, v, np.zeros(N), S0=S0)
    np.testing.assert_array_equal(S1, S0)
    np.testing.assert_allclose(out0, q @ S0, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# data-dependent scalar gate per token (GLA-style; Gated DeltaNet's alpha_t)


def _gates(shape, seed, lo=0.5):
    return np.random.default_rng(seed).uniform(lo, 1.0, shape)


def test_gated_constant_gates_are_the_per_head_decay():
    q, k, v = (_rand((2, 3, 12, 5), s) for s in (40, 41, 42))
    dec = [0.9, 0.5, 1.0]
    alpha = np.broadcast_to(np.asarray(dec)[None, :, None], (2, 3, 12))
    np.testing.assert_allclose(oracle.causal_gated(q, k, v, alpha),
                               oracle.causal(q, k, v, dec), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("fmap, norm", [(oracle.FMAP_ELU1, True), (ID, False)])
def test_gated_equals_masked_parallel_with_gate_products(fmap, norm):
    # y_i = sum_{j<=i} w_ij v_j / sum_{j<=i} w_ij with
    # w_ij = (phi(q_i) . phi(k_j)) prod_{t=j+1..i} alpha_t, written here with
    # numpy (independently of the recurrence)
    N, d = 15, 6
    q, k, v = (_rand((1, 1, N, d), s) for s in (43, 44, 45))
    a = _gates((1, 1, N), 46)
    f = (lambda x: np.where(x > 0, x + 1.0, np.exp(x))) if fmap != ID else (lambda x: x)
    fq, fk = f(q[0, 0]), f(k[0, 0])
    W = np.zeros((N, N))
    for i in range(N):
        for j in range(i + 1):
            W[i, j] = fq[i] @ fk[j] * np.prod(a[0, 0, j + 1:i + 1])
    y = W @ v[0, 0]
    if norm:
        y = y / W.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(oracle.causal_gated(q, k, v, a, fmap=fmap, normalise=norm)[0, 0],
                               y, rtol=1e-12, atol=1e-12)


def test_gated_zero_gate_resets_the_state():
    # alpha_t0 = 0 forgets everything before t0: from t0 on the outputs are
    # those of a fresh sequence starting at t0
    q, k, v = (_rand((1, 2, 20, 4), s) for s in (47, 48, 49))
    a = _gates((1, 2, 20), 50)
    a[..., 8] = 0.0
    y = oracle.causal_gated(q, k, v, a)
    y2 = oracle.causal_gated(q[..., 8:, :], k[..., 8:, :], v[..., 8:, :], a[..., 8:])
    np.testing.assert_allclose(y[..., 8:, :], y2, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# final state of the causal recurrence (the state a decode continues from)


@pytest.mark.parametrize("decay", [None, [0.96875, 0.5]])
def test_causal_state_closed_form(decay):
    # S_N = sum_t g^(N-1-t) phi(k_t) v_t^T (0-based t), z_N likewise:
    # written here with numpy's exp, independently of the oracle's phi
    B, H, N, d = 2, 2, 11, 5
    k, v = _rand((B, H, N, d), 30), _rand((B, H, N, d), 31)
    S, z = oracle.causal_state(k, v, decay)
    pk = np.where(k > 0, k + 1.0, np.exp(k))
    g = np.ones(H) if decay is None else np.asarray(decay)
    w = g[None, :, None] ** (N - 1 - np.arange(N))[None, None, :]  # [1, H, N]
    S_ref = np.einsum("bhn,bhna,bhnc->bhac", np.broadcast_to(w, (B, H, N)), pk, v)
    z_ref = np.einsum("bhn,bhna->bha", np.broadcast_to(w, (B, H, N)), pk)
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(z, z_ref, rtol=1e-12, atol=1e-12)


def test_causal_state_special_cases():
    k, v = _rand((1, 2, 9, 4), 32), _rand((1, 2, 9, 4), 33)
    # no decay: the whole-sequence sums of the non-causal form
    S, z = oracle.causal_state(k, v)
    Sn, zn = oracle.noncausal_state(k, v)
    np.testing.assert_allclose(S, Sn, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(z, zn, rtol=1e-14, atol=1e-14)
    # g = 0 keeps only the last token
    S0, z0 = oracle.causal_state(k, v, [0.0, 0.0])
    pk = np.where(k[..., -1, :] > 0, k[..., -1, :] + 1.0, np.exp(k[..., -1, :]))
    np.testing.assert_allclose(S0, pk[..., :, None] * v[..., -1, None, :], rtol=1e-15)
    np.testing.assert_allclose(z0, pk, rtol=1e-15)
    # empty sequence: the zero state
    Se, ze = oracle.causal_state(k[..., :0, :], v[..., :0, :])
    assert not Se.any() and not ze.any()


@pytest.mark.parametrize("decay", [None, [0.9, 0.6]])
def test_causal_state_is_what_the_last_output_reads(decay):
    q, k, v = (_rand((1, 2, 14, 6), s) for s in (34, 35, 36))
    S, z = oracle.causal_state(k, v, decay)
    y_last = oracle.state_read(S, z, q[..., -1:, :])[..., 0, :]
    np.testing.assert_allclose(y_last, oracle.causal(q, k, v, decay)[..., -1, :],
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("block", [1, 2, 3, 16, 64])
@pytest.mark.parametrize("segments", [1, 3])
@pytest.mark.parametrize("decay", [None, [0.96875, 0.5]])
def test_chunked_block_algebra_equals_recurrence(block, segments, decay):
    q, k, v = (_rand((1, 2, 67, 6), s, 0.7) for s in (10, 11, 12))
    yc = oracle.causal(q, k, v, decay)
    yb = oracle.chunked(q, k, v, decay, block=block, segments=segments)
    np.testing.assert_allclose(yb, yc, rtol=1e-11, atol=1e-12)


def test_decay_special_cases():
    q, k, v = (_rand((1, 2, 11, 4), s) for s in (13, 14, 15))
    # g = 1 is the undecayed recurrence
    np.testing.assert_array_equal(oracle.causal(q, k, v, [1.0, 1.0]),
                                  oracle.causal(q, k, v))
    # g = 0 forgets everything: y_t = v_t
    np.testing.assert_allclose(oracle.causal(q, k, v, [0.0, 0.0]), v,
                               rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("mode", ["causal", "noncausal", "decay"])
def test_constant_values_give_constant_output(mode):
    N, d = 23, 8
    q, k = _rand((2, N, d), 16, 3.0), _rand((2, N, d), 17, 3.0)
    u = _rand((2, 1, d), 18)
    v = np.broadcast_to(u, (2, N, d)).copy()
    if mode == "causal":
        y = oracle.causal(q, k, v)
    elif mode == "noncausal":
        y = oracle.noncausal(q, k, v)
    else:
        y = oracle.causal(q, k, v, [0.7, 0.99])
    np.testing.assert_allclose(y, np.broadcast_to(u, y.shape), rtol=1e-13,
                               atol=1e-13)


def test_outputs_are_convex_combinations_of_visible_values():
    N, d = 31, 5
    q, k, v = (_rand((1, N, d), s, 2.0) for s in (19, 20, 21))
    yc = oracle.causal(q, k, v)[0]
    for i in range(N):
        lo, hi = v[0, :i + 1].min(axis=0), v[0, :i + 1].max(axis=0)
        assert np.all(yc[i] >= lo - 1e-12) and np.all(yc[i] <= hi + 1e-12)
    yn = oracle.noncausal(q, k, v)[0]
    assert np.all(yn >= v[0].min(axis=0) - 1e-12)
    assert np.all(yn <= v[0].max(axis=0) + 1e-12)


def test_threaded_heads_match_single_thread():
    q, k, v = (_rand((3, 4, 20, 6), s) for s in (22, 23, 24))
    np.testing.assert_array_equal(oracle.causal(q, k, v, nthreads=1),
                                  oracle.causal(q, k, v, nthreads=5))
    np.testing.assert_array_equal(oracle.noncausal(q, k, v, nthreads=1),
                                  oracle.noncausal(q, k, v, nthreads=3))


def test_empty_sequence():
    q = np.zeros((2, 0, 4))
    assert oracle.causal(q, q, q).shape == (2, 0, 4)
    assert oracle.noncausal(q, q, q).shape == (2, 0, 4)
