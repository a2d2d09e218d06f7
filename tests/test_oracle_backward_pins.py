"""Pins of the float64 backward oracle (oracle.backward), none of which
re-types it:

* central finite differences of the forward C recurrence (oracle.recurrence,
  an independent implementation) for every input element of small grouped
  cases, with a random loss L = <gy, y> + <gfinal, final_state>;
* closed forms: with B = 0 and h0 = 0 the state stays zero, so
  dx = D gy, dC = 0, dA = 0, ddt = 0 and dD = sum gy x; with A = 0 (no
  decay) dx_t = sum_{s >= t} (c_s . b_t) gy_s + gfinal b_t + D gy_t, written
  with a masked matrix product;
* a mutation test: plausible mistakes planted in a copy of the adjoint
  recurrence (dropped skip term, shifted decay, pre-update state in dC, a
  missing last decay in dh0, a dropped dt-through-b term, an overwritten group
  sum) each fail the finite-difference pin.
"""
import numpy as np
import pytest

import oracle


def rand_inputs(rng, b, L, nh, P, S, ng, h0=True):
    return {
        "x": rng.standard_normal((b, L, nh, P)),
        "dt": np.exp(rng.uniform(np.log(1e-2), np.log(3e-1), (b, L, nh))),
        "A": -np.exp(rng.uniform(0.0, np.log(4.0), nh)),
        "B": rng.standard_normal((b, L, ng, S)),
        "C": rng.standard_normal((b, L, ng, S)),
        "D": rng.standard_normal(nh),
        "h0": rng.standard_normal((b, nh, P, S)) * 0.3 if h0 else None,
    }


def loss(inp, gy, gfinal):
    out = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["h0"], chunk=64)
    return float(np.sum(gy * out["y"]) + np.sum(gfinal * out["final_state"]))


def finite_differences(inp, gy, gfinal, eps=1e-6):
    grads = {}
    for k in ("x", "dt", "A", "B", "C", "D", "h0"):
        if inp[k] is None:
            continue
        g = np.zeros_like(inp[k])
        flat = inp[k].reshape(-1)
        for i in range(flat.size):
            keep = flat[i]
            flat[i] = keep + eps
            fp = loss(inp, gy, gfinal)
            flat[i] = keep - eps
            fm = loss(inp, gy, gfinal)
            flat[i] = keep
            g.reshape(-1)[i] = (fp - fm) / (2 * eps)
        grads["d" + k] = g
    return grads


def rel_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


CASES = [
    (1, 5, 2, 3, 2, 1),   # one group
    (2, 7, 4, 2, 3, 2),   # two groups of two heads
]


@pytest.fixture(scope="module")
def fd_cases():
    oracle.build()
    rng = np.random.default_rng(2024)
    out = []
    for dims in CASES:
        inp = rand_inputs(rng, *dims)
        b, L, nh, P, S, ng = dims
        gy = rng.standard_normal((b, L, nh, P))
        gfinal = rng.standard_normal((b, nh, P, S))
        out.append((inp, gy, gfinal, finite_differences(inp, gy, gfinal)))
    return out


def oracle_grads(inp, gy, gfinal, fn=None):
    fn = fn or oracle.backward
    return fn(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"], gy, gfinal)


def test_matches_finite_differences_of_the_recurrence(fd_cases):
    for inp, gy, gfinal, fd in fd_cases:
        g = oracle_grads(inp, gy, gfinal)
        for k, ref in fd.items():
            assert rel_err(g[k], ref) < 1e-7, (k, rel_err(g[k], ref))


def test_without_h0_gradient_of_h0_is_the_carried_adjoint(fd_cases):
    """With h0 absent the loss does not depend on it, but the carried
    adjoint is still returned: it equals the gradient for h0 = 0 (the loss
    is affine in h0)."""
    inp, gy, gfinal, fd = fd_cases[0]
    no_h0 = dict(inp, h0=None)
    zero_h0 = dict(inp, h0=np.zeros_like(inp["h0"]))
    g1 = oracle_grads(no_h0, gy, gfinal)
    g2 = oracle_grads(zero_h0, gy, gfinal)
    for k in g1:
        np.testing.assert_allclose(g1[k], g2[k], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g2["dh0"], fd["dh0"], rtol=1e-6, atol=1e-9)


def test_b_zero_closed_form():
    rng = np.random.default_rng(5)
    inp = rand_inputs(rng, 2, 6, 4, 3, 2, 2, h0=False)
    inp["B"] = np.zeros_like(inp["B"])
    gy = rng.standard_normal(inp["x"].shape)
    gfinal = rng.standard_normal((2, 4, 3, 2))
    g = oracle_grads(inp, gy, gfinal)
    np.testing.assert_allclose(g["dx"], inp["D"][None, None, :, None] * gy, rtol=0, atol=1e-12)
    assert np.abs(g["dC"]).max() == 0.0
    assert np.abs(g["dA"]).max() == 0.0
    assert np.abs(g["ddt"]).max() == 0.0
    np.testing.assert_allclose(g["dD"], np.einsum("blhp,blhp->h", gy, inp["x"]), rtol=1e-12)


def test_linear_attention_closed_form():
    """A = 0 (no decay): g_t = sum_{s >= t} gy_s c_s^T + gfinal, so
    dx_t = sum_{s >= t} (b_t . c_s) gy_s + gfinal b_t + D gy_t, i.e.
    dx = triu(b c^T) gy + b gfinal^T + D gy with b_t = dt_t B_t."""
    rng = np.random.default_rng(6)
    b, L, nh, P, S, ng = 1, 8, 2, 3, 4, 1
    inp = rand_inputs(rng, b, L, nh, P, S, ng)
    inp["A"] = np.zeros(nh)
    gy = rng.standard_normal((b, L, nh, P))
    gfinal = rng.standard_normal((b, nh, P, S))
    g = oracle_grads(inp, gy, gfinal)
    for h in range(nh):
        bmat = inp["dt"][0, :, h, None] * inp["B"][0, :, 0]      # [L, S], rows b_t
        cmat = inp["C"][0, :, 0]                                  # [L, S], rows c_s
        M = np.triu(bmat @ cmat.T)                                # M[t, s] = b_t . c_s, s >= t
        dx = M @ gy[0, :, h] + bmat @ gfinal[0, h].T + inp["D"][h] * gy[0, :, h]
        np.testing.assert_allclose(g["dx"][0, :, h], dx, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------------------
# mutation test: plausible mistakes planted in a copy of the adjoint
# ---------------------------------------------------------------------------

def mutated_backward(mistake):
    def fn(x, dt, A, B, C, D, h0, gy, gfinal):
        b, L, nh, P = x.shape
        ng, S = B.shape[2], B.shape[3]
        hpg = nh // ng
        out = {"dx": np.zeros_like(x), "ddt": np.zeros_like(dt), "dA": np.zeros_like(A),
               "dB": np.zeros_like(B), "dC": np.zeros_like(C), "dD": np.zeros(nh),
               "dh0": np.zeros((b, nh, P, S))}
        for bi in range(b):
            for h in range(nh):
                g = h // hpg
                hs = np.zeros((L + 1, P, S))
                if h0 is not None:
                    hs[0] = h0[bi, h]
                a = np.exp(A[h] * dt[bi, :, h])
                for t in range(L):
                    hs[t + 1] = a[t] * hs[t] + np.outer(x[bi, t, h], dt[bi, t, h] * B[bi, t, g])
                G = gfinal[bi, h].copy()
                for t in range(L - 1, -1, -1):
                    if mistake == "decay_shift":
                        G = a[t] * G
                    G = G + np.outer(gy[bi, t, h], C[bi, t, g])
                    bt = dt[bi, t, h] * B[bi, t, g]
                    skip = 0.0 if mistake == "drop_skip" else D[h] * gy[bi, t, h]
                    out["dx"][bi, t, h] = G @ bt + skip
                    db = G.T @ x[bi, t, h]
                    if mistake == "group_overwrite":
                        out["dB"][bi, t, g] = dt[bi, t, h] * db
                    else:
                        out["dB"][bi, t, g] += dt[bi, t, h] * db
                    hc = hs[t] if mistake == "pre_update_dc" else hs[t + 1]
                    out["dC"][bi, t, g] += hc.T @ gy[bi, t, h]
                    da = float(np.sum(G * hs[t]))
                    via_b = 0.0 if mistake == "drop_dt_via_b" else float(db @ B[bi, t, g])
                    out["ddt"][bi, t, h] = A[h] * a[t] * da + via_b
                    out["dA"][h] += dt[bi, t, h] * a[t] * da
                    out["dD"][h] += float(gy[bi, t, h] @ x[bi, t, h])
                    if mistake != "decay_shift":
                        G = a[t] * G
                if mistake == "dh0_no_last_decay":
                    G = G / a[0]
                out["dh0"][bi, h] = G
        return out
    return fn


MISTAKES = ["drop_skip", "decay_shift", "pre_update_dc", "dh0_no_last_decay", "drop_dt_via_b",
            "group_overwrite"]


@pytest.mark.parametrize("mistake", ["none"] + MISTAKES)
def test_pins_catch_planted_mistakes(fd_cases, mistake):
    inp, gy, gfinal, fd = fd_cases[1]  # two groups of two heads
    g = oracle_grads(inp, gy, gfinal, fn=mutated_backward(mistake))
    worst = max(rel_err(g[k], ref) for k, ref in fd.items())
    if mistake == "none":
        assert worst < 1e-7
    else:
        assert worst > 1e-3, mistake


@pytest.mark.parametrize("dims,T,h0,gf", [
    ((1, 7, 2, 3, 2, 1), 3, True, True),     # partial last chunk
    ((2, 13, 4, 2, 3, 2), 4, True, False),   # groups, no gfinal
    ((1, 20, 2, 4, 5, 1), 8, False, True),   # no h0
    ((1, 9, 3, 2, 2, 3), 9, True, True),     # one chunk, one head per group
    ((1, 16, 2, 3, 3, 1), 1, True, True),    # chunks of one token
])
def test_chunked_backward_matches_the_adjoint_recurrence(dims, T, h0, gf):
    """The chunked restatement (reverse pass over chunks, per-chunk masked
    products, dL/dl as a reverse cumsum of dL/dG) equals the token-by-token
    adjoint to rounding, whatever the chunk size."""
    rng = np.random.default_rng(31)
    inp = rand_inputs(rng, *dims, h0=h0)
    b, L, nh, P, S, ng = dims
    gy = rng.standard_normal((b, L, nh, P))
    gfinal = rng.standard_normal((b, nh, P, S)) if gf else None
    args = (inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"], gy, gfinal)
    ref = oracle.backward(*args)
    got = oracle.backward_chunked(*args, chunk=T)
    for k in ref:
        assert rel_err(got[k], ref[k]) < 1e-12, (k, rel_err(got[k], ref[k]))
