"""Pins for the float64 oracle, each independent of the oracle's own code.

Every check here follows "Accelerating Mamba-2 with High-Performance Forward
Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture" (the
recurrence, the undecayed jump and linear-attention form, the unrolled
decayed expansion, the log-space jump and the chunked output equation, and
the stability remark), or plain mathematics.  A mutation test at the end
plants plausible mistakes in a copy of the recurrence and checks that the
pins catch each of them.
"""
import math

import numpy as np
import pytest

from conftest import load_golden

RTOL = 1e-12


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def rand_inputs(rng, b, L, nh, P, S, ng, h0=True, D=True):
    """Small float64 inputs with the layer's value distributions."""
    x = rng.standard_normal((b, L, nh, P))
    dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), (b, L, nh)))
    A = -np.exp(rng.uniform(0.0, math.log(16.0), nh))
    B = rng.standard_normal((b, L, ng, S))
    C = rng.standard_normal((b, L, ng, S))
    Dv = rng.standard_normal(nh) if D else None
    H0 = 0.1 * rng.standard_normal((b, nh, P, S)) if h0 else None
    return dict(x=x, dt=dt, A=A, B=B, C=C, D=Dv, h0=H0)


# ---------------------------------------------------------------------------
# hand-worked example (tests/golden/worked_example_p2s2.txt)
# ---------------------------------------------------------------------------

def golden_inputs():
    g = load_golden("worked_example_p2s2.txt")
    inp = dict(
        x=np.array(g["x"]).reshape(1, 3, 1, 2),
        dt=np.array(g["dt"]).reshape(1, 3, 1),
        A=np.array(g["A"]),
        B=np.array(g["B"]).reshape(1, 3, 1, 2),
        C=np.array(g["C"]).reshape(1, 3, 1, 2),
        D=np.array(g["D"]),
        h0=np.array(g["h0"]).reshape(1, 1, 2, 2),
    )
    return g, inp


def test_worked_example_recurrence(oracle_mod):
    g, inp = golden_inputs()
    out = oracle_mod.recurrence(**inp, chunk=2, want=("y", "final_state", "states", "dstates", "G"))
    np.testing.assert_allclose(out["y"].ravel(), g["y"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["final_state"].ravel(), g["final_state"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["states"].ravel(), g["states"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["dstates"].ravel(), g["dstates"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["G"].ravel() / math.log(2.0), g["G_over_ln2"], rtol=1e-13)


def test_worked_example_numpy_paths(oracle_mod):
    g, inp = golden_inputs()
    y, fin = oracle_mod.recurrence_np(**inp)
    np.testing.assert_allclose(y.ravel(), g["y"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fin.ravel(), g["final_state"], rtol=1e-13, atol=1e-13)
    ch = oracle_mod.chunked(**inp, chunk=2)
    np.testing.assert_allclose(ch["y"].ravel(), g["y"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ch["states"].ravel(), g["states"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ch["dstates"].ravel(), g["dstates"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(ch["G"].ravel() / math.log(2.0), g["G_over_ln2"], rtol=1e-13)


# ---------------------------------------------------------------------------
# brute force: the unrolled decayed expansion, summed term by term
# ---------------------------------------------------------------------------

def unrolled(inp, bi, h, hpg):
    """y_i = sum_{j<=i} exp(a_{j+1}+..+a_i) (c_i . B_j) dt_j x_j
             + exp(a_1+..+a_i) h0 c_i + D x_i
       h_L = exp(a_1+..+a_L) h0 + sum_j exp(a_{j+1}+..+a_L) dt_j x_j (outer) B_j
    with every exponent summed afresh from its own terms (no running sum)."""
    x, dt, A, B, C = inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"]
    L, P = x.shape[1], x.shape[3]
    S = B.shape[3]
    g = h // hpg
    a = [A[h] * dt[bi, t, h] for t in range(L)]
    h0 = inp["h0"][bi, h] if inp["h0"] is not None else np.zeros((P, S))
    Dh = inp["D"][h] if inp["D"] is not None else 0.0
    y = np.zeros((L, P))
    for i in range(L):
        for p in range(P):
            acc = 0.0
            for j in range(i + 1):
                e = math.exp(sum(a[k] for k in range(j + 1, i + 1)))
                cb = sum(C[bi, i, g, s] * B[bi, j, g, s] for s in range(S))
                acc += e * cb * dt[bi, j, h] * x[bi, j, h, p]
            e0 = math.exp(sum(a[k] for k in range(0, i + 1)))
            acc += e0 * sum(h0[p, s] * C[bi, i, g, s] for s in range(S))
            y[i, p] = acc + Dh * x[bi, i, h, p]
    fin = math.exp(sum(a)) * h0.copy()
    for j in range(L):
        e = math.exp(sum(a[k] for k in range(j + 1, L)))
        fin += e * dt[bi, j, h] * np.outer(x[bi, j, h], B[bi, j, g])
    return y, fin


@pytest.mark.parametrize("L,P,S,nh,ng,seed", [(1, 1, 1, 1, 1, 0), (7, 2, 3, 2, 1, 1),
                                              (23, 3, 2, 2, 2, 2), (40, 4, 4, 4, 2, 3)])
def test_brute_force_unrolled_sum(oracle_mod, L, P, S, nh, ng, seed):
    rng = np.random.default_rng(seed)
    inp = rand_inputs(rng, 1, L, nh, P, S, ng)
    out = oracle_mod.recurrence(**inp, chunk=8)
    for h in range(nh):
        y_bf, fin_bf = unrolled(inp, 0, h, nh // ng)
        assert rel_err(out["y"][0, :, h], y_bf) < RTOL
        assert rel_err(out["final_state"][0, h], fin_bf) < RTOL


# ---------------------------------------------------------------------------
# special cases the page names
# ---------------------------------------------------------------------------

def test_linear_attention_when_decay_removed(oracle_mod):
    """A = 0 removes the decay: Y = C h0^T + ((C (dt B)^T) * M) X + D X and
    h_L = h0 + (dt X)^T B -- the page's undecayed jump and linear-attention
    form, computed here with plain matrix products."""
    rng = np.random.default_rng(11)
    b, L, nh, P, S, ng = 2, 50, 3, 5, 6, 1
    inp = rand_inputs(rng, b, L, nh, P, S, ng)
    inp["A"] = np.zeros(nh)
    out = oracle_mod.recurrence(**inp, chunk=16)
    M = np.tril(np.ones((L, L)))
    for bi in range(b):
        for h in range(nh):
            X = inp["x"][bi, :, h]
            Bm, Cm = inp["B"][bi, :, 0], inp["C"][bi, :, 0]
            bt = inp["dt"][bi, :, h][:, None] * Bm
            H0 = inp["h0"][bi, h]
            Y = Cm @ H0.T + ((Cm @ bt.T) * M) @ X + inp["D"][h] * X
            assert rel_err(out["y"][bi, :, h], Y) < RTOL
            assert rel_err(out["final_state"][bi, h], H0 + X.T @ bt) < RTOL


def test_no_input_B_zero(oracle_mod):
    """B = 0: only the decayed initial state remains,
    y_t = exp(g_t) h0 c_t + D x_t with g the global cumsum of a, and the
    final state is exp(g_L) h0."""
    rng = np.random.default_rng(12)
    b, L, nh, P, S, ng = 1, 300, 2, 4, 8, 1
    inp = rand_inputs(rng, b, L, nh, P, S, ng)
    inp["B"] = np.zeros_like(inp["B"])
    out = oracle_mod.recurrence(**inp, chunk=64)
    for h in range(nh):
        g = np.cumsum(inp["A"][h] * inp["dt"][0, :, h])
        H0 = inp["h0"][0, h]
        Y = np.exp(g)[:, None] * (inp["C"][0, :, 0] @ H0.T) + inp["D"][h] * inp["x"][0, :, h]
        assert rel_err(out["y"][0, :, h], Y) < RTOL
        assert rel_err(out["final_state"][0, h], math.exp(g[-1]) * H0) < RTOL


def test_dt_zero_keeps_state(oracle_mod):
    """dt = 0 leaves the state unchanged: y_t = h0 c_t + D x_t."""
    rng = np.random.default_rng(13)
    inp = rand_inputs(rng, 1, 20, 2, 3, 5, 1)
    inp["dt"] = np.zeros_like(inp["dt"])
    out = oracle_mod.recurrence(**inp, chunk=8)
    for h in range(2):
        H0 = inp["h0"][0, h]
        Y = inp["C"][0, :, 0] @ H0.T + inp["D"][h] * inp["x"][0, :, h]
        assert rel_err(out["y"][0, :, h], Y) < RTOL
        np.testing.assert_array_equal(out["final_state"][0, h], H0)


def test_cumsum_closed_form(oracle_mod):
    """With dt constant per head, the chunk-local inclusive cumsum is linear:
    G[k*T + i] = A dt (i + 1), and the padded tail repeats the last value."""
    b, L, nh, P, S, T = 1, 100, 3, 2, 2, 32
    rng = np.random.default_rng(14)
    inp = rand_inputs(rng, b, L, nh, P, S, 1)
    dts = np.array([0.01, 0.05, 0.1])
    inp["dt"] = np.broadcast_to(dts, (b, L, nh)).copy()
    out = oracle_mod.recurrence(**inp, chunk=T, want=("G",))
    for h in range(nh):
        for t in range(4 * T):
            i = (min(t, L - 1)) % T  # padded positions repeat the last real token
            np.testing.assert_allclose(out["G"][0, h, t], inp["A"][h] * dts[h] * (i + 1), rtol=1e-13)


def test_group_mapping_contiguous(oracle_mod):
    """Heads share B and C by contiguous groups: head h uses group
    h // (nheads / ngroups).  Each head of a 2-group run must equal a
    1-head, 1-group run given its own group's B and C."""
    rng = np.random.default_rng(15)
    b, L, nh, P, S, ng = 1, 33, 4, 3, 4, 2
    inp = rand_inputs(rng, b, L, nh, P, S, ng)
    full = oracle_mod.recurrence(**inp, chunk=16)
    for h in range(nh):
        g = h // (nh // ng)
        one = oracle_mod.recurrence(
            x=inp["x"][:, :, h:h + 1], dt=inp["dt"][:, :, h:h + 1], A=inp["A"][h:h + 1],
            B=inp["B"][:, :, g:g + 1], C=inp["C"][:, :, g:g + 1], D=inp["D"][h:h + 1],
            h0=inp["h0"][:, h:h + 1], chunk=16)
        np.testing.assert_array_equal(full["y"][:, :, h], one["y"][:, :, 0])
        np.testing.assert_array_equal(full["final_state"][:, h], one["final_state"][:, 0])


def test_numpy_twin_matches_c(oracle_mod):
    rng = np.random.default_rng(16)
    inp = rand_inputs(rng, 2, 37, 4, 3, 5, 2)
    out = oracle_mod.recurrence(**inp, chunk=16)
    y, fin = oracle_mod.recurrence_np(**inp)
    assert rel_err(out["y"], y) < RTOL
    assert rel_err(out["final_state"], fin) < RTOL


# ---------------------------------------------------------------------------
# chunking: the log-space jump and chunked output equal the recurrence
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,T", [(256, 256), (256, 64), (300, 128), (300, 300),
                                 (517, 256), (97, 40), (1, 64)])
def test_chunk_invariance(oracle_mod, L, T):
    rng = np.random.default_rng(L * 1000 + T)
    inp = rand_inputs(rng, 1, L, 2, 4, 6, 1)
    rec = oracle_mod.recurrence(**inp, chunk=T, want=("y", "final_state", "states", "dstates", "G"))
    ch = oracle_mod.chunked(**inp, chunk=T)
    for k in ("y", "final_state", "states", "dstates"):
        assert rel_err(ch[k], rec[k]) < RTOL, k
    assert rel_err(ch["G"], rec["G"]) < RTOL
    # jump formula between consecutive stored states:
    # states[k+1] = exp(G_last,k) states[k] + dstates[k]
    nc = rec["states"].shape[2]
    for k in range(nc - 1):
        Gl = rec["G"][..., (k + 1) * T - 1]
        pred = np.exp(Gl)[..., None, None] * rec["states"][:, :, k] + rec["dstates"][:, :, k]
        assert rel_err(pred, rec["states"][:, :, k + 1]) < RTOL


def test_one_chunk_equals_many_chunks(oracle_mod):
    rng = np.random.default_rng(17)
    inp = rand_inputs(rng, 1, 512, 2, 4, 4, 1)
    one = oracle_mod.chunked(**inp, chunk=512)
    many = oracle_mod.chunked(**inp, chunk=64)
    assert rel_err(one["y"], many["y"]) < RTOL
    assert rel_err(one["final_state"], many["final_state"]) < RTOL


def test_stability_invariant(oracle_mod):
    """With every a_t <= 0, no exponent that survives the causal mask is
    positive, both in the output's decay matrix and in the jump weights."""
    rng = np.random.default_rng(18)
    inp = rand_inputs(rng, 1, 700, 3, 2, 2, 1)
    inp["A"][0] = -16.0  # the steepest decay the distributions allow
    ch = oracle_mod.chunked(**inp, chunk=256)
    assert ch["max_kept_exponent"] <= 0.0


# ---------------------------------------------------------------------------
# padding, resume, linearity
# ---------------------------------------------------------------------------

def test_padding_partial_chunk(oracle_mod):
    """L = 4000 equals the zero-dt padded L = 4096 run restricted to its first
    4000 rows, with identical final states."""
    rng = np.random.default_rng(19)
    b, L, Lp, nh, P, S = 1, 4000, 4096, 2, 4, 4
    inp = rand_inputs(rng, b, Lp, nh, P, S, 1)
    short = {k: (v[:, :L] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    inp["dt"][:, L:] = 0.0
    inp["x"][:, L:] = 0.0
    a = oracle_mod.recurrence(**short, chunk=256)
    p = oracle_mod.recurrence(**inp, chunk=256)
    np.testing.assert_array_equal(a["y"], p["y"][:, :L])
    np.testing.assert_array_equal(a["final_state"], p["final_state"])


@pytest.mark.parametrize("L1", [100, 256, 333])
def test_resume_from_final_state(oracle_mod, L1):
    rng = np.random.default_rng(20 + L1)
    inp = rand_inputs(rng, 2, 700, 2, 3, 4, 1)
    whole = oracle_mod.recurrence(**inp, chunk=128)
    first = {k: (v[:, :L1] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    rest = {k: (v[:, L1:] if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    o1 = oracle_mod.recurrence(**first, chunk=128)
    rest["h0"] = o1["final_state"]
    o2 = oracle_mod.recurrence(**rest, chunk=128)
    assert rel_err(np.concatenate([o1["y"], o2["y"]], axis=1), whole["y"]) < RTOL
    assert rel_err(o2["final_state"], whole["final_state"]) < RTOL


def test_linearity_in_h0(oracle_mod):
    """y(h0) - y(0) = diag(exp g) C h0^T per head, g the global cumsum."""
    rng = np.random.default_rng(21)
    inp = rand_inputs(rng, 1, 200, 2, 3, 5, 1)
    with_h0 = oracle_mod.recurrence(**inp, chunk=64)
    no_h0 = oracle_mod.recurrence(**{**inp, "h0": None}, chunk=64)
    for h in range(2):
        g = np.cumsum(inp["A"][h] * inp["dt"][0, :, h])
        expect = np.exp(g)[:, None] * (inp["C"][0, :, 0] @ inp["h0"][0, h].T)
        assert rel_err(with_h0["y"][0, :, h] - no_h0["y"][0, :, h], expect) < 1e-11


def test_bh_subset_matches_full(oracle_mod):
    rng = np.random.default_rng(22)
    inp = rand_inputs(rng, 2, 64, 3, 2, 3, 1)
    full = oracle_mod.recurrence(**inp, chunk=32)
    sub = oracle_mod.recurrence(**inp, chunk=32, bh=[4, 1])
    for pair in (4, 1):
        bi, h = divmod(pair, 3)
        np.testing.assert_array_equal(sub["y"][bi, :, h], full["y"][bi, :, h])
    assert np.isnan(sub["y"][0, :, 0]).all()


def test_rejects_bad_groups(oracle_mod):
    rng = np.random.default_rng(23)
    inp = rand_inputs(rng, 1, 8, 3, 2, 2, 1)
    inp["B"] = np.zeros((1, 8, 2, 2))
    inp["C"] = np.zeros((1, 8, 2, 2))
    with pytest.raises(AssertionError):
        oracle_mod.recurrence(**inp, chunk=4)


# ---------------------------------------------------------------------------
# mutation test: plausible mistakes planted in a copy of the recurrence
# ---------------------------------------------------------------------------

def mutated_recurrence(inp, mistake):
    x, dt, A, B, C, D, h0 = (inp[k] for k in ("x", "dt", "A", "B", "C", "D", "h0"))
    b, L, nh, P = x.shape
    ng, S = B.shape[2], B.shape[3]
    y = np.zeros((b, L, nh, P))
    for bi in range(b):
        for h in range(nh):
            g = (h % ng) if mistake == "group_mod" else h // (nh // ng)
            H = h0[bi, h].copy() if h0 is not None else np.zeros((P, S))
            for t in range(L):
                a = A[h] * dt[bi, t, h]
                u = x[bi, t, h] * (1.0 if mistake == "drop_dt_in_b" else dt[bi, t, h])
                Bt = C[bi, t, g] if mistake == "swap_BC" else B[bi, t, g]
                Ct = B[bi, t, g] if mistake == "swap_BC" else C[bi, t, g]
                Hprev = H
                decay = math.exp(-a) if mistake == "sign" else math.exp(a)
                if mistake == "transpose_state":
                    H = decay * H + np.outer(u, Bt).T.reshape(P, S)
                else:
                    H = decay * H + np.outer(u, Bt)
                Hy = Hprev if mistake == "pre_update" else H
                yt = Hy @ Ct
                if mistake != "drop_D":
                    yt = yt + D[h] * x[bi, t, h]
                y[bi, t, h] = yt
    return y


@pytest.mark.parametrize("mistake", ["pre_update", "drop_D", "drop_dt_in_b", "swap_BC",
                                     "sign", "transpose_state", "group_mod"])
def test_pins_catch_planted_mistakes(oracle_mod, mistake):
    """Each planted mistake must disagree with the hand-worked example or with
    the brute-force expansion on a small grouped case."""
    g, inp = golden_inputs()
    caught = rel_err(mutated_recurrence(inp, mistake).ravel(), g["y"]) > 1e-6
    rng = np.random.default_rng(99)
    small = rand_inputs(rng, 1, 9, 4, 2, 2, 2)
    ym = mutated_recurrence(small, mistake)
    for h in range(4):
        y_bf, _ = unrolled(small, 0, h, 2)
        caught = caught or rel_err(ym[0, :, h], y_bf) > 1e-6
    assert caught, mistake
    assert rel_err(mutated_recurrence(inp, "none").ravel(), g["y"]) < 1e-13
