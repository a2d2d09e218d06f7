"""Pins for the oracle's single-token decode step (oracle.decode_step).

The step is one token of the recurrence of "Accelerating Mamba-2 with
High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section
"Mamba-2 architecture".  It is pinned by the hand-worked example of
tests/golden/ (every token, the intermediate state and the final state), by
agreement over whole sequences with the C recurrence (a separate
implementation), by the dt = 0 special case, and by planted mistakes that
those pins must catch.
"""
import math

import numpy as np
import pytest

from conftest import load_golden
from test_oracle_pins import rand_inputs


def golden():
    g = load_golden("worked_example_p2s2.txt")
    inp = dict(x=np.array(g["x"]).reshape(3, 2), dt=np.array(g["dt"]), A=np.array(g["A"]),
               B=np.array(g["B"]).reshape(3, 2), C=np.array(g["C"]).reshape(3, 2),
               D=np.array(g["D"]), h0=np.array(g["h0"]).reshape(2, 2))
    return g, inp


def step_golden(step, g, inp):
    h = inp["h0"].reshape(1, 1, 2, 2)
    ys, hs = [], []
    for t in range(3):
        y, h = step(inp["x"][t].reshape(1, 1, 2), inp["dt"][t].reshape(1, 1), inp["A"],
                    inp["B"][t].reshape(1, 1, 2), inp["C"][t].reshape(1, 1, 2), inp["D"], h)
        ys.append(y.ravel())
        hs.append(h.ravel())
    return np.concatenate(ys), hs


def test_decode_worked_example(oracle_mod):
    g, inp = golden()
    ys, hs = step_golden(oracle_mod.decode_step, g, inp)
    np.testing.assert_allclose(ys, g["y"], rtol=1e-13, atol=1e-13)
    # after two tokens the state is the start state of the second chunk
    np.testing.assert_allclose(hs[1], g["states"][4:], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(hs[2], g["final_state"], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("nh,ng,h0,D", [(2, 1, True, True), (6, 2, False, True), (3, 3, True, False)])
def test_decode_matches_c_recurrence(oracle_mod, nh, ng, h0, D):
    rng = np.random.default_rng(7 + nh)
    b, L, P, S = 2, 9, 4, 6
    inp = rand_inputs(rng, b, L, nh, P, S, ng, h0=h0, D=D)
    ref = oracle_mod.recurrence(**inp, chunk=4)
    h = inp["h0"]
    ys = []
    for t in range(L):
        y, h = oracle_mod.decode_step(inp["x"][:, t], inp["dt"][:, t], inp["A"], inp["B"][:, t],
                                      inp["C"][:, t], inp["D"], h)
        ys.append(y)
    np.testing.assert_allclose(np.stack(ys, 1), ref["y"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h, ref["final_state"], rtol=1e-11, atol=1e-12)


def test_decode_dt_zero_keeps_state(oracle_mod):
    rng = np.random.default_rng(3)
    b, nh, P, S, ng = 2, 4, 3, 5, 2
    h = rng.standard_normal((b, nh, P, S))
    x = rng.standard_normal((b, nh, P))
    C = rng.standard_normal((b, ng, S))
    D = rng.standard_normal(nh)
    y, h2 = oracle_mod.decode_step(x, np.zeros((b, nh)), -np.ones(nh),
                                   rng.standard_normal((b, ng, S)), C, D, h)
    np.testing.assert_array_equal(h2, h)
    grp = np.arange(nh) // (nh // ng)
    for bi in range(b):
        for hd in range(nh):
            np.testing.assert_allclose(y[bi, hd], h[bi, hd] @ C[bi, grp[hd]] + D[hd] * x[bi, hd],
                                       rtol=1e-13)


def _mutant(kind):
    """A copy of the decode step with one plausible mistake planted."""
    def step(x, dt, A, B, C, D, h):
        b, nh, P = x.shape
        ng = B.shape[1]
        grp = np.arange(nh) % ng if kind == "group_modulo" else np.arange(nh) // (nh // ng)
        Bh, Ch = B[:, grp], C[:, grp]
        sign = 1.0 if kind == "decay_sign" else -1.0
        decay = np.exp(sign * np.abs(A)[None, :] * dt)
        inc = (x if kind == "dt_dropped" else dt[:, :, None] * x)[:, :, :, None] * Bh[:, :, None, :]
        h_new = decay[:, :, None, None] * h + inc
        src = h if kind == "pre_update_output" else h_new
        y = np.einsum("bhps,bhs->bhp", src, Ch) + D[None, :, None] * x
        return y, h_new
    return step


@pytest.mark.parametrize("kind", ["decay_sign", "dt_dropped", "pre_update_output", "group_modulo"])
def test_decode_pins_catch_planted_mistakes(oracle_mod, kind):
    g, inp = golden()
    ys, hs = step_golden(_mutant(kind), g, inp)
    golden_ok = np.allclose(ys, g["y"], rtol=1e-9, atol=1e-9) and np.allclose(
        hs[2], g["final_state"], rtol=1e-9, atol=1e-9)
    if kind == "group_modulo":
        # one group in the golden example: the group mapping is pinned by
        # agreement with the C recurrence on several groups instead
        rng = np.random.default_rng(11)
        inp2 = rand_inputs(rng, 1, 3, 6, 2, 3, 2, h0=True, D=True)
        ref = oracle_mod.recurrence(**inp2, chunk=4)
        h = inp2["h0"]
        for t in range(3):
            y, h = _mutant(kind)(inp2["x"][:, t], inp2["dt"][:, t], inp2["A"], inp2["B"][:, t],
                                 inp2["C"][:, t], inp2["D"], h)
        golden_ok = np.allclose(h, ref["final_state"], rtol=1e-9)
    assert not golden_ok, kind
