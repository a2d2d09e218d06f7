"""GPU parity of the single-token decode step (ssd_decode_step) against the
float64 oracle: one step, several steps carrying the state, and decoding
that continues from ssd_forward's final state.

Tolerances: y as for the forward pass (tests/parity.py); the state stays
fp32 in both, so it is held to rel_l2 <= 1e-5.
"""
import numpy as np
import pytest
import torch

from parity import check_io, device_inputs, make, rel_l2, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from mamba_ssd_forward_gb300 import build
    build.build()
    oracle.build()
    import mamba_ssd_forward_gb300 as m
    return m


from mamba_ssd_forward_gb300 import inputs as W  # noqa: E402

CASES = [
    W.Workload("dec_fp32", 2, 5, 4, 16, 16, 1, 64, "fp32", True),
    W.Workload("dec_bf16_layer", 4, 5, 24, 64, 128, 1, 256, "bf16", True),
    W.Workload("dec_bf16_groups_S256", 1, 5, 48, 64, 256, 8, 256, "bf16", True),
    W.Workload("dec_fp32_odd", 3, 5, 6, 5, 12, 3, 64, "fp32", True),
    W.Workload("dec_bf16_S1024", 1, 5, 2, 8, 1024, 1, 64, "bf16", True),
    # enough (batch, head) pairs that the kernel does not slice P across CTAs
    W.Workload("dec_bf16_many_pairs", 8, 3, 80, 64, 128, 1, 256, "bf16", True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_steps_match_oracle(ssd, w):
    import oracle
    inp = make(w, seed=5)
    dev = device_inputs(inp)
    state = dev["h0"].clone()
    h = to64(inp["h0"])
    for t in range(w.seqlen):
        # fresh copies: the library takes 16-byte aligned pointers, which a
        # view into the sequence (batch 1) need not be
        sl = lambda k: dev[k][:, t].clone()  # noqa: E731
        y = ssd.decode_step(sl("x"), sl("dt"), dev["A"], sl("B"), sl("C"), dev["D"], state)
        torch.cuda.synchronize()
        y_ref, h = oracle.decode_step(to64(inp["x"][:, t]), to64(inp["dt"][:, t]), to64(inp["A"]),
                                      to64(inp["B"][:, t]), to64(inp["C"][:, t]), to64(inp["D"]), h)
        check_io(to64(y), y_ref, w.dtype, f"{w.name} y[t={t}]")
        assert rel_l2(to64(state), h) < 1e-5, f"{w.name} state[t={t}]"


def test_decode_continues_forward(ssd):
    """ssd_forward over 300 tokens, then 3 decode steps, equals the
    recurrence over all 303 tokens."""
    import oracle
    w = W.Workload("dec_after_fwd", 2, 303, 8, 64, 128, 2, 256, "bf16", True)
    inp = make(w, seed=9)
    dev = device_inputs(inp)
    L1 = 300
    sl = lambda k, a, b: dev[k][:, a:b].contiguous()  # noqa: E731
    y1, fin = ssd.forward(sl("x", 0, L1), sl("dt", 0, L1), dev["A"], sl("B", 0, L1),
                          sl("C", 0, L1), dev["D"], dev["h0"], chunk=256)
    ys = []
    for t in range(L1, w.seqlen):
        ys.append(ssd.decode_step(dev["x"][:, t].clone(), dev["dt"][:, t].clone(),
                                  dev["A"], dev["B"][:, t].clone(), dev["C"][:, t].clone(),
                                  dev["D"], fin))
    torch.cuda.synchronize()
    ref = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["h0"], chunk=256)
    check_io(to64(torch.stack(ys, 1)), ref["y"][:, L1:], w.dtype, "decoded y")
    check_io(to64(fin), ref["final_state"], w.dtype, "state after decoding")
