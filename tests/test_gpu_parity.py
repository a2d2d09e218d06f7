"""GPU parity: every entry point of the C ABI against the float64 oracle.

Small cases compare every output element; the named layer shapes and the
sweep run at full size and compare sampled (batch, head) pairs, which the
oracle computes one by one.  Tolerances are stated in tests/parity.py.
"""
import numpy as np
import pytest
import torch

from parity import (LN2, LOG2E, check_io, device_inputs, forward_checked, make, oracle_run,
                    rel_l2, sample_pairs, to64)

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


def small(name, L, nh, P, S, ng, T, dtype, h0=True, batch=1):
    return W.Workload(name, batch, L, nh, P, S, ng, T, dtype, h0)


SMALL_CASES = [
    W.TINY,
    small("tiny_bf16", 256, 2, 16, 16, 1, 64, "bf16"),
    small("one_token", 1, 2, 64, 128, 1, 256, "fp32"),
    small("one_token_bf16", 1, 3, 32, 64, 1, 64, "bf16"),
    small("shorter_than_chunk", 100, 2, 64, 64, 1, 256, "fp32"),
    small("chunk_minus_one", 255, 2, 64, 128, 1, 256, "bf16"),
    small("chunk_plus_one", 257, 2, 64, 128, 1, 256, "fp32"),
    small("ragged_T128", 333, 4, 64, 128, 2, 128, "bf16", batch=2),
    small("groups_hpg3", 300, 6, 32, 48, 2, 64, "fp32", batch=2),
    small("max_dims", 300, 2, 128, 256, 1, 256, "bf16"),
    small("max_dims_fp32", 200, 2, 128, 256, 1, 128, "fp32"),
    small("odd_multiples", 190, 3, 48, 80, 3, 64, "bf16", h0=False),
    small("no_h0_fp32", 512, 2, 64, 64, 1, 128, "fp32", h0=False),
    small("bf16_hpg6_three_heads_per_cta", 600, 12, 64, 128, 2, 256, "bf16", batch=2),
    small("bf16_S256_groups", 520, 12, 64, 256, 2, 256, "bf16"),
    small("bf16_P96_S48", 300, 4, 96, 48, 1, 128, "bf16"),
    # output pass with C B^T shared by a slice of heads: two groups, and 20
    # chunks x 24 heads, where four heads share one CTA (alternating state
    # and x buffers, the second reusing B's shared memory)
    small("bf16_chunk_two_groups", 700, 6, 64, 128, 2, 256, "bf16", batch=2),
    small("bf16_chunk_T128_S64", 500, 4, 64, 64, 1, 128, "bf16"),
    small("bf16_chunk_four_heads_per_cta", 5120, 24, 64, 128, 1, 256, "bf16"),
]


def _full_oracle(w, inp):
    return oracle_run(w, inp, want=("y", "final_state", "states", "dstates", "G"))


@pytest.mark.parametrize("w", SMALL_CASES, ids=lambda w: w.name)
def test_each_step_small(ssd, w):
    inp = make(w)
    ref = _full_oracle(w, inp)
    dev = device_inputs(inp)
    T = w.chunk

    # step 1: G in log2 units
    G = ssd.chunk_cumsum(dev["dt"], dev["A"], T, headdim=w.headdim, dstate=w.dstate)
    torch.cuda.synchronize()
    np.testing.assert_allclose(to64(G) * LN2, ref["G"], rtol=1e-5, atol=1e-6)

    # step 2: chunk-local jump terms, from the GPU's own G
    dst = ssd.chunk_state(dev["x"], dev["B"], dev["dt"], G, T)
    check_io(to64(dst), ref["dstates"], w.dtype, "dstates")

    # step 3 in isolation: fed the oracle's jump terms and G
    G_or = torch.from_numpy(ref["G"] * LOG2E).float().cuda()
    dst_or = torch.from_numpy(ref["dstates"]).float().cuda()
    h0 = dev["h0"]
    states, final = ssd.state_passing(dst_or, G_or, h0, chunk=T, seqlen=w.seqlen,
                                      ngroups=w.ngroups)
    assert rel_l2(to64(states), ref["states"]) < 1e-5
    assert rel_l2(to64(final), ref["final_state"]) < 1e-5

    # step 4 in isolation: fed the oracle's start-of-chunk states
    st_or = torch.from_numpy(ref["states"]).float().cuda()
    y = ssd.chunk_scan(dev["x"], dev["B"], dev["C"], dev["dt"], G, st_or, dev["D"], chunk=T)
    check_io(to64(y), ref["y"], w.dtype, "chunk_scan y")

    # the whole forward pass
    ssd.device_error()  # no bounded wait of the step-wise calls gave up
    y2, fin2 = forward_checked(ssd, dev, T, h0=h0)
    check_io(to64(y2), ref["y"], w.dtype, "forward y")
    check_io(to64(fin2), ref["final_state"], w.dtype, "forward final_state")
    x64 = to64(inp["x"])
    Dx = to64(inp["D"])[None, None, :, None] * x64
    check_io(to64(y2) - Dx, ref["y"] - Dx, w.dtype, "forward y - D x")


def _forward_sampled(ssd, w, seed=0):
    inp = make(w, seed)
    bh = sample_pairs(w)
    ref = oracle_run(w, inp, bh=bh)
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
    y64, fin64, x64 = to64(y), to64(fin), to64(inp["x"])
    D = to64(inp["D"])
    for pair in bh:
        b, h = divmod(pair, w.nheads)
        check_io(y64[b, :, h], ref["y"][b, :, h], w.dtype, f"{w.name} y[b={b},h={h}]")
        check_io(y64[b, :, h] - D[h] * x64[b, :, h], ref["y"][b, :, h] - D[h] * x64[b, :, h],
                 w.dtype, f"{w.name} y-Dx[b={b},h={h}]")
        check_io(fin64[b, h], ref["final_state"][b, h], w.dtype, f"{w.name} final[b={b},h={h}]")
    assert np.isfinite(y64).all()


@pytest.mark.parametrize("w", W.NAMED[1:], ids=lambda w: w.name)
def test_forward_named_full_size(ssd, w):
    _forward_sampled(ssd, w)


@pytest.mark.parametrize("w", W.sweep(), ids=lambda w: w.name)
def test_forward_sweep_full_size(ssd, w):
    _forward_sampled(ssd, w)


def test_no_writes_past_the_end(ssd):
    """y is written for t < L only: a canary tail after the output survives."""
    w = small("canary", 300, 2, 64, 64, 1, 256, "bf16")
    inp = device_inputs(make(w))
    n = inp["x"].numel()
    buf = torch.full((n + 4096,), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = buf[:n].view_as(inp["x"])
    ssd.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["h0"],
                chunk=256, y=y)
    torch.cuda.synchronize()
    assert torch.isnan(buf[n:]).all()
    assert torch.isfinite(y).all()


def test_deterministic_and_stream_aware(ssd):
    w = W.MAMBA2_130M
    inp = device_inputs(make(w))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y1, f1 = ssd.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             None, chunk=w.chunk)
        y2, f2 = ssd.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             None, chunk=w.chunk)
    s.synchronize()
    assert torch.equal(y1, y2) and torch.equal(f1, f2)


def test_resume_matches_one_shot(ssd):
    """forward on [0, L1) then on [L1, L) with h0 = the first final state
    equals one forward over [0, L) (L1 not a multiple of the chunk)."""
    w = small("resume", 700, 4, 64, 128, 1, 256, "fp32")
    inp = device_inputs(make(w))
    L1 = 333
    y, fin = ssd.forward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                         inp["h0"], chunk=256)
    sl = lambda t, a, b: t[:, a:b].contiguous()  # noqa: E731
    ya, fa = ssd.forward(sl(inp["x"], 0, L1), sl(inp["dt"], 0, L1), inp["A"],
                         sl(inp["B"], 0, L1), sl(inp["C"], 0, L1), inp["D"], inp["h0"], chunk=256)
    yb, fb = ssd.forward(sl(inp["x"], L1, 700), sl(inp["dt"], L1, 700), inp["A"],
                         sl(inp["B"], L1, 700), sl(inp["C"], L1, 700), inp["D"], fa, chunk=256)
    torch.cuda.synchronize()
    assert rel_l2(to64(torch.cat([ya, yb], 1)), to64(y)) < 2e-3
    assert rel_l2(to64(fb), to64(fin)) < 2e-3


def test_steep_decay_blocks(ssd):
    """The output pass factors the decay of a row's own 64-token block about
    the block's last token only while the block's total decay stays above
    2^-96; steeper blocks take the direct exponent.  One input with both kinds
    of block in the same chunk (and heads with only one kind), against the
    oracle."""
    w = small("bf16_steep_decay", 1024, 4, 64, 128, 1, 256, "bf16")
    inp = make(w)
    A = inp["A"].clone()
    A[0] = A[1] = -16.0
    dt = inp["dt"].double().clone()
    tok = torch.arange(w.seqlen)
    dt[0, (tok // 64) % 2 == 1, 0] = 0.5  # head 0: every other block steep
    dt[0, :, 1] = 0.1                     # head 1: every block steep
    inp["A"], inp["dt"] = A, dt.to(inp["dt"].dtype)
    a = -(A.double()[None, None, :] * inp["dt"].double()) * LOG2E
    span = a.reshape(1, w.seqlen // 64, 64, w.nheads).sum(2)
    assert (span > 96).any() and (span < 96).any()
    ref = oracle_run(w, inp)
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
    y64, x64 = to64(y), to64(inp["x"])
    Dx = to64(inp["D"])[None, None, :, None] * x64
    check_io(y64, ref["y"], w.dtype, "steep y")
    check_io(y64 - Dx, ref["y"] - Dx, w.dtype, "steep y - D x")
    check_io(to64(fin), ref["final_state"], w.dtype, "steep final_state")
