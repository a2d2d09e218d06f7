"""GPU checks of the launch plans and the timing autotuner: every candidate
plan gives results within the parity tolerance of the oracle, plans that
only change heads per CTA of the output kernel give identical bits, and the
tuner returns one of the candidates (installing nothing: later calls without
a plan keep running the default)."""
import numpy as np
import pytest
import torch

from parity import check_io, device_inputs, forward_checked, make, oracle_run, to64

pytestmark = pytest.mark.gpu

from mamba_ssd_forward_gb300 import inputs as W  # noqa: E402


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


# 8 heads per group: several chunk-jump plans and output-kernel slices
CASE = W.Workload("bf16_plans", 2, 700, 8, 64, 128, 1, 256, "bf16", True)


@pytest.fixture(scope="module")
def case(ssd):
    inp = make(CASE)
    ref = oracle_run(CASE, inp)
    dev = device_inputs(inp)
    d = ssd.dims_of(dev["x"], dev["B"], CASE.chunk)
    return inp, ref, dev, d


def test_every_candidate_plan_matches_the_oracle(ssd, case):
    inp, ref, dev, d = case
    cands = ssd.plan_candidates(d)
    assert len(cands) > 4
    by_kernel = {}
    for p in cands:
        y, fin = forward_checked(ssd, dev, CASE.chunk, h0=dev["h0"], plan=p)
        check_io(to64(y), ref["y"], "bf16", f"y {p}")
        check_io(to64(fin), ref["final_state"], "bf16", f"final_state {p}")
        key = (p["chunk_state_heads"], p["chunk_state_ctas"], p["scan_kernel"])
        by_kernel.setdefault(key, []).append(y.clone())
    # heads per CTA of the output kernel only change the launch shape
    for ys in by_kernel.values():
        for y in ys[1:]:
            assert torch.equal(y, ys[0])


def test_tune_returns_a_candidate_and_installs_nothing(ssd, case):
    inp, ref, dev, d = case
    y_def, _ = forward_checked(ssd, dev, CASE.chunk, h0=dev["h0"])
    plan, y, fin = ssd.tune(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                            dev["h0"], chunk=CASE.chunk, reps=3)
    assert plan in ssd.plan_candidates(d)
    check_io(to64(y), ref["y"], "bf16", "tuned y")
    check_io(to64(fin), ref["final_state"], "bf16", "tuned final_state")
    y2, _ = forward_checked(ssd, dev, CASE.chunk, h0=dev["h0"], plan=plan)
    assert torch.equal(y2, y)  # the returned plan reproduces the tuner's last pass
    y3, _ = forward_checked(ssd, dev, CASE.chunk, h0=dev["h0"])
    assert torch.equal(y3, y_def)  # and calls without a plan still run the default


def test_tune_from_a_cold_l2(ssd, case):
    """With a flush buffer every candidate is timed after the buffer is
    overwritten; the tuner still returns a candidate whose pass matches the
    oracle."""
    inp, ref, dev, d = case
    flush = torch.empty(160 << 20, dtype=torch.uint8, device="cuda")
    plan, y, fin = ssd.tune(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                            dev["h0"], chunk=CASE.chunk, reps=2, flush=flush)
    assert plan in ssd.plan_candidates(d)
    check_io(to64(y), ref["y"], "bf16", "cold-L2 tuned y")
    check_io(to64(fin), ref["final_state"], "bf16", "cold-L2 tuned final_state")


def test_tune_rejects_fp32(ssd):
    from mamba_ssd_forward_gb300 import _abi
    w = W.Workload("fp32_plans", 1, 256, 2, 64, 64, 1, 128, "fp32", False)
    dev = device_inputs(make(w))
    with pytest.raises(_abi.SsdError) as e:
        ssd.tune(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], None,
                 chunk=w.chunk)
    assert e.value.code == _abi.SSD_ERR_UNSUPPORTED
    assert np.isfinite(to64(dev["x"])).all()


# dstate 64 and 256: the one-tile-per-CTA output kernel (2) beside the
# others, every candidate against the oracle
@pytest.mark.parametrize("S", [64, 256])
def test_candidates_other_dstate(ssd, S):
    w = W.Workload(f"bf16_plans_S{S}", 1, 600, 6, 64, S, 2, 256, "bf16", True)
    inp = make(w)
    ref = oracle_run(w, inp)
    dev = device_inputs(inp)
    d = ssd.dims_of(dev["x"], dev["B"], w.chunk)
    cands = ssd.plan_candidates(d)
    assert any(p["scan_kernel"] == 2 for p in cands)
    assert all(p["scan_kernel"] != 1 for p in cands) or S == 64
    for p in cands:
        y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"], plan=p)
        check_io(to64(y), ref["y"], "bf16", f"y {p}")
        check_io(to64(fin), ref["final_state"], "bf16", f"final_state {p}")
