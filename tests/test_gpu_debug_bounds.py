"""The debug-bounds build (libssd_gb300_debug.so, compiled with
SSD_DEBUG_BOUNDS): every plain global load and store of the kernels checks
its index against its buffer's extent, skips an access that falls outside
and reports SSD_ERR_BOUNDS through the call's error word.  Run on small
configurations through every entry point (both I/O types, every output
kernel of the bf16 launch plans, the step-wise calls, the decode step and
the backward pass):
no check may fire, and the results still match the oracle.

The status mapping itself is checked on the release library: a debug-bounds
code written into a workspace's error word reads back as SSD_ERR_BOUNDS, a
bounded-wait code as SSD_ERR_TIMEOUT.
"""
import ctypes

import pytest
import torch

from parity import check_io, device_inputs, forward_checked, make, oracle_run, to64

pytestmark = pytest.mark.gpu

from mamba_ssd_forward_gb300 import inputs as W  # noqa: E402


@pytest.fixture(scope="module")
def ssd_debug():
    """The package bound to the debug-bounds library for the module's tests,
    the release library restored afterwards."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from mamba_ssd_forward_gb300 import _abi, build
    build.build()
    oracle.build()
    path = build.build_debug()
    import mamba_ssd_forward_gb300 as m
    release = _abi.load()
    _abi._lib = _abi.load(path)
    try:
        yield m
    finally:
        _abi._lib = release


CASES = [
    W.Workload("dbg_bf16", 2, 300, 6, 64, 128, 2, 256, "bf16", True),
    W.Workload("dbg_bf16_S256_T128", 1, 333, 4, 64, 256, 1, 128, "bf16", True),
    W.Workload("dbg_bf16_P32_T64", 1, 200, 4, 32, 64, 2, 64, "bf16", False),
    W.Workload("dbg_fp32", 2, 300, 4, 32, 64, 2, 128, "fp32", True),
    W.Workload("dbg_fp32_T256", 1, 257, 2, 64, 128, 1, 256, "fp32", True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_every_plan_in_bounds(ssd_debug, w):
    inp = make(w, seed=8)
    dev = device_inputs(inp)
    ref = oracle_run(w, inp)
    plans = [None]
    if w.dtype == "bf16":
        d = ssd_debug.dims_of(dev["x"], dev["B"], w.chunk)
        seen = set()
        for p in ssd_debug.plan_candidates(d):
            key = p["scan_kernel"]
            if key not in seen:  # one plan per output kernel
                seen.add(key)
                plans.append(p)
    for plan in plans:
        y, fin = forward_checked(ssd_debug, dev, w.chunk, h0=dev["h0"], plan=plan)
        check_io(to64(y), ref["y"], w.dtype, f"{w.name} y plan={plan}")
        check_io(to64(fin), ref["final_state"], w.dtype, f"{w.name} final plan={plan}")


@pytest.mark.parametrize("w", CASES[:1] + CASES[3:4], ids=lambda w: w.name)
def test_steps_and_decode_in_bounds(ssd_debug, w):
    inp = make(w, seed=9)
    dev = device_inputs(inp)
    T = w.chunk
    G = ssd_debug.chunk_cumsum(dev["dt"], dev["A"], T, headdim=w.headdim, dstate=w.dstate)
    dst = ssd_debug.chunk_state(dev["x"], dev["B"], dev["dt"], G, T)
    sts, fin = ssd_debug.state_passing(dst, G, dev["h0"], chunk=T, seqlen=w.seqlen,
                                       ngroups=w.ngroups)
    y = ssd_debug.chunk_scan(dev["x"], dev["B"], dev["C"], dev["dt"], G, sts, dev["D"], chunk=T)
    state = dev["h0"].clone()
    ssd_debug.decode_step(dev["x"][:, 0].clone(), dev["dt"][:, 0].clone(), dev["A"],
                          dev["B"][:, 0].clone(), dev["C"][:, 0].clone(), dev["D"], state)
    ssd_debug.device_error()
    ref = oracle_run(w, inp)
    check_io(to64(y), ref["y"], w.dtype, "step-wise y")
    check_io(to64(fin), ref["final_state"], w.dtype, "step-wise final_state")


BWD_CASES = [
    W.Workload("dbg_bwd_S128_g2", 1, 300, 4, 64, 128, 2, 256, "fp32", True),
    W.Workload("dbg_bwd_S64_T64_hpg1", 2, 150, 2, 64, 64, 2, 64, "fp32", False),
    W.Workload("dbg_bwd_S256_T128", 1, 200, 2, 64, 256, 1, 128, "fp32", True),
]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: w.name)
def test_backward_in_bounds(ssd_debug, w):
    """ssd_backward (all eight launches) with every check compiled in: no
    check fires and every gradient still matches the oracle's adjoint."""
    import oracle
    inp = make(w, seed=10)
    dev = device_inputs(inp)
    g = torch.Generator(device="cpu")
    g.manual_seed(10)
    gy = torch.randn(inp["x"].shape, generator=g)
    gfinal = torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g)
    ws = ssd_debug.new_workspace(
        ssd_debug.backward_workspace_size(dev["x"], dev["B"], w.chunk), "cuda")
    out = ssd_debug.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                             dev["h0"], gy.cuda(), gfinal.cuda(), chunk=w.chunk, workspace=ws)
    ssd_debug.workspace_error(ws)
    ref = oracle.backward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                          inp["h0"], gy.double().numpy(), gfinal.double().numpy())
    for n in ("dx", "ddt", "dA", "dB", "dC", "dD", "dh0"):
        check_io(to64(out[n]), ref[n], "fp32", f"{w.name} {n}")


def test_error_codes_map_to_statuses():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_forward_gb300 import _abi, build
    import mamba_ssd_forward_gb300 as m
    build.build()
    lib = _abi.load()
    ws = m.new_workspace(4096, "cuda")
    h = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for code, status in ((2001, _abi.SSD_ERR_BOUNDS), (150, _abi.SSD_ERR_TIMEOUT), (0, _abi.SSD_OK)):
        ws[:4].view(torch.int32).fill_(code)
        torch.cuda.synchronize()
        assert lib.ssd_workspace_error(ctypes.c_void_p(ws.data_ptr()), h) == status
        assert int(ws[:4].view(torch.int32).item()) == 0  # read and cleared
