"""The bounded device-side waits: a wait that nothing satisfies gives up
after its limit, the host reads SSD_ERR_TIMEOUT, and the context stays
usable (a forward pass afterwards matches the oracle).  The wait is made to
run out by a barrier that nothing arrives on, with a 2 ms limit; no kernel
faults, traps or hangs."""
import ctypes

import pytest
import torch

from parity import check_io, device_inputs, make, oracle_run, to64

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


def test_wait_gives_up_and_context_recovers(ssd):
    from mamba_ssd_forward_gb300 import _abi
    lib = _abi.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ssd.device_error()  # nothing recorded before
    try:
        assert lib.ssd_selftest_bounded_wait(2_000_000, st) == _abi.SSD_OK
        with pytest.raises(_abi.SsdError) as e:
            ssd.device_error()
        assert e.value.code == _abi.SSD_ERR_TIMEOUT
    finally:
        lib.ssd_device_error(st)  # cleared whatever happened
    ssd.device_error()  # and stays clear
    w = W.Workload("after_timeout", 1, 300, 4, 64, 128, 1, 256, "bf16", True)
    inp = make(w)
    ref = oracle_run(w, inp)
    dev = device_inputs(inp)
    y, fin = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                         chunk=w.chunk)
    ssd.device_error()
    check_io(to64(y), ref["y"], "bf16", "y after a timed-out wait")
    check_io(to64(fin), ref["final_state"], "bf16", "final_state after a timed-out wait")
