"""The bounded device-side waits: a wait that nothing satisfies gives up
after its limit, the host reads SSD_ERR_TIMEOUT from the error word the wait
reported to, and the context stays usable (a forward pass afterwards matches
the oracle).  Each workspace has its own error word: a wait that gives up on
one stream, reporting to one workspace, leaves the word of a forward pass
running on another stream with another workspace clear.  The wait is made to
run out by a barrier that nothing arrives on, with a 2 ms limit; no kernel
faults, traps or hangs."""
import ctypes

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


CASE = W.Workload("after_timeout", 1, 300, 4, 64, 128, 1, 256, "bf16", True)


def _vp(t):
    return ctypes.c_void_p(t.data_ptr())


def test_library_word_gives_up_and_context_recovers(ssd):
    from mamba_ssd_forward_gb300 import _abi
    lib = _abi.load()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ssd.device_error()  # nothing recorded before
    try:
        assert lib.ssd_selftest_bounded_wait(2_000_000, None, st) == _abi.SSD_OK
        with pytest.raises(_abi.SsdError) as e:
            ssd.device_error()
        assert e.value.code == _abi.SSD_ERR_TIMEOUT
    finally:
        lib.ssd_device_error(st)  # cleared whatever happened
    ssd.device_error()  # and stays clear
    inp = make(CASE)
    ref = oracle_run(CASE, inp)
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, CASE.chunk, h0=dev["h0"])
    check_io(to64(y), ref["y"], "bf16", "y after a timed-out wait")
    check_io(to64(fin), ref["final_state"], "bf16", "final_state after a timed-out wait")


def test_workspace_words_are_independent(ssd):
    """A wait that gives up on stream 1, reporting to workspace 1, while a
    forward pass runs on stream 2 with workspace 2: only workspace 1 reads
    SSD_ERR_TIMEOUT, and the forward pass matches the oracle."""
    from mamba_ssd_forward_gb300 import _abi
    lib = _abi.load()
    inp = make(CASE)
    ref = oracle_run(CASE, inp)
    dev = device_inputs(inp)
    need = ssd.workspace_size(dev["x"], dev["B"], CASE.chunk)
    ws1, ws2 = ssd.new_workspace(need, "cuda"), ssd.new_workspace(need, "cuda")
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    h1, h2 = ctypes.c_void_p(s1.cuda_stream), ctypes.c_void_p(s2.cuda_stream)
    try:
        assert lib.ssd_selftest_bounded_wait(20_000_000, _vp(ws1), h1) == _abi.SSD_OK
        with torch.cuda.stream(s2):
            y, fin = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                                 dev["h0"], chunk=CASE.chunk, workspace=ws2)
        assert lib.ssd_workspace_error(_vp(ws2), h2) == _abi.SSD_OK
        assert lib.ssd_workspace_error(_vp(ws1), h1) == _abi.SSD_ERR_TIMEOUT
    finally:
        lib.ssd_workspace_error(_vp(ws1), h1)
    assert lib.ssd_workspace_error(_vp(ws1), h1) == _abi.SSD_OK  # cleared by the read
    assert lib.ssd_device_error(h1) == _abi.SSD_OK  # the library-wide word untouched
    check_io(to64(y), ref["y"], "bf16", "y beside a timed-out wait")
    check_io(to64(fin), ref["final_state"], "bf16", "final_state beside a timed-out wait")
