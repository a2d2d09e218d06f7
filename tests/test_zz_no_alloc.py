"""ssd_forward_noalloc against ssd_forward on the GPU.

The no-allocation entry point runs the forward pass with its workspace in the
library's fixed scratch array.  It must give what ssd_forward gives (with a
caller workspace) on the same inputs, within the parity tolerances of
tests/parity.py, on two calls in a row: the second call reuses the array the
first left dirty, which checks that nothing in it has to start at zero.  The
file is named to be collected last, so it also runs after every other GPU
test in the same process.
"""
import ctypes

import numpy as np
import pytest
import torch

from parity import check_io, device_inputs, make, to64
from mamba_ssd_forward_gb300 import inputs as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_forward_gb300 import _abi, build
    build.build()
    return _abi.load()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _run(lib, w, dev, noalloc, ws=None):
    from mamba_ssd_forward_gb300 import _abi
    d = _abi.SsdDims(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk)
    io = _abi.SSD_BF16 if w.dtype == "bf16" else _abi.SSD_F32
    y = torch.full_like(dev["x"], float("nan"))
    fin = torch.full((w.batch, w.nheads, w.headdim, w.dstate), float("nan"),
                     dtype=torch.float32, device="cuda")
    ins = [_vp(dev[k]) for k in ("x", "dt", "A", "B", "C", "D", "h0")]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        rc = lib.ssd_forward_noalloc(ctypes.byref(d), io, *ins, _vp(y), _vp(fin), stream)
    else:
        rc = lib.ssd_forward(ctypes.byref(d), io, *ins, _vp(y), _vp(fin), _vp(ws), ws.numel(),
                             stream)
    torch.cuda.synchronize()
    assert rc == _abi.SSD_OK, lib.ssd_status_string(rc).decode()
    # the no-allocation call reports to the library-wide error word, the
    # other to its workspace's word
    if noalloc:
        assert lib.ssd_device_error(stream) == _abi.SSD_OK
    else:
        assert lib.ssd_workspace_error(_vp(ws), stream) == _abi.SSD_OK
    return to64(y), to64(fin)


CASES = [
    W.MAMBA2_130M,
    W.TINY,
    W.Workload("noalloc_bf16_ragged_h0", 2, 777, 6, 64, 128, 2, 256, "bf16", True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_forward_twice(lib, w):
    from mamba_ssd_forward_gb300 import _abi
    d = _abi.SsdDims(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk)
    io = _abi.SSD_BF16 if w.dtype == "bf16" else _abi.SSD_F32
    need = lib.ssd_forward_workspace_size(ctypes.byref(d), io)
    assert 0 < need <= _abi.SSD_NOALLOC_SCRATCH_BYTES
    dev = device_inputs(make(w, seed=3))
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws[:_abi.SSD_WS_HEADER_BYTES].zero_()  # a new workspace's error word starts clear
    y_ref, f_ref = _run(lib, w, dev, noalloc=False, ws=ws)
    for call in (1, 2):
        y, f = _run(lib, w, dev, noalloc=True)
        assert np.isfinite(y).all() and np.isfinite(f).all()
        check_io(y, y_ref, w.dtype, f"{w.name} noalloc call {call} y")
        check_io(f, f_ref, w.dtype, f"{w.name} noalloc call {call} final_state")


def test_noalloc_rejects_oversize(lib):
    from mamba_ssd_forward_gb300 import _abi
    w = W.MAMBA2_2P7B
    d = _abi.SsdDims(w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, w.chunk)
    assert lib.ssd_forward_workspace_size(ctypes.byref(d), _abi.SSD_BF16) > \
        _abi.SSD_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = lib.ssd_forward_noalloc(ctypes.byref(d), _abi.SSD_BF16, fake, fake, fake, fake, fake,
                                 None, None, fake, None, None)
    assert rc == _abi.SSD_ERR_UNSUPPORTED
