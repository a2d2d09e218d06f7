"""GPU tests of ssd_forward_host_overlapped: host buffers in and out, the
work cut into slices whose copies overlap the computation.  The results
must equal ssd_forward's on the device (same kernels, same chunking; slices
along the batch, or along whole chunks of tokens resuming from the previous
slice's final state) and the float64 oracle within the parity tolerances."""
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
    (W.Workload("ov_batch4_bf16", 4, 700, 8, 64, 128, 2, 256, "bf16", True), 4),
    (W.Workload("ov_batch3_slices2_fp32", 3, 300, 4, 32, 64, 1, 128, "fp32", True), 2),
    (W.Workload("ov_tokens_bf16", 1, 1500, 6, 64, 128, 3, 256, "bf16", True), 4),
    (W.Workload("ov_tokens_no_h0_bf16", 1, 777, 4, 64, 64, 1, 128, "bf16", False), 3),
    (W.Workload("ov_one_slice_bf16", 2, 400, 4, 64, 128, 1, 256, "bf16", True), 1),
]


@pytest.mark.parametrize("w,n", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_overlapped_matches_device_forward(ssd, w, n):
    import oracle
    inp = make(w, seed=4)
    dev = device_inputs(inp)
    y_dev, f_dev = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"],
                               dev["h0"], chunk=w.chunk)
    h = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    y = torch.full_like(h["x"], float("nan")).pin_memory()
    fin = torch.full((w.batch, w.nheads, w.headdim, w.dstate), float("nan")).pin_memory()
    ws = ssd.new_workspace(ssd.host_overlapped_workspace_size(h["x"], h["B"], w.chunk, n, True,
                                                              h["h0"] is not None, True),
                           "cuda")
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ssd.forward_host_overlapped(h["x"], h["dt"], h["A"], h["B"], h["C"], h["D"], h["h0"],
                                w.chunk, ws, y, fin, n_slices=n, h2d_stream=s_in,
                                d2h_stream=s_out)
    torch.cuda.current_stream().synchronize()
    ssd.workspace_error(ws)
    assert torch.isfinite(y.float()).all() and torch.isfinite(fin).all()
    assert rel_l2(to64(y), to64(y_dev)) < 1e-6
    assert rel_l2(to64(fin), to64(f_dev)) < 1e-6
    ref = oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                            inp["h0"], chunk=w.chunk)
    check_io(to64(y), ref["y"], w.dtype, f"{w.name} y")
    check_io(to64(fin), ref["final_state"], w.dtype, f"{w.name} final_state")
