"""Shared helpers of the GPU parity tests: tolerances and sampled oracle runs.

Tolerances (relative L2 over the compared elements):
  fp32 I/O (TF32 tensor-core products): rel_l2 <= 2e-3 and
      max|got - ref| <= 1e-2 * max|ref|
  bf16 I/O (bf16 operands, fp32 accumulation): rel_l2 <= 1e-2
The same bounds apply to the final state, and to y - D x (the skip term is
O(1) and could hide an error in the state-space part).
"""
import numpy as np
import torch

import oracle
from mamba_ssd_forward_gb300 import inputs as ssd_inputs

LN2 = float(np.log(2.0))
LOG2E = 1.0 / LN2


def to64(t):
    return t.detach().to("cpu").double().numpy()


def rel_l2(got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def check_io(got, ref, dtype, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    if dtype == "fp32":
        m = float(np.abs(got - ref).max()) if got.size else 0.0
        lim = 1e-2 * float(np.abs(ref).max()) if ref.size else 0.0
        assert r <= 2e-3 and m <= lim, f"{what}: rel_l2 {r:.3e} max_abs {m:.3e} (limit {lim:.3e})"
    else:
        assert r <= 1e-2, f"{what}: rel_l2 {r:.3e}"
    return r


def sample_pairs(w, n=4):
    """A few (batch, head) pairs spread over the tensor, as flat indices."""
    total = w.batch * w.nheads
    if total <= n:
        return list(range(total))
    cand = [0, total - 1, total // 2, (w.nheads // 3) + (w.batch - 1) * w.nheads]
    out = []
    for c in cand:
        if c not in out and 0 <= c < total:
            out.append(c)
    return out[:n]


def device_inputs(inp, device="cuda"):
    return {k: (None if v is None else v.to(device).contiguous()) for k, v in inp.items()}


def oracle_run(w, inp, bh=None, want=("y", "final_state")):
    return oracle.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                             inp["h0"], chunk=w.chunk, bh=bh, want=want)


def make(w, seed=0):
    return ssd_inputs.make_inputs(w, seed)


def forward_checked(ssd, dev, chunk, h0=None, plan=None, workspace=None, y=None,
                    final_state=None):
    """ssd.forward on device inputs `dev` with a workspace of its own (or the
    given one), then the workspace's error word must be clear: no bounded
    device-side wait of the call gave up."""
    if workspace is None:
        workspace = ssd.new_workspace(ssd.workspace_size(dev["x"], dev["B"], chunk),
                                      dev["x"].device)
    out = ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], h0,
                      chunk=chunk, workspace=workspace, y=y, final_state=final_state, plan=plan)
    ssd.workspace_error(workspace)
    return out
