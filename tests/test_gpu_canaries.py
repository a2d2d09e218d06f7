"""Canaries: every output buffer of the C ABI sits between two guard regions
(NaN for floating-point outputs, a byte pattern after the forward's
workspace) that the call must leave untouched, while the output itself
matches the oracle.  Covers the forward pass in both I/O types (y, the final
state and the workspace holding G, the jump terms and the start states),
each step-wise entry point (G, dstates, states, the final state, y) and the
decode step (y and the state).  A kernel writing past either end of a
buffer, or leaving part of it unwritten (a NaN left over), fails here.
"""
import numpy as np
import pytest
import torch

from parity import LN2, check_io, device_inputs, make, oracle_run, rel_l2, to64

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements of guard before and after each output


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


class Guarded:
    """A tensor of `shape` inside a NaN-filled buffer with GUARD elements on
    each side (the offset keeps the 16-byte alignment the library needs)."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.full((GUARD + n + GUARD,), float("nan"), dtype=dtype, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        assert torch.isnan(self.buf[:GUARD]).all(), f"{what}: written before the start"
        assert torch.isnan(self.buf[-GUARD:]).all(), f"{what}: written past the end"
        assert torch.isfinite(self.t).all(), f"{what}: elements left unwritten or non-finite"


CASES = [
    W.Workload("canary_bf16", 2, 300, 6, 64, 128, 2, 256, "bf16", True),
    W.Workload("canary_bf16_S256_T128", 1, 333, 4, 64, 256, 1, 128, "bf16", True),
    W.Workload("canary_fp32", 2, 300, 4, 32, 64, 2, 128, "fp32", True),
    W.Workload("canary_fp32_T64", 1, 130, 3, 48, 80, 3, 64, "fp32", False),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_forward_writes_inside_its_buffers(ssd, w):
    inp = make(w, seed=3)
    dev = device_inputs(inp)
    io = dev["x"].dtype
    y = Guarded(tuple(dev["x"].shape), io)
    fin = Guarded((w.batch, w.nheads, w.headdim, w.dstate), torch.float32)
    need = ssd.workspace_size(dev["x"], dev["B"], w.chunk)
    wsbuf = ssd.new_workspace(need + 65536, "cuda")
    wsbuf[need:].fill_(0xA5)
    ws = wsbuf[:need]
    ssd.forward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                chunk=w.chunk, workspace=ws, y=y.t, final_state=fin.t)
    ssd.workspace_error(ws)
    y.check("forward y")
    fin.check("forward final_state")
    assert bool((wsbuf[need:] == 0xA5).all()), "forward: written past the workspace"
    ref = oracle_run(w, inp)
    check_io(to64(y.t), ref["y"], w.dtype, "forward y")
    check_io(to64(fin.t), ref["final_state"], w.dtype, "forward final_state")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_steps_write_inside_their_buffers(ssd, w):
    inp = make(w, seed=4)
    dev = device_inputs(inp)
    io = dev["x"].dtype
    T = w.chunk
    nc = -(-w.seqlen // T)
    ref = oracle_run(w, inp, want=("y", "final_state", "states", "dstates", "G"))

    G = Guarded((w.batch, w.nheads, nc * T), torch.float32)
    ssd.chunk_cumsum(dev["dt"], dev["A"], T, headdim=w.headdim, dstate=w.dstate, out=G.t)
    G.check("chunk_cumsum G")
    # the oracle's G covers the real tokens; padding tokens repeat the last
    Gt = to64(G.t).reshape(w.batch, w.nheads, nc, T) * LN2
    Gr = ref["G"].reshape(w.batch, w.nheads, nc, T)
    np.testing.assert_allclose(Gt, Gr, rtol=1e-5, atol=1e-6)

    dst = Guarded((w.batch, w.nheads, nc, w.headdim, w.dstate), torch.float32)
    ssd.chunk_state(dev["x"], dev["B"], dev["dt"], G.t, T, out=dst.t)
    dst.check("chunk_state dstates")
    check_io(to64(dst.t), ref["dstates"], w.dtype, "chunk_state dstates")

    sts = Guarded((w.batch, w.nheads, nc, w.headdim, w.dstate), torch.float32)
    fin = Guarded((w.batch, w.nheads, w.headdim, w.dstate), torch.float32)
    ssd.state_passing(dst.t, G.t, dev["h0"], chunk=T, seqlen=w.seqlen, ngroups=w.ngroups,
                      states=sts.t, final_state=fin.t)
    sts.check("state_passing states")
    fin.check("state_passing final_state")
    check_io(to64(sts.t), ref["states"], w.dtype, "state_passing states")
    check_io(to64(fin.t), ref["final_state"], w.dtype, "state_passing final_state")

    y = Guarded(tuple(dev["x"].shape), io)
    ssd.chunk_scan(dev["x"], dev["B"], dev["C"], dev["dt"], G.t, sts.t, dev["D"], chunk=T,
                   y=y.t)
    y.check("chunk_scan y")
    check_io(to64(y.t), ref["y"], w.dtype, "chunk_scan y")
    ssd.device_error()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_writes_inside_its_buffers(ssd, dtype):
    import oracle
    w = W.Workload("canary_dec", 3, 1, 6, 32, 64, 3, 64, dtype, True)
    inp = make(w, seed=6)
    dev = device_inputs(inp)
    io = dev["x"].dtype
    st = Guarded((w.batch, w.nheads, w.headdim, w.dstate), torch.float32)
    st.t.copy_(dev["h0"])
    y = Guarded((w.batch, w.nheads, w.headdim), io)
    x1, dt1 = dev["x"][:, 0].clone(), dev["dt"][:, 0].clone()
    B1, C1 = dev["B"][:, 0].clone(), dev["C"][:, 0].clone()
    ssd.decode_step(x1, dt1, dev["A"], B1, C1, dev["D"], st.t, y=y.t)
    y.check("decode y")
    st.check("decode state")
    y_ref, h = oracle.decode_step(to64(inp["x"][:, 0]), to64(inp["dt"][:, 0]), to64(inp["A"]),
                                  to64(inp["B"][:, 0]), to64(inp["C"][:, 0]), to64(inp["D"]),
                                  to64(inp["h0"]))
    check_io(to64(y.t), y_ref, dtype, "decode y")
    assert rel_l2(to64(st.t), h) < 1e-5
    ssd.device_error()
