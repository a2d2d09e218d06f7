"""The backward pass (ssd_backward, fp32 I/O) against the oracle's adjoint
recurrence, which is pinned to finite differences of the forward
recurrence: dx, ddt, dA, dB, dC, dD and dh0 for a loss
L = <gy, y> + <gfinal, final_state> with seeded gy and gfinal.  Cases: every
supported dstate, chunks of 64 (the step-kernel forward), 128 and 256,
ragged last chunks, one token, several heads per group (dB, dC summed over
heads) and one (written directly), with and without h0, gfinal and D,
chunks steep enough to underflow their decay, repeated calls (fixed
summation order: the same bits), and the full-size shapes the bench times,
checked on one group of one batch."""
import pytest
import torch

from parity import check_io, device_inputs, make, rel_l2, to64

pytestmark = pytest.mark.gpu

from mamba_ssd_forward_gb300 import inputs as W  # noqa: E402


@pytest.fixture(scope="module")
def ssd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mamba_ssd_forward_gb300 import build
    build.build()
    import mamba_ssd_forward_gb300 as m
    return m


CASES = [
    # name, b, L, nh, P, S, ng, T, dtype, h0
    W.Workload("bwd_S128_T256", 2, 1300, 8, 64, 128, 1, 256, "fp32", True),
    W.Workload("bwd_S64_T128_g2_hpg3", 1, 515, 6, 64, 64, 2, 128, "fp32", False),
    W.Workload("bwd_S256_T256", 1, 700, 4, 64, 256, 1, 256, "fp32", True),
    W.Workload("bwd_S128_T64_g2", 1, 333, 4, 64, 128, 2, 64, "fp32", True),
    W.Workload("bwd_S64_T256_hpg1", 2, 600, 4, 64, 64, 4, 256, "fp32", True),
    W.Workload("bwd_one_token", 1, 1, 2, 64, 128, 1, 256, "fp32", True),
    W.Workload("bwd_S256_T128_g2", 1, 400, 4, 64, 256, 2, 128, "fp32", False),
]

NAMES = ("dx", "ddt", "dA", "dB", "dC", "dD", "dh0")


def grads_in(w, seed):
    """Seeded dL/dy and dL/dfinal_state, fp32 values held in float64 on the
    CPU (the library and the oracle see the same numbers)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 + seed)
    gy = torch.randn((w.batch, w.seqlen, w.nheads, w.headdim), generator=g, dtype=torch.float64)
    gfinal = torch.randn((w.batch, w.nheads, w.headdim, w.dstate), generator=g,
                         dtype=torch.float64)
    return gy.float().double(), gfinal.float().double()


def run(ssd, w, inp, gy, gfinal):
    dev = device_inputs(inp)
    gyd = gy.float().cuda().contiguous()
    gfd = None if gfinal is None else gfinal.float().cuda().contiguous()
    ws = ssd.new_workspace(ssd.backward_workspace_size(dev["x"], dev["B"], w.chunk), "cuda")
    out = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                       gyd, gfd, chunk=w.chunk, workspace=ws)
    ssd.workspace_error(ws)
    return out


def reference(inp, gy, gfinal):
    import oracle
    return oracle.backward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                           inp["h0"], gy.numpy(), None if gfinal is None else gfinal.numpy())


def compare(out, ref, what):
    for n in NAMES:
        check_io(to64(out[n]), ref[n], "fp32", f"{what} {n}")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_matches_the_adjoint(ssd, w):
    inp = make(w, seed=31)
    gy, gfinal = grads_in(w, 31)
    out = run(ssd, w, inp, gy, gfinal)
    compare(out, reference(inp, gy, gfinal), w.name)


NEAR_FP32 = [CASES[0], CASES[1], CASES[2], CASES[3]]


@pytest.mark.parametrize("w", NEAR_FP32, ids=lambda w: w.name)
def test_backward_near_fp32(ssd, w):
    """The GEMM-shaped products (the chunks' jump terms and the state terms
    of every token) run on the tensor cores with each fp32 operand split
    into a TF32 high part and its remainder (three products per fp32 one,
    about 2^-21 relative error each); the rest in fp32.  Every gradient
    stays within 5e-5 relative L2 of the float64 oracle (measured: 1e-6 to
    6e-6).  Plain TF32 products would leave dx near 4e-4 and dA at 5e-3 or
    more, far outside this bound."""
    inp = make(w, seed=31)
    gy, gfinal = grads_in(w, 31)
    out = run(ssd, w, inp, gy, gfinal)
    ref = reference(inp, gy, gfinal)
    for n in NAMES:
        r = rel_l2(to64(out[n]), ref[n])
        assert r <= 5e-5, f"{w.name} {n}: relative L2 {r:.3e}"


def test_backward_without_D_and_gfinal(ssd):
    """D = None (no skip term; dD is still sum gy . x) and gfinal = None."""
    w = W.Workload("bwd_noD", 1, 520, 4, 64, 128, 1, 256, "fp32", True)
    inp = make(w, seed=32)
    inp["D"] = None
    gy, _ = grads_in(w, 32)
    out = run(ssd, w, inp, gy, None)
    compare(out, reference(inp, gy, None), "no D, no gfinal")


def test_backward_steep_chunks(ssd):
    """Heads 0 and 1 decay by far more than 2^-180 within a chunk: every
    factor exp2(G_s - G_t) the backward forms has a non-positive exponent,
    so these only underflow to zero, as the exact values do."""
    w = W.Workload("bwd_steep", 1, 768, 4, 64, 128, 1, 256, "fp32", True)
    inp = make(w, seed=33)
    A = inp["A"].clone()
    A[0] = A[1] = -16.0
    dt = inp["dt"].clone()
    dt[0, :, 0] = 0.5
    dt[0, 300:, 1] = 0.1
    inp["A"], inp["dt"] = A, dt
    gy, gfinal = grads_in(w, 33)
    out = run(ssd, w, inp, gy, gfinal)
    compare(out, reference(inp, gy, gfinal), "steep")


REPEAT = [W.Workload("bwd_repeat", 2, 1024, 8, 64, 64, 2, 256, "fp32", True),
          # the long-context layer's group shape on a shorter sequence: the
          # GEMM kernel's CTAs each take several tiles through one pipeline
          W.Workload("bwd_repeat_S256_g8", 1, 2048, 48, 64, 256, 8, 256, "fp32", True)]


@pytest.mark.parametrize("w", REPEAT, ids=lambda w: w.name)
def test_backward_is_deterministic(ssd, w):
    """dB, dC, dA and dD are sums in a fixed order, and every GEMM tile is
    computed by one CTA in a fixed order: repeated calls on the same inputs
    give the same bits."""
    inp = make(w, seed=34)
    gy, gfinal = grads_in(w, 34)
    first = run(ssd, w, inp, gy, gfinal)
    for _ in range(2):
        again = run(ssd, w, inp, gy, gfinal)
        for n in NAMES:
            assert torch.equal(first[n], again[n]), n


def test_backward_rejects_unsupported(ssd):
    w = W.Workload("bwd_P32", 1, 256, 2, 32, 128, 1, 256, "fp32", False)
    inp = device_inputs(make(w, seed=0))
    assert ssd.backward_workspace_size(inp["x"], inp["B"], 256) == 0
    with pytest.raises(ssd.SsdError):
        ssd.backward(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], None,
                     torch.zeros_like(inp["x"]), None, chunk=256)


BF16 = [
    W.Workload("bwd_bf16_S128_T256_g2", 1, 700, 8, 64, 128, 2, 256, "bf16", True),
    W.Workload("bwd_bf16_S64_T128_hpg1", 2, 333, 4, 64, 64, 4, 128, "bf16", False),
    W.Workload("bwd_bf16_S256_T256", 1, 520, 4, 64, 256, 1, 256, "bf16", True),
]


@pytest.mark.parametrize("w", BF16, ids=lambda w: w.name)
def test_backward_bf16_io(ssd, w):
    """bf16 I/O: the same fp32 computation on the bf16 inputs (gy rounded to
    bf16 as well), dx, ddt, dB, dC rounded to bf16 at the end and held to
    the bf16 bound; dA, dD, dh0 stay fp32 and keep the fp32 bound."""
    inp = make(w, seed=36)
    gy, gfinal = grads_in(w, 36)
    gy = gy.to(torch.bfloat16)
    dev = device_inputs(inp)
    ws = ssd.new_workspace(ssd.backward_workspace_size(dev["x"], dev["B"], w.chunk), "cuda")
    out = ssd.backward(dev["x"], dev["dt"], dev["A"], dev["B"], dev["C"], dev["D"], dev["h0"],
                       gy.cuda(), gfinal.float().cuda(), chunk=w.chunk, workspace=ws)
    ssd.workspace_error(ws)
    ref = reference(inp, gy.double(), gfinal)
    for n in ("dx", "ddt", "dB", "dC"):
        assert out[n].dtype == torch.bfloat16
        check_io(to64(out[n]), ref[n], "bf16", f"{w.name} {n}")
    for n in ("dA", "dD", "dh0"):
        check_io(to64(out[n]), ref[n], "fp32", f"{w.name} {n}")


FULL = [W.LONG_32K.with_(name=W.LONG_32K.name.replace("bf16", "fp32"), dtype="fp32"),
        W.Workload("sweep_fp32_S128_L16384_T256", 2, 16384, 32, 64, 128, 1, 256, "fp32", True)]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_backward_full_size_sampled(ssd, w):
    """The full-size shapes the bench times (the long-context layer in fp32
    and a sweep shape), in the bench's launch configuration: every output
    of one group of one batch -- dx, ddt, dA, dD, dh0 of its heads and the
    group's dB, dC (sums over exactly those heads) -- against the oracle's
    chunked backward on that slice (pinned to the adjoint recurrence)."""
    import oracle
    inp = make(w, seed=35)
    gy, gfinal = grads_in(w, 35)
    out = run(ssd, w, inp, gy, gfinal)
    hpg = w.nheads // w.ngroups
    bi, g = w.batch - 1, w.ngroups // 2
    hs = slice(g * hpg, (g + 1) * hpg)
    sl = lambda t: None if t is None else t[bi:bi + 1, :, hs]
    ref = oracle.backward_chunked(
        sl(inp["x"]), sl(inp["dt"]), inp["A"][hs], inp["B"][bi:bi + 1, :, g:g + 1],
        inp["C"][bi:bi + 1, :, g:g + 1], inp["D"][hs],
        None if inp["h0"] is None else inp["h0"][bi:bi + 1, hs], sl(gy).numpy(),
        gfinal[bi:bi + 1, hs].numpy(), chunk=w.chunk)
    got = {"dx": out["dx"][bi:bi + 1, :, hs], "ddt": out["ddt"][bi:bi + 1, :, hs],
           "dB": out["dB"][bi:bi + 1, :, g:g + 1], "dC": out["dC"][bi:bi + 1, :, g:g + 1],
           "dh0": out["dh0"][bi:bi + 1, hs]}
    for n, v in got.items():
        check_io(to64(v), ref[n], "fp32", f"{w.name} {n}")
    if w.batch == 1:  # dA and dD sum over the batch
        check_io(to64(out["dA"][hs]), ref["dA"], "fp32", f"{w.name} dA")
        check_io(to64(out["dD"][hs]), ref["dD"], "fp32", f"{w.name} dD")


def test_autograd_function(ssd):
    """ssd.ssd() under torch.autograd: the gradients of a loss
    <gy, y> + <gfinal, final_state> reach every input and match the oracle's
    adjoint recurrence; inputs that do not require grad get none."""
    w = W.Workload("bwd_autograd", 1, 400, 4, 64, 64, 2, 128, "fp32", True)
    inp = make(w, seed=37)
    gy, gfinal = grads_in(w, 37)
    dev = device_inputs(inp)
    leaves = {k: dev[k].clone().requires_grad_(k != "D") for k in
              ("x", "dt", "A", "B", "C", "D", "h0")}
    y, fin = ssd.ssd(leaves["x"], leaves["dt"], leaves["A"], leaves["B"], leaves["C"],
                     leaves["D"], leaves["h0"], chunk=w.chunk)
    loss = (y * gy.float().cuda()).sum() + (fin * gfinal.float().cuda()).sum()
    loss.backward()
    ref = reference(inp, gy, gfinal)
    names = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "h0": "dh0"}
    for k, n in names.items():
        check_io(to64(leaves[k].grad), ref[n], "fp32", f"autograd {n}")
    assert leaves["D"].grad is None
