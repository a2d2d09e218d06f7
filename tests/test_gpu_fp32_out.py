"""The fp32 kernels (fwd_chunk_state_tf32: the chunk jump terms with every
landed box transposed in place for kind::tf32; fwd_out_tf32: the masked
C B^T of a 128-row tile shared by a slice of heads, the in-chunk decay
factored about one anchor per chunk and head, an exact per-element path for
steep chunks) through ssd_forward with fp32 I/O, against the oracle: every
supported
dstate and chunk size, ragged last chunks, several groups, with and without
h0, and chunks steep enough to need the exact path (alone and beside
ordinary heads of the same CTA).  The relative error of y - D x is checked
as well, so that the skip term cannot hide an error in the state-space
part."""
import pytest
import torch

from parity import LOG2E, check_io, device_inputs, forward_checked, make, oracle_run, to64

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


CASES = [
    W.Workload("fp32_S128_T256", 2, 1300, 8, 64, 128, 1, 256, "fp32", True),
    W.Workload("fp32_S64_T256_g2", 1, 900, 6, 64, 64, 2, 256, "fp32", False),
    W.Workload("fp32_S32_T128", 2, 700, 4, 64, 32, 1, 128, "fp32", True),
    W.Workload("fp32_S96_T128_g3", 1, 515, 6, 64, 96, 3, 128, "fp32", True),
    # the second row tile of the last chunk lies past the sequence
    W.Workload("fp32_short_tail", 1, 600, 4, 64, 128, 1, 256, "fp32", True),
    W.Workload("fp32_one_token", 1, 1, 2, 64, 128, 1, 256, "fp32", True),
    # the tf32 chunk-jump kernel with two slices of S and one head per item
    # (three heads per group), beside the step output kernel
    W.Workload("fp32_S256_hpg3", 1, 700, 3, 64, 256, 1, 256, "fp32", True),
    W.Workload("fp32_S256_T128_g2", 2, 333, 4, 64, 256, 2, 128, "fp32", False),
]


def check(w, inp, y, fin, what):
    ref = oracle_run(w, inp)
    y64 = to64(y)
    Dx = to64(inp["D"])[None, None, :, None] * to64(inp["x"])
    check_io(y64, ref["y"], "fp32", f"{what} y")
    check_io(y64 - Dx, ref["y"] - Dx, "fp32", f"{what} y - D x")
    check_io(to64(fin), ref["final_state"], "fp32", f"{what} final_state")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp32_forward_matches_the_oracle(ssd, w):
    inp = make(w, seed=21)
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
    check(w, inp, y, fin, w.name)


@pytest.mark.parametrize("T", [128, 256])
def test_fp32_steep_chunks(ssd, T):
    """Heads 0 and 1 decay by far more than 2^-180 within a chunk (every
    chunk of head 1, every other chunk of head 0) and take the exact path;
    heads 2 and 3 keep the factored path in the same CTAs."""
    w = W.Workload(f"fp32_steep_T{T}", 1, 1024, 4, 64, 128, 1, T, "fp32", True)
    inp = make(w, seed=5)
    A = inp["A"].clone()
    A[0] = A[1] = -16.0
    dt = inp["dt"].double().clone()
    tok = torch.arange(w.seqlen)
    dt[0, (tok // T) % 2 == 1, 0] = 0.5
    dt[0, :, 1] = 0.1
    inp["A"], inp["dt"] = A, dt.to(inp["dt"].dtype)
    span = -(A.double()[None, None, :] * inp["dt"].double() * LOG2E)
    span = span.reshape(1, w.seqlen // T, T, w.nheads).sum(2)
    assert (span[..., :2] > 180).any() and (span[..., 2:] < 180).all()
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
    check(w, inp, y, fin, f"steep T={T}")


def test_fp32_zero_dt_tokens(ssd):
    """Tokens with dt = 0 contribute nothing and do not decay: their factor
    v_j is zero whatever the anchor, and the chunk keeps the factored path."""
    w = W.Workload("fp32_dt0", 1, 768, 4, 64, 128, 1, 256, "fp32", True)
    inp = make(w, seed=6)
    dt = inp["dt"].clone()
    dt[0, 100:300, :] = 0.0
    inp["dt"] = dt
    dev = device_inputs(inp)
    y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
    check(w, inp, y, fin, "dt = 0 span")


def test_fp32_forward_is_deterministic(ssd):
    """Many heads per CTA over many chunks (the sweep's shape at dstate 64):
    repeated calls give the same bits, and every call matches the oracle on
    sampled (batch, head) pairs."""
    from parity import sample_pairs
    w = W.Workload("fp32_repeat", 2, 4096, 32, 64, 64, 1, 256, "fp32", True)
    inp = make(w, seed=0)
    dev = device_inputs(inp)
    pairs = sample_pairs(w)
    ref = oracle_run(w, inp, bh=pairs)
    first = None
    for _ in range(4):
        y, fin = forward_checked(ssd, dev, w.chunk, h0=dev["h0"])
        if first is None:
            first = (y.clone(), fin.clone())
            y64 = to64(y)
            for pair in pairs:
                b, h = divmod(pair, w.nheads)
                check_io(y64[b, :, h], ref["y"][b, :, h], "fp32", f"y[b={b},h={h}]")
        else:
            assert torch.equal(y, first[0]) and torch.equal(fin, first[1])
