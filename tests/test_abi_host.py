"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol include/ssd.h declares, and rejects bad arguments before launching
anything (so these run without a GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mamba_ssd_forward_gb300 import _abi, build
    build.build()
    return _abi.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"SSD_API\s+[\w\s\*]+?\b(\w+)\s*\(", src))
    return names


def test_header_declares_the_five_steps():
    names = declared_functions()
    for n in ("ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing",
              "ssd_chunk_scan", "ssd_forward", "ssd_forward_workspace_size",
              "ssd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from mamba_ssd_forward_gb300 import _abi
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(_abi.EXPORTS) == declared_functions()


def test_status_strings(lib):
    for code in range(6):
        s = lib.ssd_status_string(code).decode()
        assert s.startswith("SSD_") and "UNKNOWN" not in s
    assert lib.ssd_status_string(77).decode() == "SSD_ERR_UNKNOWN"


def dims(**kw):
    from mamba_ssd_forward_gb300 import _abi
    base = dict(batch=2, seqlen=1000, nheads=8, headdim=64, dstate=128, ngroups=2, chunk=256)
    base.update(kw)
    return _abi.SsdDims(**base)


def test_workspace_size(lib):
    d = dims()
    nc = 4
    hdr = 256  # SSD_WS_HEADER_BYTES: the call's error word
    # bf16: the per-chunk start states in bf16
    ws = lib.ssd_forward_workspace_size(ctypes.byref(d), 1)
    assert ws >= hdr + 2 * 2 * 8 * nc * 64 * 128
    assert ws % 256 == 0
    # fp32: G, the chunk jump terms and the states, fp32
    ws = lib.ssd_forward_workspace_size(ctypes.byref(d), 0)
    assert ws >= hdr + 4 * 2 * 8 * nc * 256 + 2 * 4 * 2 * 8 * nc * 64 * 128
    assert ws % 256 == 0
    assert lib.ssd_forward_workspace_size(ctypes.byref(d), 7) == 0
    assert lib.ssd_forward_workspace_size(None, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(ngroups=3), 1),            # nh % ng != 0
    (dict(batch=0), 1),
    (dict(seqlen=0), 1),
    (dict(headdim=48 + 1), 2),       # not a multiple of 16
    (dict(headdim=144), 2),          # > 128
    (dict(dstate=272), 2),           # > 256
    (dict(dstate=8), 2),
    (dict(chunk=96), 2),
    (dict(chunk=512), 2),
])
def test_rejects_bad_dims_before_launch(lib, kw, code):
    d = dims(**kw)
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), 1, fake, fake, fake, None) == code
    assert lib.ssd_forward_workspace_size(ctypes.byref(d), 1) == 0
    rc = lib.ssd_forward(ctypes.byref(d), 1, fake, fake, fake, fake, fake, None, None, fake,
                         None, fake, 1 << 40, None)
    assert rc == code


def test_rejects_null_and_misaligned_pointers(lib):
    d = dims()
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), 1, None, ok, ok, None) == 1
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), 1, bad, ok, ok, None) == 1
    assert lib.ssd_chunk_cumsum(ctypes.byref(d), 5, ok, ok, ok, None) == 1  # dtype
    assert lib.ssd_chunk_state(ctypes.byref(d), 1, ok, ok, ok, ok, None, None) == 1
    assert lib.ssd_state_passing(ctypes.byref(d), ok, ok, bad, ok, None, None) == 1
    assert lib.ssd_chunk_scan(ctypes.byref(d), 1, ok, ok, ok, ok, ok, ok, bad, ok, None) == 1
    ws = lib.ssd_forward_workspace_size(ctypes.byref(d), 1)
    # workspace too small, and workspace not 256-byte aligned
    assert lib.ssd_forward(ctypes.byref(d), 1, ok, ok, ok, ok, ok, None, None, ok, None,
                           ok, ws - 1, None) == 1
    assert lib.ssd_forward(ctypes.byref(d), 1, ok, ok, ok, ok, ok, None, None, ok, None,
                           ctypes.c_void_p((1 << 20) + 16), ws, None) == 1
    assert lib.ssd_chunk_cumsum(None, 1, ok, ok, ok, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    from mamba_ssd_forward_gb300 import _abi
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load(str(tmp_path / "nope.so"))


def test_product_path_never_touches_the_oracle():
    """The package and the CUDA sources do not import, load or name the
    oracle; the oracle does not import the package."""
    pkg = os.path.join(ROOT, "mamba_ssd_forward_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                for pat in (r"\bimport\s+oracle", r"\bfrom\s+oracle", r"ssd_oracle",
                            r"libssd_oracle"):
                    assert not re.search(pat, src), (fn, pat)
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith((".py", ".c")):
            src = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "mamba_ssd_forward_gb300" not in src, fn


def test_noalloc_limit_and_rejections(lib):
    """ssd_forward_noalloc: the header's scratch size matches the binding's,
    and oversize or invalid dims are rejected before any CUDA call (so this
    runs without a GPU)."""
    from mamba_ssd_forward_gb300 import _abi
    hdr = open(os.path.join(ROOT, "include", "ssd.h")).read()
    m = re.search(r"#define\s+SSD_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", hdr)
    assert m and int(m.group(1)) << int(m.group(2)) == _abi.SSD_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    big = dims(batch=2, seqlen=4096, nheads=80, ngroups=1)
    assert lib.ssd_forward_workspace_size(ctypes.byref(big), 1) > _abi.SSD_NOALLOC_SCRATCH_BYTES
    args = [fake, fake, fake, fake, fake, None, None, fake, None, None]
    assert lib.ssd_forward_noalloc(ctypes.byref(big), 1, *args) == _abi.SSD_ERR_UNSUPPORTED
    # pointers are checked before the size, with ssd_forward's codes
    null_x = [None] + args[1:]
    assert lib.ssd_forward_noalloc(ctypes.byref(big), 1, *null_x) == _abi.SSD_ERR_INVALID_ARG
    odd_y = args[:7] + [ctypes.c_void_p((1 << 20) + 4)] + args[8:]
    assert lib.ssd_forward_noalloc(ctypes.byref(big), 1, *odd_y) == _abi.SSD_ERR_INVALID_ARG
    assert lib.ssd_forward_noalloc(ctypes.byref(dims(ngroups=3)), 1, *args) == 1
    assert lib.ssd_forward_noalloc(ctypes.byref(dims(chunk=96)), 1, *args) == 2
    assert lib.ssd_forward_noalloc(ctypes.byref(dims()), 7, *args) == 1
    assert lib.ssd_forward_noalloc(None, 1, *args) == 1


def test_decode_step_rejections(lib):
    """ssd_decode_step validates before launching: seqlen must be 1, S a
    multiple of 4 up to 1024, nh a multiple of ng, pointers aligned."""
    from mamba_ssd_forward_gb300 import _abi
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    args = lambda st, y: [ok, ok, ok, ok, ok, None, st, y, None]  # noqa: E731
    d1 = dims(seqlen=1)
    assert lib.ssd_decode_step(ctypes.byref(dims(seqlen=2)), 1, *args(ok, ok)) == 1
    assert lib.ssd_decode_step(ctypes.byref(dims(seqlen=1, dstate=6)), 1, *args(ok, ok)) == 2
    assert lib.ssd_decode_step(ctypes.byref(dims(seqlen=1, dstate=1028)), 1, *args(ok, ok)) == 2
    assert lib.ssd_decode_step(ctypes.byref(dims(seqlen=1, ngroups=3)), 1, *args(ok, ok)) == 1
    assert lib.ssd_decode_step(ctypes.byref(d1), 1, *args(bad, ok)) == 1
    assert lib.ssd_decode_step(ctypes.byref(d1), 1, *args(ok, None)) == 1
    assert lib.ssd_decode_step(ctypes.byref(d1), 9, *args(ok, ok)) == 1
    assert lib.ssd_decode_step(None, 1, *args(ok, ok)) == 1
    assert _abi.SSD_OK == 0


def test_host_overlapped_sizes_and_rejections(lib):
    """ssd_forward_host_overlapped: a workspace size for both slicing modes,
    and bad arguments rejected before anything is enqueued."""
    d4 = dims(batch=4, seqlen=1000)
    d1 = dims(batch=1, seqlen=1000)
    for d in (d4, d1):
        for n in (1, 2, 4):
            assert lib.ssd_forward_host_overlapped_workspace_size(ctypes.byref(d), 1, 1, 1, 1, n) > 0
    assert lib.ssd_forward_host_overlapped_workspace_size(ctypes.byref(d4), 1, 1, 1, 1, 0) == 0
    assert lib.ssd_forward_host_overlapped_workspace_size(ctypes.byref(dims(chunk=96)), 1, 1, 1,
                                                          1, 2) == 0
    ok = ctypes.c_void_p(1 << 20)
    host = [ok] * 5 + [None, None, ok, None]
    ws = lib.ssd_forward_host_overlapped_workspace_size(ctypes.byref(d4), 1, 0, 0, 0, 2)
    assert lib.ssd_forward_host_overlapped(ctypes.byref(d4), 1, *host, ok, ws, 0, None, None,
                                           None, None) == 1  # n_slices
    assert lib.ssd_forward_host_overlapped(ctypes.byref(d4), 1, *host, ok, ws - 256, 2, None,
                                           None, None, None) == 1  # workspace too small
    assert lib.ssd_forward_host_overlapped(ctypes.byref(dims(headdim=144)), 1, *host, ok, ws, 2,
                                           None, None, None, None) == 2
    # a plan that is not a candidate, rejected before any copy is enqueued
    from mamba_ssd_forward_gb300 import _abi
    bad = _abi.SsdPlan(3, 1, 1, 3)
    assert lib.ssd_forward_host_overlapped(ctypes.byref(d4), 1, *host, ok, ws, 2,
                                           ctypes.byref(bad), None, None, None) == 1
    # any plan with fp32 I/O
    good = _abi.SsdPlan(**__import__("mamba_ssd_forward_gb300").default_plan(d4))
    ws32 = lib.ssd_forward_host_overlapped_workspace_size(ctypes.byref(d4), 0, 0, 0, 0, 2)
    assert lib.ssd_forward_host_overlapped(ctypes.byref(d4), 0, *host, ok, ws32, 2,
                                           ctypes.byref(good), None, None, None) == 1


def _dims(b, L, nh, P, S, ng, T):
    from mamba_ssd_forward_gb300 import _abi
    return _abi.SsdDims(b, L, nh, P, S, ng, T)


@pytest.mark.parametrize("shape", [
    (4, 2048, 24, 64, 128, 1, 256),   # 130M-like layer
    (2, 4096, 80, 64, 128, 1, 256),   # 2.7B-like layer
    (1, 32768, 48, 64, 256, 8, 256),  # long context, S = 256
    (2, 500, 12, 32, 64, 3, 128),     # P = 32: only the per-slice output kernel
    (1, 300, 2, 128, 256, 1, 256),    # largest P and S
])
def test_plan_candidates_are_valid_and_hold_the_default(lib, shape):
    import mamba_ssd_forward_gb300 as m
    b, L, nh, P, S, ng, T = shape
    d = _dims(*shape)
    cands = m.plan_candidates(d)
    assert cands
    hpg = nh // ng
    chunk_kernel_ok = P == 64 and S in (64, 128) and T in (128, 256)
    split_kernel_ok = P == 64 and S in (64, 128, 256) and T in (128, 256)
    factored_ok = P == 64 and S % 64 == 0 and S <= 256 and T in (128, 256)
    for c in cands:
        assert c["chunk_state_ctas"] in (1, 2)
        hmax = 4 if c["chunk_state_ctas"] == 1 else 2
        assert 1 <= c["chunk_state_heads"] <= hmax and hpg % c["chunk_state_heads"] == 0
        assert c["chunk_state_heads"] * P <= (256 if c["chunk_state_ctas"] == 1 else 128)
        assert c["scan_kernel"] in (0, 1, 2, 3) and hpg % c["scan_heads"] == 0
        if c["scan_kernel"] == 3:
            assert factored_ok
        elif c["scan_kernel"] == 1:
            assert chunk_kernel_ok
        elif c["scan_kernel"] == 2:
            assert split_kernel_ok
        else:
            assert c["scan_heads"] <= 4 and c["scan_heads"] * P <= 256
    assert len({tuple(c.values()) for c in cands}) == len(cands)
    default = m.default_plan(d)
    assert default in cands
    expect = 3 if factored_ok else 1 if chunk_kernel_ok else 2 if split_kernel_ok else 0
    assert default["scan_kernel"] == expect
    # the factored output kernel takes every divisor of the heads per group
    if factored_ok:
        assert {c["scan_heads"] for c in cands if c["scan_kernel"] == 3} == \
            {h for h in range(1, hpg + 1) if hpg % h == 0}


def test_plan_rejections(lib):
    import mamba_ssd_forward_gb300 as m
    from mamba_ssd_forward_gb300 import _abi
    d = _dims(2, 4096, 80, 64, 128, 1, 256)
    assert m.plan_candidates(d, io=0) == []  # fp32 I/O has no plan
    with pytest.raises(_abi.SsdError) as e:
        m.default_plan(d, io=0)
    assert e.value.code == _abi.SSD_ERR_UNSUPPORTED
    assert m.plan_candidates(_dims(2, 4096, 80, 64, 128, 3, 256)) == []  # nh % ng
    assert m.plan_candidates(_dims(2, 4096, 80, 64, 128, 1, 100)) == []  # chunk
    bad = [
        {"chunk_state_heads": 3, "chunk_state_ctas": 1, "scan_kernel": 1, "scan_heads": 20},
        {"chunk_state_heads": 4, "chunk_state_ctas": 2, "scan_kernel": 1, "scan_heads": 20},
        {"chunk_state_heads": 4, "chunk_state_ctas": 1, "scan_kernel": 1, "scan_heads": 3},
        {"chunk_state_heads": 4, "chunk_state_ctas": 1, "scan_kernel": 0, "scan_heads": 8},
        {"chunk_state_heads": 4, "chunk_state_ctas": 1, "scan_kernel": 4, "scan_heads": 1},
        {"chunk_state_heads": 4, "chunk_state_ctas": 1, "scan_kernel": 3, "scan_heads": 3},
    ]
    # a plan that is not a candidate is rejected by every call taking one,
    # before anything is launched (fake aligned pointers, never dereferenced)
    ok = ctypes.c_void_p(1 << 20)
    ws = lib.ssd_forward_workspace_size(ctypes.byref(d), 1)
    args = [ok, ok, ok, ok, ok, None, None, ok, None, ok, ws]
    n = ctypes.c_int(-1)
    for p in bad:
        assert p not in m.plan_candidates(d)
        ref = ctypes.byref(_abi.SsdPlan(**p))
        assert lib.ssd_forward_ex(ctypes.byref(d), 1, *args, ref, None) == 1
        assert lib.ssd_forward_profiled(ctypes.byref(d), 1, *args, ref, None, None, 0,
                                        ctypes.byref(n)) == 1
        assert n.value == -1  # nothing launched, nothing reported
        assert lib.ssd_forward_host(ctypes.byref(d), 1, *args, ref, None) == 1
    # fp32 calls take no plan
    good = ctypes.byref(_abi.SsdPlan(**m.default_plan(d)))
    ws32 = lib.ssd_forward_workspace_size(ctypes.byref(d), 0)
    assert lib.ssd_forward_ex(ctypes.byref(d), 0, *args[:-1], ws32, good, None) == 1
    # events promised but missing
    assert lib.ssd_forward_profiled(ctypes.byref(d), 1, *args, None, None, None, 2, None) == 1
    rc = lib.ssd_forward_tune(ctypes.byref(d), 1, *([None] * 10), 0, 5, None, 0, None, None)
    assert rc == _abi.SSD_ERR_INVALID_ARG
    # a tuner call with valid arguments but nowhere to put the chosen plan
    rc = lib.ssd_forward_tune(ctypes.byref(d), 1, *args, 5, None, 0, None, None)
    assert rc == _abi.SSD_ERR_INVALID_ARG
    # a flush buffer of zero bytes
    plan = ctypes.byref(_abi.SsdPlan())
    rc = lib.ssd_forward_tune(ctypes.byref(d), 1, *args, 5, ctypes.c_void_p(4096), 0, None, plan)
    assert rc == _abi.SSD_ERR_INVALID_ARG


def test_selftest_and_error_reads_reject_bad_arguments(lib):
    from mamba_ssd_forward_gb300 import _abi
    for bad in (0, 999, 1_000_000_001):
        assert lib.ssd_selftest_bounded_wait(bad, None, None) == _abi.SSD_ERR_INVALID_ARG
    # an error word must be 4-byte aligned
    assert lib.ssd_selftest_bounded_wait(2_000_000, ctypes.c_void_p((1 << 20) + 2), None) == 1
    # a workspace's error word: NULL or misaligned workspaces are rejected
    assert lib.ssd_workspace_error(None, None) == 1
    assert lib.ssd_workspace_error(ctypes.c_void_p((1 << 20) + 16), None) == 1


def test_library_keeps_no_plan_table():
    """Launch plans are arguments, never stored: the plan code holds no
    table, and the header declares no call that installs one."""
    src = open(os.path.join(ROOT, "mamba_ssd_forward_gb300", "csrc", "ssd_plan.cu")).read()
    assert "std::map" not in src and "mutex" not in src and "static" not in src
    names = declared_functions()
    assert "ssd_forward_set_plan" not in names and "ssd_forward_get_plan" not in names


def test_debug_bounds_library_builds_with_every_export():
    """The debug-bounds variant (SSD_DEBUG_BOUNDS) compiles from the same
    sources and exports the same C ABI; the GPU tests run it."""
    import ctypes
    from mamba_ssd_forward_gb300 import _abi, build
    path = build.build_debug()
    lib = ctypes.CDLL(path)
    for n in _abi.EXPORTS:
        assert hasattr(lib, n), n
    assert path != _abi.LIB_PATH


def test_backward_workspace_and_rejections(lib):
    """ssd_backward: its workspace holds at least G, the jump terms, the
    start and adjoint states and the c . B blocks (and the fp32 copies with
    bf16 I/O); unsupported dims give 0 / SSD_ERR_UNSUPPORTED, bad pointers,
    a short or misaligned workspace SSD_ERR_INVALID_ARG, all before any
    launch."""
    from mamba_ssd_forward_gb300 import _abi
    d = dims()  # b2 L1000 h8 P64 S128 ng2 T256 (nc = 4)
    nc, T = 4, 256
    ws32 = lib.ssd_backward_workspace_size(ctypes.byref(d), 0)
    st = 4 * 2 * 8 * nc * 64 * 128
    assert ws32 >= 256 + 4 * 2 * 8 * nc * T + 3 * st + 4 * 2 * 2 * nc * T * T
    assert ws32 % 256 == 0
    ws16 = lib.ssd_backward_workspace_size(ctypes.byref(d), 1)
    assert ws16 >= ws32 + 4 * 2 * 1000 * (2 * 8 * 64 + 2 * 2 * 128)  # fp32 copies of x, gy, B, C
    assert lib.ssd_backward_workspace_size(ctypes.byref(d), 7) == 0
    for bad in (dims(headdim=32), dims(dstate=96), dims(headdim=128),
                # chunk lengths other than 64, 128 and 256
                dims(dstate=256, chunk=96), dims(chunk=32), dims(chunk=512)):
        assert lib.ssd_backward_workspace_size(ctypes.byref(bad), 0) == 0
    for good in (dims(chunk=64), dims(dstate=256, chunk=64), dims(dstate=64, chunk=128)):
        assert lib.ssd_backward_workspace_size(ctypes.byref(good), 0) > 0
    ok = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    args = [ok, ok, ok, ok, ok, None, None, ok, None, ok, ok, ok, ok, ok, None, None]

    def call(dd, dtype, a, wsp, nbytes):
        return lib.ssd_backward(ctypes.byref(dd), dtype, *a, wsp, nbytes, None)

    assert call(dims(dstate=96), 0, args, ok, ws32) == _abi.SSD_ERR_UNSUPPORTED
    for i in range(len(args)):  # x dt A B C D h0 gy gfinal dx ddt dA dB dC dD dh0
        a = list(args)
        if args[i] is not None:  # required: NULL is rejected
            a[i] = None
            assert call(d, 0, a, ok, ws32) == _abi.SSD_ERR_INVALID_ARG, i
        a[i] = odd  # required or optional: misaligned is rejected
        assert call(d, 0, a, ok, ws32) == _abi.SSD_ERR_INVALID_ARG, i
    assert call(d, 0, args, ok, ws32 - 1) == _abi.SSD_ERR_INVALID_ARG
    assert call(d, 0, args, ctypes.c_void_p((1 << 20) + 16), ws32) == _abi.SSD_ERR_INVALID_ARG
    assert call(d, 1, args, ok, ws16 - 1) == _abi.SSD_ERR_INVALID_ARG
    assert lib.ssd_backward_profiled(ctypes.byref(d), 0, *args, ok, ws32, None, None, 2,
                                     None) == _abi.SSD_ERR_INVALID_ARG  # events NULL, n 2
