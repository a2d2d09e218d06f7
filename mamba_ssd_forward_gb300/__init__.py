"""Mamba-2 chunked SSD forward pass for GB300 (sm_103a).

Thin Python binding over the C ABI in include/ssd.h: it infers the
dimensions from tensor shapes, allocates outputs and workspace with torch on
the current CUDA stream, and passes raw device pointers.  All arithmetic runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback.

Tensor layouts (all contiguous, on one CUDA device):
    x [b, L, nh, P], dt [b, L, nh], B/C [b, L, ng, S] -- float32 or bfloat16
    A [nh], D [nh], h0 [b, nh, P, S]                   -- float32
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import SSD_BF16, SSD_F32, SsdError  # noqa: F401

__all__ = ["forward", "chunk_cumsum", "chunk_state", "state_passing", "chunk_scan",
           "decode_step", "workspace_size", "new_workspace", "workspace_error", "dims_of",
           "backward", "backward_workspace_size", "ssd",
           "SsdError"]


def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SSD_F32
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    raise TypeError(f"I/O tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors passed to the SSD library must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _f32(t, name):
    if t is not None and t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def dims_of(x: torch.Tensor, B: torch.Tensor, chunk: int) -> _abi.SsdDims:
    b, L, nh, P = x.shape
    ng, S = B.shape[2], B.shape[3]
    return _abi.SsdDims(b, L, nh, P, S, ng, int(chunk))


def _nchunks(d: _abi.SsdDims) -> int:
    return (d.seqlen + d.chunk - 1) // d.chunk


def workspace_size(x: torch.Tensor, B: torch.Tensor, chunk: int = 256) -> int:
    d = dims_of(x, B, chunk)
    return int(_abi.load().ssd_forward_workspace_size(ctypes.byref(d), _io_code(x)))


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """A uint8 device workspace of `nbytes` bytes with its error-word header
    (the first SSD_WS_HEADER_BYTES) zeroed, as every workspace of the forward
    calls must be before its first use."""
    ws = torch.empty(max(int(nbytes), _abi.SSD_WS_HEADER_BYTES), dtype=torch.uint8,
                     device=device)
    ws[:_abi.SSD_WS_HEADER_BYTES].zero_()
    return ws


def _plan_ref(plan):
    """ctypes reference to an ssd_plan from a dict of its four fields, or
    None (the default plan)."""
    if plan is None:
        return None
    return ctypes.byref(_abi.SsdPlan(**{k: int(v) for k, v in plan.items()}))


def forward(x, dt, A, B, C, D=None, h0=None, chunk: int = 256, workspace=None,
            y=None, final_state=None, return_final_state: bool = True, plan=None):
    """y, final_state = the SSD forward pass (ssd_forward_ex).

    `workspace`, `y` and `final_state` may be preallocated (a uint8 CUDA
    tensor of at least workspace_size() bytes made by new_workspace(), and
    outputs of the right shape and dtype); otherwise they are allocated here.
    `plan` is a launch plan dict (bf16 only; None = the default)."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    io = _io_code(x)
    ws_need = lib.ssd_forward_workspace_size(ctypes.byref(d), io)
    if ws_need == 0:
        raise SsdError("ssd_forward_workspace_size", _abi.SSD_ERR_UNSUPPORTED,
                       "dimensions are invalid or unsupported")
    if workspace is None:
        workspace = new_workspace(ws_need, x.device)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate),
                                  dtype=torch.float32, device=x.device)
    _abi.check("ssd_forward_ex", lib.ssd_forward_ex(
        ctypes.byref(d), io, _ptr(x), _ptr(dt), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
        _ptr(_f32(D, "D")), _ptr(_f32(h0, "h0")), _ptr(y), _ptr(final_state),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _plan_ref(plan),
        _stream()))
    return y, final_state


def backward_workspace_size(x: torch.Tensor, B: torch.Tensor, chunk: int = 256) -> int:
    """Bytes of workspace ssd_backward needs (0: unsupported dims or dtype)."""
    d = dims_of(x, B, chunk)
    return int(_abi.load().ssd_backward_workspace_size(ctypes.byref(d), _io_code(x)))


def backward(x, dt, A, B, C, D=None, h0=None, gy=None, gfinal=None, chunk: int = 256,
             workspace=None, want_dD: bool = True, want_dh0: bool = True, out=None,
             events=None) -> dict:
    """Gradients of a loss through forward() given gy = dL/dy and gfinal =
    dL/dfinal_state (None = 0), by ssd_backward (fp32 or bf16 I/O, computed in
    fp32): a dict of dx, ddt, dB, dC (in the I/O dtype), dA, dD, dh0 (fp32;
    the last two None unless wanted).  `workspace`
    may be a preallocated new_workspace(backward_workspace_size(...)) and
    `out` a dict returned by an earlier call (its tensors are reused).  With
    `events` (torch.cuda.Event, enable_timing) the call is
    ssd_backward_profiled, recording them around its launches."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    io = _io_code(x)
    ws_need = lib.ssd_backward_workspace_size(ctypes.byref(d), io)
    if ws_need == 0:
        raise SsdError("ssd_backward_workspace_size", _abi.SSD_ERR_UNSUPPORTED,
                       "dimensions or dtype are invalid or unsupported by the backward")
    if gy is None:
        raise ValueError("gy (dL/dy) is required")
    if workspace is None:
        workspace = new_workspace(ws_need, x.device)
    if out is None:
        out = {"dx": torch.empty_like(x), "ddt": torch.empty_like(dt),
               "dA": torch.empty_like(A), "dB": torch.empty_like(B), "dC": torch.empty_like(C),
               "dD": torch.empty_like(A) if want_dD else None,
               "dh0": (torch.empty((d.batch, d.nheads, d.headdim, d.dstate),
                                   dtype=torch.float32, device=x.device) if want_dh0 else None)}
    args = [ctypes.byref(d), io, _ptr(x), _ptr(dt), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
            _ptr(_f32(D, "D")), _ptr(_f32(h0, "h0")), _ptr(gy), _ptr(_f32(gfinal, "gfinal")),
            _ptr(out["dx"]), _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]),
            _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dh0"]), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream()]
    if events is None:
        _abi.check("ssd_backward", lib.ssd_backward(*args))
        return out
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    n = ctypes.c_int(0)
    _abi.check("ssd_backward_profiled", lib.ssd_backward_profiled(
        *args, handles, len(events), ctypes.byref(n)))
    out["n_launches"] = n.value
    return out


def chunk_cumsum(dt, A, chunk: int, headdim: int = 16, dstate: int = 16, out=None):
    """G [b, nh, nc*T] float32 (log2 units) = ssd_chunk_cumsum.  headdim and
    dstate only need to lie in the supported range; they do not affect G.
    `out` may be a preallocated G."""
    lib = _abi.load()
    b, L, nh = dt.shape
    d = _abi.SsdDims(b, L, nh, headdim, dstate, 1, int(chunk))
    G = out if out is not None else torch.empty(
        (b, nh, _nchunks(d) * d.chunk), dtype=torch.float32, device=dt.device)
    _abi.check("ssd_chunk_cumsum", lib.ssd_chunk_cumsum(
        ctypes.byref(d), _io_code(dt), _ptr(dt), _ptr(_f32(A, "A")), _ptr(G), _stream()))
    return G


def chunk_state(x, B, dt, G, chunk: int, out=None):
    """dstates [b, nh, nc, P, S] float32 = ssd_chunk_state (`out` may be a
    preallocated dstates)."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    if out is None:
        out = torch.empty((d.batch, d.nheads, _nchunks(d), d.headdim, d.dstate),
                          dtype=torch.float32, device=x.device)
    _abi.check("ssd_chunk_state", lib.ssd_chunk_state(
        ctypes.byref(d), _io_code(x), _ptr(x), _ptr(B), _ptr(dt), _ptr(_f32(G, "G")),
        _ptr(out), _stream()))
    return out


def state_passing(dstates, G, h0=None, chunk: int = 256, seqlen: int | None = None,
                  ngroups: int = 1, return_final_state: bool = True, states=None,
                  final_state=None):
    """states [b, nh, nc, P, S], final_state [b, nh, P, S] = ssd_state_passing
    (`states` and `final_state` may be preallocated)."""
    lib = _abi.load()
    b, nh, nc, P, S = dstates.shape
    L = seqlen if seqlen is not None else nc * chunk
    d = _abi.SsdDims(b, L, nh, P, S, ngroups, int(chunk))
    if states is None:
        states = torch.empty_like(dstates)
    final = final_state
    if final is None and return_final_state:
        final = torch.empty((b, nh, P, S), dtype=torch.float32, device=dstates.device)
    _abi.check("ssd_state_passing", lib.ssd_state_passing(
        ctypes.byref(d), _ptr(_f32(dstates, "dstates")), _ptr(_f32(G, "G")),
        _ptr(_f32(h0, "h0")), _ptr(states), _ptr(final), _stream()))
    return states, final


def chunk_scan(x, B, C, dt, G, states, D=None, chunk: int = 256, y=None):
    """y [b, L, nh, P] (I/O dtype) = ssd_chunk_scan (`y` may be preallocated)."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    if y is None:
        y = torch.empty_like(x)
    _abi.check("ssd_chunk_scan", lib.ssd_chunk_scan(
        ctypes.byref(d), _io_code(x), _ptr(x), _ptr(B), _ptr(C), _ptr(dt),
        _ptr(_f32(G, "G")), _ptr(_f32(states, "states")), _ptr(_f32(D, "D")), _ptr(y),
        _stream()))
    return y


def decode_step(x, dt, A, B, C, D, state, y=None):
    """y [b, nh, P] (I/O dtype) = ssd_decode_step: one token for every
    (batch, head) state.  x [b, nh, P], dt [b, nh], B/C [b, ng, S] in the I/O
    dtype; state [b, nh, P, S] float32 is updated in place."""
    lib = _abi.load()
    b, nh, P = x.shape
    ng, S = B.shape[1], B.shape[2]
    d = _abi.SsdDims(b, 1, nh, P, S, ng, 256)
    if y is None:
        y = torch.empty_like(x)
    _abi.check("ssd_decode_step", lib.ssd_decode_step(
        ctypes.byref(d), _io_code(x), _ptr(x), _ptr(dt), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
        _ptr(_f32(D, "D")), _ptr(_f32(state, "state")), _ptr(y), _stream()))
    return y


def forward_profiled(x, dt, A, B, C, D, h0, chunk, workspace, y, final_state, events,
                     plan=None):
    """ssd_forward recording `events` (torch.cuda.Event, enable_timing) around
    each of its launches on the current stream; returns the launch count."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    n = ctypes.c_int(0)
    _abi.check("ssd_forward_profiled", lib.ssd_forward_profiled(
        ctypes.byref(d), _io_code(x), _ptr(x), _ptr(dt), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
        _ptr(_f32(D, "D")), _ptr(_f32(h0, "h0")), _ptr(y), _ptr(final_state), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _plan_ref(plan), _stream(), handles,
        len(events), ctypes.byref(n)))
    return n.value


def host_workspace_size(x, B, chunk, has_D=True, has_h0=False, want_final_state=True) -> int:
    d = dims_of(x, B, chunk)
    return int(_abi.load().ssd_forward_host_workspace_size(
        ctypes.byref(d), _io_code(x), int(has_D), int(has_h0), int(want_final_state)))


def _host_ptr(t):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError("ssd_forward_host takes contiguous host tensors")
    return ctypes.c_void_p(t.data_ptr())


def forward_host(x, dt, A, B, C, D, h0, chunk, workspace, y, final_state=None, plan=None):
    """ssd_forward_host: host tensors in (x, dt, A, B, C, D, h0) and out (y,
    final_state), a device uint8 `workspace` of host_workspace_size() bytes.
    Enqueued on the current stream; synchronise before reading y."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    if not workspace.is_cuda:
        raise ValueError("the workspace of ssd_forward_host lives on the device")
    _abi.check("ssd_forward_host", lib.ssd_forward_host(
        ctypes.byref(d), _io_code(x), _host_ptr(x), _host_ptr(dt), _host_ptr(A), _host_ptr(B),
        _host_ptr(C), _host_ptr(D), _host_ptr(h0), _host_ptr(y), _host_ptr(final_state),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _plan_ref(plan), _stream()))


def host_overlapped_workspace_size(x, B, chunk, n_slices, has_D=True, has_h0=False,
                                   want_final_state=True) -> int:
    d = dims_of(x, B, chunk)
    return int(_abi.load().ssd_forward_host_overlapped_workspace_size(
        ctypes.byref(d), _io_code(x), int(has_D), int(has_h0), int(want_final_state),
        int(n_slices)))


def forward_host_overlapped(x, dt, A, B, C, D, h0, chunk, workspace, y, final_state=None,
                            n_slices=4, h2d_stream=None, d2h_stream=None, plan=None):
    """ssd_forward_host_overlapped: as forward_host, cut into up to n_slices
    slices whose uploads (h2d_stream), forward passes (current stream) and
    downloads (d2h_stream) overlap.  Streams are torch.cuda.Stream or None."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    if not workspace.is_cuda:
        raise ValueError("the workspace of ssd_forward_host_overlapped lives on the device")
    sh = lambda s: None if s is None else ctypes.c_void_p(s.cuda_stream)  # noqa: E731
    _abi.check("ssd_forward_host_overlapped", lib.ssd_forward_host_overlapped(
        ctypes.byref(d), _io_code(x), _host_ptr(x), _host_ptr(dt), _host_ptr(A), _host_ptr(B),
        _host_ptr(C), _host_ptr(D), _host_ptr(h0), _host_ptr(y), _host_ptr(final_state),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), int(n_slices),
        _plan_ref(plan), _stream(), sh(h2d_stream), sh(d2h_stream)))


def plan_candidates(d: _abi.SsdDims, io: int = 1) -> list[dict]:
    """Every valid launch plan for dims `d` (ssd_forward_plan_candidates);
    empty for fp32 I/O (io 0), which has none."""
    lib = _abi.load()
    n = lib.ssd_forward_plan_candidates(ctypes.byref(d), int(io), None, 0)
    arr = (_abi.SsdPlan * max(n, 1))()
    lib.ssd_forward_plan_candidates(ctypes.byref(d), int(io), arr, n)
    return [arr[i].as_dict() for i in range(n)]


def default_plan(d: _abi.SsdDims, io: int = 1) -> dict:
    """The cost-model launch plan (ssd_forward_default_plan)."""
    p = _abi.SsdPlan()
    _abi.check("ssd_forward_default_plan",
               _abi.load().ssd_forward_default_plan(ctypes.byref(d), int(io), ctypes.byref(p)))
    return p.as_dict()


def tune(x, dt, A, B, C, D=None, h0=None, chunk: int = 256, reps: int = 5, workspace=None,
         flush=None):
    """Time every launch plan on these inputs (ssd_forward_tune).  Returns
    (plan dict, y, final_state) of the final pass with the fastest plan; pass
    the plan to later calls (forward(..., plan=...)): nothing is installed.
    `flush`, a device tensor larger than the L2 (e.g. 256 MB), makes every
    candidate launch run from a cold L2 (the buffer is overwritten before
    each, outside the timing); without it the launches run back to back."""
    lib = _abi.load()
    d = dims_of(x, B, chunk)
    io = _io_code(x)
    if workspace is None:
        workspace = new_workspace(lib.ssd_forward_workspace_size(ctypes.byref(d), io), x.device)
    y = torch.empty_like(x)
    final_state = torch.empty((d.batch, d.nheads, d.headdim, d.dstate), dtype=torch.float32,
                              device=x.device)
    p = _abi.SsdPlan()
    _abi.check("ssd_forward_tune", lib.ssd_forward_tune(
        ctypes.byref(d), io, _ptr(x), _ptr(dt), _ptr(_f32(A, "A")), _ptr(B), _ptr(C),
        _ptr(_f32(D, "D")), _ptr(_f32(h0, "h0")), _ptr(y), _ptr(final_state),
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(reps),
        _ptr(flush), 0 if flush is None else flush.numel() * flush.element_size(), _stream(),
        ctypes.byref(p)))
    return p.as_dict(), y, final_state


def workspace_error(workspace) -> None:
    """Synchronise the current stream and raise SsdError if a kernel of a
    call that used `workspace` gave up a bounded wait since the last check
    (ssd_workspace_error); clears the workspace's error word."""
    _abi.check("ssd_workspace_error", _abi.load().ssd_workspace_error(_ptr(workspace), _stream()))


def device_error() -> None:
    """Synchronise the current stream and raise SsdError if a call without a
    workspace (the step-wise entry points, ssd_forward_noalloc) gave up a
    bounded wait since the last check (ssd_device_error)."""
    _abi.check("ssd_device_error", _abi.load().ssd_device_error(_stream()))


class _SsdFunction(torch.autograd.Function):
    """forward() and backward() as one differentiable operation: the forward
    pass through ssd_forward, the gradients of every tensor input through
    ssd_backward (which recomputes the forward's intermediates itself, so
    only the inputs are saved)."""

    @staticmethod
    def forward(ctx, x, dt, A, B, C, D, h0, chunk):
        y, final_state = forward(x, dt, A, B, C, D, h0, chunk=chunk)
        ctx.save_for_backward(x, dt, A, B, C, D, h0)
        ctx.chunk = chunk
        return y, final_state

    @staticmethod
    def backward(ctx, gy, gfinal):
        x, dt, A, B, C, D, h0 = ctx.saved_tensors
        need = ctx.needs_input_grad
        if gy is None:
            gy = torch.zeros_like(x)
        g = backward(x, dt, A, B, C, D, h0, gy.contiguous(),
                     None if gfinal is None else gfinal.float().contiguous(), chunk=ctx.chunk,
                     want_dD=D is not None and need[5], want_dh0=h0 is not None and need[6])
        return (g["dx"] if need[0] else None, g["ddt"] if need[1] else None,
                g["dA"] if need[2] else None, g["dB"] if need[3] else None,
                g["dC"] if need[4] else None, g["dD"] if D is not None and need[5] else None,
                g["dh0"] if h0 is not None and need[6] else None, None)


def ssd(x, dt, A, B, C, D=None, h0=None, chunk: int = 256):
    """y, final_state = the SSD forward pass, differentiable with respect to
    x, dt, A, B, C, D and h0 (autograd; the backward pass is ssd_backward,
    P = 64, S in {64, 128, 256})."""
    return _SsdFunction.apply(x, dt, A, B, C, D, h0, chunk)
