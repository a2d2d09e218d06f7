"""Float64 oracle: ctypes driver for the C recurrence and numpy restatements.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Shapes (row-major):
    x [b,L,nh,P]   dt [b,L,nh]   A [nh]   B, C [b,L,ng,S]   D [nh]
    h0 / final_state [b,nh,P,S]   states / dstates [b,nh,nc,P,S]
    y [b,L,nh,P]   G [b,nh,nc*T]  (natural-log units; the CUDA path stores
    G times log2(e))
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "libssd_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ssd_oracle.c into a shared library next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, dp = ctypes.c_int64, ctypes.c_void_p
        lib.ssd_oracle_forward.restype = ctypes.c_int
        lib.ssd_oracle_forward.argtypes = [i64] * 7 + [dp] * 7 + [dp, i64] + [dp] * 5
        _lib = lib
        # libgomp is linked into the library; its thread controls are
        # reachable through the same handle.
        _lib.omp_set_num_threads.argtypes = [ctypes.c_int]
        _lib.omp_get_max_threads.restype = ctypes.c_int
    return _lib


def set_threads(n: int) -> None:
    """Number of OpenMP threads the C recurrence uses from now on."""
    _load().omp_set_num_threads(int(n))


def max_threads() -> int:
    return int(_load().omp_get_max_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _dims(x, dt, A, B):
    b, L, nh, P = x.shape
    ng, S = B.shape[2], B.shape[3]
    assert dt.shape == (b, L, nh) and A.shape == (nh,) and B.shape == (b, L, ng, S)
    assert nh % ng == 0
    return b, L, nh, P, S, ng


def recurrence(x, dt, A, B, C, D=None, h0=None, chunk=256, bh=None,
               want=("y", "final_state")):
    """Run the C token-by-token recurrence.  Returns a dict with the requested
    outputs among y, final_state, states, dstates, G (float64 numpy)."""
    x, dt, A, B, C, D, h0 = map(_f64, (x, dt, A, B, C, D, h0))
    b, L, nh, P, S, ng = _dims(x, dt, A, B)
    assert C.shape == B.shape
    T = int(chunk)
    nc = (L + T - 1) // T
    shapes = {
        "y": (b, L, nh, P),
        "final_state": (b, nh, P, S),
        "states": (b, nh, nc, P, S),
        "dstates": (b, nh, nc, P, S),
        "G": (b, nh, nc * T),
    }
    out = {k: np.full(shapes[k], np.nan) for k in want}
    bh_arr = None if bh is None else np.ascontiguousarray(bh, dtype=np.int64)

    def ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    rc = _load().ssd_oracle_forward(
        b, L, nh, P, S, ng, T,
        ptr(x), ptr(dt), ptr(A), ptr(B), ptr(C), ptr(D), ptr(h0),
        ptr(bh_arr), 0 if bh_arr is None else len(bh_arr),
        ptr(out.get("y")), ptr(out.get("final_state")), ptr(out.get("states")),
        ptr(out.get("dstates")), ptr(out.get("G")))
    if rc != 0:
        raise ValueError(f"ssd_oracle_forward rejected its arguments (code {rc})")
    return out


def recurrence_np(x, dt, A, B, C, D=None, h0=None):
    """The same recurrence in numpy, vectorised over (P, S) only; for tiny
    inputs.  Returns (y, final_state)."""
    x, dt, A, B, C, D, h0 = map(_f64, (x, dt, A, B, C, D, h0))
    b, L, nh, P, S, ng = _dims(x, dt, A, B)
    hpg = nh // ng
    y = np.zeros((b, L, nh, P))
    final = np.zeros((b, nh, P, S))
    for bi in range(b):
        for h in range(nh):
            g = h // hpg
            H = np.zeros((P, S)) if h0 is None else h0[bi, h].copy()
            for t in range(L):
                H = np.exp(A[h] * dt[bi, t, h]) * H + np.outer(dt[bi, t, h] * x[bi, t, h], B[bi, t, g])
                y[bi, t, h] = H @ C[bi, t, g] + (0.0 if D is None else D[h]) * x[bi, t, h]
            final[bi, h] = H
    return y, final


def decode_step(x, dt, A, B, C, D=None, h=None):
    """One token of the recurrence ("Mamba-2 architecture": the state update
    h_t = exp(A dt_t) h_{t-1} + (dt_t x_t) outer B_t, output taken from the
    updated state, y_t = h_t . c_t + D x_t), float64, for a batch of
    (batch, head) states at once.

    Shapes: x [b,nh,P], dt [b,nh], A [nh], B, C [b,ng,S], D [nh] or None,
    h [b,nh,P,S] or None (zero).  Head hd reads group hd // (nh // ng).
    Returns (y [b,nh,P], h_new [b,nh,P,S])."""
    x, dt, A, B, C, D, h = map(_f64, (x, dt, A, B, C, D, h))
    b, nh, P = x.shape
    ng, S = B.shape[1], B.shape[2]
    if nh % ng:
        raise ValueError("nheads must be a multiple of ngroups")
    grp = np.arange(nh) // (nh // ng)
    Bh, Ch = B[:, grp], C[:, grp]                       # [b, nh, S]
    decay = np.exp(A[None, :] * dt)                     # [b, nh]
    h_prev = np.zeros((b, nh, P, S)) if h is None else h
    h_new = decay[:, :, None, None] * h_prev + (dt[:, :, None] * x)[:, :, :, None] * Bh[:, :, None, :]
    y = np.einsum("bhps,bhs->bhp", h_new, Ch)
    if D is not None:
        y = y + D[None, :, None] * x
    return y, h_new


def chunked(x, dt, A, B, C, D=None, h0=None, chunk=256):
    """The chunked log-space formulas, float64, per (batch, head, chunk):

        G      = inclusive cumsum of a = A*dt inside the chunk
        Y      = exp(G) * (C h^T) + ((C B^T) * exp(G_i - G_j) * M) (dt * X) + D X
        h_next = exp(G_last) h + (exp(G_last - G) * dt * X)^T B      (P x S)

    with M the causal mask including the diagonal.  Returns a dict with y,
    final_state, states (start of chunk), dstates (chunk-local jump term),
    G (natural log, padded like the recurrence) and max_kept_exponent, the
    largest exponent that survives the mask (non-positive by construction
    when every a_t <= 0)."""
    x, dt, A, B, C, D, h0 = map(_f64, (x, dt, A, B, C, D, h0))
    b, L, nh, P, S, ng = _dims(x, dt, A, B)
    hpg = nh // ng
    T = int(chunk)
    nc = (L + T - 1) // T
    y = np.zeros((b, L, nh, P))
    final = np.zeros((b, nh, P, S))
    states = np.zeros((b, nh, nc, P, S))
    dstates = np.zeros((b, nh, nc, P, S))
    Gall = np.zeros((b, nh, nc * T))
    kept = -np.inf
    for bi in range(b):
        for h in range(nh):
            g = h // hpg
            H = np.zeros((P, S)) if h0 is None else h0[bi, h].copy()
            for k in range(nc):
                lo, hi = k * T, min((k + 1) * T, L)
                n = hi - lo
                X = x[bi, lo:hi, h]            # n x P
                Bc = B[bi, lo:hi, g]           # n x S
                Cc = C[bi, lo:hi, g]           # n x S
                d = dt[bi, lo:hi, h]           # n
                G = np.cumsum(A[h] * d)        # n
                Gall[bi, h, lo:lo + n] = G
                Gall[bi, h, lo + n:(k + 1) * T] = G[-1]
                states[bi, h, k] = H
                mask = np.tril(np.ones((n, n), dtype=bool))
                expo = G[:, None] - G[None, :]
                if n:
                    kept = max(kept, expo[mask].max())
                decay = np.where(mask, np.exp(np.where(mask, expo, 0.0)), 0.0)
                Yc = np.exp(G)[:, None] * (Cc @ H.T)
                Yc += ((Cc @ Bc.T) * decay) @ (d[:, None] * X)
                if D is not None:
                    Yc += D[h] * X
                y[bi, lo:hi, h] = Yc
                w = np.exp(G[-1] - G) * d      # exp(G_last - G) * dt
                kept = max(kept, (G[-1] - G).max())
                dH = (w[:, None] * X).T @ Bc   # P x S
                dstates[bi, h, k] = dH
                H = np.exp(G[-1]) * H + dH
            final[bi, h] = H
    return {"y": y, "final_state": final, "states": states, "dstates": dstates,
            "G": Gall, "max_kept_exponent": kept}


def backward(x, dt, A, B, C, D=None, h0=None, gy=None, gfinal=None):
    """Gradients of a loss L(y, final_state) through the forward recurrence,
    given gy = dL/dy [b, L, nh, P] and gfinal = dL/dfinal_state [b, nh, P, S]
    (None = 0), in float64 by the adjoint recurrence token by token (tiny
    inputs only).

    Forward ("Mamba-2 architecture"): a_t = exp(A dt_t), b_t = dt_t B_t,
    h_t = a_t h_{t-1} + x_t b_t^T (P x S), y_t = h_t c_t + D x_t.  With
    g_t = dL/dh_t (P x S), going backwards from g = gfinal:
        g_t    = gy_t c_t^T + a_{t+1} g_{t+1}
        dx_t   = g_t b_t + D gy_t
        db_t   = g_t^T x_t            -> dB_t = dt_t db_t,   dt_t += <db_t, B_t>
        dc_t   = h_t^T gy_t
        da_t   = <g_t, h_{t-1}>       -> dt_t += A a_t da_t, dA += dt_t a_t da_t
        dD    += <gy_t, x_t>,  dh0 = a_1 g_1 (the g carried past t = 1).
    The gradients of B and C sum over the heads of a group.  Returns a dict
    of dx, ddt, dA, dB, dC, dD, dh0 (float64)."""
    x, dt, A, B, C, D, h0, gy, gfinal = map(_f64, (x, dt, A, B, C, D, h0, gy, gfinal))
    b, L, nh, P, S, ng = _dims(x, dt, A, B)
    hpg = nh // ng
    out = {"dx": np.zeros_like(x), "ddt": np.zeros_like(dt), "dA": np.zeros_like(A),
           "dB": np.zeros_like(B), "dC": np.zeros_like(C), "dD": np.zeros(nh),
           "dh0": np.zeros((b, nh, P, S))}
    for bi in range(b):
        for h in range(nh):
            g = h // hpg
            # forward, keeping every state: hs[t + 1] = h_t, hs[0] = h0
            hs = np.zeros((L + 1, P, S))
            if h0 is not None:
                hs[0] = h0[bi, h]
            a = np.exp(A[h] * dt[bi, :, h])
            for t in range(L):
                hs[t + 1] = a[t] * hs[t] + np.outer(x[bi, t, h], dt[bi, t, h] * B[bi, t, g])
            Dh = 0.0 if D is None else D[h]
            G = np.zeros((P, S)) if gfinal is None else gfinal[bi, h].copy()
            for t in range(L - 1, -1, -1):
                G = G + np.outer(gy[bi, t, h], C[bi, t, g])    # dL/dh_t, complete
                bt = dt[bi, t, h] * B[bi, t, g]
                out["dx"][bi, t, h] = G @ bt + Dh * gy[bi, t, h]
                db = G.T @ x[bi, t, h]
                out["dB"][bi, t, g] += dt[bi, t, h] * db
                out["dC"][bi, t, g] += hs[t + 1].T @ gy[bi, t, h]
                da = float(np.sum(G * hs[t]))
                out["ddt"][bi, t, h] = A[h] * a[t] * da + float(db @ B[bi, t, g])
                out["dA"][h] += dt[bi, t, h] * a[t] * da
                out["dD"][h] += float(gy[bi, t, h] @ x[bi, t, h])
                G = a[t] * G                                      # dL/dh_{t-1} from h_t
            out["dh0"][bi, h] = G
    return out


def backward_chunked(x, dt, A, B, C, D=None, h0=None, gy=None, gfinal=None, chunk=256):
    """The gradients of ``backward`` by the chunked formulas a chunk-parallel
    kernel would use (numpy float64; derived from the forward of
    "Mamba-2 architecture", its chunked output equation and state jump).
    Per (batch, head), with G the inclusive in-chunk cumsum of l_t = A dt_t,
    h_k the state entering chunk k and R_k = dL/dh_{k+1} coming from the
    chunks after k (R of the last chunk = gfinal):

      R_{k-1} = exp(G_last) R_k + sum_{s in k} exp(G_s) gy_s c_s^T   (dh0 = R_{-1})
      dx_t  = dt_t [sum_{s>=t} exp(G_s - G_t) (B_t . C_s) gy_s + exp(G_last - G_t) R_k B_t] + D gy_t
      q_t   = sum_{s>=t} exp(G_s - G_t) (gy_s . x_t) C_s + exp(G_last - G_t) R_k^T x_t
      dB_t += dt_t q_t,   dC_t += exp(G_t) h_k^T gy_t + sum_{j<=t} exp(G_t - G_j) (gy_t . x_j) dt_j B_j
      dL/dG_i = gy_i . ysm_i - x_i . dxsm_i  (+ <R_k, h_{k+1}> at the chunk's last token)
      eta_t = dL/dl_t = sum_{i>=t in k} dL/dG_i
      ddt_t = A eta_t + q_t . B_t,   dA += sum_t dt_t eta_t,   dD += sum_t gy_t . x_t
    where ysm = y - D x and dxsm = dx - D gy.  Sums over heads of a group for
    dB and dC.  Used to pin the chunked restatement against the adjoint
    recurrence (``backward``)."""
    x, dt, A, B, C, D, h0, gy, gfinal = map(_f64, (x, dt, A, B, C, D, h0, gy, gfinal))
    b, L, nh, P, S, ng = _dims(x, dt, A, B)
    hpg = nh // ng
    T = int(chunk)
    nc = -(-L // T)
    out = {"dx": np.zeros_like(x), "ddt": np.zeros_like(dt), "dA": np.zeros_like(A),
           "dB": np.zeros_like(B), "dC": np.zeros_like(C), "dD": np.zeros(nh),
           "dh0": np.zeros((b, nh, P, S))}
    for bi in range(b):
        for h in range(nh):
            g = h // hpg
            Dh = 0.0 if D is None else D[h]
            spans = [(k * T, min(T, L - k * T)) for k in range(nc)]
            G = [np.cumsum(A[h] * dt[bi, t0:t0 + v, h]) for t0, v in spans]
            # forward: the state entering each chunk (hk[nc] = final state)
            hk = np.zeros((nc + 1, P, S))
            if h0 is not None:
                hk[0] = h0[bi, h]
            for k, (t0, v) in enumerate(spans):
                w = np.exp(G[k][-1] - G[k]) * dt[bi, t0:t0 + v, h]
                hk[k + 1] = np.exp(G[k][-1]) * hk[k] + \
                    (x[bi, t0:t0 + v, h] * w[:, None]).T @ B[bi, t0:t0 + v, g]
            # backward over chunks: R[k] = dL/dh_{k+1} from the later chunks
            R = np.zeros((nc, P, S))
            carry = np.zeros((P, S)) if gfinal is None else gfinal[bi, h].copy()
            for k in range(nc - 1, -1, -1):
                t0, v = spans[k]
                R[k] = carry
                carry = np.exp(G[k][-1]) * carry + \
                    (gy[bi, t0:t0 + v, h] * np.exp(G[k])[:, None]).T @ C[bi, t0:t0 + v, g]
            out["dh0"][bi, h] = carry
            for k, (t0, v) in enumerate(spans):
                Gk, GL = G[k], G[k][-1]
                xs, gys, dts = x[bi, t0:t0 + v, h], gy[bi, t0:t0 + v, h], dt[bi, t0:t0 + v, h]
                Bs, Cs = B[bi, t0:t0 + v, g], C[bi, t0:t0 + v, g]
                up = np.triu(np.exp(Gk[None, :] - Gk[:, None]))   # [t, s]: exp(G_s - G_t), s >= t
                low = np.tril(np.exp(Gk[:, None] - Gk[None, :]))  # [t, j]: exp(G_t - G_j), j <= t
                back = np.exp(GL - Gk)[:, None]
                dxsm = dts[:, None] * ((up * (Bs @ Cs.T)) @ gys + back * (Bs @ R[k].T))
                q = (up * (xs @ gys.T)) @ Cs + back * (xs @ R[k])
                ysm = np.exp(Gk)[:, None] * (Cs @ hk[k].T) + \
                    ((low * (Cs @ Bs.T)) * dts[None, :]) @ xs
                dG = np.sum(gys * ysm, 1) - np.sum(xs * dxsm, 1)
                dG[-1] += np.sum(R[k] * hk[k + 1])
                eta = np.cumsum(dG[::-1])[::-1]
                out["dx"][bi, t0:t0 + v, h] = dxsm + Dh * gys
                out["dB"][bi, t0:t0 + v, g] += dts[:, None] * q
                out["dC"][bi, t0:t0 + v, g] += np.exp(Gk)[:, None] * (gys @ hk[k]) + \
                    ((low * (gys @ xs.T)) * dts[None, :]) @ Bs
                out["ddt"][bi, t0:t0 + v, h] = A[h] * eta + np.sum(q * Bs, 1)
                out["dA"][h] += float(np.sum(dts * eta))
                out["dD"][h] += float(np.sum(gys * xs))
    return out
