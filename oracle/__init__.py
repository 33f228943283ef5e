"""Float64 CPU oracle for the Mamba (S6) selective scan and the Mamba-2 SSD layer.

TEST INFRASTRUCTURE ONLY.  This package is the slow, obviously correct
reference that the CUDA kernels are checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the CUDA path and never imports it.

The arithmetic lives in ``ssm_oracle.c`` (plain C, IEEE double, libm
``exp``/``expm1``/``log1p``, OpenMP over independent channels).  This module
only loads that library, widens the stored input values (fp32, or bf16 given
as its raw 16-bit patterns) exactly to float64, and slices inputs.

Sources: the pages "State-space models" (rayaq.ca; sections Discretization,
Recurrence and convolution, Mamba: selection, The parallel scan, Implementation)
and "Structured State Space Models and Mamba" (llms.blog; sections Discretization
Mechanics, the S6 section, Hardware-Aware Parallel Associative Scan, State Space
Duality and Mamba-2).

Every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

RULE_EULER, RULE_BILINEAR, RULE_ZOH, RULE_ZOH_SIMPLE = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into liboracle.so (gcc, -O2, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SSM_ORACLE_LIB lets the mutation test load a deliberately broken
            # copy of this library in a child process.
            lib = ctypes.CDLL(os.environ.get("SSM_ORACLE_LIB") or build())
            d, i64, i32 = ctypes.c_double, ctypes.c_int64, ctypes.c_int
            pd = ctypes.POINTER(ctypes.c_double)
            lib.oracle_softplus.restype = d
            lib.oracle_softplus.argtypes = [d]
            lib.oracle_discretize_scalar.restype = i32
            lib.oracle_discretize_scalar.argtypes = [d, d, d, i32, pd, pd]
            lib.oracle_selective_scan_f64.restype = i32
            lib.oracle_selective_scan_f64.argtypes = (
                [pd] * 10 + [i64] * 4 + [i32] * 5)
            lib.oracle_lti_kernel.restype = i32
            lib.oracle_lti_kernel.argtypes = [pd] * 5 + [i64] * 3 + [i32]
            lib.oracle_causal_conv.restype = i32
            lib.oracle_causal_conv.argtypes = [pd] * 4 + [i64] * 3 + [i32]
            lib.oracle_conv_silu.restype = i32
            lib.oracle_conv_silu.argtypes = [pd] * 6 + [i64] * 4 + [i32]
            lib.oracle_selective_scan_bwd_f64.restype = i32
            lib.oracle_selective_scan_bwd_f64.argtypes = [pd] * 20 + [i64] * 4 + [i32] * 2
            lib.oracle_ssd_f64.restype = i32
            lib.oracle_ssd_f64.argtypes = [pd] * 10 + [i64] * 6 + [i32] * 3
            lib.oracle_max_threads.restype = i32
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def widen(a, io_dtype: str = "f32") -> np.ndarray:
    """Exact float64 copy of stored values.

    ``io_dtype == "bf16"``: ``a`` holds raw bfloat16 bit patterns (uint16);
    a bfloat16 is the top half of a float32, so the value is the uint16
    shifted into the high 16 bits of a float32 word.
    """
    if a is None:
        return None
    a = np.asarray(a)
    if io_dtype == "bf16":
        assert a.dtype == np.uint16, "bf16 values are passed as uint16 bit patterns"
        f32 = (a.astype(np.uint32) << 16).view(np.float32)
        return np.ascontiguousarray(f32, dtype=np.float64)
    return np.ascontiguousarray(a, dtype=np.float64)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def softplus(v: float) -> float:
    """log(1 + e^v), evaluated in double."""
    return float(_load().oracle_softplus(float(v)))


def discretize(a: float, b: float, dt: float, rule: int):
    """Scalar (abar, bbar) for h' = a h + b u with step dt.

    rule: RULE_EULER, RULE_BILINEAR, RULE_ZOH (exact), RULE_ZOH_SIMPLE
    (abar = e^{dt a}, bbar = dt b).
    """
    ab, bb = ctypes.c_double(), ctypes.c_double()
    rc = _load().oracle_discretize_scalar(float(a), float(b), float(dt), int(rule),
                                          ctypes.byref(ab), ctypes.byref(bb))
    if rc != 0:
        raise ValueError(f"unknown discretisation rule {rule}")
    return ab.value, bb.value


def selective_scan(x, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None,
                   *, delta_softplus: bool = True, bbar_mode: int = 0,
                   per_channel_bc: bool = False, io_dtype: str = "f32",
                   threads: int = 0):
    """Run the selective scan in float64.

    Shapes: x, delta, z: (batch, L, dim); A: (dim, N); B, C: (batch, L, N), or
    (dim, N) with ``per_channel_bc``; D, delta_bias: (dim,); h0: (batch, dim, N).
    ``io_dtype`` says how x, delta, z and time-varying B, C are stored ("f32"
    or "bf16" as uint16 bits); A, D, delta_bias, h0 and per-channel B, C are
    always fp32/fp64 values.
    Returns (out, final_state) as float64 arrays.
    """
    return _scan64(widen(x, io_dtype), delta, A, B, C, D, z, delta_bias, h0,
                   delta_softplus=delta_softplus, bbar_mode=bbar_mode,
                   per_channel_bc=per_channel_bc, io_dtype=io_dtype, threads=threads)


def _scan64(x64, delta, A, B, C, D, z, delta_bias, h0, *, delta_softplus, bbar_mode,
            per_channel_bc, io_dtype, threads):
    """selective_scan with x already widened to float64."""
    dl64 = widen(delta, io_dtype)
    z64 = widen(z, io_dtype)
    bc_dtype = "f32" if per_channel_bc else io_dtype
    B64, C64 = widen(B, bc_dtype), widen(C, bc_dtype)
    A64, D64, bias64 = widen(A), widen(D), widen(delta_bias)
    batch, L, dim = x64.shape
    N = A64.shape[1]
    assert dl64.shape == x64.shape and A64.shape == (dim, N)
    if per_channel_bc:
        assert B64.shape == (dim, N) and C64.shape == (dim, N)
    else:
        assert B64.shape == (batch, L, N) and C64.shape == (batch, L, N)
    if z64 is not None:
        assert z64.shape == x64.shape
    state = (np.array(h0, dtype=np.float64, order="C", copy=True) if h0 is not None
             else np.zeros((batch, dim, N), dtype=np.float64))
    assert state.shape == (batch, dim, N)
    out = np.empty((batch, L, dim), dtype=np.float64)
    rc = _load().oracle_selective_scan_f64(
        _ptr(x64), _ptr(dl64), _ptr(A64), _ptr(B64), _ptr(C64), _ptr(D64),
        _ptr(z64), _ptr(bias64), _ptr(out), _ptr(state),
        batch, L, dim, N, int(per_channel_bc), int(delta_softplus),
        int(h0 is not None), int(bbar_mode), int(threads))
    if rc != 0:
        raise ValueError("oracle_selective_scan_f64 rejected its arguments")
    return out, state


def selective_scan_channels(channels, x, delta, A, B, C, D=None, z=None,
                            delta_bias=None, h0=None, **kw):
    """Scan only the listed channels ``[(b, d), ...]`` over the full length.

    Inputs are sliced per batch row (no arithmetic); returns
    ``{(b, d): (out[L], final_state[N])}``.
    """
    per_channel_bc = kw.get("per_channel_bc", False)
    by_b = {}
    for b, d in channels:
        by_b.setdefault(int(b), []).append(int(d))
    res = {}
    for b, ds in by_b.items():
        ds = sorted(set(ds))
        sel = np.asarray(ds)
        sl = lambda a: None if a is None else np.ascontiguousarray(a[b:b + 1][:, :, sel])
        o, s = selective_scan(
            sl(x), sl(delta), np.asarray(A)[sel],
            np.asarray(B)[sel] if per_channel_bc else np.asarray(B)[b:b + 1],
            np.asarray(C)[sel] if per_channel_bc else np.asarray(C)[b:b + 1],
            None if D is None else np.asarray(D)[sel], sl(z),
            None if delta_bias is None else np.asarray(delta_bias)[sel],
            None if h0 is None else np.asarray(h0)[b:b + 1][:, sel], **kw)
        for j, d in enumerate(ds):
            res[(b, d)] = (o[0, :, j].copy(), s[0, j].copy())
    return res


def lti_kernel(A, B, C, dt, L: int, bbar_mode: int = 0):
    """K[d, k] = sum_n C[d,n] e^{k dt_d A[d,n]} bbar[d,n], shape (dim, L)."""
    A64, B64, C64, dt64 = widen(A), widen(B), widen(C), widen(dt)
    dim, N = A64.shape
    K = np.empty((dim, L), dtype=np.float64)
    rc = _load().oracle_lti_kernel(_ptr(A64), _ptr(B64), _ptr(C64), _ptr(dt64),
                                   _ptr(K), dim, N, L, int(bbar_mode))
    if rc != 0:
        raise ValueError("oracle_lti_kernel rejected its arguments")
    return K


def selective_scan_bwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, h0=None, *,
                       dout, dfinal=None, delta_softplus: bool = True, io_dtype: str = "f32",
                       threads: int = 0):
    """Gradients of ``selective_scan`` (bbar_mode 0, time-varying B and C) in float64.

    ``dout``: (batch, L, dim) gradient of out; ``dfinal``: (batch, dim, N) gradient
    of the final state or None.  Stored inputs are widened as in ``selective_scan``
    (``dout`` is float64 or fp32 values).  Returns a dict with dx, ddelta, dA, dB,
    dC, dD, dz (None without a gate), dbias and dh0, all float64.
    """
    x64, dl64, z64 = widen(x, io_dtype), widen(delta, io_dtype), widen(z, io_dtype)
    B64, C64 = widen(B, io_dtype), widen(C, io_dtype)
    A64, D64, bias64, h64 = widen(A), widen(D), widen(delta_bias), widen(h0)
    g64, gf64 = widen(dout), widen(dfinal)
    batch, L, dim = x64.shape
    N = A64.shape[1]
    assert B64.shape == (batch, L, N) and C64.shape == (batch, L, N) and g64.shape == x64.shape
    r = {k: np.zeros(s_, dtype=np.float64) for k, s_ in (
        ("dx", x64.shape), ("ddelta", x64.shape), ("dA", (dim, N)), ("dB", (batch, L, N)),
        ("dC", (batch, L, N)), ("dD", (dim,)), ("dz", x64.shape), ("dbias", (dim,)),
        ("dh0", (batch, dim, N)))}
    rc = _load().oracle_selective_scan_bwd_f64(
        _ptr(x64), _ptr(dl64), _ptr(A64), _ptr(B64), _ptr(C64), _ptr(D64), _ptr(z64), _ptr(bias64),
        _ptr(h64), _ptr(g64), _ptr(gf64), _ptr(r["dx"]), _ptr(r["ddelta"]), _ptr(r["dA"]),
        _ptr(r["dB"]), _ptr(r["dC"]), _ptr(r["dD"]), _ptr(r["dz"]), _ptr(r["dbias"]), _ptr(r["dh0"]),
        batch, L, dim, N, int(delta_softplus), int(threads))
    if rc != 0:
        raise ValueError("oracle_selective_scan_bwd_f64 rejected its arguments")
    if z64 is None:
        r["dz"] = None
    return r


CONV_WIDTH = 4  # taps of the Mamba block's depthwise causal convolution


def conv_silu(x, w, cb=None, hist=None, io_dtype: str = "f32", threads: int = 0):
    """u = silu(sum_k w[d,k] x[t-k] + cb[d]) with the W-1 inputs before the
    sequence taken from ``hist`` (batch, dim, W-1), oldest first (zeros when None).

    x: (batch, L, dim) stored as ``io_dtype``; w: (dim, W); cb: (dim,) or None.
    Returns (u, hist_out) in float64; hist_out holds the last W-1 inputs of the
    history-extended sequence, oldest first.
    """
    x64 = widen(x, io_dtype)
    w64, cb64 = widen(w), widen(cb)
    batch, L, dim = x64.shape
    W = w64.shape[1]
    assert w64.shape == (dim, W)
    h64 = None if hist is None else widen(hist)
    if h64 is not None:
        assert h64.shape == (batch, dim, W - 1)
    u = np.empty_like(x64)
    hout = np.empty((batch, dim, W - 1), dtype=np.float64)
    rc = _load().oracle_conv_silu(_ptr(x64), _ptr(w64), _ptr(cb64), _ptr(h64), _ptr(u),
                                  _ptr(hout), batch, L, dim, W, int(threads))
    if rc != 0:
        raise ValueError("oracle_conv_silu rejected its arguments")
    return u, hout


def conv_selective_scan(x, conv_w, conv_b, conv_hist, delta, A, B, C, D=None, z=None,
                        delta_bias=None, h0=None, *, delta_softplus: bool = True,
                        bbar_mode: int = 0, per_channel_bc: bool = False,
                        io_dtype: str = "f32", threads: int = 0):
    """The block prologue followed by the selective scan on its output:
    u = conv_silu(x, ...), then selective_scan with x := u (the scan input and the
    D skip both take u).  Returns (out, final_state, conv_hist_out) in float64."""
    u, hout = conv_silu(x, conv_w, conv_b, conv_hist, io_dtype=io_dtype, threads=threads)
    out, st = _scan64(u, delta, A, B, C, D, z, delta_bias, h0,
                      delta_softplus=delta_softplus, bbar_mode=bbar_mode,
                      per_channel_bc=per_channel_bc, io_dtype=io_dtype, threads=threads)
    return out, st, hout


def causal_conv(x, K, D=None, io_dtype: str = "f32", threads: int = 0):
    """out[b,t,d] = sum_{k<=t} K[d,k] x[b,t-k,d] + D[d] x[b,t,d]."""
    x64 = widen(x, io_dtype)
    K64, D64 = widen(K), widen(D)
    batch, L, dim = x64.shape
    assert K64.shape == (dim, L)
    out = np.empty_like(x64)
    rc = _load().oracle_causal_conv(_ptr(x64), _ptr(K64), _ptr(D64), _ptr(out),
                                    batch, L, dim, int(threads))
    if rc != 0:
        raise ValueError("oracle_causal_conv rejected its arguments")
    return out


def ssd(x, dt, A, B, C, D=None, z=None, dt_bias=None, h0=None, *, dt_softplus: bool = True,
        io_dtype: str = "bf16", threads: int = 0):
    """Mamba-2 SSD layer (scalar decay per head) stepped as a recurrence, float64.

    Shapes: x, z: (batch, L, H, P); dt: (batch, L, H); A, D, dt_bias: (H,);
    B, C: (batch, L, G, N) with head h reading group h // (H // G);
    h0: (batch, H, P, N).  x, dt, z, B, C are stored as ``io_dtype``; A, D,
    dt_bias and h0 are fp32/fp64 values.  Returns (out, final_state).
    """
    x64, dt64, z64 = widen(x, io_dtype), widen(dt, io_dtype), widen(z, io_dtype)
    B64, C64 = widen(B, io_dtype), widen(C, io_dtype)
    A64, D64, bias64 = widen(A), widen(D), widen(dt_bias)
    batch, L, H, P = x64.shape
    G, N = B64.shape[2], B64.shape[3]
    assert dt64.shape == (batch, L, H) and A64.shape == (H,)
    assert B64.shape == (batch, L, G, N) and C64.shape == B64.shape
    if z64 is not None:
        assert z64.shape == x64.shape
    state = (np.array(h0, dtype=np.float64, order="C", copy=True) if h0 is not None
             else np.zeros((batch, H, P, N), dtype=np.float64))
    assert state.shape == (batch, H, P, N)
    out = np.empty_like(x64)
    rc = _load().oracle_ssd_f64(
        _ptr(x64), _ptr(dt64), _ptr(A64), _ptr(B64), _ptr(C64), _ptr(D64), _ptr(z64),
        _ptr(bias64), _ptr(out), _ptr(state), batch, L, H, P, G, N, int(dt_softplus),
        int(h0 is not None), int(threads))
    if rc != 0:
        raise ValueError("oracle_ssd_f64 rejected its arguments")
    return out, state
