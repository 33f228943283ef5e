"""B300-native (sm_103a) Mamba S6 selective scan and Mamba-2 SSD layer.

The compute lives in the C-ABI library ``libssmscan.so`` built from ``csrc/``
(declarations in ``include/ssm_scan.h`` and ``include/ssm_ssd.h``).  This package only marshals PyTorch
tensors (used for device memory and streams) into that ABI; it never computes
any part of the scan itself and has no CPU fallback.
"""
from __future__ import annotations

from . import _abi
from ._abi import (SSM_BC_PER_CHANNEL, SSM_BC_TIME_VARYING, SSM_BF16, SSM_F32, SSM_OK,
                   SSMError, SsdDims, SsmDims)

__all__ = ["ssm_selective_scan_fwd", "ssm_conv_selective_scan_fwd", "ssm_selective_scan_bwd",
           "ssm_selective_scan_fwd_noalloc",
           "ssm_check_status", "ssm_status_string",
           "ssm_release_workspace", "ssm_workspace_reserved_bytes", "ssm_kernel_launches",
           "ssm_set_option",
           "ssm_profile_enable", "ssm_profile_read", "ssm_ssd_fwd", "SSMError", "SsmDims",
           "SsdDims"]


def _torch():
    import torch
    return torch


def _addr(t):
    return 0 if t is None else int(t.data_ptr())


def ssm_selective_scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                           out=None, final_state=None, *, delta_softplus: bool = True,
                           state_in: bool = False, bbar_mode: int = 0,
                           return_final_state: bool = True, stream=None, _noalloc: bool = False):
    """Selective-scan forward on the current CUDA device.

    x, delta, z: (batch, L, dim) float32 or bfloat16 CUDA tensors, contiguous.
    A: (dim, N) float32.  B, C: (batch, L, N) in the io dtype (time-varying,
    shared by all channels) or (dim, N) float32 (constant per channel).
    D, delta_bias: (dim,) float32 or None.  With ``state_in`` the initial state
    is read from ``final_state`` (batch, dim, N) float32, which is then
    overwritten with the final state.  Returns ``(out, final_state)``; the
    call is asynchronous on ``stream`` (default: torch's current stream).
    """
    return _scan(x, delta, A, B, C, D, z, delta_bias, out, final_state, None,
                 delta_softplus=delta_softplus, state_in=state_in, bbar_mode=bbar_mode,
                 return_final_state=return_final_state, stream=stream, noalloc=_noalloc)


def ssm_conv_selective_scan_fwd(x, conv_w, conv_b, conv_state, delta, A, B, C, D=None, z=None,
                                delta_bias=None, out=None, final_state=None, *,
                                delta_softplus: bool = True, state_in: bool = False,
                                return_final_state: bool = True, stream=None):
    """Selective-scan forward with the Mamba-block prologue on x:
    u = silu(sum_k conv_w[d,k] x[t-k] + conv_b[d]) feeds the scan in place of x.

    conv_w: (dim, 4) float32 (tap k multiplies the input k steps back); conv_b: (dim,)
    float32 or None; conv_state: (batch, dim, 3) float32 or None, read first as the
    three inputs before the sequence when ``state_in`` and overwritten with the last
    three inputs.  Other arguments as ``ssm_selective_scan_fwd`` (time-varying B, C).
    Returns ``(out, final_state)``.
    """
    torch = _torch()
    dim = x.shape[-1]
    for name, t, shp in (("conv_w", conv_w, (dim, 4)), ("conv_b", conv_b, (dim,)),
                         ("conv_state", conv_state, (x.shape[0], dim, 3))):
        if t is None:
            continue
        if t.dtype != torch.float32 or tuple(t.shape) != shp:
            raise ValueError(f"{name}: expected float32 {shp}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if conv_w is None:
        raise ValueError("conv_w is required")
    return _scan(x, delta, A, B, C, D, z, delta_bias, out, final_state,
                 (conv_w, conv_b, conv_state), delta_softplus=delta_softplus, state_in=state_in,
                 bbar_mode=0, return_final_state=return_final_state, stream=stream, noalloc=False)


def ssm_selective_scan_bwd(x, delta, A, B, C, D, z, delta_bias, h_init, dout, dfinal_state=None,
                           *, delta_softplus: bool = True, stream=None, grads=None):
    """Gradients of ``ssm_selective_scan_fwd`` (time-varying B, C; bbar_mode 0).

    Inputs as the forward (h_init: (batch, dim, N) float32 or None); dout: gradient of
    out, same shape and dtype as x; dfinal_state: gradient of the final state (float32)
    or None.  Returns a dict: dx, ddelta, dz (io dtype; dz None without a gate),
    dA (dim, N), dB, dC (batch, L, N), dD, ddelta_bias (dim,), dh_init (batch, dim, N)
    -- all float32 except dx, ddelta, dz; dD / ddelta_bias / dh_init are None when D /
    delta_bias / h_init are.  ``grads``: such a dict from an earlier call with the same
    shapes, whose tensors are overwritten instead of allocating new ones.
    """
    torch = _torch()
    if x.dtype == torch.float32:
        io = SSM_F32
    elif x.dtype == torch.bfloat16:
        io = SSM_BF16
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    batch, L, dim = x.shape
    N = A.shape[-1]
    if B.dim() != 3:
        raise ValueError("the backward pass takes time-varying B and C (batch, L, N)")
    for name, t, dt, shp in (
            ("delta", delta, x.dtype, x.shape), ("z", z, x.dtype, x.shape), ("dout", dout, x.dtype, x.shape),
            ("A", A, torch.float32, (dim, N)), ("D", D, torch.float32, (dim,)),
            ("delta_bias", delta_bias, torch.float32, (dim,)), ("B", B, x.dtype, (batch, L, N)),
            ("C", C, x.dtype, (batch, L, N)), ("h_init", h_init, torch.float32, (batch, dim, N)),
            ("dfinal_state", dfinal_state, torch.float32, (batch, dim, N))):
        if t is None:
            continue
        if t.dtype != dt or tuple(t.shape) != tuple(shp):
            raise ValueError(f"{name}: expected {dt} {tuple(shp)}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    f32 = dict(dtype=torch.float32, device=x.device)
    g = grads if grads is not None else {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x),
         "dz": torch.empty_like(x) if z is not None else None,
         "dA": torch.empty((dim, N), **f32), "dB": torch.empty((batch, L, N), **f32),
         "dC": torch.empty((batch, L, N), **f32),
         "dD": torch.empty((dim,), **f32) if D is not None else None,
         "ddelta_bias": torch.empty((dim,), **f32) if delta_bias is not None else None,
         "dh_init": torch.empty((batch, dim, N), **f32) if h_init is not None else None}
    dims = SsmDims(batch=batch, seqlen=L, dim=dim, dstate=N, io_dtype=io, bc_layout=SSM_BC_TIME_VARYING,
                   delta_softplus=int(bool(delta_softplus)), state_in=0, bbar_mode=0, reserved=0)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    addrs = [_addr(t) for t in (x, delta, A, B, C, D, z, delta_bias, h_init, dout, dfinal_state,
                                g["dx"], g["ddelta"], g["dA"], g["dB"], g["dC"], g["dD"], g["dz"],
                                g["ddelta_bias"], g["dh_init"])]
    rc = _abi.call_bwd(addrs, dims, int(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_selective_scan_bwd")
    return g


def _scan(x, delta, A, B, C, D, z, delta_bias, out, final_state, conv, *, delta_softplus,
          state_in, bbar_mode, return_final_state, stream, noalloc):
    torch = _torch()
    if x.dtype == torch.float32:
        io = SSM_F32
    elif x.dtype == torch.bfloat16:
        io = SSM_BF16
    else:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    if x.dim() != 3:
        raise ValueError("x must be (batch, L, dim)")
    batch, L, dim = x.shape
    N = A.shape[-1]
    per_channel = B.dim() == 2
    for name, t, dt, shp in (
            ("delta", delta, x.dtype, x.shape), ("z", z, x.dtype, x.shape),
            ("A", A, torch.float32, (dim, N)), ("D", D, torch.float32, (dim,)),
            ("delta_bias", delta_bias, torch.float32, (dim,)),
            ("B", B, torch.float32 if per_channel else x.dtype, (dim, N) if per_channel else (batch, L, N)),
            ("C", C, torch.float32 if per_channel else x.dtype, (dim, N) if per_channel else (batch, L, N))):
        if t is None:
            continue
        if t.dtype != dt or tuple(t.shape) != tuple(shp):
            raise ValueError(f"{name}: expected {dt} {tuple(shp)}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    if final_state is None and (state_in or return_final_state):
        if state_in:
            raise ValueError("state_in needs final_state holding the initial state")
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=x.device)
    dims = SsmDims(batch=batch, seqlen=L, dim=dim, dstate=N, io_dtype=io,
                   bc_layout=SSM_BC_PER_CHANNEL if per_channel else SSM_BC_TIME_VARYING,
                   delta_softplus=int(bool(delta_softplus)), state_in=int(bool(state_in)),
                   bbar_mode=int(bbar_mode), reserved=0)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    if conv is not None:
        cw, cb, cs = conv
        rc = _abi.call_conv_fwd(_addr(x), _addr(cw), _addr(cb), _addr(cs), _addr(delta), _addr(A),
                                _addr(B), _addr(C), _addr(D), _addr(z), _addr(delta_bias),
                                _addr(out), _addr(final_state), dims, int(stream))
        what = "ssm_conv_selective_scan_fwd"
    else:
        rc = _abi.call_fwd(_addr(x), _addr(delta), _addr(A), _addr(B), _addr(C), _addr(D),
                           _addr(z), _addr(delta_bias), _addr(out), _addr(final_state), dims,
                           int(stream), noalloc=noalloc)
        what = "ssm_selective_scan_fwd_noalloc" if noalloc else "ssm_selective_scan_fwd"
    if rc != SSM_OK:
        raise SSMError(rc, what)
    return out, final_state


def ssm_ssd_fwd(x, dt, A, B, C, D=None, z=None, dt_bias=None, out=None, final_state=None, *,
                dt_softplus: bool = True, state_in: bool = False, return_final_state: bool = True,
                stream=None):
    """Mamba-2 SSD layer forward on the current CUDA device.

    x, z: (batch, L, H, P) bfloat16; dt: (batch, L, H) bfloat16 (raw step);
    A, D, dt_bias: (H,) float32 (D, dt_bias may be None); B, C: (batch, L, G, N)
    bfloat16, head h reading group h // (H // G).  With ``state_in`` the initial
    state is read from ``final_state`` (batch, H, P, N) float32, which is then
    overwritten with the final state.  Returns ``(out, final_state)``.
    """
    torch = _torch()
    if x.dim() != 4:
        raise ValueError("x must be (batch, L, heads, headdim)")
    batch, L, H, P = x.shape
    if B.dim() != 4:
        raise ValueError("B must be (batch, L, groups, dstate)")
    G, N = B.shape[2], B.shape[3]
    io = SSM_BF16 if x.dtype == torch.bfloat16 else SSM_F32
    for name, t, dty, shp in (
            ("dt", dt, x.dtype, (batch, L, H)), ("z", z, x.dtype, x.shape),
            ("A", A, torch.float32, (H,)), ("D", D, torch.float32, (H,)),
            ("dt_bias", dt_bias, torch.float32, (H,)),
            ("B", B, x.dtype, (batch, L, G, N)), ("C", C, x.dtype, (batch, L, G, N))):
        if t is None:
            continue
        if t.dtype != dty or tuple(t.shape) != tuple(shp):
            raise ValueError(f"{name}: expected {dty} {tuple(shp)}, got {t.dtype} {tuple(t.shape)}")
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError("x must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty_like(x)
    if final_state is None and (state_in or return_final_state):
        if state_in:
            raise ValueError("state_in needs final_state holding the initial state")
        final_state = torch.empty((batch, H, P, N), dtype=torch.float32, device=x.device)
    dims = SsdDims(batch=batch, seqlen=L, nheads=H, headdim=P, ngroups=G, dstate=N, io_dtype=io,
                   dt_softplus=int(bool(dt_softplus)), state_in=int(bool(state_in)), reserved=0)
    if stream is None:
        stream = torch.cuda.current_stream(x.device).cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    rc = _abi.call_ssd(_addr(x), _addr(dt), _addr(A), _addr(B), _addr(C), _addr(D), _addr(z),
                       _addr(dt_bias), _addr(out), _addr(final_state), dims, int(stream))
    if rc != SSM_OK:
        raise SSMError(rc, "ssm_ssd_fwd")
    return out, final_state


def ssm_selective_scan_fwd_noalloc(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                                   out=None, final_state=None, **kw):
    """Same call as ``ssm_selective_scan_fwd`` through the library entry point that
    allocates no device memory for its own work: the chunk-carry workspace sits in a
    fixed 16 MiB device array inside the library (shared by all such calls on a device,
    so calls that overlap on the GPU race), and problems that need more raise SSMError
    with code SSM_ERR_SCRATCH.  It is meant for callers that cannot let a library
    allocate.  ``out`` and ``final_state`` should be passed in by such callers; when
    they are omitted, this binding creates them with torch, as the other entry point
    does."""
    return ssm_selective_scan_fwd(x, delta, A, B, C, D, z, delta_bias, out, final_state,
                                  _noalloc=True, **kw)


def ssm_check_status(stream=None) -> int:
    if stream is None:
        stream = _torch().cuda.current_stream().cuda_stream
    elif hasattr(stream, "cuda_stream"):
        stream = stream.cuda_stream
    return _abi.check_status(int(stream))


ssm_status_string = _abi.status_string
ssm_release_workspace = _abi.release_workspace
ssm_workspace_reserved_bytes = _abi.workspace_reserved_bytes
ssm_kernel_launches = _abi.kernel_launches
ssm_set_option = _abi.set_option
ssm_profile_enable = _abi.profile_enable
ssm_profile_read = _abi.profile_read
