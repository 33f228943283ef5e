"""Shared test helpers: move a Workload to the GPU, run the CUDA path through the
C ABI, run the oracle, and compare with the floored relative error."""
from __future__ import annotations

import numpy as np

import oracle
from oracle.metrics import TOL, report


def to_torch(a, device="cuda"):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def device_inputs(w, device="cuda"):
    import torch
    dev = {k: to_torch(getattr(w, k), device)
           for k in ("x", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    dev["final_state"] = (to_torch(w.h0, device) if w.h0 is not None else
                          torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device=device))
    return dev


def run_gpu(w, dev=None, out=None, bbar_mode=0):
    """Run the CUDA path; return (out, final_state) as float64 numpy arrays."""
    import torch
    import selective_state_space_112_b300 as ssm
    dev = dev or device_inputs(w)
    fs = dev["final_state"].clone() if w.h0 is not None else dev["final_state"]
    o, f = ssm.ssm_selective_scan_fwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"],
                                      dev["D"], dev["z"], dev["delta_bias"], out=out,
                                      final_state=fs, delta_softplus=w.delta_softplus,
                                      state_in=w.h0 is not None, bbar_mode=bbar_mode)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), f.cpu().numpy().astype(np.float64)


def run_oracle(w, threads=0, bbar_mode=0):
    return oracle.selective_scan(w.x, w.delta, w.A, w.B, w.C, D=w.D, z=w.z,
                                 delta_bias=w.delta_bias, h0=w.h0,
                                 delta_softplus=w.delta_softplus,
                                 per_channel_bc=w.per_channel_bc, io_dtype=w.io,
                                 threads=threads, bbar_mode=bbar_mode)


def assert_close(got, ref, io, what="", floor=None):
    r = report(got, ref, floor)
    assert r["err"] <= TOL[io], f"{what}: {r} (tol {TOL[io]})"
    return r
