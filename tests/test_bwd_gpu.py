"""The backward pass (gradients with the states rebuilt) against the float64 oracle.

Every gradient (dx, ddelta, dz, dA, dB, dC, dD, the step-bias gradient and the
initial-state gradient) is compared element by element with the floored relative
error, at the forward's tolerances (1e-5 for fp32 inputs, 2e-2 for bf16), on seeded
inputs with an upstream gradient dout ~ N(0, 1) and a final-state gradient.
"""
import zlib

import numpy as np
import pytest

import oracle
from selective_state_space_112_b300.workloads import (bf16_bits_to_f32, f32_to_bf16_bits,
                                                      make_workload)

from helpers import assert_close, device_inputs, to_torch

pytestmark = pytest.mark.gpu

NAMES = [("dx", "dx"), ("ddelta", "ddelta"), ("dz", "dz"), ("dA", "dA"), ("dB", "dB"),
         ("dC", "dC"), ("dD", "dD"), ("ddelta_bias", "dbias"), ("dh_init", "dh0")]


def grads(w, seed, with_dfinal=True):
    """Run the CUDA backward and the oracle on the same inputs and upstream gradients."""
    import torch
    import selective_state_space_112_b300 as ssm
    rng = np.random.default_rng(seed)
    dout = rng.standard_normal(w.x.shape, dtype=np.float32)
    dout_stored = f32_to_bf16_bits(dout) if w.io == "bf16" else dout
    dout64 = bf16_bits_to_f32(dout_stored).astype(np.float64) if w.io == "bf16" else dout.astype(np.float64)
    dfinal = rng.standard_normal((w.batch, w.dim, w.dstate), dtype=np.float32) if with_dfinal else None
    dev = device_inputs(w)
    g = ssm.ssm_selective_scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                   dev["z"], dev["delta_bias"],
                                   dev["final_state"] if w.h0 is not None else None,
                                   to_torch(dout_stored), to_torch(dfinal),
                                   delta_softplus=w.delta_softplus)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    got = {k: (None if v is None else v.float().cpu().numpy().astype(np.float64)) for k, v in g.items()}
    ref = oracle.selective_scan_bwd(w.x, w.delta, w.A, w.B, w.C, w.D, w.z, w.delta_bias, w.h0,
                                    dout=dout64, dfinal=dfinal, delta_softplus=w.delta_softplus,
                                    io_dtype=w.io)
    return got, ref


def check(w, what, seed=0, with_dfinal=True):
    got, ref = grads(w, seed, with_dfinal)
    for gk, rk in NAMES:
        if got[gk] is None:
            continue
        assert_close(got[gk], ref[rk], w.io, f"{what}: {gk}")


CASES = [
    # (name, workload kwargs, forced chunks)
    ("auto", dict(batch=2, seqlen=300, dim=96, dstate=16), 0),
    ("chunks3_h0", dict(batch=2, seqlen=400, dim=64, dstate=16, state_in=True), 3),
    ("chunks7_ragged", dict(batch=1, seqlen=455, dim=136, dstate=16, state_in=True), 7),
    ("N8", dict(batch=2, seqlen=130, dim=72, dstate=8), 2),
    ("N4", dict(batch=3, seqlen=97, dim=40, dstate=4), 2),
    ("N13", dict(batch=2, seqlen=96, dim=64, dstate=13), 2),
    ("no_gate_D_bias", dict(batch=2, seqlen=150, dim=48, dstate=16, gate=False, with_D=False,
                            with_bias=False), 2),
    ("L2_h0", dict(batch=2, seqlen=2, dim=40, dstate=16, state_in=True), 0),
    ("L1", dict(batch=4, seqlen=1, dim=40, dstate=16), 0),
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("name,kw,chunks", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(name, kw, chunks, io):
    import selective_state_space_112_b300 as ssm
    w = make_workload(name, io=io, seed=zlib.crc32(name.encode()) % 1000, **kw)
    try:
        ssm.ssm_set_option("chunks", chunks)
        check(w, f"{name}/{io}", seed=len(name))
    finally:
        ssm.ssm_set_option("chunks", 0)


def test_backward_without_softplus_or_final_gradient():
    """Raw steps (small, positive; no bias) and no final-state gradient."""
    import selective_state_space_112_b300 as ssm
    w = make_workload("nosp", batch=2, seqlen=200, dim=64, dstate=16, io="f32", seed=4)
    w.delta = (np.abs(w.delta) * 0.05).astype(np.float32)
    w.delta_bias = None
    w.delta_softplus = False
    try:
        ssm.ssm_set_option("chunks", 3)
        check(w, "no softplus", with_dfinal=False)
    finally:
        ssm.ssm_set_option("chunks", 0)


def test_backward_of_an_empty_sequence():
    """L = 0: the final state is the initial one, so dh_init = dfinal_state and the
    parameter gradients are zero."""
    import torch
    import selective_state_space_112_b300 as ssm
    w = make_workload("e", batch=2, seqlen=0, dim=32, dstate=16, io="f32", seed=2, state_in=True)
    dev = device_inputs(w)
    dfin = torch.randn((w.batch, w.dim, w.dstate), device="cuda")
    g = ssm.ssm_selective_scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                   dev["z"], dev["delta_bias"], dev["final_state"], dev["x"], dfin)
    torch.cuda.synchronize()
    assert torch.equal(g["dh_init"], dfin)
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(g[k]).item() == 0, k
