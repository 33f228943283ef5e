"""The Mamba-block prologue (depthwise causal conv of width 4 + silu on x) fused into
the scan, against the float64 oracle (prologue, then the scan on its output).

Outputs, the final state and the three-input history are compared element by
element with the floored relative error (1e-5 for fp32 inputs, 2e-2 for bf16).
"""
import zlib

import numpy as np
import pytest

import oracle
from selective_state_space_112_b300.workloads import make_conv, make_workload

from helpers import assert_close, device_inputs, to_torch

pytestmark = pytest.mark.gpu


def run_conv_gpu(w, cv, dev=None):
    import torch
    import selective_state_space_112_b300 as ssm
    dev = dev or device_inputs(w)
    fs = dev["final_state"].clone()
    cs = (to_torch(cv.hist) if cv.hist is not None else
          torch.full((w.batch, w.dim, 3), float("nan"), dtype=torch.float32, device="cuda"))
    o, f = ssm.ssm_conv_selective_scan_fwd(
        dev["x"], to_torch(cv.w), to_torch(cv.b), cs, dev["delta"], dev["A"], dev["B"], dev["C"],
        dev["D"], dev["z"], dev["delta_bias"], final_state=fs, delta_softplus=w.delta_softplus,
        state_in=w.h0 is not None)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    return f64(o), f64(f), f64(cs)


def run_conv_oracle(w, cv):
    return oracle.conv_selective_scan(w.x, cv.w, cv.b, cv.hist, w.delta, w.A, w.B, w.C, D=w.D,
                                      z=w.z, delta_bias=w.delta_bias, h0=w.h0,
                                      delta_softplus=w.delta_softplus, io_dtype=w.io)


def check(w, cv, what):
    out, st, cs = run_conv_gpu(w, cv)
    ref, ref_st, ref_cs = run_conv_oracle(w, cv)
    assert_close(out, ref, w.io, f"{what}: out")
    assert_close(st, ref_st, w.io, f"{what}: final state")
    np.testing.assert_array_equal(cs, ref_cs, err_msg=f"{what}: conv history")


CASES = [
    # (name, workload kwargs, conv kwargs, forced chunks, tma)
    ("ragged_D", dict(batch=2, seqlen=300, dim=136, dstate=16), {}, 0, 1),
    ("chunks5_hist", dict(batch=2, seqlen=700, dim=96, dstate=16, state_in=True), dict(hist=True), 5, 1),
    ("chunks3_hist_generic", dict(batch=2, seqlen=400, dim=72, dstate=16, state_in=True),
     dict(hist=True), 3, 0),
    ("ragged_L", dict(batch=3, seqlen=77, dim=64, dstate=16), {}, 0, 1),
    ("ragged_L_generic", dict(batch=3, seqlen=77, dim=64, dstate=16), {}, 2, 0),
    ("no_gate_no_bias", dict(batch=2, seqlen=200, dim=48, dstate=16, gate=False, with_bias=False),
     dict(with_bias=False), 2, 1),
    ("N8", dict(batch=2, seqlen=150, dim=200, dstate=8), {}, 2, 1),
    ("N4", dict(batch=2, seqlen=150, dim=64, dstate=4), {}, 0, 1),
    ("N13", dict(batch=2, seqlen=96, dim=64, dstate=13), {}, 2, 1),
    ("L2_hist", dict(batch=2, seqlen=2, dim=40, dstate=16, state_in=True), dict(hist=True), 0, 1),
    ("L1_hist_step", dict(batch=4, seqlen=1, dim=40, dstate=16, state_in=True), dict(hist=True), 0, 1),
    ("L1_step", dict(batch=4, seqlen=1, dim=40, dstate=16), {}, 0, 1),
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("name,kw,ckw,chunks,tma", CASES, ids=[c[0] for c in CASES])
def test_conv_prologue_parity(name, kw, ckw, chunks, tma, io):
    import selective_state_space_112_b300 as ssm
    w = make_workload(name, io=io, seed=zlib.crc32(name.encode()) % 1000, **kw)
    cv = make_conv(w, **ckw)
    try:
        ssm.ssm_set_option("chunks", chunks)
        ssm.ssm_set_option("tma", tma)
        check(w, cv, f"{name}/{io}")
    finally:
        ssm.ssm_set_option("chunks", 0)
        ssm.ssm_set_option("tma", 1)


LANE_CASES = [
    # (name, workload kwargs, conv kwargs, forced chunks, tma, lanes per channel)
    ("g2_ragged_D", dict(batch=2, seqlen=300, dim=136, dstate=16), {}, 0, 1, 2),
    ("g2_chunks5_hist", dict(batch=2, seqlen=700, dim=96, dstate=16, state_in=True),
     dict(hist=True), 5, 1, 2),
    ("g2_chunks3_generic", dict(batch=2, seqlen=400, dim=72, dstate=16, state_in=True),
     dict(hist=True), 3, 0, 2),
    ("g4_ragged_L", dict(batch=3, seqlen=77, dim=64, dstate=16), {}, 2, 1, 4),
    ("g4_N13", dict(batch=2, seqlen=96, dim=64, dstate=13), {}, 0, 1, 4),
    ("g2_N32_hist", dict(batch=2, seqlen=260, dim=80, dstate=32, state_in=True), dict(hist=True), 3, 1, 2),
    ("g4_N64", dict(batch=2, seqlen=140, dim=48, dstate=64), {}, 2, 1, 4),
    ("g4_N24_generic", dict(batch=2, seqlen=150, dim=40, dstate=24, gate=False, with_bias=False),
     dict(with_bias=False), 0, 0, 4),
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("name,kw,ckw,chunks,tma,lanes", LANE_CASES, ids=[c[0] for c in LANE_CASES])
def test_conv_prologue_lanes_per_channel(name, kw, ckw, chunks, tma, lanes, io):
    """Two and four lanes per channel (each lane gathers its channel's raw inputs of
    a group of rounds by shuffles and keeps the convolution at its own steps), and
    states past 16 (N 24, 32, 64), which only those layouts cover."""
    import selective_state_space_112_b300 as ssm
    w = make_workload(name, io=io, seed=zlib.crc32(name.encode()) % 1000, **kw)
    cv = make_conv(w, **ckw)
    try:
        ssm.ssm_set_option("chunks", chunks)
        ssm.ssm_set_option("tma", tma)
        ssm.ssm_set_option("lanes", lanes)
        check(w, cv, f"{name}/{io}")
    finally:
        ssm.ssm_set_option("chunks", 0)
        ssm.ssm_set_option("tma", 1)
        ssm.ssm_set_option("lanes", 0)


def test_conv_prologue_without_softplus_ragged():
    """Steps past the sequence end without softplus take the per-step test path.
    The steps are given directly (small positive values, no bias)."""
    from selective_state_space_112_b300.workloads import f32_to_bf16_bits
    w = make_workload("nosp", batch=2, seqlen=45, dim=64, dstate=16, io="bf16", seed=3)
    steps = np.abs(np.random.default_rng(3).standard_normal(w.delta.shape)).astype(np.float32) * 0.05
    w.delta = f32_to_bf16_bits(steps)
    w.delta_bias = None
    w.delta_softplus = False
    check(w, make_conv(w), "no softplus")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_prologue_continuation(io):
    """A sequence run as two calls, the second with state_in and both states (the
    SSM state and the three-input history) carried, matches one call over the whole
    sequence, and the oracle."""
    import torch
    import selective_state_space_112_b300 as ssm
    L1, L2 = 130, 97
    w = make_workload("cont", batch=2, seqlen=L1 + L2, dim=96, dstate=16, io=io, seed=17)
    cv = make_conv(w)
    dev = device_inputs(w)
    cw, cb = to_torch(cv.w), to_torch(cv.b)
    full = ssm.ssm_conv_selective_scan_fwd(dev["x"], cw, cb, None, dev["delta"], dev["A"], dev["B"],
                                           dev["C"], dev["D"], dev["z"], dev["delta_bias"])[0]
    part = lambda t, a, b: None if t is None else t[:, a:b].contiguous()
    fs = torch.zeros((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
    cs = torch.zeros((w.batch, w.dim, 3), dtype=torch.float32, device="cuda")
    outs = []
    for a, b in ((0, L1), (L1, L1 + L2)):
        o, _ = ssm.ssm_conv_selective_scan_fwd(
            part(dev["x"], a, b), cw, cb, cs, part(dev["delta"], a, b), dev["A"], part(dev["B"], a, b),
            part(dev["C"], a, b), dev["D"], part(dev["z"], a, b), dev["delta_bias"], final_state=fs,
            state_in=True)
        outs.append(o)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    got = torch.cat(outs, dim=1).float().cpu().numpy().astype(np.float64)
    ref, ref_st, ref_cs = run_conv_oracle(w, cv)
    assert_close(got, ref, io, "continued")
    assert_close(full.float().cpu().numpy().astype(np.float64), ref, io, "one call")
    assert_close(fs.cpu().numpy().astype(np.float64), ref_st, io, "continued final state")
    np.testing.assert_array_equal(cs.cpu().numpy().astype(np.float64), ref_cs)


def test_conv_history_of_an_empty_sequence():
    """seqlen 0 keeps the history with state_in and zero-fills it without."""
    import torch
    import selective_state_space_112_b300 as ssm
    w = make_workload("empty", batch=2, seqlen=0, dim=32, dstate=16, io="f32", seed=1)
    cv = make_conv(w, hist=True)
    dev = device_inputs(w)
    hist = to_torch(cv.hist)
    for state_in, expect in ((True, cv.hist), (False, np.zeros_like(cv.hist))):
        cs = hist.clone()
        fs = torch.randn((w.batch, w.dim, w.dstate), device="cuda")
        ssm.ssm_conv_selective_scan_fwd(dev["x"], to_torch(cv.w), to_torch(cv.b), cs, dev["delta"],
                                        dev["A"], dev["B"], dev["C"], dev["D"], dev["z"],
                                        dev["delta_bias"], final_state=fs, state_in=state_in)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(cs.cpu().numpy(), expect)
