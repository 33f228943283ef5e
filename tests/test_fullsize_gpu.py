"""The fused block prologue and the backward pass at the sizes the benchmark times.

The small cases of test_conv_gpu.py and test_bwd_gpu.py check every element; these
run the full-size layers in the launch configuration (automatic lane split, chunk
plan and, for the backward, sub-chunks of the reverse carry) that bench.py times:
  * the prologue + scan on the long-context layer (1 x 131072 x 2560, N 16, bf16) and
    the 1.4B-shaped layer (4 x 4096 x 4096): every output and the final state of
    sampled channels against the oracle run on those channels over their whole
    length (the prologue and the scan are independent across channels);
  * the backward pass on a layer of the long-context width (1 x 16384 x 2560, N 16,
    bf16; the automatic plan cuts it into 29 chunks): every gradient element, the
    sums over channels (dB, dC) included, against the oracle over all channels.
Bars as everywhere: floored max relative error <= 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest

import oracle
from selective_state_space_112_b300.workloads import (bf16_bits_to_f32, config, f32_to_bf16_bits,
                                                      make_conv, make_workload)

from helpers import assert_close, device_inputs, to_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    import selective_state_space_112_b300 as ssm
    for k, v in dict(chunks=0, pow_path=1, tma=1, lanes=0).items():
        ssm.ssm_set_option(k, v)
    yield


def _prologue_sampled(name, nsample, seed):
    import torch
    import selective_state_space_112_b300 as ssm
    w = config(name)
    cv = make_conv(w)
    dev = device_inputs(w)
    out, fs = ssm.ssm_conv_selective_scan_fwd(dev["x"], to_torch(cv.w), to_torch(cv.b), None,
                                              dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                              dev["z"], dev["delta_bias"])
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    by_b = {}
    for _ in range(nsample):
        by_b.setdefault(int(rng.integers(w.batch)), set()).add(int(rng.integers(w.dim)))
    by_b.setdefault(0, set()).add(0)
    by_b.setdefault(w.batch - 1, set()).add(w.dim - 1)
    for b, ds in sorted(by_b.items()):
        sel = np.array(sorted(ds))
        sl = lambda a: np.ascontiguousarray(a[b:b + 1][:, :, sel])
        r_out, r_fs, _ = oracle.conv_selective_scan(
            sl(w.x), cv.w[sel], cv.b[sel], None, sl(w.delta), w.A[sel], w.B[b:b + 1], w.C[b:b + 1],
            D=w.D[sel], z=sl(w.z), delta_bias=w.delta_bias[sel], io_dtype=w.io)
        g_out = out[b:b + 1][:, :, torch.as_tensor(sel, device=out.device)].float().cpu().numpy()
        g_fs = fs[b:b + 1][:, torch.as_tensor(sel, device=fs.device)].cpu().numpy()
        assert_close(g_out.astype(np.float64), r_out, w.io, f"{name} prologue, row {b}: out")
        assert_close(g_fs.astype(np.float64), r_fs, w.io, f"{name} prologue, row {b}: final state")
    assert bool(torch.isfinite(out.float()).all())


def test_prologue_long_bf16_sampled():
    _prologue_sampled("long_bf16", 24, 41)


def test_prologue_mamba1p4b_bf16_sampled():
    _prologue_sampled("mamba1p4b_bf16", 48, 42)


def test_backward_long_context_width():
    import torch
    import selective_state_space_112_b300 as ssm
    w = make_workload("bwd_wide", batch=1, seqlen=16384, dim=2560, dstate=16, io="bf16", seed=44)
    rng = np.random.default_rng(45)
    dout = f32_to_bf16_bits(rng.standard_normal(w.x.shape, dtype=np.float32))
    dfinal = rng.standard_normal((w.batch, w.dim, w.dstate), dtype=np.float32)
    dev = device_inputs(w)
    g = ssm.ssm_selective_scan_bwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"],
                                   dev["z"], dev["delta_bias"], None, to_torch(dout), to_torch(dfinal))
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    got = {k: (None if v is None else v.float().cpu().numpy().astype(np.float64)) for k, v in g.items()}
    del g, dev
    torch.cuda.empty_cache()
    ref = oracle.selective_scan_bwd(w.x, w.delta, w.A, w.B, w.C, w.D, w.z, w.delta_bias, None,
                                    dout=bf16_bits_to_f32(dout).astype(np.float64), dfinal=dfinal,
                                    io_dtype=w.io)
    for gk, rk in (("dx", "dx"), ("ddelta", "ddelta"), ("dz", "dz"), ("dA", "dA"), ("dB", "dB"),
                   ("dC", "dC"), ("dD", "dD"), ("ddelta_bias", "dbias")):
        assert_close(got[gk], ref[rk], w.io, f"backward 1x16384x2560: {gk}")
