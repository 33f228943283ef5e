"""The Mamba-2 SSD layer (ssm_ssd_fwd) against the float64 oracle's recurrence.

Outputs and the final state are compared element by element with the floored
relative error at the bf16 bar (2e-2): inputs are bf16, and the kernel's tensor
core operands (the masked decay matrix, the decay-weighted inputs, the carried
state) are pairs of bf16 values with fp32 accumulation.  Sizes span several 128-step
chunks and ragged tails; the full-size layer is checked on sampled heads.
"""
import zlib

import numpy as np
import pytest

import oracle
from selective_state_space_112_b300.workloads import SSD_CONFIGS, f32_to_bf16_bits, make_ssd

from helpers import assert_close, to_torch

pytestmark = pytest.mark.gpu


def ssd_gpu(w, h0=None):
    import torch
    import selective_state_space_112_b300 as ssm
    h0 = w.h0 if h0 is None else h0
    fs = (to_torch(h0).clone() if h0 is not None else
          torch.full((w.batch, w.nheads, w.headdim, w.dstate), float("nan"), device="cuda"))
    o, f = ssm.ssm_ssd_fwd(to_torch(w.x), to_torch(w.dt), to_torch(w.A), to_torch(w.B), to_torch(w.C),
                           to_torch(w.D), to_torch(w.z), to_torch(w.dt_bias), final_state=fs,
                           dt_softplus=w.dt_softplus, state_in=h0 is not None)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    return o.float().cpu().numpy().astype(np.float64), f.cpu().numpy().astype(np.float64)


def ssd_oracle(w):
    return oracle.ssd(w.x, w.dt, w.A, w.B, w.C, D=w.D, z=w.z, dt_bias=w.dt_bias, h0=w.h0,
                      dt_softplus=w.dt_softplus)


CASES = [
    # name, make_ssd kwargs
    ("n64_ragged", dict(batch=2, seqlen=200, nheads=4, headdim=64, dstate=64)),
    ("n128_groups_state", dict(batch=2, seqlen=256, nheads=6, headdim=64, dstate=128, ngroups=2,
                               state_in=True)),
    ("n256_no_gate_state", dict(batch=1, seqlen=130, nheads=3, headdim=64, dstate=256, ngroups=3,
                                gate=False, state_in=True)),
    ("n128_short", dict(batch=3, seqlen=5, nheads=2, headdim=64, dstate=128)),
    ("n64_one_chunk", dict(batch=1, seqlen=64, nheads=2, headdim=64, dstate=64)),
    ("n64_one_step_state", dict(batch=2, seqlen=1, nheads=2, headdim=64, dstate=64, state_in=True)),
    ("n128_no_D_no_bias", dict(batch=1, seqlen=100, nheads=2, headdim=64, dstate=128, with_D=False,
                               with_bias=False)),
    ("n128_long", dict(batch=1, seqlen=2048, nheads=8, headdim=64, dstate=128, ngroups=2)),
    ("n256_long_groups", dict(batch=2, seqlen=777, nheads=4, headdim=64, dstate=256, ngroups=2,
                              state_in=True)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_ssd_parity(name, kw):
    w = make_ssd(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    out, st = ssd_gpu(w)
    ref, ref_st = ssd_oracle(w)
    assert_close(out, ref, "bf16", f"{name}: out")
    assert_close(st, ref_st, "bf16", f"{name}: final state")


def test_ssd_without_softplus():
    """The raw step taken as given (small positive steps, no bias)."""
    w = make_ssd("nosp", batch=2, seqlen=150, nheads=3, headdim=64, dstate=64, seed=5)
    steps = np.abs(np.random.default_rng(5).standard_normal(w.dt.shape)).astype(np.float32) * 0.05
    w.dt = f32_to_bf16_bits(steps)
    w.dt_bias = None
    w.dt_softplus = False
    out, st = ssd_gpu(w)
    ref, ref_st = ssd_oracle(w)
    assert_close(out, ref, "bf16", "no softplus: out")
    assert_close(st, ref_st, "bf16", "no softplus: final state")


def test_ssd_fast_decay_takes_the_unsplit_path():
    """Large steps on a fast-decaying head: a chunk's range of S (the running sum of
    step * A) far above 160, where the kernel forms each decay exp(S_i - S_j) with its
    own exponential instead of the split product; most decays underflow to zero."""
    w = make_ssd("fast", batch=1, seqlen=300, nheads=3, headdim=64, dstate=128, seed=8,
                 state_in=True)
    w.dt_bias = np.full(w.nheads, 2.0, np.float32)          # steps near 2
    w.A = np.array([-1.5, -0.05, -3.0], np.float32)          # ranges ~380, ~13, ~770 per chunk
    out, st = ssd_gpu(w)
    ref, ref_st = ssd_oracle(w)
    assert_close(out, ref, "bf16", "fast decay: out")
    assert_close(st, ref_st, "bf16", "fast decay: final state")


SPLIT_CASES = [
    ("n64_ragged_parts", dict(batch=2, seqlen=200, nheads=4, headdim=64, dstate=64)),
    ("n128_groups_state_parts", dict(batch=2, seqlen=700, nheads=6, headdim=64, dstate=128, ngroups=2,
                                     state_in=True)),
    ("n256_state_parts", dict(batch=1, seqlen=777, nheads=4, headdim=64, dstate=256, ngroups=2,
                              state_in=True)),
]


@pytest.mark.parametrize("name,kw", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_ssd_sequence_parts(name, kw):
    """Each sequence cut into 2 and 4 parts of consecutive chunks, taken in order by
    persistent CTAs with the state handed over through the carry: the result equals
    the one-part run bit for bit (the carry is the sum of the state's accumulators
    that every chunk start forms anyway) and the oracle at the bf16 bar."""
    import selective_state_space_112_b300 as ssm
    w = make_ssd(name, seed=zlib.crc32(name.encode()) % 1000, **kw)
    try:
        ssm.ssm_set_option("ssd_split", 1)
        out1, st1 = ssd_gpu(w)
        for parts in (2, 4):
            ssm.ssm_set_option("ssd_split", parts)
            out, st = ssd_gpu(w)
            assert np.array_equal(out, out1), f"{name}: {parts} parts: out"
            assert np.array_equal(st, st1), f"{name}: {parts} parts: final state"
    finally:
        ssm.ssm_set_option("ssd_split", 0)
    ref, ref_st = ssd_oracle(w)
    assert_close(out1, ref, "bf16", f"{name}: out")
    assert_close(st1, ref_st, "bf16", f"{name}: final state")


def test_ssd_part_handover_timeout_is_reported_and_the_context_stays_usable():
    """The hand-over between sequence parts without a GPU fault: the first part of one
    unit is told never to release its state, so the wait of its second part runs out
    (after 2 s).  The kernel returns, ssm_check_status reports SSM_ERR_TIMEOUT once, and
    the next call matches the oracle."""
    import selective_state_space_112_b300 as ssm
    w = make_ssd("hold_part", batch=1, seqlen=512, nheads=2, headdim=64, dstate=64, seed=31)
    t = lambda a: to_torch(a)
    try:
        ssm.ssm_set_option("ssd_split", 2)
        ssm.ssm_set_option("ssd_hold_part", 2)
        ssm.ssm_ssd_fwd(t(w.x), t(w.dt), t(w.A), t(w.B), t(w.C), t(w.D), t(w.z), t(w.dt_bias))
        assert ssm.ssm_check_status() == -9  # SSM_ERR_TIMEOUT
        assert ssm.ssm_check_status() == 0
    finally:
        ssm.ssm_set_option("ssd_hold_part", 0)
        ssm.ssm_set_option("ssd_split", 0)
    out, st = ssd_gpu(w)
    ref, ref_st = ssd_oracle(w)
    assert_close(out, ref, "bf16", "after the hand-over timeout: out")
    assert_close(st, ref_st, "bf16", "after the hand-over timeout: final state")


def test_ssd_continuation_and_determinism():
    """Two calls carrying the state equal one call over the whole sequence (the
    split falls inside a chunk), and a repeated call is bitwise identical."""
    from dataclasses import replace
    w = make_ssd("cont", batch=2, seqlen=300, nheads=4, headdim=64, dstate=128, ngroups=2, seed=7,
                 state_in=True)
    out, st = ssd_gpu(w)
    out2, st2 = ssd_gpu(w)
    assert np.array_equal(out, out2) and np.array_equal(st, st2)
    cut = 141
    part = lambda a, s: a[:, s]
    w1 = replace(w, x=part(w.x, slice(0, cut)), dt=part(w.dt, slice(0, cut)), B=part(w.B, slice(0, cut)),
                 C=part(w.C, slice(0, cut)), z=part(w.z, slice(0, cut)))
    o1, s1 = ssd_gpu(w1)
    w2 = replace(w, x=part(w.x, slice(cut, None)), dt=part(w.dt, slice(cut, None)),
                 B=part(w.B, slice(cut, None)), C=part(w.C, slice(cut, None)), z=part(w.z, slice(cut, None)))
    o2, s2 = ssd_gpu(w2, h0=s1.astype(np.float32))
    ref, ref_st = ssd_oracle(w)
    assert_close(np.concatenate([o1, o2], axis=1), ref, "bf16", "continued: out")
    assert_close(s2, ref_st, "bf16", "continued: final state")


def test_ssd_empty_sequence():
    """L = 0 writes the final state: zeros without state_in, h_{-1} kept with it."""
    import torch
    import selective_state_space_112_b300 as ssm
    w = make_ssd("empty", batch=2, seqlen=0, nheads=2, headdim=64, dstate=64, seed=1)
    t = lambda a: to_torch(a)
    fs = torch.full((2, 2, 64, 64), 3.0, device="cuda")
    ssm.ssm_ssd_fwd(t(w.x), t(w.dt), t(w.A), t(w.B), t(w.C), t(w.D), t(w.z), t(w.dt_bias), final_state=fs)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs).item() == 0
    fs.fill_(3.0)
    ssm.ssm_ssd_fwd(t(w.x), t(w.dt), t(w.A), t(w.B), t(w.C), t(w.D), t(w.z), t(w.dt_bias), final_state=fs,
                    state_in=True)
    torch.cuda.synchronize()
    assert bool((fs == 3.0).all())


def _full_size_sampled(name, npairs, seed):
    import torch
    cfg = SSD_CONFIGS[name]
    w = make_ssd(name, **cfg)
    out, st = ssd_gpu(w)
    G = w.ngroups
    rng = np.random.default_rng(seed)
    pairs = [(0, 0), (w.batch - 1, w.nheads - 1)] + [
        (int(b), int(h)) for b, h in zip(np.arange(npairs - 2) % w.batch,
                                         rng.choice(w.nheads, npairs - 2, replace=False))]
    for b, h in pairs:
        g = h // (w.nheads // G)
        sl = make_ssd("slice", batch=1, seqlen=1, nheads=1, headdim=64, dstate=w.dstate, seed=0)
        sl.batch, sl.seqlen, sl.nheads, sl.ngroups = 1, w.seqlen, 1, 1
        sl.x = w.x[b:b + 1, :, h:h + 1]
        sl.dt = w.dt[b:b + 1, :, h:h + 1]
        sl.A, sl.D, sl.dt_bias = w.A[h:h + 1], w.D[h:h + 1], w.dt_bias[h:h + 1]
        sl.B, sl.C = w.B[b:b + 1, :, g:g + 1], w.C[b:b + 1, :, g:g + 1]
        sl.z = w.z[b:b + 1, :, h:h + 1]
        sl.h0 = None
        ref, ref_st = ssd_oracle(sl)
        assert_close(out[b:b + 1, :, h:h + 1], ref, "bf16", f"{name}, b {b} head {h}: out")
        assert_close(st[b:b + 1, h:h + 1], ref_st, "bf16", f"{name}, b {b} head {h}: final state")
    del out
    torch.cuda.empty_cache()


def test_ssd_full_size_sampled_heads():
    """The 2.7B-shaped layer (4 x 4096 steps, 80 heads of 64, N 128) in one call, as
    the benchmark launches it; sixteen (batch row, head) pairs spread over every batch
    row and the head range (the first and last head included) against the oracle run
    on that head's slice of the inputs."""
    _full_size_sampled("mamba2_2p7b_bf16", 16, 2700)


def test_ssd_full_size_parts_bitwise():
    """The 2.7B-shaped layer as the benchmark launches it (more sequences than
    resident CTAs: parts taken in order by persistent CTAs) equals the one-part launch
    of 640 CTAs and the four-part launch bit for bit."""
    import torch
    import selective_state_space_112_b300 as ssm
    w = make_ssd("mamba2_2p7b_bf16", **SSD_CONFIGS["mamba2_2p7b_bf16"])
    res = []
    try:
        for parts in (0, 1, 4):
            ssm.ssm_set_option("ssd_split", parts)
            res.append(ssd_gpu(w))
    finally:
        ssm.ssm_set_option("ssd_split", 0)
    for (o, s), parts in zip(res[1:], (1, 4)):
        assert np.array_equal(o, res[0][0]), f"{parts} parts: out"
        assert np.array_equal(s, res[0][1]), f"{parts} parts: final state"
    del res
    torch.cuda.empty_cache()


def test_ssd_full_size_n256_sampled_heads():
    """The N = 256 layer (4 x 4096 steps, 80 heads of 64) as the benchmark launches it
    (the kernel for 256 state rows: two blocks of 128 per product), eight (batch row,
    head) pairs against the oracle."""
    _full_size_sampled("mamba2_n256_bf16", 8, 2560)
