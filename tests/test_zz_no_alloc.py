"""The entry point that allocates no device memory, against the regular one.

ssm_selective_scan_fwd_noalloc serves callers that cannot let a library allocate
device memory (an arena that owns all device memory, a serving loop that forbids
allocation after warm-up).  It keeps the chunk-carry workspace of long sequences in a
fixed device array inside the library instead of the memory pool.  Each case here is
forced into several sequence chunks so that the workspace is really used, and two
calls in a row must both agree with the regular entry point within the parity
tolerance (1e-5 for fp32 inputs, 2e-2 for bf16).  This file is collected last so that
a run stopping at its first failure has run every other test before it.
"""
import numpy as np
import pytest

from oracle.metrics import TOL, floored_rel_err
from selective_state_space_112_b300.workloads import make_workload

from helpers import device_inputs

pytestmark = pytest.mark.gpu

CASES = [
    # (name, make_workload kwargs, forced chunk count)
    ("bf16_state_in", dict(batch=2, seqlen=3000, dim=96, dstate=16, io="bf16", state_in=True), 6),
    ("f32_gate", dict(batch=1, seqlen=2100, dim=136, dstate=16, io="f32"), 5),
    ("f32_N8_lti", dict(batch=2, seqlen=1000, dim=64, dstate=8, io="f32", lti=True,
                         with_bias=False), 4),
]


def _run(ssm, w, dev, noalloc):
    import torch
    fs = dev["final_state"].clone()
    fn = ssm.ssm_selective_scan_fwd_noalloc if noalloc else ssm.ssm_selective_scan_fwd
    out = torch.empty_like(dev["x"])
    fn(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"], dev["D"], dev["z"],
       dev["delta_bias"], out=out, final_state=fs, delta_softplus=w.delta_softplus,
       state_in=w.h0 is not None)
    assert ssm.ssm_check_status() == 0
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), fs.double().cpu().numpy()


@pytest.mark.parametrize("name,kw,chunks", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_regular_entry_point(name, kw, chunks):
    import selective_state_space_112_b300 as ssm
    w = make_workload(name, seed=21, **kw)
    dev = device_inputs(w)
    try:
        ssm.ssm_set_option("chunks", chunks)
        ref_out, ref_fs = _run(ssm, w, dev, noalloc=False)
        for _ in range(2):  # the shared scratch keeps the previous call's contents
            got_out, got_fs = _run(ssm, w, dev, noalloc=True)
            assert floored_rel_err(got_out, ref_out) <= TOL[w.io], name
            assert floored_rel_err(got_fs, ref_fs) <= TOL[w.io], name
            assert np.all(np.isfinite(got_out))
    finally:
        ssm.ssm_set_option("chunks", 0)


def test_noalloc_allocates_nothing():
    """Forced into chunks, the no-allocation entry point leaves the library's memory pool
    untouched: with the pool trimmed to nothing first, it still holds nothing after two
    calls; the regular entry point, given the same call, takes its workspace from it."""
    import selective_state_space_112_b300 as ssm
    w = make_workload("pool", batch=1, seqlen=4000, dim=512, dstate=16, io="bf16", seed=5,
                      state_in=True)
    dev = device_inputs(w)
    try:
        ssm.ssm_set_option("chunks", 8)
        _run(ssm, w, dev, noalloc=True)          # first call on the device: set-up
        assert ssm.ssm_release_workspace() == 0
        before = ssm.ssm_workspace_reserved_bytes()
        assert before == 0
        for _ in range(2):
            _run(ssm, w, dev, noalloc=True)
            assert ssm.ssm_workspace_reserved_bytes() == before
        _run(ssm, w, dev, noalloc=False)
        assert ssm.ssm_workspace_reserved_bytes() > before
    finally:
        ssm.ssm_set_option("chunks", 0)


def test_noalloc_rejects_a_workspace_beyond_its_scratch():
    """A forced chunk count whose workspace ((chunks - 1) * batch * dim * (2 N + 1) * 4
    bytes and the carry flags) is above the 16 MiB array: the call returns
    SSM_ERR_SCRATCH before launching anything.  (An automatic chunk count shrinks until
    its workspace fits instead.)"""
    import torch
    import selective_state_space_112_b300 as ssm
    from selective_state_space_112_b300._abi import SSM_ERR_SCRATCH, SSM_NOALLOC_SCRATCH_BYTES
    batch, dim, N, chunks = 1, 4096, 16, 80
    L = chunks * 32
    assert (chunks - 1) * batch * dim * (N + 1) * 4 > SSM_NOALLOC_SCRATCH_BYTES
    w = make_workload("big", batch=batch, seqlen=L, dim=dim, dstate=N, io="bf16", seed=3)
    dev = device_inputs(w)
    launches = ssm.ssm_kernel_launches()
    try:
        ssm.ssm_set_option("chunks", chunks)
        with pytest.raises(ssm.SSMError) as e:
            ssm.ssm_selective_scan_fwd_noalloc(dev["x"], dev["delta"], dev["A"], dev["B"],
                                               dev["C"], dev["D"], dev["z"], dev["delta_bias"])
        assert e.value.code == SSM_ERR_SCRATCH
        assert ssm.ssm_kernel_launches() == launches
        # the regular entry point takes the same call
        ssm.ssm_selective_scan_fwd(dev["x"], dev["delta"], dev["A"], dev["B"], dev["C"],
                                   dev["D"], dev["z"], dev["delta_bias"])
        torch.cuda.synchronize()
        assert ssm.ssm_check_status() == 0
    finally:
        ssm.ssm_set_option("chunks", 0)
