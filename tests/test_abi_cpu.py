"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/*.h declares, and rejects bad arguments on the host before
touching the device."""
import os
import re

import pytest

from selective_state_space_112_b300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("ssm_scan.h", "ssm_ssd.h")]


def header_functions():
    names = set()
    for hdr in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(hdr).read(), flags=re.S)
        names.update(re.findall(r"\b(ssm_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_every_header_is_checked():
    assert sorted(HEADERS) == sorted(
        os.path.join(ROOT, "include", h) for h in os.listdir(os.path.join(ROOT, "include")) if h.endswith(".h"))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert set(names) == set(_abi.EXPORTS), names
    L = _abi.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings():
    for code in list(_abi.STATUS) + [-99]:
        s = _abi.status_string(code)
        assert isinstance(s, str) and s
    assert _abi.status_string(0) == "ok"


def dims(**kw):
    base = dict(batch=2, seqlen=16, dim=8, dstate=4, io_dtype=0, bc_layout=0,
                delta_softplus=1, state_in=0, bbar_mode=0, reserved=0)
    base.update(kw)
    return _abi.SsmDims(**base)


# Fake, never dereferenced device addresses: validation happens first on the host.
BASE = 1 << 40
P = {k: BASE + i * (1 << 30) for i, k in enumerate(
    ["x", "delta", "A", "B", "C", "D", "z", "bias", "out", "fs"])}


def call(d, **over):
    q = dict(P)
    q.update(over)
    return _abi.call_fwd(q["x"], q["delta"], q["A"], q["B"], q["C"], q["D"], q["z"],
                         q["bias"], q["out"], q["fs"], d, 0)


def test_null_dims():
    L = _abi.lib()
    assert L.ssm_selective_scan_fwd(*([None] * 10), None, None) == -1


@pytest.mark.parametrize("bad", [dict(batch=0), dict(dim=0), dict(dstate=0), dict(dstate=65),
                                 dict(seqlen=-1), dict(io_dtype=2), dict(bc_layout=3),
                                 dict(delta_softplus=2), dict(state_in=5), dict(reserved=1),
                                 dict(bbar_mode=9)])
def test_bad_dims(bad):
    assert call(dims(**bad)) == -2


def test_state_in_needs_state():
    assert call(dims(state_in=1), fs=0) == -2


def test_null_required_pointer():
    for k in ("x", "delta", "A", "B", "C", "out"):
        assert call(dims(), **{k: 0}) == -1, k


def test_misaligned():
    for k in ("x", "delta", "A", "B", "C", "D", "z", "bias", "out", "fs"):
        assert call(dims(), **{k: P[k] + 4}) == -3, k


def test_overlap():
    assert call(dims(), out=P["x"] + 16) == -6
    assert call(dims(), fs=P["out"]) == -6
    assert call(dims(), fs=P["A"]) == -6


def test_exact_zoh_accepted_on_the_host():
    """bbar_mode 1 (exact ZOH) passes host validation: without a GPU the call fails
    only at the device (SSM_ERR_CUDA), never with SSM_ERR_UNSUPPORTED."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(dims(bbar_mode=1)) == -5


CP = {k: BASE + (12 + i) * (1 << 30) for i, k in enumerate(["cw", "cb", "cs"])}


def call_conv(d, **over):
    q = dict(P)
    q.update(CP)
    q.update(over)
    return _abi.call_conv_fwd(q["x"], q["cw"], q["cb"], q["cs"], q["delta"], q["A"], q["B"], q["C"],
                              q["D"], q["z"], q["bias"], q["out"], q["fs"], d, 0)


def test_conv_entry_host_checks():
    """The block-prologue entry checks its own arguments on the host: taps are
    required, every pointer 16-byte aligned, the history disjoint from the other
    tensors; the forms it is not built for (constant B and C, the exact-ZOH term)
    are SSM_ERR_UNSUPPORTED before anything touches the device."""
    assert call_conv(dims(), cw=0) == -1
    for k in ("cw", "cb", "cs"):
        assert call_conv(dims(), **{k: CP[k] + 4}) == -3, k
    assert call_conv(dims(), cs=P["out"]) == -6
    assert call_conv(dims(), cs=P["fs"]) == -6
    assert call_conv(dims(bc_layout=1)) == -4
    assert call_conv(dims(bbar_mode=1)) == -4
    assert call_conv(dims(dstate=65)) == -2


def test_conv_entry_accepts_wide_states_on_the_host():
    """N up to 64 (two and four lanes per channel) passes the prologue entry's host
    validation: without a GPU the call fails only at the device (SSM_ERR_CUDA)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for n in (24, 32, 64):
        assert call_conv(dims(dstate=n)) == -5, n


def test_no_cpu_fallback():
    """A valid call without a usable GPU must fail, never compute on the host."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(dims()) == -5


def test_options():
    with pytest.raises(_abi.SSMError):
        _abi.set_option("no_such_option", 1)
    with pytest.raises(_abi.SSMError):
        _abi.set_option("chunks", -1)
    for name in ("chunks", "min_chunk_len", "lanes"):
        _abi.set_option(name, 0)
    for v in (2, 4, 1, 0):
        _abi.set_option("ssd_split", v)
    with pytest.raises(_abi.SSMError):
        _abi.set_option("ssd_split", 3)
    _abi.set_option("ssd_hold_part", 0)
    with pytest.raises(_abi.SSMError):
        _abi.set_option("ssd_hold_part", -1)
    _abi.set_option("min_chunk_len", 64)
    _abi.set_option("lane_threads", 36864)
    _abi.set_option("ctas_per_sm", 3)
    _abi.set_option("inject_stall", 0)
    _abi.set_option("pow_path", 1)
    _abi.set_option("tma", 1)
    assert _abi.profile_read() == {}


# ---------------------------------------------------------------- Mamba-2 SSD entry

SP = {k: BASE + (20 + i) * (1 << 30) for i, k in enumerate(
    ["x", "dt", "A", "B", "C", "D", "z", "bias", "out", "fs"])}


def sdims(**kw):
    base = dict(batch=2, seqlen=100, nheads=4, headdim=64, ngroups=2, dstate=128, io_dtype=1,
                dt_softplus=1, state_in=0, reserved=0)
    base.update(kw)
    return _abi.SsdDims(**base)


def call_ssd(d, **over):
    q = dict(SP)
    q.update(over)
    return _abi.call_ssd(q["x"], q["dt"], q["A"], q["B"], q["C"], q["D"], q["z"], q["bias"],
                         q["out"], q["fs"], d, 0)


def test_ssd_entry_host_checks():
    """ssm_ssd_fwd rejects bad arguments on the host: NULL dims and required
    pointers, bad sizes and flags, misaligned pointers, overlapping outputs, and the
    forms this build does not cover (fp32 io, head dimension other than 64, N other
    than 64, 128 or 256)."""
    L = _abi.lib()
    assert L.ssm_ssd_fwd(*([None] * 10), None, None) == -1
    for k in ("x", "dt", "A", "B", "C", "out"):
        assert call_ssd(sdims(), **{k: 0}) == -1, k
    for bad in (dict(batch=0), dict(batch=65536), dict(seqlen=-1), dict(nheads=0), dict(headdim=0),
                dict(ngroups=0), dict(ngroups=3), dict(dstate=0), dict(io_dtype=2),
                dict(dt_softplus=2), dict(state_in=2), dict(reserved=1)):
        assert call_ssd(sdims(**bad)) == -2, bad
    assert call_ssd(sdims(state_in=1), fs=0) == -2
    for k in SP:
        assert call_ssd(sdims(), **{k: SP[k] + 4}) == -3, k
    assert call_ssd(sdims(), out=SP["x"] + 16) == -6
    assert call_ssd(sdims(), fs=SP["out"]) == -6
    assert call_ssd(sdims(), fs=SP["B"]) == -6
    for bad in (dict(io_dtype=0), dict(headdim=32), dict(dstate=16), dict(dstate=96)):
        assert call_ssd(sdims(**bad)) == -4, bad


def test_ssd_entry_reaches_the_device():
    """A valid SSD call passes host validation (N 64, 128, 256, with and without
    groups): without a GPU it fails only at the device (SSM_ERR_CUDA)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for n in (64, 128, 256):
        assert call_ssd(sdims(dstate=n)) == -5, n
    assert call_ssd(sdims(ngroups=1, D=0, z=0, bias=0, fs=0)) == -5
