"""The one-launch chunk carry of the forward kernel, emulated on the CPU in float64.

The kernel cuts the sequence into chunks; each chunk's first scan starts from a zero
state (the first chunk from the initial state, so that its end state is the true one)
and publishes its step sum S_c and end state H_c; a chunk's carry-in is then folded
from all earlier chunks in a fixed order, from the previous chunk back to the first,
  H_acc += exp(A S_acc) H_j,  S_acc += S_j   (j = c-1, c-2, ..., 1; then chunk 0's
  true end state is added as exp(A S_acc) H_0).
This is the associative combine of the per-step maps ("State-space models", The
parallel scan; "Structured State Space Models and Mamba", Hardware-Aware Parallel
Associative Scan) applied to chunk aggregates.  The walk may also stop early at any
chunk whose true end state (inclusive prefix) is known: the emulation checks every
such mix, and that the prefix a chunk would publish, exp(A S_c) h_in + H_c, is its
true end state.  The aggregates come from the oracle run on each chunk alone; the
carry-ins must equal the oracle's own states at the chunk boundaries.
"""
import itertools

import numpy as np
import pytest

import oracle
from selective_state_space_112_b300.workloads import bf16_bits_to_f32, make_workload


def _steps(w):
    """Per-(b, t, d) step sizes softplus(delta + bias) in float64."""
    dl = bf16_bits_to_f32(w.delta) if w.io == "bf16" else w.delta
    v = dl.astype(np.float64) + (0.0 if w.delta_bias is None else w.delta_bias.astype(np.float64))
    return np.logaddexp(0.0, v) if w.delta_softplus else v


def _piece(w, t0, t1, h0):
    sl = lambda a: None if a is None else np.ascontiguousarray(a[:, t0:t1])
    return oracle.selective_scan(sl(w.x), sl(w.delta), w.A, sl(w.B), sl(w.C), D=w.D, z=sl(w.z),
                                 delta_bias=w.delta_bias, h0=h0, delta_softplus=w.delta_softplus,
                                 io_dtype=w.io)


@pytest.mark.parametrize("io,state_in", [("f32", False), ("bf16", True)])
def test_lookback_fold_gives_the_chunk_boundary_states(io, state_in):
    w = make_workload("lb", batch=2, seqlen=6 * 32, dim=5, dstate=4, io=io, seed=17, state_in=state_in)
    k, ln = 6, 32
    A = w.A.astype(np.float64)
    steps = _steps(w)
    # true states at the chunk boundaries (one oracle run per prefix)
    true = [w.h0.astype(np.float64) if state_in else np.zeros((w.batch, w.dim, w.dstate))]
    for c in range(k):
        _, st = _piece(w, 0, (c + 1) * ln, w.h0)
        true.append(st)
    # the chunks' first scans: from zero, the first chunk from the initial state
    H, S = [], []
    for c in range(k):
        _, st = _piece(w, c * ln, (c + 1) * ln, w.h0 if c == 0 else None)
        H.append(st)
        S.append(steps[:, c * ln:(c + 1) * ln, :].sum(axis=1))      # (batch, dim)
    np.testing.assert_allclose(H[0], true[1], rtol=1e-12, atol=1e-12)

    def walk(c, published):
        """Carry-in of chunk c; published[j] is True where chunk j's prefix is out."""
        Hacc = np.zeros_like(H[0])
        Sacc = np.zeros_like(S[0])
        for j in range(c - 1, -1, -1):
            if published[j] or j == 0:            # the first chunk always publishes a prefix
                P = H[0] if j == 0 else true[j + 1]
                return Hacc + np.exp(A[None] * Sacc[..., None]) * P
            Hacc = Hacc + np.exp(A[None] * Sacc[..., None]) * H[j]
            Sacc = Sacc + S[j]
        raise AssertionError("the walk must end at chunk 0")

    for c in range(1, k):
        for pub in itertools.product([False, True], repeat=c):
            hin = walk(c, pub)
            np.testing.assert_allclose(hin, true[c], rtol=1e-10, atol=1e-12)
        # the inclusive prefix the chunk then publishes is its true end state
        hin = walk(c, (False,) * c)
        P = np.exp(A[None] * S[c][..., None]) * hin + H[c]
        np.testing.assert_allclose(P, true[c + 1], rtol=1e-10, atol=1e-12)
    # the last chunk's second scan from its carry-in gives the call's outputs
    out_full, st_full = _piece(w, 0, k * ln, w.h0)
    o_last, st_last = _piece(w, (k - 1) * ln, k * ln, walk(k - 1, (False,) * (k - 1)))
    np.testing.assert_allclose(o_last, out_full[:, (k - 1) * ln:], rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(st_last, st_full, rtol=1e-10, atol=1e-12)
