"""m3_ssm_prefill_noalloc, the prefill for callers that may not allocate device memory
(plugin hosts and serving loops that forbid cudaMalloc once running, code whose memory
belongs to a pool it does not control).  It runs the same kernels as m3_ssm_prefill but
takes its scratch from a static array in the library's device image.

Called through the C ABI twice in a row on different inputs (the second call must not
see the first call's scratch contents), each time against m3_ssm_prefill with its own
workspace, within the bf16 tolerance the parity tests use.  This file sorts last so
that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import state_space_sequence_trapezoidal_b300 as m3
from state_space_sequence_trapezoidal_b300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,R", [(128, 1), (64, 4)])
def test_noalloc_prefill_matches_workspace_prefill_twice(N, R):
    B, H, Pd = 2, 3, 64
    T = 3 * (128 // R) + 5
    for call, seed in enumerate((4100 + N + R, 4200 + N + R)):
        inp = synth.make_inputs(B, T, H, Pd, N, R, seed, "bf16")
        d = P.to_device(inp, "bf16")
        st0 = P.state_to_device(P.random_state(B, H, N, Pd, R, "bf16", seed), "bf16")

        ref_state = m3.State.zeros(B, H, N, Pd, R)
        y_ref = m3.m3_ssm_prefill(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"],
                                  d["theta"], st0, hT=ref_state)

        y = torch.full_like(y_ref, float("nan"))
        got_state = m3.State.zeros(B, H, N, Pd, R)
        m3.m3_ssm_prefill_noalloc(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"],
                                  d["theta"], st0, y=y, hT=got_state)
        torch.cuda.synchronize()

        e = P.rel_err(y.cpu().numpy(), y_ref.cpu().numpy())
        assert e <= P.TOL["bf16"], (call, e)
        eh = P.rel_err(got_state.h.cpu().numpy(), ref_state.h.cpu().numpy())
        assert eh <= P.TOL["bf16"], (call, eh)
        assert P.phi_err(got_state.phi.cpu().numpy(), ref_state.phi.cpu().numpy()) <= P.PHI_TOL["bf16"]
        assert torch.equal(got_state.prev_B, ref_state.prev_B)
        assert torch.equal(got_state.prev_x, ref_state.prev_x)
        assert np.isfinite(y.cpu().numpy()).all()
