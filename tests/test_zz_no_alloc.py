"""m3_ssm_prefill_noalloc, the prefill for callers that may not allocate device memory
(plugin hosts and serving loops that forbid cudaMalloc once running, code whose memory
belongs to a pool it does not control).  It runs the same kernels as m3_ssm_prefill but
takes its scratch from a static array in the library's device image.

Called through the C ABI twice in a row on different inputs (the second call must not
see the first call's scratch contents), each time against m3_ssm_prefill with its own
workspace.  Both calls run the same deterministic kernels on the same inputs, so the
results must agree bit for bit.  The shapes include long sequences over few (batch row,
head) pairs, which the prefill splits into segments whose per-segment states live in the
scratch; a shape whose scratch would exceed the array is refused.  This file sorts last
so that a run stopping at the first failure has already run every other test."""
import pytest
import torch

import state_space_sequence_trapezoidal_b300 as m3
from state_space_sequence_trapezoidal_b300 import synth
from tests import parity as P

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20  # the array's size, as the header states


@pytest.mark.parametrize("B,H,N,R,T", [
    (2, 3, 128, 1, 3 * 128 + 5),   # one segment: only the status word is used
    (2, 3, 64, 4, 3 * 32 + 5),
    (1, 2, 128, 1, 1024),          # segmented: per-segment states in the scratch
    (1, 4, 128, 1, 1500),
    (1, 2, 64, 4, 300),
])
def test_noalloc_prefill_matches_workspace_prefill_twice(B, H, N, R, T):
    Pd = 64
    segmented = (B, H, T) not in ((2, 3, 3 * 128 + 5), (2, 3, 3 * 32 + 5))
    for call, seed in enumerate((4100 + N + R + T, 4200 + N + R + T)):
        inp = synth.make_inputs(B, T, H, Pd, N, R, seed, "bf16")
        d = P.to_device(inp, "bf16")
        ws = m3.prefill_workspace(d["x"], d["dt"], d["theta"])
        assert (ws.numel() > 256) == segmented
        assert ws.numel() <= SCRATCH_BYTES
        st0 = P.state_to_device(P.prior_state(B, H, N, Pd, R, "bf16", seed), "bf16")

        ref_state = m3.State.zeros(B, H, N, Pd, R)
        y_ref = m3.m3_ssm_prefill(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"],
                                  d["theta"], st0, hT=ref_state, workspace=ws)

        y = torch.full_like(y_ref, float("nan"))
        got_state = m3.State.zeros(B, H, N, Pd, R)
        got_state.h.fill_(float("nan"))
        m3.m3_ssm_prefill_noalloc(d["x"], d["B"], d["C"], d["dt"], d["A"], d["lambda"],
                                  d["theta"], st0, y=y, hT=got_state)
        torch.cuda.synchronize()
        assert m3.m3_ssm_device_status(ws) == m3.M3_OK

        assert torch.equal(y, y_ref), (call, (y - y_ref).abs().max().item())
        assert torch.equal(got_state.h, ref_state.h), call
        assert torch.equal(got_state.phi, ref_state.phi), call
        assert torch.equal(got_state.prev_B, ref_state.prev_B)
        assert torch.equal(got_state.prev_x, ref_state.prev_x)
        # and both against the oracle, at the bf16 tolerance
        sl = P.all_slices(B, H)
        yr, _ = P.run_oracle(inp, sl, P.state_to_host(st0))
        e = P.rel_err(P.pick(y.cpu().numpy(), sl, True), yr)
        assert e <= P.TOL["bf16"], (call, e)


def test_noalloc_refuses_shapes_beyond_the_scratch():
    """B1 T16384 H32 N128 needs about 16 MiB of per-segment state: refused before any launch
    (the inputs are only shape- and pointer-checked, so they are left uninitialised)."""
    B, T, H, Pd, N, R = 1, 16384, 32, 64, 128, 1
    bf = dict(dtype=torch.bfloat16, device="cuda")
    x = torch.empty(B, T, H, R, Pd, **bf)
    Bm = torch.empty(B, T, H, R, N, **bf)
    dt = torch.empty(B, T, H, **bf)
    theta = torch.empty(B, T, H, N // 2, **bf)
    A = torch.empty(H, dtype=torch.float32, device="cuda")
    assert m3.prefill_workspace(x, dt, theta).numel() > SCRATCH_BYTES
    y = torch.empty(B, T, H, R, Pd, dtype=torch.float32, device="cuda")
    with pytest.raises(m3.M3Error) as e:
        m3.m3_ssm_prefill_noalloc(x, Bm, Bm, dt, A, dt, theta, y=y)
    assert e.value.status == m3.M3_ERR_WORKSPACE
