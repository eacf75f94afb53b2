"""Failure detection on the GPU without a fault: bounded waits that expire.

Every wait inside the tensor-core kernels (for a copy, a product or another
role of the block) is bounded.  nsp_set_wait_timeout_cycles shortens the
bound to a few cycles, so the first wait of a call that is not already
satisfied expires: the kernel records NSP_ERR_TIMEOUT in the workspace
status word, every role stops, waits for the copies and products it issued,
frees its tensor memory and returns.  The test then checks that the status
reaches the host, that the context is still usable and that the next call on
the same workspace, with the default bound, matches the oracle.  Nothing here
hangs or faults: the expiring waits are the kernels' own bounded waits.
"""
import pytest
import torch

import oracle
from gpu_common import TOL_GRAD, assert_fwd_close, f64, oracle_inputs, rel_l2, to_dev
from variable_length_sequence_gb300 import nsp as nsp_mod
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

SHORT_BOUND = 100          # GPU cycles: shorter than any copy or product takes


def _short_bound(nsp, fn):
    prev = nsp.nsp_set_wait_timeout_cycles(SHORT_BOUND)
    try:
        return fn()
    finally:
        nsp.nsp_set_wait_timeout_cycles(prev)


def test_setter_returns_previous_bound(nsp):
    prev = nsp.nsp_set_wait_timeout_cycles(12345)
    try:
        assert nsp.nsp_set_wait_timeout_cycles(-1) == 12345
        assert nsp.nsp_set_wait_timeout_cycles(-1) == 4000000000     # the default
    finally:
        nsp.nsp_set_wait_timeout_cycles(prev)


def test_forward_wait_expires_then_recovers(nsp):
    w = make_custom([700, 300, 57, 1], 8, 2, 128, seed=81, with_dout=False)
    d = to_dev(w)
    scale = 128 ** -0.5
    ws = torch.empty(nsp.nsp_attn_fwd_workspace_size(w.T, w.T, 8, 2, 128), dtype=torch.uint8,
                     device="cuda")
    _short_bound(nsp, lambda: nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=scale,
                                           workspace=ws))
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_ERR_TIMEOUT
    torch.cuda.synchronize()                        # the context is still usable
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=scale, workspace=ws)
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_OK
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, scale, True)
    assert_fwd_close(f64(out), f64(lse), ro, rl, label="after a timed-out call")


def test_backward_wait_expires_then_recovers(nsp):
    w = make_custom([600, 129, 300], 8, 2, 128, seed=82)
    d = to_dev(w)
    scale = 128 ** -0.5
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=scale)
    ws = torch.empty(nsp.nsp_attn_bwd_workspace_size(w.T, 8, 2, 128, nsp_mod.NSP_BF16),
                     dtype=torch.uint8, device="cuda")
    _short_bound(nsp, lambda: nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"],
                                           scale=scale, workspace=ws))
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_ERR_TIMEOUT
    dq, dk, dv = nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], scale=scale,
                              workspace=ws)
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_OK
    q, k, v, do = oracle_inputs(w)
    ref = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert rel_l2(f64(g), r) <= TOL_GRAD, name
