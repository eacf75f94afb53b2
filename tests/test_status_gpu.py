"""Device-side error reporting: a malformed cu_seqlens is caught by the
first kernel, recorded in the workspace status word and makes the other
kernels no-ops; the next valid call resets it.  Host-side errors come back
before anything is enqueued."""
import numpy as np
import pytest
import torch

from variable_length_sequence_gb300 import nsp as nsp_mod
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bad", ["nonmonotone", "first_nonzero", "short_total"])
def test_bad_cu_seqlens_reported(nsp, bad):
    w = make_custom([50, 70, 80], 4, 2, 128, seed=1)
    q, k, v, do = (getattr(w, n).cuda() for n in ("q", "k", "v", "dout"))
    cu = w.cu_seqlens.copy()
    if bad == "nonmonotone":
        cu[1], cu[2] = cu[2], cu[1]
    elif bad == "first_nonzero":
        cu[0] = 3
    else:
        cu[-1] = 150
    cu_d = torch.from_numpy(cu).cuda()
    ws = torch.empty(nsp.nsp_attn_fwd_workspace_size(200, 200, 4, 2, 128), dtype=torch.uint8,
                     device="cuda")
    out, lse = nsp.attn_fwd(q, k, v, cu_d, workspace=ws)
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_ERR_INVALID
    # a valid call on the same workspace resets the status
    nsp.attn_fwd(q, k, v, torch.from_numpy(w.cu_seqlens).cuda(), workspace=ws)
    assert nsp.nsp_status_query(ws) == nsp_mod.NSP_OK
    wsb = torch.empty(nsp.nsp_attn_bwd_workspace_size(200, 4, 2, 128, nsp_mod.NSP_BF16),
                      dtype=torch.uint8, device="cuda")
    nsp.attn_bwd(q, k, v, out, do, lse, cu_d, workspace=wsb)
    assert nsp.nsp_status_query(wsb) == nsp_mod.NSP_ERR_INVALID


def test_host_errors_raise(nsp):
    w = make_custom([10], 4, 2, 128, seed=2)
    q, k, v = (getattr(w, n).cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nsp_mod.NspError) as e:
        nsp.attn_fwd(q, k, v, cu, workspace=small)
    assert e.value.status == nsp_mod.NSP_ERR_WORKSPACE
    with pytest.raises(nsp_mod.NspError) as e:
        nsp.attn_fwd(q[:, :3].contiguous(), k, v, cu)      # Hq=3 not a multiple of Hkv=2
    assert e.value.status == nsp_mod.NSP_ERR_INVALID
    with pytest.raises(ValueError):
        nsp.attn_fwd(q[:, :2], k, v, cu)                   # strided view


def test_empty_stream(nsp):
    q = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    out, lse = nsp.attn_fwd(q, k, k, cu, workspace=ws)
    assert out.shape == (0, 4, 128) and nsp.nsp_status_query(ws) == nsp_mod.NSP_OK
