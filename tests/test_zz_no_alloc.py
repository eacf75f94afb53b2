"""nsp_attn_fwd_noalloc: the forward for callers that cannot allocate device
memory (allocator callbacks, plugins whose host framework owns every device
allocation, fixed-footprint processes).  Its scheduler scratch is the
library's static device array, shared by all calls, so two calls in a row
with different document layouts must each match the workspace entry point.

This file is collected last on purpose: it must pass alone in a fresh
process and after every other test."""
import numpy as np
import pytest
import torch

from gpu_common import TOL_LSE, TOL_OUT, TOL_OUT_F32, TOL_LSE_F32, f64, max_abs
from variable_length_sequence_gb300 import nsp as nsp_mod
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu


def _run_both(nsp, w, out_dtype=None, q_start=0, q_len=None, kv_start=0, kv_len=None):
    q, k, v = (getattr(w, n).cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    q_len = T - q_start if q_len is None else q_len
    kv_len = T - kv_start if kv_len is None else kv_len
    qs, ks, vs = q[q_start:q_start + q_len], k[kv_start:kv_start + kv_len], v[kv_start:kv_start + kv_len]
    ref_o, ref_l = nsp.attn_fwd(qs, ks, vs, cu, scale=d ** -0.5, out_dtype=out_dtype,
                                q_start=q_start, kv_start=kv_start)
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    nsp.nsp_attn_fwd_noalloc(qs, ks, vs, cu, w.ndoc, q_start, q_len, kv_start, kv_len, Hq, Hkv,
                             d, d ** -0.5, True, out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == nsp_mod.NSP_OK
    return out, lse, ref_o, ref_l


def test_noalloc_matches_workspace_entry_point_twice(nsp):
    # call 1: tensor-core path, ragged documents; call 2: different layout and length
    w1 = make_custom([300, 1, 77, 500, 2], 8, 2, 128, seed=41, with_dout=False)
    w2 = make_custom([40] * 30 + [1200, 3], 16, 4, 128, seed=42, with_dout=False)
    for w in (w1, w2):
        out, lse, ro, rl = _run_both(nsp, w)
        assert max_abs(f64(out), f64(ro)) <= TOL_OUT
        assert max_abs(f64(lse), f64(rl)) <= TOL_LSE


def test_noalloc_partial_and_fp32_paths(nsp):
    # a float32 ring partial (key range ends mid-document), then float32 inputs
    w = make_custom([600, 250, 170], 8, 2, 128, seed=43, with_dout=False)
    out, lse, ro, rl = _run_both(nsp, w, out_dtype=torch.float32, q_start=512, q_len=508,
                                 kv_start=0, kv_len=700)
    assert max_abs(f64(out), f64(ro)) <= TOL_OUT
    assert max_abs(f64(lse), f64(rl)) <= TOL_LSE
    w32 = make_custom([90, 150], 4, 2, 64, dtype="f32", seed=44, with_dout=False)
    out, lse, ro, rl = _run_both(nsp, w32)
    assert max_abs(f64(out), f64(ro)) <= TOL_OUT_F32
    assert max_abs(f64(lse), f64(rl)) <= TOL_LSE_F32


def test_noalloc_rejects_sizes_beyond_its_scratch(nsp):
    lib = nsp_mod.load()
    big = 1 << 24                                     # 16M query tokens: above 1 MiB of scratch
    st = lib.nsp_attn_fwd_noalloc(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 0, big, 0, big, 8, 2,
                                  128, 0.088, 1, nsp_mod.NSP_BF16, 1 << 20, nsp_mod.NSP_BF16,
                                  None, None, None)
    assert st == nsp_mod.NSP_ERR_WORKSPACE
