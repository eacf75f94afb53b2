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


def _call(nsp, w, cu_np, out, lse, status):
    q, k, v = (getattr(w, n).cuda() for n in ("q", "k", "v"))
    T, Hq, d = q.shape
    cu = torch.from_numpy(cu_np).cuda()
    nsp.nsp_attn_fwd_noalloc(q, k, v, cu, len(cu_np) - 1, 0, T, 0, T, Hq, k.shape[1], d,
                             d ** -0.5, True, out, lse, status)
    torch.cuda.synchronize()
    return int(status.item())


def test_noalloc_bad_cu_seqlens_reported_then_cleared(nsp):
    """A malformed cu_seqlens reaches the caller through device_status; the
    next valid call on the shared scratch starts afresh and matches."""
    w = make_custom([120, 90, 300], 8, 2, 128, seed=45, with_dout=False)
    out = torch.empty((w.T, 8, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, w.T), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for bad in ("decreasing", "first_nonzero"):
        cu = w.cu_seqlens.copy()
        if bad == "decreasing":
            cu[1], cu[2] = cu[2], cu[1]
        else:
            cu[0] = 5
        assert _call(nsp, w, cu, out, lse, status) == nsp_mod.NSP_ERR_INVALID, bad
        o, l, ro, rl = _run_both(nsp, w)
        assert max_abs(f64(o), f64(ro)) <= TOL_OUT and max_abs(f64(l), f64(rl)) <= TOL_LSE


def test_noalloc_empty_query_range(nsp):
    """q_len = 0: only the scheduler and the status copy run."""
    w = make_custom([64, 64], 4, 2, 128, seed=46, with_dout=False)
    q, k, v = (getattr(w, n).cuda() for n in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    out = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((4, 0), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    nsp.nsp_attn_fwd_noalloc(q[:0], k, v, cu, w.ndoc, 0, 0, 0, w.T, 4, 2, 128, 128 ** -0.5, True,
                             out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == nsp_mod.NSP_OK


def test_noalloc_device_memory_unchanged(nsp):
    """After the set-up of a device (its first call looks the scratch up),
    calls of any size up to the limit leave the device's free memory exactly
    where it was: the entry point allocates nothing."""
    ws = [make_custom([300, 1, 77, 500, 2], 8, 2, 128, seed=47, with_dout=False),
          make_custom([40] * 30 + [1200, 3], 16, 4, 128, seed=48, with_dout=False)]
    bufs = []
    for w in ws:
        q, k, v = (getattr(w, n).cuda() for n in ("q", "k", "v"))
        bufs.append((w, q, k, v, torch.from_numpy(w.cu_seqlens).cuda(),
                     torch.empty_like(q), torch.empty((q.shape[1], w.T), dtype=torch.float32,
                                                      device="cuda")))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    def run(b):
        w, q, k, v, cu, out, lse = b
        nsp.nsp_attn_fwd_noalloc(q, k, v, cu, w.ndoc, 0, w.T, 0, w.T, q.shape[1], k.shape[1], 128,
                                 128 ** -0.5, True, out, lse, status)

    run(bufs[0])                       # set-up of this device (if not done yet)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for b in bufs:
            run(b)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert int(status.item()) == nsp_mod.NSP_OK
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_sizes_beyond_its_scratch(nsp):
    lib = nsp_mod.load()
    big = 1 << 24                                     # 16M query tokens: above 1 MiB of scratch
    st = lib.nsp_attn_fwd_noalloc(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 0, big, 0, big, 8, 2,
                                  128, 0.088, 1, nsp_mod.NSP_BF16, 1 << 20, nsp_mod.NSP_BF16,
                                  None, None, None)
    assert st == nsp_mod.NSP_ERR_WORKSPACE
