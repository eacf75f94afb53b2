"""Races and stray writes, without a sanitizer (none is available here).

* Grid independence: the persistent attention kernels take work items
  dynamically, and each item is computed whole by one CTA, so the results
  must be bit-identical whatever the number of CTAs.  The grid is shrunk
  through the NSP_PERSISTENT_CTAS environment variable; a race between CTAs
  (a shared buffer, a counter, a schedule read before it is written) shows
  up as a bit difference.  One entry point is grid-dependent by design: the
  ring-block backward splits its dK/dV items over query-head subsets when
  the block has few key tiles for the grid, and the subsets add into the
  float32 accumulators with atomics, so its dk/dv may differ in the last
  bits between grids; it is compared within the gradient bar instead.
* Guard zones: every output is a view into a larger buffer whose guard bytes
  before and after hold a pattern; after the calls the guards must be
  unchanged, so no kernel writes past the rows, heads or tiles it owns.
"""
import os

import pytest
import torch

from gpu_common import f64, rel_l2, to_dev
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

GUARD = 4096           # bytes on each side; keeps every view 16-byte aligned
PATTERN = 0x5A


def _run_all(nsp, w, dev):
    """Bit-identical across grids: forward, backward (recomputing and with
    the dS cache), a ring partial block, the ring accumulation in place, the
    head-grouped forward, the forward without a workspace, two batched
    blocks, and the forward and backward at head dimension 64.  Returned
    last: the ring-block backward's (dq, dk, dv), grid-dependent in the last
    bits."""
    sc = w.cfg.d ** -0.5
    T, Hq, Hkv = w.T, w.cfg.Hq, w.cfg.Hkv
    out, lse = nsp.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], scale=sc)
    dq, dk, dv = nsp.attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                              scale=sc)
    qa, ka = 200, 64
    po, pl = nsp.attn_fwd(dev["q"][qa:], dev["k"][ka:], dev["v"][ka:], dev["cu"], scale=sc,
                          out_dtype=torch.float32, q_start=qa, kv_start=ka)
    acc, lacc = nsp.ring_accumulate_init(T - qa, Hq, w.cfg.d, "cuda")
    for a, b in ((ka, T), (0, ka)):
        nsp.attn_fwd_accumulate(dev["q"][qa:], dev["k"][a:b], dev["v"][a:b], dev["cu"], acc, lacc,
                                scale=sc, q_start=qa, kv_start=a)
    og, lg = nsp.attn_fwd_headgroups(nsp.seq2head(dev["q"], 2), dev["k"], dev["v"], dev["cu"],
                                     scale=sc)
    bl = [(qa, T - qa, ka, T - ka, torch.empty((T - qa, Hq, w.cfg.d), device="cuda"),
           torch.empty((Hq, T - qa), device="cuda")),
          (0, qa, 0, qa, torch.empty((qa, Hq, w.cfg.d), device="cuda"),
           torch.empty((Hq, qa), device="cuda"))]
    nsp.attn_fwd_blocks(dev["q"], dev["k"], dev["v"], dev["cu"], bl, scale=sc)
    on, ln = torch.empty_like(out), torch.empty_like(lse)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    nsp.nsp_attn_fwd_noalloc(dev["q"], dev["k"], dev["v"], dev["cu"], len(w.lengths), 0, T, 0, T,
                             Hq, Hkv, w.cfg.d, sc, True, on, ln, st)
    gq = torch.zeros((T - qa, Hq, w.cfg.d), dtype=torch.float32, device="cuda")
    gk = torch.zeros((T - ka, Hkv, w.cfg.d), dtype=torch.float32, device="cuda")
    gv = torch.zeros_like(gk)
    nsp.attn_bwd_accumulate(dev["q"][qa:], dev["k"][ka:], dev["v"][ka:], out[qa:], dev["dout"][qa:],
                            lse[:, qa:].contiguous(), dev["cu"], gq, gk, gv, scale=sc,
                            q_start=qa, kv_start=ka)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, Hq)
    ws_c = nsp.bwd_workspace(T, Hq, Hkv, w.cfg.d, "cuda", ds_cache_bytes=need)
    cq, ck, cv = nsp.attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                              scale=sc, workspace=ws_c)
    assert nsp.nsp_bwd_ds_cache_used(ws_c)
    # head dimension 64: the first half of every head's columns as its own problem
    h64 = {n: dev[n][:, :, :64].contiguous() for n in ("q", "k", "v", "dout")}
    o64, l64 = nsp.attn_fwd(h64["q"], h64["k"], h64["v"], dev["cu"])
    g64 = nsp.attn_bwd(h64["q"], h64["k"], h64["v"], o64, h64["dout"], l64, dev["cu"])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ([out, lse, dq, dk, dv, po, pl, acc, lacc, og, lg, on, ln] + [t for b in bl for t in b[4:]]
            + [cq, ck, cv, o64, l64, *g64], (gq, gk, gv))


@pytest.mark.parametrize("lens", [[100, 1, 300, 60, 250, 0, 517], [33] * 40 + [700]],
                         ids=["mixed", "short_docs"])
def test_results_do_not_depend_on_the_grid(nsp, lens):
    w = make_custom(lens, 8, 2, 128, seed=70)
    dev = to_dev(w)
    ref, ref_ring = _run_all(nsp, w, dev)
    old = os.environ.get("NSP_PERSISTENT_CTAS")
    try:
        for ctas in ("1", "7", "64"):
            os.environ["NSP_PERSISTENT_CTAS"] = ctas
            got, got_ring = _run_all(nsp, w, dev)
            for i, (a, b) in enumerate(zip(ref, got)):
                assert torch.equal(a, b), f"output {i} differs with {ctas} CTAs"
            for name, a, b in zip(("dq", "dk", "dv"), ref_ring, got_ring):
                e = rel_l2(f64(b), f64(a))
                assert e <= 1e-5, f"ring-block {name} differs by {e} with {ctas} CTAs"
    finally:
        if old is None:
            os.environ.pop("NSP_PERSISTENT_CTAS", None)
        else:
            os.environ["NSP_PERSISTENT_CTAS"] = old


def _guarded(shape, dtype):
    n = torch.Size(shape).numel() * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(dtype).view(shape)


def _guards_intact(buf):
    return bool((buf[:GUARD] == PATTERN).all()) and bool((buf[-GUARD:] == PATTERN).all())


def test_outputs_stay_inside_their_buffers(nsp):
    w = make_custom([100, 1, 300, 60, 250, 0, 129], 8, 2, 128, seed=71)
    dev = to_dev(w)
    T, Hq, Hkv, d = w.T, 8, 2, 128
    sc = d ** -0.5
    bufs = {}

    def g(name, shape, dtype):
        b, t = _guarded(shape, dtype)
        bufs[name] = b
        return t

    ws_f = g("ws_f", (nsp.nsp_attn_fwd_workspace_size(T, T, Hq, Hkv, d),), torch.uint8)
    ws_b = g("ws_b", (nsp.nsp_attn_bwd_workspace_size(T, Hq, Hkv, d),), torch.uint8)
    out, lse = g("out", (T, Hq, d), torch.bfloat16), g("lse", (Hq, T), torch.float32)
    nsp.nsp_attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], len(w.lengths), 0, T, 0, T, Hq,
                     Hkv, d, sc, True, out, lse, ws_f)
    dq = g("dq", (T, Hq, d), torch.bfloat16)
    dk, dv = g("dk", (T, Hkv, d), torch.bfloat16), g("dv", (T, Hkv, d), torch.bfloat16)
    nsp.nsp_attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                     len(w.lengths), T, Hq, Hkv, d, sc, True, dq, dk, dv, ws_b)
    # a ring block: partial, in-place accumulation, block backward
    qa, ka, n = 256, 0, T - 256
    po, pl = g("po", (n, Hq, d), torch.float32), g("pl", (Hq, n), torch.float32)
    ws_r = g("ws_r", (nsp.nsp_attn_fwd_workspace_size(n, n, Hq, Hkv, d),), torch.uint8)
    nsp.nsp_attn_fwd(dev["q"][qa:], dev["k"][ka:ka + n], dev["v"][ka:ka + n], dev["cu"],
                     len(w.lengths), qa, n, ka, n, Hq, Hkv, d, sc, True, po, pl, ws_r)
    nsp.nsp_attn_fwd_accumulate(dev["q"][qa:], dev["k"][ka:ka + n], dev["v"][ka:ka + n],
                                dev["cu"], len(w.lengths), qa, n, ka, n, Hq, Hkv, d, sc, True,
                                po, pl, ws_r)
    gq = g("gq", (n, Hq, d), torch.float32)
    gk, gv = g("gk", (n, Hkv, d), torch.float32), g("gv", (n, Hkv, d), torch.float32)
    for t in (gq, gk, gv):
        t.zero_()
    ws_ba = g("ws_ba", (nsp.nsp_attn_bwd_accumulate_workspace_size(n, n, Hq, Hkv, d),),
              torch.uint8)
    nsp.nsp_attn_bwd_accumulate(dev["q"][qa:], dev["k"][ka:ka + n], dev["v"][ka:ka + n],
                                out[qa:], dev["dout"][qa:], lse[:, qa:].contiguous(), dev["cu"],
                                len(w.lengths), qa, n, ka, n, Hq, Hkv, d, sc, True, gq, gk, gv,
                                ws_ba)
    # merge (single and batched) and the permutation both ways
    mo, ml = g("mo", (n, Hq, d), torch.bfloat16), g("ml", (Hq, n), torch.float32)
    nsp.nsp_lse_merge([po, po], [pl, pl], mo, ml)
    mb, mbl = g("mb", (n, Hq, d), torch.float32), g("mbl", (Hq, n), torch.float32)
    mb2 = g("mb2", (n, Hq, d), torch.float32)
    nsp.nsp_lse_merge_batch([([po], [pl]), ([po, po], [pl, pl])], [mb, mb2], [mbl, None])
    # two batched blocks of the whole stream, and the subgroup permutation
    b1o, b1l = g("b1o", (n, Hq, d), torch.float32), g("b1l", (Hq, n), torch.float32)
    b2o, b2l = g("b2o", (qa, Hq, d), torch.float32), g("b2l", (Hq, qa), torch.float32)
    blocks = [(qa, n, ka, n, b1o, b1l), (0, qa, 0, qa, b2o, b2l)]
    ws_bl = g("ws_bl", (nsp.nsp_attn_fwd_blocks_workspace_size(blocks, Hq, Hkv, d),), torch.uint8)
    nsp.nsp_attn_fwd_blocks(dev["q"], dev["k"], dev["v"], dev["cu"], len(w.lengths), T, blocks,
                            Hq, Hkv, d, sc, True, False, ws_bl)
    Tg = T - T % 3
    pg = g("pg", (3, 2, Tg // 3, Hq // 2, d), torch.bfloat16)
    nsp.nsp_seq2head_permute_groups(dev["q"][:Tg], pg, 3, Tg // 3, Hq, d, 2, False)
    perm = g("perm", (4, T, Hq // 4, d), torch.bfloat16)
    back = g("back", (T, Hq, d), torch.bfloat16)
    nsp.nsp_seq2head_permute(dev["q"], perm, T, Hq, d, 4, False)
    nsp.nsp_seq2head_permute(perm, back, T, Hq, d, 4, True)
    # the backward with an exactly sized dS cache (the guard follows its last
    # slot), and the forward and backward at head dimension 64
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, Hq)
    base = (nsp.nsp_attn_bwd_workspace_size(T, Hq, Hkv, d) + 1023) // 1024 * 1024
    ws_c = g("ws_c", (base + need,), torch.uint8)
    cq = g("cq", (T, Hq, d), torch.bfloat16)
    ck, cv = g("ck", (T, Hkv, d), torch.bfloat16), g("cv", (T, Hkv, d), torch.bfloat16)
    nsp.nsp_attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                     len(w.lengths), T, Hq, Hkv, d, sc, True, cq, ck, cv, ws_c)
    assert nsp.nsp_bwd_ds_cache_used(ws_c)
    h64 = {n: dev[n][:, :, :64].contiguous() for n in ("q", "k", "v", "dout")}
    o64, l64 = g("o64", (T, Hq, 64), torch.bfloat16), g("l64", (Hq, T), torch.float32)
    ws_f64 = g("ws_f64", (nsp.nsp_attn_fwd_workspace_size(T, T, Hq, Hkv, 64),), torch.uint8)
    nsp.nsp_attn_fwd(h64["q"], h64["k"], h64["v"], dev["cu"], len(w.lengths), 0, T, 0, T, Hq,
                     Hkv, 64, 64 ** -0.5, True, o64, l64, ws_f64)
    q64 = g("q64", (T, Hq, 64), torch.bfloat16)
    k64, v64 = g("k64", (T, Hkv, 64), torch.bfloat16), g("v64", (T, Hkv, 64), torch.bfloat16)
    base64 = (nsp.nsp_attn_bwd_workspace_size(T, Hq, Hkv, 64) + 1023) // 1024 * 1024
    ws_b64 = g("ws_b64", (base64 + need,), torch.uint8)
    nsp.nsp_attn_bwd(h64["q"], h64["k"], h64["v"], o64, h64["dout"], l64, dev["cu"],
                     len(w.lengths), T, Hq, Hkv, 64, 64 ** -0.5, True, q64, k64, v64, ws_b64)
    torch.cuda.synchronize()
    bad = [name for name, b in bufs.items() if not _guards_intact(b)]
    assert not bad, f"guard bytes overwritten around: {bad}"
    assert torch.equal(back, dev["q"])
