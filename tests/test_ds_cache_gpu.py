"""Backward with the dS cache: nsp_attn_bwd given workspace past
nsp_attn_bwd_workspace_size keeps every dS = P (dP - delta) tile that the
dK/dV kernel builds and computes dQ = scale dS K from the cached tiles
instead of recomputing S and dP (the recomputation NSP Sec. 2.3 weighs
against memory).

Against the fp64 oracle: every element of small cases (GQA, MHA, odd
query-head groups, causal and not, empty and one-token documents, ragged
tails), config 5 whole with the per-row bar, config 2 on sampled dQ rows.
dK and dV must equal the recomputing backward's bit for bit (the cache only
adds a copy of a tile the kernel already builds); the cached dQ is
deterministic; a cache one tile short falls back to recomputation (bit for
bit the backward without cache); the head-grouped layout equals the packed
one with dq permuted.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (TOL_GRAD, assert_rows_close, f64, oracle_inputs, rel_l2, sample_rows,
                        timed, to_dev, workload)
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

TILE = 128 * 128 * 2


def _fwd(nsp, d, causal):
    return nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)


def _bwd(nsp, w, d, out, lse, causal, cache_bytes):
    T, Hq, hd = d["q"].shape
    ws = nsp.bwd_workspace(T, Hq, d["k"].shape[1], hd, "cuda", ds_cache_bytes=cache_bytes)
    g = nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], causal=causal,
                     workspace=ws)
    torch.cuda.synchronize()
    return g, nsp.nsp_bwd_ds_cache_used(ws)


SMALL = [
    ([1, 5, 0, 3], 4, 2, True),
    ([130, 1, 200], 8, 2, True),
    ([257, 300], 8, 1, False),
    ([33] * 12, 32, 4, True),
    ([600, 129, 300, 1, 500], 4, 4, True),
    ([600, 129, 300, 1, 500], 4, 4, False),
    ([400, 129], 6, 2, True),
    ([0, 5, 0, 260, 0, 1], 2, 2, True),
    ([1100, 77], 8, 2, False),
]


@pytest.mark.parametrize("lens,Hq,Hkv,causal", SMALL,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_{'c' if c[3] else 'nc'}"
                              for c in SMALL])
def test_small_whole(nsp, lens, Hq, Hkv, causal):
    w = make_custom(lens, Hq, Hkv, 128, seed=3 + sum(lens) + Hq)
    d = to_dev(w)
    out, lse = _fwd(nsp, d, causal)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, Hq, causal)
    (dq0, dk0, dv0), used0 = _bwd(nsp, w, d, out, lse, causal, 0)
    (dq, dk, dv), used = _bwd(nsp, w, d, out, lse, causal, need)
    (dq2, _, _), _ = _bwd(nsp, w, d, out, lse, causal, need)
    assert not used0 and used, (used0, used)
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0), "dK/dV changed by the cache copy"
    assert torch.equal(dq, dq2), "cached dQ not deterministic"
    q, k, v, do = oracle_inputs(w)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, 128 ** -0.5, causal)
    for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_l2(f64(g), r)
        print(f"[{lens} {n} cached] rel L2 {e:.3e}")
        assert e <= TOL_GRAD, n
    assert_rows_close(f64(dq), rq, label=f"{lens} dq cached per row")


def test_cache_one_tile_short_recomputes(nsp):
    w = make_custom([700, 129, 33, 400], 8, 2, 128, seed=61)
    d = to_dev(w)
    out, lse = _fwd(nsp, d, True)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, 8)
    (dq0, dk0, dv0), _ = _bwd(nsp, w, d, out, lse, True, 0)
    (dq, dk, dv), used = _bwd(nsp, w, d, out, lse, True, need - TILE)
    assert not used
    assert torch.equal(dq, dq0) and torch.equal(dk, dk0) and torch.equal(dv, dv0)
    (_, _, _), used = _bwd(nsp, w, d, out, lse, True, need)
    assert used


@pytest.mark.parametrize("P", [2, 4])
def test_headgroups_equals_packed(nsp, P):
    w = make_custom([700, 129, 33], 8, 2, 128, seed=62)
    d = to_dev(w)
    out, lse = _fwd(nsp, d, True)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, 8)
    (dq, dk, dv), used = _bwd(nsp, w, d, out, lse, True, need)
    assert used
    T = w.T
    ws = nsp.bwd_workspace(T, 8, 2, 128, "cuda", ds_cache_bytes=need)
    dqg, dkg, dvg = nsp.attn_bwd_headgroups(nsp.seq2head(d["q"], P), d["k"], d["v"],
                                            nsp.seq2head(out, P), nsp.seq2head(d["dout"], P),
                                            lse, d["cu"], workspace=ws)
    torch.cuda.synchronize()
    assert nsp.nsp_bwd_ds_cache_used(ws)
    assert torch.equal(dqg, nsp.seq2head(dq, P)) and torch.equal(dkg, dk) and torch.equal(dvg, dv)


def test_config5_whole(nsp):
    w = workload(5)
    d = to_dev(w)
    out, lse = _fwd(nsp, d, True)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, w.cfg.Hq)
    (dq, dk, dv), used = _bwd(nsp, w, d, out, lse, True, need)
    assert used
    q, k, v, do = oracle_inputs(w)
    rq, rk, rv = timed("oracle bwd C5", oracle.attn_bwd, q, k, v, do, w.cu_seqlens,
                       128 ** -0.5, True)
    for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_l2(f64(g), r)
        print(f"[C5 {n} cached] rel L2 {e:.3e}")
        assert e <= TOL_GRAD, n
        assert_rows_close(f64(g), r, label=f"C5 {n} cached per row")


def test_config2_sampled(nsp):
    w = workload(2)
    d = to_dev(w)
    out, lse = _fwd(nsp, d, True)
    need = nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, w.cfg.Hq)
    (dq0, dk0, dv0), _ = _bwd(nsp, w, d, out, lse, True, 0)
    (dq, dk, dv), used = _bwd(nsp, w, d, out, lse, True, need)
    assert used
    assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
    del dq0, dk0, dv0
    q, k, v, do = oracle_inputs(w)
    cu = w.cu_seqlens
    # rows of the longest document (up to 64 key tiles each) and seeded rows
    b = int(np.argmax(np.diff(cu)))
    rows = np.unique(np.concatenate([sample_rows(cu, 384, seed=72),
                                     np.arange(int(cu[b + 1]) - 64, int(cu[b + 1]))]))
    rq = timed(f"oracle dq C2 {len(rows)} rows", oracle.attn_bwd_dq_rows, q, k, v, do, cu,
               128 ** -0.5, True, rows)
    got = f64(dq[torch.from_numpy(rows).cuda()])
    e = rel_l2(got, rq)
    print(f"[C2 dq rows cached] rel L2 {e:.3e}")
    assert e <= TOL_GRAD
    assert_rows_close(got, rq, label="C2 dq rows cached")
