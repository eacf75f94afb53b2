"""Batched ring-block backward (nsp_attn_bwd_blocks): the contributions of
many (query range, key range) blocks added into whole-stream float32
gradient accumulators in one launch of each backward kernel (HSAP Sec.
2.2.1 ring InterSP; Sec. 3.2 blocks).

Checked against one nsp_attn_bwd_accumulate call per block (the same
arithmetic per block; only the order of the float additions differs), against
the oracle's ring-block backward summed over the blocks, and, for every
block of a ring (causal and not), against the oracle's whole-stream
gradients.  Config 2 as a ring of 8 shards in one call is compared with the
whole-stream backward and the oracle on sampled rows and keys.  With a dS
cache (every block's dS tiles kept, dQ from them), the batched backward is
compared with the same call without it and with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TOL_GRAD, f64, oracle_inputs, rel_l2, sample_rows, to_dev, workload
from variable_length_sequence_gb300.workloads import make_custom, shard_bounds

pytestmark = pytest.mark.gpu


def _zeros(w):
    T, Hq, Hkv, d = w.T, w.cfg.Hq, w.cfg.Hkv, w.cfg.d
    return (torch.zeros((T, Hq, d), device="cuda"), torch.zeros((T, Hkv, d), device="cuda"),
            torch.zeros((T, Hkv, d), device="cuda"))


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_blocks_equal_per_block_calls_and_oracle(nsp, causal):
    w = make_custom([600, 129, 300, 1, 500], 8, 2, 128, seed=111)
    d = to_dev(w)
    T = w.T
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)
    ranges = [(0, 400, 0, 400), (400, 400, 0, 400), (400, 400, 400, 400), (800, 300, 0, 800),
              (800, 730, 800, 730), (4, 1, 0, 1000), (128, 700, 650, 300), (0, 0, 0, 10),
              (400, 400, 0, 400)]                                   # a repeated block adds twice
    dq, dk, dv = _zeros(w)
    nsp.attn_bwd_blocks(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], ranges, dq, dk, dv,
                        causal=causal)
    rq, rk, rv = _zeros(w)
    for qa, ql, ka, kl in ranges:
        if ql == 0 or kl == 0:
            continue
        nsp.attn_bwd_accumulate(d["q"][qa:qa + ql], d["k"][ka:ka + kl], d["v"][ka:ka + kl],
                                out[qa:qa + ql], d["dout"][qa:qa + ql],
                                lse[:, qa:qa + ql].contiguous(), d["cu"], rq[qa:qa + ql],
                                rk[ka:ka + kl], rv[ka:ka + kl], causal=causal, q_start=qa,
                                kv_start=ka)
    torch.cuda.synchronize()
    for name, a, b in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_l2(f64(a), f64(b))
        print(f"[blocks vs per-block calls] {name} rel L2 {e:.2e}")
        assert e <= 1e-5, name
    q, k, v, do = oracle_inputs(w)
    oq, ok, ov = (np.zeros(t.shape) for t in (dq, dk, dv))
    for qa, ql, ka, kl in ranges:
        if ql == 0 or kl == 0:
            continue
        bq, bk, bv = oracle.attn_bwd_block(q, k, v, do, w.cu_seqlens, 128 ** -0.5, causal,
                                           (qa, qa + ql), (ka, ka + kl))
        oq[qa:qa + ql] += bq
        ok[ka:ka + kl] += bk
        ov[ka:ka + kl] += bv
    for name, a, r in (("dq", dq, oq), ("dk", dk, ok), ("dv", dv, ov)):
        e = rel_l2(f64(a), r)
        print(f"[blocks vs oracle] {name} rel L2 {e:.2e}")
        assert e <= TOL_GRAD, name


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_whole_ring_one_call(nsp, causal):
    """Every (query shard, key shard) block of a 6-shard ring in one call adds
    up to the whole-stream gradients."""
    w = make_custom([700, 33, 400, 129, 250], 8, 2, 128, seed=112)
    d = to_dev(w)
    n = 6
    T = w.T - w.T % (4 * n)
    cu = np.minimum(w.cu_seqlens, T)
    cu_d = torch.from_numpy(cu).cuda()
    q, k, v, do = (t[:T].contiguous() for t in (d["q"], d["k"], d["v"], d["dout"]))
    out, lse = nsp.attn_fwd(q, k, v, cu_d, causal=causal)
    bounds = shard_bounds(T, n)
    ranges = [(qa, qb - qa, ka, kb - ka) for qa, qb in bounds for ka, kb in bounds]
    dq = torch.zeros((T, 8, 128), device="cuda")
    dk, dv = torch.zeros((T, 2, 128), device="cuda"), torch.zeros((T, 2, 128), device="cuda")
    nsp.attn_bwd_blocks(q, k, v, out, do, lse, cu_d, ranges, dq, dk, dv, causal=causal)
    torch.cuda.synchronize()
    qo, ko, vo, doo = (x[:T] for x in oracle_inputs(w))
    ref = oracle.attn_bwd(qo, ko, vo, doo, cu, 128 ** -0.5, causal)
    for name, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        e = rel_l2(f64(a), r)
        print(f"[ring of {n} in one call, causal={causal}] {name} rel L2 {e:.2e}")
        assert e <= TOL_GRAD, name


def test_config2_ring_one_call(nsp):
    """Config 2 as a ring of 8 shards of 4096 tokens: the 36 causal blocks in
    one call, against nsp_attn_bwd and the oracle (sampled rows and keys)."""
    w = workload(2)
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"])
    gq, gk, gv = nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"])
    bounds = shard_bounds(w.T, 8)
    ranges = [(qa, qb - qa, ka, kb - ka) for i, (qa, qb) in enumerate(bounds)
              for ka, kb in bounds[:i + 1]]
    dq, dk, dv = _zeros(w)
    nsp.attn_bwd_blocks(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], ranges, dq, dk, dv)
    torch.cuda.synchronize()
    for name, a, b in (("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
        e = rel_l2(f64(a), f64(b))
        print(f"[C2 ring vs whole-stream backward] {name} rel L2 {e:.2e}")
        assert e <= 5e-3, name
    q, k, v, do = oracle_inputs(w)
    rows = sample_rows(w.cu_seqlens, 128, seed=113)
    rq = oracle.attn_bwd_dq_rows(q, k, v, do, w.cu_seqlens, 128 ** -0.5, True, rows)
    assert rel_l2(f64(dq[torch.from_numpy(rows).cuda()]), rq) <= TOL_GRAD
    keys = np.sort(np.random.default_rng(114).choice(w.T, 24, replace=False))
    rk, rv = oracle.attn_bwd_dkv_rows(q, k, v, do, w.cu_seqlens, 128 ** -0.5, True, keys, 1)
    kidx = torch.from_numpy(keys).cuda()
    assert rel_l2(f64(dk[kidx, 1]), rk) <= TOL_GRAD
    assert rel_l2(f64(dv[kidx, 1]), rv) <= TOL_GRAD


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_blocks_with_ds_cache(nsp, causal):
    """The batched backward with a dS cache sized by
    nsp_attn_bwd_blocks_ds_cache_size: the cache is used, and the gradients
    match the batched backward without it (1e-5: only the order of the float
    additions differs) and the oracle's blocks summed."""
    w = make_custom([600, 129, 300, 1, 500], 8, 2, 128, seed=115)
    d = to_dev(w)
    T = w.T
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)
    ranges = [(0, 400, 0, 400), (400, 400, 0, 400), (400, 400, 400, 400), (800, 300, 0, 800),
              (800, 730, 800, 730), (4, 1, 0, 1000), (128, 700, 650, 300), (0, 0, 0, 10),
              (400, 400, 0, 400)]
    need = nsp.nsp_attn_bwd_blocks_ds_cache_size(w.cu_seqlens, ranges, 8, causal)
    assert need > 0
    base = (nsp.nsp_attn_bwd_blocks_workspace_size(T, ranges, 8, 2, 128) + 1023) // 1024 * 1024
    res = {}
    for cache in (0, need):
        ws = torch.empty(base + cache, dtype=torch.uint8, device="cuda")
        g = _zeros(w)
        nsp.attn_bwd_blocks(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], ranges, *g,
                            causal=causal, workspace=ws)
        torch.cuda.synchronize()
        assert nsp.nsp_bwd_ds_cache_used(ws) == (cache > 0)
        res[cache > 0] = g
    for name, a, b in zip(("dq", "dk", "dv"), res[True], res[False]):
        e = rel_l2(f64(a), f64(b))
        print(f"[blocks cached vs not] {name} rel L2 {e:.2e}")
        assert e <= 1e-5, name
    q, k, v, do = oracle_inputs(w)
    oq, ok, ov = (np.zeros(t.shape) for t in res[True])
    for qa, ql, ka, kl in ranges:
        if ql == 0 or kl == 0:
            continue
        bq, bk, bv = oracle.attn_bwd_block(q, k, v, do, w.cu_seqlens, 128 ** -0.5, causal,
                                           (qa, qa + ql), (ka, ka + kl))
        oq[qa:qa + ql] += bq
        ok[ka:ka + kl] += bk
        ov[ka:ka + kl] += bv
    for name, a, r in zip(("dq", "dk", "dv"), res[True], (oq, ok, ov)):
        assert rel_l2(f64(a), r) <= TOL_GRAD, name


def test_config2_ring_one_call_ds_cache(nsp):
    """Config 2's 36-block ring in one call with the dS cache: used, and
    within 1e-5 of the same call without it."""
    w = workload(2)
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"])
    bounds = shard_bounds(w.T, 8)
    ranges = [(qa, qb - qa, ka, kb - ka) for i, (qa, qb) in enumerate(bounds)
              for ka, kb in bounds[:i + 1]]
    need = nsp.nsp_attn_bwd_blocks_ds_cache_size(w.cu_seqlens, ranges, w.cfg.Hq)
    base = (nsp.nsp_attn_bwd_blocks_workspace_size(w.T, ranges, 32, 4, 128) + 1023) // 1024 * 1024
    res = {}
    for cache in (0, need):
        ws = torch.empty(base + cache, dtype=torch.uint8, device="cuda")
        g = _zeros(w)
        nsp.attn_bwd_blocks(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], ranges, *g,
                            workspace=ws)
        torch.cuda.synchronize()
        assert nsp.nsp_bwd_ds_cache_used(ws) == (cache > 0)
        res[cache > 0] = g
        del ws
    for name, a, b in zip(("dq", "dk", "dv"), res[True], res[False]):
        e = rel_l2(f64(a), f64(b))
        print(f"[C2 ring cached vs not] {name} rel L2 {e:.2e}")
        assert e <= 1e-5, name
