"""Head dimension 64 on the tensor cores (bf16), against the fp64 oracle:
the same kernels with 64-column Q, K, V (and dOut) tiles and 64-column O,
dQ, dK, dV accumulators.  Forward, checked at every element: GQA with an
even and an odd number of query heads per KV head (multi-head attention
among them), causal and not, ragged tails, zero-length and one-token
documents, a document ending inside a tile; ring partial blocks (float32
out) and accumulation in place; the batched block call (bit-identical to one
call per block); the head-grouped layout (bit-identical to the packed
forward followed by the permutation).  Backward: whole-stream gradients,
recomputing and with the dS cache, and a ring's blocks batched and one per
call.  Every call launches tensor-core kernels only.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_fwd_close, f64, oracle_inputs, to_dev
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

D = 64
CASES = [
    # lengths, Hq, Hkv, causal
    ([1, 1, 1], 2, 1, True),
    ([77, 128, 129, 255, 256, 257], 8, 2, True),
    ([77, 128, 129, 255, 256, 257], 8, 2, False),
    ([1500, 3, 700], 4, 4, True),
    ([0, 5, 0, 260, 0, 1], 2, 2, True),
    ([400, 129], 6, 2, False),
    ([33] * 20, 16, 2, True),
]


def _tc_only(nsp, fn):
    tc0, cc0 = nsp.nsp_path_launches(True), nsp.nsp_path_launches(False)
    r = fn()
    torch.cuda.synchronize()
    assert nsp.nsp_path_launches(False) == cc0, "a CUDA-core attention kernel ran"
    assert nsp.nsp_path_launches(True) > tc0
    return r


@pytest.mark.parametrize("lens,Hq,Hkv,causal", CASES,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_{'c' if c[3] else 'nc'}" for c in CASES])
def test_forward_whole(nsp, lens, Hq, Hkv, causal):
    w = make_custom(lens, Hq, Hkv, D, seed=sum(lens) + 3 * Hq, with_dout=False)
    d = to_dev(w)
    out, lse = _tc_only(nsp, lambda: nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal))
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, D ** -0.5, causal)
    assert_fwd_close(f64(out), f64(lse), ro, rl, label=f"d64 {lens} h{Hq}kv{Hkv}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4)], ids=["gqa", "mha"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_ring_partials_and_accumulate(nsp, Hq, Hkv, causal):
    w = make_custom([600, 129, 300, 1], Hq, Hkv, D, seed=95 + Hq, with_dout=False)
    d = to_dev(w)
    q, k, v, _ = oracle_inputs(w)
    T = w.T
    for qa, qb, ka, kb in ((0, T, 0, T), (300, 900, 0, 400), (129, 257, 600, T), (5, 6, 0, T)):
        po, pl = _tc_only(nsp, lambda: nsp.attn_fwd(
            d["q"][qa:qb], d["k"][ka:kb], d["v"][ka:kb], d["cu"], causal=causal,
            out_dtype=torch.float32, q_start=qa, kv_start=ka))
        ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, D ** -0.5, causal, q_range=(qa, qb),
                                 kv_range=(ka, kb))
        assert_fwd_close(f64(po), f64(pl), ro, rl, label=f"d64 partial q{qa}:{qb} k{ka}:{kb}")
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, D ** -0.5, causal)
    rng = np.random.default_rng(96)
    cuts = np.unique(np.concatenate([[0, T], rng.integers(1, T, 5)]))
    blocks = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
    acc, lacc = nsp.ring_accumulate_init(T, Hq, D, "cuda")
    for ka, kb in [blocks[i] for i in rng.permutation(len(blocks))]:
        nsp.attn_fwd_accumulate(d["q"], d["k"][ka:kb], d["v"][ka:kb], d["cu"], acc, lacc,
                                causal=causal, kv_start=ka)
    torch.cuda.synchronize()
    assert_fwd_close(f64(acc), f64(lacc), ro, rl, label="d64 ring accumulate")


def test_blocks_equal_single_calls(nsp):
    w = make_custom([600, 129, 300, 1, 500], 8, 2, D, seed=97, with_dout=False)
    d = to_dev(w)
    ranges = [(0, 400, 0, 400), (400, 400, 0, 400), (800, 300, 800, 300), (5, 1, 0, 1000),
              (129, 700, 650, 300)]
    bl = []
    for qa, ql, ka, kl in ranges:
        bl.append((qa, ql, ka, kl,
                   torch.full((ql, 8, D), float("nan"), dtype=torch.float32, device="cuda"),
                   torch.full((8, ql), float("nan"), device="cuda")))
    _tc_only(nsp, lambda: nsp.attn_fwd_blocks(d["q"], d["k"], d["v"], d["cu"], bl))
    for qa, ql, ka, kl, out, lse in bl:
        so, sl = nsp.attn_fwd(d["q"][qa:qa + ql], d["k"][ka:ka + kl], d["v"][ka:ka + kl], d["cu"],
                              out_dtype=torch.float32, q_start=qa, kv_start=ka)
        torch.cuda.synchronize()
        assert torch.equal(out, so) and torch.equal(lse, sl), (qa, ql, ka, kl)


def test_headgroups(nsp):
    w = make_custom([700, 129, 33], 8, 2, D, seed=98, with_dout=False)
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"])
    for P in (2, 4, 8):
        og, lg = _tc_only(nsp, lambda: nsp.attn_fwd_headgroups(nsp.seq2head(d["q"], P), d["k"],
                                                                d["v"], d["cu"]))
        assert torch.equal(og, nsp.seq2head(out, P)) and torch.equal(lg, lse), P


BWD = [
    ([77, 128, 129, 255, 256, 257], 8, 2, True),
    ([600, 129, 300, 1], 4, 4, False),
    ([0, 5, 0, 260, 0, 1], 6, 2, True),
    ([1, 5, 0, 3], 4, 2, True),
]


@pytest.mark.parametrize("lens,Hq,Hkv,causal", BWD,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_{'c' if c[3] else 'nc'}" for c in BWD])
def test_backward_whole_and_ds_cache(nsp, lens, Hq, Hkv, causal):
    """The tensor-core backward at d = 64, recomputing and with the dS
    cache: every element against the oracle's gradients, dK/dV equal bit
    for bit between the two."""
    from gpu_common import TOL_GRAD, assert_rows_close, rel_l2
    w = make_custom(lens, Hq, Hkv, D, seed=7 + sum(lens) + Hq)
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)
    T = w.T
    res = {}
    for cache in (0, nsp.nsp_attn_bwd_ds_cache_size(w.cu_seqlens, Hq, causal)):
        ws = nsp.bwd_workspace(T, Hq, Hkv, D, "cuda", ds_cache_bytes=cache)
        res[cache > 0] = _tc_only(nsp, lambda: nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"],
                                                            lse, d["cu"], causal=causal,
                                                            workspace=ws))
        assert nsp.nsp_bwd_ds_cache_used(ws) == (cache > 0)
    q, k, v, do = oracle_inputs(w)
    ref = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, D ** -0.5, causal)
    for cached, grads in res.items():
        for name, g, r in zip(("dq", "dk", "dv"), grads, ref):
            e = rel_l2(f64(g), r)
            print(f"[d64 {lens} {name} cache={cached}] rel L2 {e:.3e}")
            assert e <= TOL_GRAD, (name, cached)
        assert_rows_close(f64(grads[0]), ref[0], label=f"d64 dq cache={cached}")
    assert torch.equal(res[True][1], res[False][1]) and torch.equal(res[True][2], res[False][2])


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_ring_backward_blocks(nsp, causal):
    """Every block of a 4-shard ring in one batched call (and one call per
    block) adds up to the oracle's whole-stream gradients."""
    from gpu_common import TOL_GRAD, rel_l2
    w = make_custom([600, 129, 300, 1, 570], 8, 2, D, seed=99)
    d = to_dev(w)
    T = w.T
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)
    n = T // 4
    ranges = [(i * n, n, j * n, n) for i in range(4) for j in range(4) if not causal or j <= i]
    acc = [torch.zeros((T, 8, D), device="cuda"), torch.zeros((T, 2, D), device="cuda"),
           torch.zeros((T, 2, D), device="cuda")]
    _tc_only(nsp, lambda: nsp.attn_bwd_blocks(d["q"], d["k"], d["v"], out, d["dout"], lse,
                                              d["cu"], ranges, *acc, causal=causal))
    per = [torch.zeros_like(t) for t in acc]
    for qa, ql, ka, kl in ranges:
        nsp.attn_bwd_accumulate(d["q"][qa:qa + ql], d["k"][ka:ka + kl], d["v"][ka:ka + kl],
                                out[qa:qa + ql], d["dout"][qa:qa + ql],
                                lse[:, qa:qa + ql].contiguous(), d["cu"], per[0][qa:qa + ql],
                                per[1][ka:ka + kl], per[2][ka:ka + kl], causal=causal, q_start=qa,
                                kv_start=ka)
    torch.cuda.synchronize()
    q, k, v, do = oracle_inputs(w)
    ref = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, D ** -0.5, causal)
    for name, a, b, r in zip(("dq", "dk", "dv"), acc, per, ref):
        assert rel_l2(f64(a), f64(b)) <= 1e-5, name
        e = rel_l2(f64(a), r)
        print(f"[d64 ring blocks {name}] rel L2 {e:.3e}")
        assert e <= TOL_GRAD, name
