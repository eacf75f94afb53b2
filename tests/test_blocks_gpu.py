"""Batched ring blocks (nsp_attn_fwd_blocks): many (query range, key range)
blocks of one packed stream in one schedule and one launch (HSAP Sec.
2.2.1, InterSP ring; Sec. 3.2, attention blocks).

Every block's output must equal, bit for bit, nsp_attn_fwd on that block
alone (the same kernel walks the same tiles in the same order); the blocks
are also compared with the oracle's partials, and a ring accumulated step by
step (one batched call per step, one block per query shard) with the
oracle's unchunked attention.  Config 3's whole ring (every non-empty causal
block of 8 shards of 16384 tokens) runs as one call.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_fwd_close, f64, oracle_inputs, to_dev, workload
from variable_length_sequence_gb300.workloads import make_custom, shard_bounds

pytestmark = pytest.mark.gpu

SHAPES = [  # lengths, Hq, Hkv, d, dtype: tcgen05 GQA, tcgen05 paired tiles (MHA), CUDA cores
    ([600, 129, 300, 1, 500], 8, 2, 128, "bf16"),
    ([600, 129, 300, 1, 500], 4, 4, 128, "bf16"),
    ([300, 77, 150], 4, 2, 64, "f32"),
]
RANGES = [(0, 400, 0, 400), (400, 400, 0, 400), (400, 400, 400, 400), (800, 300, 0, 800),
          (800, 300, 800, 300), (5, 1, 0, 1000), (129, 700, 650, 300), (0, 0, 0, 10),
          (1000, 30, 0, 0)]


def _blocks(w, d, dev, ranges, accumulate=False):
    Hq, hd = w.cfg.Hq, w.cfg.d
    bl = []
    for qa, ql, ka, kl in ranges:
        if accumulate:
            out, lse = torch.zeros((ql, Hq, hd), dtype=torch.float32, device=dev), \
                torch.full((Hq, ql), float("-inf"), device=dev)
        else:
            out = torch.full((ql, Hq, hd), float("nan"), dtype=torch.float32, device=dev)
            lse = torch.full((Hq, ql), float("nan"), device=dev)
        bl.append((qa, ql, ka, kl, out, lse))
    return bl


@pytest.mark.parametrize("lens,Hq,Hkv,hd,dt", SHAPES,
                         ids=[f"h{s[1]}kv{s[2]}_d{s[3]}_{s[4]}" for s in SHAPES])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_blocks_equal_single_calls(nsp, lens, Hq, Hkv, hd, dt, causal):
    w = make_custom(lens, Hq, Hkv, hd, dtype=dt, seed=101, with_dout=False)
    d = to_dev(w)
    T = w.T
    ranges = [r for r in RANGES if r[0] + r[1] <= T and r[2] + r[3] <= T]
    bl = _blocks(w, d, "cuda", ranges)
    nsp.attn_fwd_blocks(d["q"], d["k"], d["v"], d["cu"], bl, causal=causal)
    torch.cuda.synchronize()
    q, k, v, _ = oracle_inputs(w)
    for qa, ql, ka, kl, out, lse in bl:
        if ql == 0:
            continue
        so, sl = nsp.attn_fwd(d["q"][qa:qa + ql], d["k"][ka:ka + kl], d["v"][ka:ka + kl], d["cu"],
                              causal=causal, out_dtype=torch.float32, q_start=qa, kv_start=ka)
        torch.cuda.synchronize()
        assert torch.equal(out, so) and torch.equal(lse, sl), (qa, ql, ka, kl)
        ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, hd ** -0.5, causal,
                                 q_range=(qa, qa + ql), kv_range=(ka, ka + kl))
        assert_fwd_close(f64(out), f64(lse), ro, rl, f32=(dt == "f32"),
                         label=f"block q{qa}+{ql} k{ka}+{kl}")


@pytest.mark.parametrize("lens,Hq,Hkv,hd,dt", SHAPES[:2],
                         ids=[f"h{s[1]}kv{s[2]}" for s in SHAPES[:2]])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_ring_steps_accumulate(nsp, lens, Hq, Hkv, hd, dt, causal):
    """A ring of 6 shards: step s meets query shard i with key shard
    (i - s) mod 6, one batched call per step (step 0 writes, the others
    merge in place); the result is unchunked attention."""
    w = make_custom(lens, Hq, Hkv, hd, dtype=dt, seed=102, with_dout=False)
    d = to_dev(w)
    n = 6
    T = w.T - w.T % n
    bounds = shard_bounds(T, n)
    acc = [(torch.empty((T // n, Hq, hd), dtype=torch.float32, device="cuda"),
            torch.empty((Hq, T // n), dtype=torch.float32, device="cuda")) for _ in range(n)]
    for s in range(n):
        bl = []
        for i in range(n):
            (qa, qb), (ka, kb) = bounds[i], bounds[(i - s) % n]
            bl.append((qa, qb - qa, ka, kb - ka, acc[i][0], acc[i][1]))
        nsp.attn_fwd_blocks(d["q"], d["k"], d["v"], d["cu"], bl, causal=causal, accumulate=s > 0)
    torch.cuda.synchronize()
    q, k, v, _ = oracle_inputs(w)
    cu = np.minimum(w.cu_seqlens, T)
    ro, rl = oracle.attn_fwd(q[:T], k[:T], v[:T], cu, hd ** -0.5, causal)
    out = torch.cat([a for a, _ in acc])
    lse = torch.cat([l for _, l in acc], dim=1)
    assert_fwd_close(f64(out), f64(lse), ro, rl, label=f"ring steps causal={causal}")


def test_config3_whole_ring_one_call(nsp):
    """Config 3: all non-empty causal (q-shard, kv-shard) blocks of 8 shards
    of 16384 tokens in one call, bit-identical to one call per block."""
    w = workload(3)
    d = to_dev(w)
    bounds = shard_bounds(w.T, 8)
    cu = w.cu_seqlens.astype(np.int64)
    ranges = []
    for i, (qa, qb) in enumerate(bounds):
        for (ka, kb) in bounds[:i + 1]:
            # non-empty: some document has a query in [qa, qb) and a key in [ka, kb)
            if any(max(cu[b], qa) < min(cu[b + 1], qb) and max(cu[b], ka) < min(cu[b + 1], kb)
                   for b in range(len(cu) - 1)):
                ranges.append((qa, qb - qa, ka, kb - ka))
    bl = _blocks(w, d, "cuda", ranges)
    nsp.attn_fwd_blocks(d["q"], d["k"], d["v"], d["cu"], bl)
    torch.cuda.synchronize()
    for qa, ql, ka, kl, out, lse in bl:
        so, sl = nsp.attn_fwd(d["q"][qa:qa + ql], d["k"][ka:ka + kl], d["v"][ka:ka + kl], d["cu"],
                              out_dtype=torch.float32, q_start=qa, kv_start=ka)
        torch.cuda.synchronize()
        assert torch.equal(out, so) and torch.equal(lse, sl), (qa, ka)
        del so, sl
    print(f"[C3] {len(ranges)} blocks in one call, bit-identical to single calls")
