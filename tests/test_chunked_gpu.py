"""Ring-style chunk partials on the GPU: a query shard against a key shard
(global token ids compared with cu_seqlens), rows with no allowed key give
lse = -inf and out = 0; merging a shard's partials reproduces unchunked
attention (config 3: 8 shards of 16384 tokens)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (assert_fwd_close, f64, max_abs, oracle_inputs, sample_rows, timed,
                        to_dev, workload)
from variable_length_sequence_gb300.workloads import make_custom, shard_bounds

pytestmark = pytest.mark.gpu


def partial(nsp, d, w, qa, qb, ka, kb, causal=True):
    q = d["q"][qa:qb]
    k, v = d["k"][ka:kb], d["v"][ka:kb]
    return nsp.attn_fwd(q, k, v, d["cu"], scale=w.cfg.d ** -0.5, causal=causal,
                        out_dtype=torch.float32, q_start=qa, kv_start=ka)


@pytest.mark.parametrize("causal", [True, False])
def test_partials_small_vs_oracle(nsp, causal):
    w = make_custom([100, 1, 300, 60, 250], 8, 2, 128, seed=3, with_dout=False)
    d = to_dev(w)
    q, k, v, _ = oracle_inputs(w)
    T = w.T
    for (qa, qb), (ka, kb) in [((0, 256), (0, 256)), ((256, 711), (0, 256)),
                               ((128, 500), (300, 640)), ((400, 711), (0, 129)),
                               ((0, 100), (100, 711)), ((5, 6), (0, 711))]:
        out, lse = partial(nsp, d, w, qa, qb, ka, kb, causal)
        torch.cuda.synchronize()
        ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 128 ** -0.5, causal, q_range=(qa, qb),
                                 kv_range=(ka, kb))
        assert_fwd_close(f64(out), f64(lse), ro, rl, label=f"partial q{qa}:{qb} k{ka}:{kb}")
        empty = np.isneginf(rl)
        assert np.all(f64(out)[empty.T] == 0.0)


def _nonempty(cu, qa, qb, ka, kb):
    """Some query of [qa, qb) may see some key of [ka, kb) (causal): the
    first query at or after ka whose document starts before kb."""
    lo = max(qa, ka)
    if lo >= qb:
        return False
    b_lo = int(np.searchsorted(cu, lo, side="right") - 1)
    return cu[b_lo] < kb


def test_config3_ring_merge(nsp):
    w = workload(3)
    d = to_dev(w)
    cu = w.cu_seqlens.astype(np.int64)
    bounds = shard_bounds(w.T, w.cfg.shards)
    whole_o, whole_l = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=128 ** -0.5)
    merged_o = torch.empty_like(whole_o)
    merged_l = torch.empty_like(whole_l)
    n_pairs = 0
    for qs, (qa, qb) in enumerate(bounds):
        outs, lses = [], []
        for ks, (ka, kb) in enumerate(bounds[:qs + 1]):
            if not _nonempty(cu, qa, qb, ka, kb):
                continue
            o, l = partial(nsp, d, w, qa, qb, ka, kb)
            outs.append(o)
            lses.append(l)
        n_pairs += len(outs)
        mo, ml = nsp.lse_merge(outs, lses, out_dtype=torch.bfloat16)
        merged_o[qa:qb] = mo
        merged_l[:, qa:qb] = ml
    torch.cuda.synchronize()
    print(f"[C3: {n_pairs} non-empty (q-shard, kv-shard) pairs]")
    # merged == unchunked (both GPU), at every element
    eo = max_abs(f64(merged_o), f64(whole_o))
    el = max_abs(f64(merged_l), f64(whole_l))
    print(f"[C3 merged vs unchunked] out {eo:.3e} lse {el:.3e}")
    assert eo <= 2e-2 and el <= 1e-3
    # merged vs the oracle on sampled rows
    rows = sample_rows(cu, 256, seed=33, extra=[b[0] for b in bounds] + [b[1] - 1 for b in bounds])
    q, k, v, _ = oracle_inputs(w)
    ro, rl = timed("oracle C3 rows", oracle.attn_fwd_rows, q, k, v, cu, 128 ** -0.5, True, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_fwd_close(f64(merged_o[idx]), f64(merged_l[:, idx]), ro, rl, label="C3 ring merged")


def test_config3_shuffled_shards_match_oracle(nsp):
    """The long document at a seeded random position, so shard edges cut it
    (cross-up / cross-right / corner blocks)."""
    w = workload(3, shuffle=True)
    d = to_dev(w)
    cu = w.cu_seqlens.astype(np.int64)
    bounds = shard_bounds(w.T, w.cfg.shards)
    q, k, v, _ = oracle_inputs(w)
    r = np.random.default_rng(77)
    for qs in (3, 6):
        qa, qb = bounds[qs]
        outs, lses = [], []
        for (ka, kb) in bounds[:qs + 1]:
            o, l = partial(nsp, d, w, qa, qb, ka, kb)     # empty pairs included: neutral
            outs.append(o)
            lses.append(l)
        mo, ml = nsp.lse_merge(outs, lses, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        rows = np.unique(np.concatenate([[qa, qb - 1], r.integers(qa, qb, 96)]))
        ro, rl = oracle.attn_fwd_rows(q, k, v, cu, 128 ** -0.5, True, rows)
        idx = torch.from_numpy(rows - qa).cuda()
        assert_fwd_close(f64(mo[idx]), f64(ml[:, idx]), ro, rl, label=f"C3 shuffled shard {qs}")
