"""Varlen attention forward on the GPU against the fp64 oracle: every
element on small and edge-case inputs, whole configs 1 and 5, sampled rows
(first/last row of every document plus random rows, all heads) at the full
sizes of configs 2-4."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (assert_fwd_close, f64, oracle_inputs, sample_rows, timed, to_dev,
                        workload)
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu


def run_fwd(nsp, w, causal=True):
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=w.cfg.d ** -0.5,
                            causal=causal)
    torch.cuda.synchronize()
    return out, lse


def test_config1_fp32_whole(nsp):
    w = workload(1)
    out, lse = run_fwd(nsp, w)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 64 ** -0.5, True)
    assert out.dtype == torch.float32
    assert_fwd_close(f64(out), f64(lse), ro, rl, f32=True, label="C1 fp32")


EDGE = [
    # lengths, Hq, Hkv, d, causal, dtype
    ([1], 4, 4, 128, True, "bf16"),
    ([1, 1, 1], 2, 1, 64, True, "bf16"),
    ([0, 5, 0, 0, 3, 0], 8, 2, 128, True, "bf16"),        # zero-length documents
    ([127], 8, 1, 128, True, "bf16"),
    ([128], 8, 8, 128, True, "bf16"),
    ([129], 8, 2, 128, False, "bf16"),
    ([300, 1, 2, 250], 32, 4, 128, True, "bf16"),
    ([1000], 16, 2, 128, True, "bf16"),
    ([77, 128, 129, 255, 256, 257], 8, 2, 64, True, "bf16"),
    ([77, 128, 129, 255, 256, 257], 8, 2, 128, False, "bf16"),
    ([33] * 20, 32, 4, 128, True, "bf16"),                # many short docs in one tile
    ([500, 13], 4, 2, 64, True, "f32"),
    ([200, 300], 4, 1, 128, False, "f32"),
]


@pytest.mark.parametrize("lens,Hq,Hkv,d,causal,dt", EDGE,
                         ids=[f"{len(e[0])}docs_T{sum(e[0])}_h{e[1]}kv{e[2]}_d{e[3]}_"
                              f"{'c' if e[4] else 'nc'}_{e[5]}" for e in EDGE])
def test_edge_cases_whole(nsp, lens, Hq, Hkv, d, causal, dt):
    w = make_custom(lens, Hq, Hkv, d, dtype=dt, seed=sum(lens) + Hq, with_dout=False)
    out, lse = run_fwd(nsp, w, causal)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, d ** -0.5, causal)
    assert_fwd_close(f64(out), f64(lse), ro, rl, f32=(dt == "f32"), label=f"edge {lens}")


def test_config5_whole(nsp):
    w = workload(5)
    out, lse = run_fwd(nsp, w)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = timed("oracle fwd C5", oracle.attn_fwd, q, k, v, w.cu_seqlens, 128 ** -0.5, True)
    assert_fwd_close(f64(out), f64(lse), ro, rl, label="C5 whole")


def _sampled(nsp, cid, n_random, shuffle=False):
    w = workload(cid, shuffle)
    out, lse = run_fwd(nsp, w)
    rows = sample_rows(w.cu_seqlens, n_random, seed=cid)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = timed(f"oracle fwd C{cid} {len(rows)} rows", oracle.attn_fwd_rows, q, k, v,
                   w.cu_seqlens, 128 ** -0.5, True, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_fwd_close(f64(out[idx]), f64(lse[:, idx]), ro, rl, label=f"C{cid} sampled")


def test_config2_sampled(nsp):
    _sampled(nsp, 2, 512)


def test_config3_sampled(nsp):
    _sampled(nsp, 3, 256)


@pytest.mark.slow
def test_config4_sampled(nsp):
    _sampled(nsp, 4, 128)
