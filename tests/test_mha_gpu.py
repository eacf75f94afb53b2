"""Multi-head attention (Hq = Hkv, BASP Sec. II-A "Multi-Head Attention")
and other odd numbers of query heads per KV head on the tensor-core
forward, against the fp64 oracle.

For an odd group size the tensor-core forward pairs two adjacent 128-row
query tiles of one head per work item (they read the same K/V tiles), on a
schedule of 256-row tiles whose key range is the union of the two halves'.
Checked at every element: ragged tails (a 256-row tile with an empty second
half), tiles whose halves lie in different documents, zero-length and
one-token documents, causal and not; ring partial blocks, accumulation in
place and the head-grouped layout; and that these calls launch tensor-core
kernels only.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_fwd_close, f64, oracle_inputs, to_dev
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, Hq, Hkv, causal
    ([129], 4, 4, True),
    ([300], 4, 4, False),
    ([1500, 3, 700], 4, 4, True),
    ([77, 128, 129, 255, 256, 257], 8, 8, True),
    ([77, 128, 129, 255, 256, 257], 8, 8, False),
    ([33] * 20, 4, 4, True),
    ([0, 5, 0, 260, 0, 1], 2, 2, True),
    ([400, 129], 6, 2, True),              # 3 query heads per KV head
    ([700, 200], 10, 2, False),            # 5 query heads per KV head
    ([1], 3, 3, True),
]


@pytest.mark.parametrize("lens,Hq,Hkv,causal", CASES,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_{'c' if c[3] else 'nc'}" for c in CASES])
def test_forward_whole_on_tensor_cores(nsp, lens, Hq, Hkv, causal):
    w = make_custom(lens, Hq, Hkv, 128, seed=sum(lens) + 7 * Hq, with_dout=False)
    d = to_dev(w)
    tc0, cc0 = nsp.nsp_path_launches(True), nsp.nsp_path_launches(False)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], causal=causal)
    torch.cuda.synchronize()
    assert nsp.nsp_path_launches(False) == cc0, "the CUDA-core forward ran"
    assert nsp.nsp_path_launches(True) == tc0 + 1
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 128 ** -0.5, causal)
    assert_fwd_close(f64(out), f64(lse), ro, rl, label=f"MHA {lens} h{Hq}kv{Hkv}")


@pytest.mark.parametrize("causal", [True, False])
def test_ring_partials_and_accumulate(nsp, causal):
    w = make_custom([600, 129, 300, 1], 4, 4, 128, seed=91, with_dout=False)
    d = to_dev(w)
    q, k, v, _ = oracle_inputs(w)
    T = w.T
    for qa, qb, ka, kb in ((0, T, 0, T), (300, 900, 0, 400), (129, 257, 600, T), (5, 6, 0, T)):
        po, pl = nsp.attn_fwd(d["q"][qa:qb], d["k"][ka:kb], d["v"][ka:kb], d["cu"],
                              causal=causal, out_dtype=torch.float32, q_start=qa, kv_start=ka)
        torch.cuda.synchronize()
        ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 128 ** -0.5, causal, q_range=(qa, qb),
                                 kv_range=(ka, kb))
        assert_fwd_close(f64(po), f64(pl), ro, rl, label=f"MHA partial q{qa}:{qb} k{ka}:{kb}")
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 128 ** -0.5, causal)
    rng = np.random.default_rng(92)
    cuts = np.unique(np.concatenate([[0, T], rng.integers(1, T, 5)]))
    blocks = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
    acc, lacc = nsp.ring_accumulate_init(T, 4, 128, "cuda")
    for ka, kb in [blocks[i] for i in rng.permutation(len(blocks))]:
        nsp.attn_fwd_accumulate(d["q"], d["k"][ka:kb], d["v"][ka:kb], d["cu"], acc, lacc,
                                causal=causal, kv_start=ka)
    torch.cuda.synchronize()
    assert_fwd_close(f64(acc), f64(lacc), ro, rl, label="MHA ring accumulate")


def test_headgroups_layout(nsp):
    """The grouped layout on the paired-tile path: bit-identical to the packed
    forward followed by the permutation."""
    w = make_custom([700, 129, 33], 8, 8, 128, seed=93, with_dout=False)
    d = to_dev(w)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"])
    for P in (2, 4, 8):
        og, lg = nsp.attn_fwd_headgroups(nsp.seq2head(d["q"], P), d["k"], d["v"], d["cu"])
        torch.cuda.synchronize()
        assert torch.equal(og, nsp.seq2head(out, P)) and torch.equal(lg, lse), P


def test_backward_mha_on_tensor_cores(nsp):
    """The backward already took MHA on the tensor cores; with the forward's
    out and lse from the paired-tile path it matches the oracle."""
    from gpu_common import TOL_GRAD, rel_l2
    w = make_custom([500, 129, 1], 4, 4, 128, seed=94)
    d = to_dev(w)
    cc0 = nsp.nsp_path_launches(False)
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"])
    dq, dk, dv = nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"])
    torch.cuda.synchronize()
    assert nsp.nsp_path_launches(False) == cc0
    q, k, v, do = oracle_inputs(w)
    ref = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, 128 ** -0.5, True)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert rel_l2(f64(g), r) <= TOL_GRAD, name
