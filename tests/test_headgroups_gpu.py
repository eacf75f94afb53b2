"""Forward in the Ulysses receive layout (nsp_attn_fwd_headgroups): q and
out as [P][T][Hq/P][d] (HSAP Sec. 2.2.2 IntraSP all-to-all; BASP Sec. II-C),
k and v packed.  It must equal nsp_attn_fwd on the packed layout followed
by the seq->head permutation, bit for bit, and the oracle within the stated
tolerances."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_fwd_close, f64, oracle_inputs, sample_rows, timed, to_dev, workload
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, Hq, Hkv, d, dtype, P, causal
    ([100, 1, 300, 60, 250], 8, 2, 128, "bf16", 2, True),    # tensor cores
    ([100, 1, 300, 60, 250], 8, 2, 128, "bf16", 4, True),    # tensor cores, 2 heads per group
    ([257, 300], 8, 1, 128, "bf16", 4, False),               # non-causal
    ([33] * 12, 32, 4, 128, "bf16", 8, True),                # config 3's grouping, short docs
    ([130, 1, 200], 8, 2, 128, "bf16", 8, True),             # 1 head per group: CUDA cores
    ([17, 64, 100, 200], 4, 4, 64, "f32", 2, True),          # fp32, d = 64: CUDA cores
]


@pytest.mark.parametrize("lens,Hq,Hkv,d,dt,P,causal", CASES,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_d{c[3]}_{c[4]}_P{c[5]}"
                              f"{'' if c[6] else '_nc'}" for c in CASES])
def test_headgroups_small(nsp, lens, Hq, Hkv, d, dt, P, causal):
    w = make_custom(lens, Hq, Hkv, d, dtype=dt, seed=50 + P, with_dout=False)
    dev = to_dev(w)
    out, lse = nsp.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], scale=d ** -0.5,
                            causal=causal)
    qg = nsp.seq2head(dev["q"], P)
    og, lg = nsp.attn_fwd_headgroups(qg, dev["k"], dev["v"], dev["cu"], scale=d ** -0.5,
                                     causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(og, nsp.seq2head(out, P)), "grouped output differs from permuted output"
    assert torch.equal(lg, lse)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, d ** -0.5, causal)
    # the grouped output against the oracle's output moved by the oracle's permutation
    assert_fwd_close(f64(og), f64(lg), oracle.seq2head(ro, P), rl, f32=(dt == "f32"),
                     label=f"headgroups P={P}")


def test_config3_headgroups(nsp):
    """Config 3's [131072, 32, 128] stream as 8 head groups of 4 heads."""
    w = workload(3)
    dev = to_dev(w)
    P = w.cfg.permute_groups
    qg = nsp.seq2head(dev["q"], P)
    og, lg = nsp.attn_fwd_headgroups(qg, dev["k"], dev["v"], dev["cu"], scale=128 ** -0.5)
    out, lse = nsp.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], scale=128 ** -0.5)
    torch.cuda.synchronize()
    assert torch.equal(og, nsp.seq2head(out, P))
    assert torch.equal(lg, lse)
    cu = w.cu_seqlens.astype(np.int64)
    rows = sample_rows(cu, 128, seed=51)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = timed("oracle C3 rows", oracle.attn_fwd_rows, q, k, v, cu, 128 ** -0.5, True, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_fwd_close(f64(nsp.head2seq(og)[idx]), f64(lg[:, idx]), ro, rl, label="C3 headgroups")


BWD_CASES = [
    # lengths, Hq, Hkv, d, dtype, P, causal
    ([100, 1, 300, 60, 250], 8, 2, 128, "bf16", 4, True),    # tensor cores, 2 heads per group
    ([130, 1, 200], 8, 2, 128, "bf16", 8, True),             # 1 head per group
    ([257, 300], 8, 1, 128, "bf16", 2, False),               # non-causal
    ([128, 129], 4, 4, 128, "f32", 2, True),                 # CUDA cores (fp32)
]


@pytest.mark.parametrize("lens,Hq,Hkv,d,dt,P,causal", BWD_CASES,
                         ids=[f"T{sum(c[0])}_h{c[1]}kv{c[2]}_d{c[3]}_{c[4]}_P{c[5]}"
                              f"{'' if c[6] else '_nc'}" for c in BWD_CASES])
def test_headgroups_backward(nsp, lens, Hq, Hkv, d, dt, P, causal):
    """The backward in the receive layout equals nsp_attn_bwd + permutation
    (bit for bit on the tensor cores; the CUDA-core dq sums with float
    atomics, so there within float32 rounding) and the oracle's gradients."""
    from gpu_common import TOL_GRAD, rel_l2
    w = make_custom(lens, Hq, Hkv, d, dtype=dt, seed=60 + P)
    dev = to_dev(w)
    sc = d ** -0.5
    out, lse = nsp.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu"], scale=sc, causal=causal)
    dq, dk, dv = nsp.attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                              scale=sc, causal=causal)
    qg, og, dog = (nsp.seq2head(x, P) for x in (dev["q"], out, dev["dout"]))
    dqg, dkg, dvg = nsp.attn_bwd_headgroups(qg, dev["k"], dev["v"], og, dog, lse, dev["cu"],
                                            scale=sc, causal=causal)
    torch.cuda.synchronize()
    if dt == "bf16":
        assert torch.equal(dqg, nsp.seq2head(dq, P))
        assert torch.equal(dkg, dk) and torch.equal(dvg, dv)
    else:
        for a, b in ((dqg, nsp.seq2head(dq, P)), (dkg, dk), (dvg, dv)):
            assert rel_l2(f64(a), f64(b)) <= 1e-6
    q, k, v, do = oracle_inputs(w)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, sc, causal)
    for name, g, r in (("dq", f64(dqg), oracle.seq2head(rq, P)), ("dk", f64(dkg), rk),
                       ("dv", f64(dvg), rv)):
        e = rel_l2(g, r)
        print(f"[headgroups bwd P={P} {name}] rel L2 {e:.3e} (tol {TOL_GRAD})")
        assert e <= TOL_GRAD
