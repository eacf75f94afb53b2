"""Ring-block backward on the GPU (nsp_attn_bwd_accumulate): one (query
range, key range) block's share of dq/dk/dv, added into float32
accumulators (HSAP Sec. 2.2.1 ring InterSP, the backward that meets every
circulating key/value block once).

Each block is checked against the fp64 oracle's block backward, and the sum
of the blocks of a chunking against the oracle's whole-stream gradients and
the GPU's own nsp_attn_bwd.  Relative L2 per tensor <= 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TOL_GRAD, f64, oracle_inputs, rel_l2, sample_rows, timed, to_dev, workload
from variable_length_sequence_gb300.workloads import make_custom, shard_bounds

pytestmark = pytest.mark.gpu


def _check(name, got, ref, tol=TOL_GRAD):
    e = rel_l2(got, ref)
    print(f"[{name}] rel L2 {e:.3e} (tol {tol})")
    assert e <= tol, f"{name}: rel L2 {e}"


def _fwd(nsp, w, d, causal=True):
    return nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=w.cfg.d ** -0.5, causal=causal)


def _accumulators(w, qlen, klen):
    dq = torch.zeros((qlen, w.cfg.Hq, w.cfg.d), dtype=torch.float32, device="cuda")
    dk = torch.zeros((klen, w.cfg.Hkv, w.cfg.d), dtype=torch.float32, device="cuda")
    return dq, dk, torch.zeros_like(dk)


def _block(nsp, w, d, out, lse, qr, kr, acc, causal=True):
    (qa, qb), (ka, kb) = qr, kr
    dq, dk, dv = acc
    nsp.attn_bwd_accumulate(d["q"][qa:qb], d["k"][ka:kb], d["v"][ka:kb], out[qa:qb],
                            d["dout"][qa:qb], lse[:, qa:qb].contiguous(), d["cu"], dq, dk, dv,
                            scale=w.cfg.d ** -0.5, causal=causal, q_start=qa, kv_start=ka)


def _chunks(T, n_cuts, r):
    cuts = np.unique(np.concatenate([[0, T], r.integers(1, T, n_cuts)]))
    return [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]


SMALL = [
    # lengths, Hq, Hkv, d, causal, dtype
    ([100, 1, 300, 60, 250], 8, 2, 128, True, "bf16"),      # tensor cores, GQA 4
    ([257, 300], 8, 1, 128, False, "bf16"),                  # tensor cores, non-causal
    ([33] * 12, 32, 4, 128, True, "bf16"),                   # many short documents
    ([17, 64, 100, 200], 4, 4, 64, True, "f32"),             # CUDA cores, fp32, d = 64
]


@pytest.mark.parametrize("lens,Hq,Hkv,d,causal,dt", SMALL,
                         ids=[f"T{sum(e[0])}_h{e[1]}kv{e[2]}_d{e[3]}_{'c' if e[4] else 'nc'}_{e[5]}"
                              for e in SMALL])
def test_blocks_vs_oracle(nsp, lens, Hq, Hkv, d, causal, dt):
    w = make_custom(lens, Hq, Hkv, d, dtype=dt, seed=40 + sum(lens))
    dev = to_dev(w)
    out, lse = _fwd(nsp, w, dev, causal)
    q, k, v, do = oracle_inputs(w)
    T = w.T
    r = np.random.default_rng(41)
    # single blocks against the oracle's block backward
    for qr, kr in (((0, T), (0, T)), ((130, T - 20), (64, min(400, T))),
                   ((T // 2, T), (0, T // 2)), ((5, 6), (0, T))):
        acc = _accumulators(w, qr[1] - qr[0], kr[1] - kr[0])
        _block(nsp, w, dev, out, lse, qr, kr, acc, causal)
        torch.cuda.synchronize()
        ref = oracle.attn_bwd_block(q, k, v, do, w.cu_seqlens, d ** -0.5, causal, qr, kr)
        for n, g, rf in zip(("dq", "dk", "dv"), acc, ref):
            if np.abs(rf).max() == 0:
                assert float(g.abs().max()) == 0.0, f"{n} of an empty block is not zero"
                continue
            _check(f"block q{qr} k{kr} {n}", f64(g), rf)
    # a chunking, blocks in random order, summed in place
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, d ** -0.5, causal)
    qc, kc = _chunks(T, 3, r), _chunks(T, 4, r)
    blocks = [(a, b) for a in qc for b in kc]
    acc = _accumulators(w, T, T)
    for i in r.permutation(len(blocks)):
        qr, kr = blocks[i]
        part = _accumulators(w, qr[1] - qr[0], kr[1] - kr[0])
        _block(nsp, w, dev, out, lse, qr, kr, part, causal)
        acc[0][qr[0]:qr[1]] += part[0]
        acc[1][kr[0]:kr[1]] += part[1]
        acc[2][kr[0]:kr[1]] += part[2]
    torch.cuda.synchronize()
    for n, g, rf in zip(("dq", "dk", "dv"), acc, (rq, rk, rv)):
        _check(f"sum of {len(blocks)} blocks {n}", f64(g), rf)


def test_empty_block_leaves_accumulators(nsp):
    """Causal: queries of the first document against keys of the second."""
    w = make_custom([200, 311], 8, 2, 128, seed=43)
    dev = to_dev(w)
    out, lse = _fwd(nsp, w, dev)
    g = torch.Generator(device="cuda").manual_seed(5)
    acc = tuple(torch.randn(s, generator=g, device="cuda") for s in
                ((150, 8, 128), (311, 2, 128), (311, 2, 128)))
    before = tuple(a.clone() for a in acc)
    _block(nsp, w, dev, out, lse, (0, 150), (200, 511), acc)
    torch.cuda.synchronize()
    for a, b in zip(acc, before):
        assert torch.equal(a, b)


def test_config2_ring_backward(nsp):
    """Config 2 split into 8 shards of 4096 tokens: every causal (q-shard,
    kv-shard) block accumulated in place; the sums equal nsp_attn_bwd of the
    whole stream and the oracle on sampled rows and keys."""
    w = workload(2)
    dev = to_dev(w)
    out, lse = _fwd(nsp, w, dev)
    whole = nsp.attn_bwd(dev["q"], dev["k"], dev["v"], out, dev["dout"], lse, dev["cu"],
                         scale=128 ** -0.5)
    bounds = shard_bounds(w.T, 8)
    n = w.T // 8
    dq = torch.zeros((w.T, 32, 128), dtype=torch.float32, device="cuda")
    dk = torch.zeros((w.T, 4, 128), dtype=torch.float32, device="cuda")
    dv = torch.zeros_like(dk)
    ws = torch.empty(nsp.nsp_attn_bwd_accumulate_workspace_size(n, n, 32, 4, 128),
                     dtype=torch.uint8, device="cuda")
    lse_sh = [lse[:, a:b].contiguous() for a, b in bounds]
    for qs, (qa, qb) in enumerate(bounds):
        for (ka, kb) in bounds[:qs + 1]:
            nsp.nsp_attn_bwd_accumulate(dev["q"][qa:qb], dev["k"][ka:kb], dev["v"][ka:kb],
                                        out[qa:qb], dev["dout"][qa:qb], lse_sh[qs], dev["cu"],
                                        len(w.lengths), qa, n, ka, n, 32, 4, 128, 128 ** -0.5,
                                        True, dq[qa:qb], dk[ka:kb], dv[ka:kb], ws)
    torch.cuda.synchronize()
    for name, g, ref in (("dq", dq, whole[0]), ("dk", dk, whole[1]), ("dv", dv, whole[2])):
        _check(f"C2 ring vs whole-stream {name}", f64(g), f64(ref))
    q, k, v, do = oracle_inputs(w)
    cu = w.cu_seqlens
    rows = sample_rows(cu, 128, seed=44, extra=[b[0] for b in bounds] + [b[1] - 1 for b in bounds])
    rq = timed("oracle dq C2 rows", oracle.attn_bwd_dq_rows, q, k, v, do, cu, 128 ** -0.5, True,
               rows)
    _check("C2 ring dq rows", f64(dq[torch.from_numpy(rows).cuda()]), rq)
    keys = np.unique(np.concatenate([[b[1] - 1 for b in bounds],
                                     np.random.default_rng(45).integers(0, w.T, 24)]))
    rk, rv = timed("oracle dkv C2 g1", oracle.attn_bwd_dkv_rows, q, k, v, do, cu, 128 ** -0.5,
                   True, keys, 1)
    kidx = torch.from_numpy(keys).cuda()
    _check("C2 ring dk keys g1", f64(dk[kidx, 1]), rk)
    _check("C2 ring dv keys g1", f64(dv[kidx, 1]), rv)
