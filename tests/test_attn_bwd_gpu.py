"""Varlen attention backward on the GPU against the fp64 oracle's analytic
gradients: every element on small inputs and on config 5, sampled dQ rows
and dK/dV key rows (all heads) on configs 2 and 4.  Relative L2 per tensor
<= 1e-2; on config 5, also every (row, head) within the internal per-row
bar.  The sampled key rows include keys deep inside the longest documents,
whose key-stationary work items accumulate over many query tiles and heads:
the first keys of config 2's longest document (seen by all of its queries)
and, on config 4, keys about 2560 queries before the end of the
262144-token document."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (TOL_GRAD, assert_rows_close, f64, oracle_inputs, rel_l2, sample_rows,
                        timed, to_dev, workload)
from variable_length_sequence_gb300.workloads import make_custom

pytestmark = pytest.mark.gpu


def run_fwd_bwd(nsp, w, causal=True):
    d = to_dev(w)
    scale = w.cfg.d ** -0.5
    out, lse = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=scale, causal=causal)
    dq, dk, dv = nsp.attn_bwd(d["q"], d["k"], d["v"], out, d["dout"], lse, d["cu"], scale=scale,
                              causal=causal)
    torch.cuda.synchronize()
    return dq, dk, dv


def _check(name, got, ref):
    e = rel_l2(got, ref)
    print(f"[{name}] rel L2 {e:.3e} (tol {TOL_GRAD})")
    assert e <= TOL_GRAD, f"{name}: rel L2 {e}"


SMALL = [
    ([1, 5, 0, 3], 4, 2, 64, True, "bf16"),
    ([130, 1, 200], 8, 2, 128, True, "bf16"),
    ([257, 300], 8, 1, 128, False, "bf16"),
    ([33] * 12, 32, 4, 128, True, "bf16"),
    ([128, 129], 4, 4, 128, True, "f32"),
]


@pytest.mark.parametrize("lens,Hq,Hkv,d,causal,dt", SMALL,
                         ids=[f"T{sum(e[0])}_h{e[1]}kv{e[2]}_d{e[3]}_{'c' if e[4] else 'nc'}_{e[5]}"
                              for e in SMALL])
def test_bwd_small_whole(nsp, lens, Hq, Hkv, d, causal, dt):
    w = make_custom(lens, Hq, Hkv, d, dtype=dt, seed=7 + sum(lens))
    dq, dk, dv = run_fwd_bwd(nsp, w, causal)
    q, k, v, do = oracle_inputs(w)
    rq, rk, rv = oracle.attn_bwd(q, k, v, do, w.cu_seqlens, d ** -0.5, causal)
    for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check(f"{lens} {n}", f64(g), r)


def test_config5_whole(nsp):
    w = workload(5)
    dq, dk, dv = run_fwd_bwd(nsp, w)
    q, k, v, do = oracle_inputs(w)
    rq, rk, rv = timed("oracle bwd C5", oracle.attn_bwd, q, k, v, do, w.cu_seqlens,
                       128 ** -0.5, True)
    for n, g, r in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        _check(f"C5 {n}", f64(g), r)
        assert_rows_close(f64(g), r, label=f"C5 {n} per row")


def deep_keys(cu, depth: int, seed: int, n_random: int = 8) -> list:
    """Keys of the longest document whose visible queries reach `depth` rows
    deep: the 4 keys `depth` rows before the document's end and seeded keys
    between there and the end (a depth of the whole document gives its first
    keys, seen by every query of it)."""
    lens = np.diff(cu)
    b = int(np.argmax(lens))
    start = int(cu[b + 1]) - min(depth, int(lens[b]))
    keys = set(range(start, start + 4))
    rng = np.random.default_rng(seed)
    keys.update(int(x) for x in rng.integers(start, int(cu[b + 1]), n_random))
    return sorted(keys)


def _sampled(nsp, cid, n_rows, n_keys, depth):
    w = workload(cid)
    dq, dk, dv = run_fwd_bwd(nsp, w)
    q, k, v, do = oracle_inputs(w)
    cu = w.cu_seqlens
    rows = sample_rows(cu, n_rows, seed=10 + cid)
    rq = timed(f"oracle dq C{cid} {len(rows)} rows", oracle.attn_bwd_dq_rows, q, k, v, do, cu,
               128 ** -0.5, True, rows)
    _check(f"C{cid} dq rows", f64(dq[torch.from_numpy(rows).cuda()]), rq)
    # key rows: the last rows of every document (cheap: few queries see them)
    # plus random keys inside documents shorter than 4096
    lens = np.diff(cu)
    keys = set()
    for b in range(len(lens)):
        if lens[b] > 0:
            keys.update(range(int(cu[b + 1]) - min(8, int(lens[b])), int(cu[b + 1])))
    short = [b for b in range(len(lens)) if 0 < lens[b] < 4096]
    r = np.random.default_rng(20 + cid)
    for b in r.choice(short, min(len(short), n_keys), replace=False):
        keys.add(int(r.integers(cu[b], cu[b + 1])))
    deep = deep_keys(cu, depth, seed=30 + cid)
    print(f"[C{cid}] deep keys {deep[:4]}.. (up to {depth} queries of the longest document "
          f"see them)")
    keys.update(deep)
    keys = np.array(sorted(keys))
    kidx = torch.from_numpy(keys).cuda()
    for g in range(w.cfg.Hkv):
        rk, rv = timed(f"oracle dkv C{cid} g{g}", oracle.attn_bwd_dkv_rows, q, k, v, do, cu,
                       128 ** -0.5, True, keys, g)
        _check(f"C{cid} dk g{g}", f64(dk[kidx, g]), rk)
        _check(f"C{cid} dv g{g}", f64(dv[kidx, g]), rv)


def test_config2_sampled(nsp):
    # depth = whole document: its first keys, seen by all of its queries
    _sampled(nsp, 2, 512, 24, depth=1 << 30)


@pytest.mark.slow
def test_config4_sampled(nsp):
    _sampled(nsp, 4, 128, 16, depth=2560)
