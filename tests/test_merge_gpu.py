"""LSE merge on the GPU against the oracle merge, and the chunking identity:
merging partials of a key chunking reproduces unchunked attention."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import TOL_LSE, TOL_OUT, assert_fwd_close, f64, max_abs

pytestmark = pytest.mark.gpu


def _partials(seed, lens, Hq, Hkv, d, cuts, q_range):
    r = np.random.default_rng(seed)
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q, k, v = (r.standard_normal((T, h, d)) for h in (Hq, Hkv, Hkv))
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        o, l = oracle.attn_fwd(q, k, v, cu, d ** -0.5, True, q_range=q_range, kv_range=(a, b))
        outs.append(o.astype(np.float32))
        lses.append(l.astype(np.float32))
    whole = oracle.attn_fwd(q, k, v, cu, d ** -0.5, True, q_range=q_range)
    return outs, lses, whole


@pytest.mark.parametrize("n_cuts", [1, 2, 5, 9])
@pytest.mark.parametrize("d", [64, 128])
def test_merge_matches_oracle(nsp, n_cuts, d):
    lens = [40, 1, 130, 7, 200, 33]
    T = sum(lens)
    cuts = [0] + sorted(np.random.default_rng(n_cuts).choice(np.arange(1, T), n_cuts - 1,
                                                             replace=False).tolist()) + [T]
    outs, lses, whole = _partials(n_cuts, lens, 8, 2, d, cuts, (0, T))
    ref_o, ref_l = oracle.lse_merge([o.astype(np.float64) for o in outs],
                                    [l.astype(np.float64) for l in lses])
    go, gl = nsp.lse_merge([torch.from_numpy(o).cuda() for o in outs],
                           [torch.from_numpy(l).cuda() for l in lses], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert max_abs(f64(go), ref_o) <= 1e-5
    assert max_abs(f64(gl), ref_l) <= 1e-5
    # and against unchunked attention, with a bf16 output
    gob, glb = nsp.lse_merge([torch.from_numpy(o).cuda() for o in outs],
                             [torch.from_numpy(l).cuda() for l in lses],
                             out_dtype=torch.bfloat16)
    assert_fwd_close(f64(gob), f64(glb), whole[0], whole[1], label=f"merge n={n_cuts}")


def test_merge_edge_rows(nsp):
    """n = 1 is the identity; -inf partials are neutral; all -inf gives 0/-inf."""
    r = np.random.default_rng(5)
    T, H, d = 70, 4, 128
    o1 = r.standard_normal((T, H, d)).astype(np.float32)
    l1 = r.standard_normal((H, T)).astype(np.float32)
    l1[:, 3] = -np.inf
    o1[3] = 0.0
    o2 = np.zeros_like(o1)
    l2 = np.full_like(l1, -np.inf)
    go, gl = nsp.lse_merge([torch.from_numpy(o1).cuda()], [torch.from_numpy(l1).cuda()])
    assert max_abs(f64(go), o1) <= 1e-6 and max_abs(f64(gl), l1) <= 1e-6
    go, gl = nsp.lse_merge([torch.from_numpy(o1).cuda(), torch.from_numpy(o2).cuda()],
                           [torch.from_numpy(l1).cuda(), torch.from_numpy(l2).cuda()])
    assert max_abs(f64(go), o1) <= 1e-6 and max_abs(f64(gl), l1) <= 1e-6
    go, gl = nsp.lse_merge([torch.from_numpy(o2).cuda()] * 3, [torch.from_numpy(l2).cuda()] * 3)
    assert torch.all(go == 0) and torch.all(torch.isneginf(gl))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_batch_equals_single_merges(nsp, out_dtype):
    """nsp_lse_merge_batch: 5 segments of 1-9 partials in one launch give the
    same bits as one nsp_lse_merge per segment, and the oracle merge."""
    r = np.random.default_rng(8)
    T, H, d = 333, 8, 128
    segments, refs = [], []
    for g, n in enumerate((1, 3, 9, 2, 4)):
        outs = [torch.from_numpy(r.standard_normal((T, H, d)).astype(np.float32)).cuda()
                for _ in range(n)]
        lses = []
        for i in range(n):
            l = r.standard_normal((H, T)).astype(np.float32) * 3
            l[:, r.integers(0, T, 20)] = -np.inf                 # rows without keys
            if g == 3:
                l[:, :7] = -np.inf                               # rows that saw nothing at all
            lses.append(torch.from_numpy(l).cuda())
        segments.append((outs, lses))
        refs.append(nsp.lse_merge(outs, lses, out_dtype=out_dtype))
    outs_m = [torch.empty((T, H, d), dtype=out_dtype, device="cuda") for _ in segments]
    lses_m = [torch.empty((H, T), dtype=torch.float32, device="cuda") for _ in segments]
    nsp.nsp_lse_merge_batch(segments, outs_m, lses_m)
    torch.cuda.synchronize()
    for (ro, rl), go, gl, (outs, lses) in zip(refs, outs_m, lses_m, segments):
        assert torch.equal(go, ro) and torch.equal(gl, rl)
        oo, ol = oracle.lse_merge([f64(o) for o in outs], [f64(l) for l in lses])
        tol = 1e-5 if out_dtype == torch.float32 else 2e-2
        assert max_abs(f64(go), oo) <= tol and max_abs(f64(gl), ol) <= 1e-5
