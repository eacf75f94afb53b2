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
