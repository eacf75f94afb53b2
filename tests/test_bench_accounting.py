"""bench.py's work accounting on the host (no GPU): the allowed pairs it
credits to each ring block agree with the library's cost hook over the same
ranges, and the whole-stream useful FLOP is 4 d Hq (forward) and 10 d Hq
(backward) times the allowed pairs."""
import numpy as np
import pytest

from variable_length_sequence_gb300 import build as nsp_build
from variable_length_sequence_gb300 import nsp
from variable_length_sequence_gb300.workloads import (CONFIGS, draw_lengths, cu_from_lengths,
                                                       seed_of, shard_bounds)


@pytest.fixture(scope="module")
def lib():
    nsp_build.build()
    return nsp.load()


@pytest.mark.parametrize("cid", [2, 3])
def test_ring_block_pairs_match_cost_hook(lib, cid):
    import bench
    cfg = CONFIGS[cid]
    cu = cu_from_lengths(draw_lengths(cfg, np.random.default_rng(seed_of(cid))))
    bounds = shard_bounds(int(cu[-1]), 8)
    pairs = bench.allowed_pairs_blocks(cu, bounds)
    listed = {(qs, ks): n for qs, ks, n in pairs}
    for qs, (qa, qb) in enumerate(bounds):
        for ks, (ka, kb) in enumerate(bounds[:qs + 1]):
            c = nsp.nsp_attn_cost(cu, cfg.Hq, cfg.Hkv, cfg.d, True, nsp.NSP_BF16, qa, qb - qa, ka,
                                  kb - ka)
            assert listed.get((qs, ks), 0) == c["pairs"], (qs, ks)
    # every causal pair of the stream lies in exactly one block
    whole = nsp.nsp_attn_cost(cu, cfg.Hq, cfg.Hkv, cfg.d, True)
    assert sum(n for _, _, n in pairs) == whole["pairs"] == nsp.nsp_attn_pairs(cu, True)
    assert whole["fwd_flop"] == 4 * cfg.d * cfg.Hq * whole["pairs"]
    assert whole["bwd_flop"] == 10 * cfg.d * cfg.Hq * whole["pairs"]
