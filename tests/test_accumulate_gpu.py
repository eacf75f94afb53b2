"""Ring accumulation in place (nsp_attn_fwd_accumulate): each key block's
partial is merged into a running float32 (acc, lse_acc) by the attention
epilogue itself (HSAP Sec. 2.2.1 online accumulation, with the receive-side
rescale fused as HSAP's Limitations section proposes).

After every block of a key chunking, in any order, acc must be the
unchunked attention output and lse_acc its log-sum-exp; rows that see no key
of any block keep acc = 0 and lse_acc = -inf.  Checked against the fp64
oracle (unchunked), and against the GPU's own partials + nsp_lse_merge."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import (TOL_LSE, TOL_OUT, assert_fwd_close, f64, max_abs, oracle_inputs,
                        sample_rows, timed, to_dev, workload)
from variable_length_sequence_gb300.workloads import make_custom, shard_bounds

pytestmark = pytest.mark.gpu


def ring(nsp, d, w, qa, qb, blocks, causal=True):
    """Accumulate the key blocks [(ka, kb), ...] of the query range [qa, qb)."""
    acc, lse = nsp.ring_accumulate_init(qb - qa, w.cfg.Hq, w.cfg.d, "cuda")
    for ka, kb in blocks:
        nsp.attn_fwd_accumulate(d["q"][qa:qb], d["k"][ka:kb], d["v"][ka:kb], d["cu"], acc, lse,
                                scale=w.cfg.d ** -0.5, causal=causal, q_start=qa, kv_start=ka)
    torch.cuda.synchronize()
    return acc, lse


def random_blocks(T, n_cuts, rng):
    cuts = np.unique(np.concatenate([[0, T], rng.integers(1, T, n_cuts)]))
    blocks = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
    order = rng.permutation(len(blocks))
    return [blocks[i] for i in order]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qr", [(0, 711), (128, 500), (5, 6)])
def test_random_chunkings_tc_vs_oracle(nsp, causal, qr):
    """bf16, d = 128, 4 query heads per KV head: the tcgen05 kernel."""
    w = make_custom([100, 1, 300, 60, 250], 8, 2, 128, seed=3, with_dout=False)
    d = to_dev(w)
    q, k, v, _ = oracle_inputs(w)
    qa, qb = qr
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 128 ** -0.5, causal, q_range=(qa, qb))
    rng = np.random.default_rng(11 + qa)
    for n_cuts in (1, 3, 8):
        acc, lse = ring(nsp, d, w, qa, qb, random_blocks(w.T, n_cuts, rng), causal)
        assert_fwd_close(f64(acc), f64(lse), ro, rl,
                         label=f"accumulate q{qa}:{qb} causal={causal} cuts={n_cuts}")


def test_random_chunkings_simt_f32_vs_oracle(nsp):
    """float32 I/O, d = 64, MHA (config 1's shape): the CUDA-core kernel."""
    w = workload(1)
    d = to_dev(w)
    q, k, v, _ = oracle_inputs(w)
    ro, rl = oracle.attn_fwd(q, k, v, w.cu_seqlens, 64 ** -0.5, True)
    rng = np.random.default_rng(5)
    for n_cuts in (1, 4, 9):
        acc, lse = ring(nsp, d, w, 0, w.T, random_blocks(w.T, n_cuts, rng))
        assert_fwd_close(f64(acc), f64(lse), ro, rl, f32=True, label=f"C1 accumulate cuts={n_cuts}")


@pytest.mark.parametrize("hkv,d_head,dtype", [(2, 128, "bf16"), (4, 64, "f32")])
def test_rows_without_keys_unchanged(nsp, hkv, d_head, dtype):
    """Causal blocks whose keys all lie after the queries leave acc/lse as they were."""
    w = make_custom([200, 311], 4, hkv, d_head, dtype=dtype, seed=9, with_dout=False)
    d = to_dev(w)
    acc, lse = ring(nsp, d, w, 0, 150, [(300, 511), (160, 300)])
    assert torch.all(acc == 0) and torch.all(torch.isneginf(lse))
    # a partially visible block: rows before the block's first key unchanged
    acc, lse = ring(nsp, d, w, 0, 200, [(120, 200)])
    assert torch.all(acc[:120] == 0) and torch.all(torch.isneginf(lse[:, :120]))
    assert torch.all(torch.isfinite(lse[:, 120:]))


def test_config3_ring_accumulate(nsp):
    """Config 3: every causal (q-shard, kv-shard) block of 8 shards of 16384
    tokens accumulated in place equals the unchunked forward at every element,
    the partials + nsp_lse_merge route, and the oracle on sampled rows."""
    w = workload(3)
    d = to_dev(w)
    cu = w.cu_seqlens.astype(np.int64)
    bounds = shard_bounds(w.T, w.cfg.shards)
    whole_o, whole_l = nsp.attn_fwd(d["q"], d["k"], d["v"], d["cu"], scale=128 ** -0.5,
                                    out_dtype=torch.float32)
    acc_all = torch.empty_like(whole_o)
    lse_all = torch.empty_like(whole_l)
    for qs, (qa, qb) in enumerate(bounds):
        # the diagonal block last: a ring receives its own block first or last
        blocks = list(bounds[:qs]) + [bounds[qs]]
        acc, lse = ring(nsp, d, w, qa, qb, blocks)
        acc_all[qa:qb] = acc
        lse_all[:, qa:qb] = lse
        if qs in (2, 7):
            outs, lses = [], []
            for ka, kb in blocks:
                o, l = nsp.attn_fwd(d["q"][qa:qb], d["k"][ka:kb], d["v"][ka:kb], d["cu"],
                                    scale=128 ** -0.5, out_dtype=torch.float32, q_start=qa,
                                    kv_start=ka)
                outs.append(o)
                lses.append(l)
            mo, ml = nsp.lse_merge(outs, lses, out_dtype=torch.float32)
            torch.cuda.synchronize()
            eo, el = max_abs(f64(acc), f64(mo)), max_abs(f64(lse), f64(ml))
            print(f"[C3 shard {qs}: accumulate vs partials+merge] out {eo:.3e} lse {el:.3e}")
            # both round P to bf16, against different reference maxima (a
            # partial's own maximum; the running maximum in place): they
            # agree far inside the 2e-2 bar, not to float32 rounding
            assert eo <= 1e-3 and el <= 1e-5
    eo = max_abs(f64(acc_all), f64(whole_o))
    el = max_abs(f64(lse_all), f64(whole_l))
    print(f"[C3 accumulate vs unchunked] out {eo:.3e} lse {el:.3e}")
    assert eo <= TOL_OUT and el <= TOL_LSE
    rows = sample_rows(cu, 256, seed=34, extra=[b[0] for b in bounds] + [b[1] - 1 for b in bounds])
    q, k, v, _ = oracle_inputs(w)
    ro, rl = timed("oracle C3 rows", oracle.attn_fwd_rows, q, k, v, cu, 128 ** -0.5, True, rows)
    idx = torch.from_numpy(rows).cuda()
    assert_fwd_close(f64(acc_all[idx]), f64(lse_all[:, idx]), ro, rl, label="C3 ring accumulate")
