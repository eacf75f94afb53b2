"""Pins that tie the fp64 oracle to what the pages and the mathematics fix.

Each ``pin_*`` takes the oracle's modules (``att`` = attention, ``mrg`` =
merge, ``prm`` = permute) and raises AssertionError on a mismatch, so the
same checks run against the real oracle (tests/test_oracle.py) and against
copies with a planted mistake (tests/test_oracle_mutants.py).

None of these retypes the oracle's own formula: they use worked examples
derived by hand (tests/golden/closed_forms.json), closed forms, invariants,
library routines on special cases (torch scaled_dot_product_attention and
autograd in float64, scipy logsumexp) and finite differences.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")


def _ev(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, {"log": math.log, "sqrt": math.sqrt,
                                                   "inf": math.inf}))
    if isinstance(x, list):
        return [_ev(e) for e in x]
    return float(x)


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(seed, lens, Hq, Hkv, d):
    r = _rng(seed)
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return (cu, r.standard_normal((T, Hq, d)), r.standard_normal((T, Hkv, d)),
            r.standard_normal((T, Hkv, d)), r.standard_normal((T, Hq, d)))


# --------------------------------------------------------------------------- forward


def pin_golden_attention(att, mrg, prm):
    for case in golden()["attention"]:
        q, k, v = (np.array(_ev(case[n])) for n in ("q", "k", "v"))
        d = q.shape[-1]
        out, lse = att.attn_fwd(q, k, v, np.array(case["cu_seqlens"]), 1.0 / math.sqrt(d),
                                case["causal"])
        np.testing.assert_allclose(out, np.array(_ev(case["out"])), rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse, np.array(_ev(case["lse"])), rtol=0, atol=1e-12,
                                   err_msg=case["name"])


def pin_length_one_docs(att, mrg, prm):
    """A one-token document: out = v, lse = scale <q, k> (single allowed key)."""
    cu, q, k, v, _ = _rand(1, [1, 5, 1, 1, 3], 4, 2, 8)
    scale = 0.37
    out, lse = att.attn_fwd(q, k, v, cu, scale, True)
    for t in (0, 6, 7):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(out[t, h], v[t, g], rtol=0, atol=1e-12)
            assert abs(lse[h, t] - scale * float(q[t, h] @ k[t, g])) < 1e-12


def pin_zero_queries(att, mrg, prm):
    """Q = 0: uniform weights, out_t = mean of v over J(t), lse = ln |J(t)|."""
    lens = [3, 7, 1, 5]
    cu, q, k, v, _ = _rand(2, lens, 4, 2, 8)
    q[:] = 0.0
    for causal in (True, False):
        out, lse = att.attn_fwd(q, k, v, cu, 0.5, causal)
        for b in range(len(lens)):
            s, e = int(cu[b]), int(cu[b + 1])
            for t in range(s, e):
                hi = t + 1 if causal else e
                for h in range(4):
                    g = h // 2
                    np.testing.assert_allclose(out[t, h], v[s:hi, g].mean(0), atol=1e-12)
                    assert abs(lse[h, t] - math.log(hi - s)) < 1e-12


def pin_constant_v(att, mrg, prm):
    """Constant V (every row c_g) returns c_g for every query."""
    cu, q, k, v, _ = _rand(3, [4, 9, 2], 4, 2, 8)
    c = _rng(30).standard_normal((2, 8))
    v[:] = c[None]
    out, _ = att.attn_fwd(q, k, v, cu, 0.35, True)
    for h in range(4):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(c[h // 2], out[:, h].shape),
                                   atol=1e-12)


def pin_rows_sum_to_one(att, mrg, prm):
    """Softmax rows sum to 1, masked entries are 0, and out = P V."""
    lens = [5, 1, 8, 3]
    cu, q, k, v, _ = _rand(4, lens, 2, 1, 4)
    for causal in (True, False):
        out, _ = att.attn_fwd(q, k, v, cu, 0.5, causal)
        for h in range(2):
            P = att.attn_probs(q, k, cu, 0.5, causal, h)
            np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-13)
            for t in range(q.shape[0]):
                b = int(np.searchsorted(cu, t, side="right") - 1)
                lo, hi = int(cu[b]), (t + 1 if causal else int(cu[b + 1]))
                assert np.all(P[t, :lo] == 0) and np.all(P[t, hi:] == 0)
            np.testing.assert_allclose(out[:, h], P @ v[:, 0], atol=1e-12)


def pin_packed_equals_alone(att, mrg, prm):
    """Packed stream == each document run as its own stream (no cross-contamination)."""
    lens = [7, 1, 12, 4, 9]
    cu, q, k, v, _ = _rand(5, lens, 4, 2, 8)
    for causal in (True, False):
        out, lse = att.attn_fwd(q, k, v, cu, 0.3, causal)
        for b in range(len(lens)):
            s, e = int(cu[b]), int(cu[b + 1])
            o1, l1 = att.attn_fwd(q[s:e], k[s:e], v[s:e], np.array([0, e - s]), 0.3, causal)
            np.testing.assert_allclose(out[s:e], o1, atol=1e-12)
            np.testing.assert_allclose(lse[:, s:e], l1, atol=1e-12)


def _sdpa_masked(q, k, v, cu, scale, causal, Hkv):
    """torch SDPA (float64, CPU) on the packed stream with an explicit boolean
    block-diagonal (and causal) mask; GQA through enable_gqa."""
    T = q.shape[0]
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    mask = doc[:, None] == doc[None, :]
    if causal:
        mask &= np.arange(T)[None, :] <= np.arange(T)[:, None]
    Q = torch.from_numpy(q).permute(1, 0, 2)[None]
    K = torch.from_numpy(k).permute(1, 0, 2)[None]
    V = torch.from_numpy(v).permute(1, 0, 2)[None]
    return Q, K, V, torch.from_numpy(mask)


def pin_sdpa_library(att, mrg, prm):
    """Special case reducing to a library routine: torch SDPA, float64."""
    F = torch.nn.functional
    lens = [6, 13, 1, 10]
    for Hq, Hkv in ((4, 4), (8, 2)):
        cu, q, k, v, _ = _rand(6 + Hkv, lens, Hq, Hkv, 16)
        for causal in (True, False):
            out, _ = att.attn_fwd(q, k, v, cu, 0.25, causal)
            Q, K, V, M = _sdpa_masked(q, k, v, cu, 0.25, causal, Hkv)
            ref = F.scaled_dot_product_attention(Q, K, V, attn_mask=M, scale=0.25,
                                                 enable_gqa=(Hq != Hkv))
            np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), atol=1e-12)
            # one document alone: the library's own causal flag
            s, e = int(cu[1]), int(cu[2])
            o1, _ = att.attn_fwd(q[s:e], k[s:e], v[s:e], np.array([0, e - s]), 0.25, causal)
            r1 = F.scaled_dot_product_attention(Q[:, :, s:e], K[:, :, s:e], V[:, :, s:e],
                                                is_causal=causal, scale=0.25,
                                                enable_gqa=(Hq != Hkv))
            np.testing.assert_allclose(o1, r1[0].permute(1, 0, 2).numpy(), atol=1e-12)


def pin_lse_library(att, mrg, prm):
    """lse of a bidirectional single document equals scipy's logsumexp of the
    scaled scores of all its keys (library routine, special case)."""
    from scipy.special import logsumexp
    cu, q, k, v, _ = _rand(9, [11], 4, 2, 8)
    _, lse = att.attn_fwd(q, k, v, cu, 0.4, False)
    for h in range(4):
        for t in range(11):
            assert abs(lse[h, t] - logsumexp(0.4 * (k[:, h // 2] @ q[t, h]))) < 1e-12


def pin_rows_variant(att, mrg, prm):
    """Sampled-row forward equals the whole-stream forward on those rows."""
    cu, q, k, v, _ = _rand(10, [5, 17, 1, 9], 4, 2, 8)
    out, lse = att.attn_fwd(q, k, v, cu, 0.3, True)
    rows = np.array([0, 3, 5, 21, 22, 31, 12])
    o2, l2 = att.attn_fwd_rows(q, k, v, cu, 0.3, True, rows)
    np.testing.assert_allclose(o2, out[rows], atol=1e-13)
    np.testing.assert_allclose(l2, lse[:, rows], atol=1e-13)


# --------------------------------------------------------------------------- chunks + merge


def pin_golden_merge(att, mrg, prm):
    for case in golden()["merge"]:
        outs = [np.array(_ev(o)) for o in case["outs"]]
        lses = [np.array(_ev(l)) for l in case["lses"]]
        out, lse = mrg.lse_merge(outs, lses)
        np.testing.assert_allclose(out, np.array(_ev(case["out"])), atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse, np.array(_ev(case["lse"])), atol=1e-12,
                                   err_msg=case["name"])


def pin_chunk_merge_equals_whole(att, mrg, prm):
    """Merging the partials of any key chunking equals unchunked attention."""
    lens = [9, 1, 20, 3, 14, 1, 6]
    cu, q, k, v, _ = _rand(11, lens, 4, 2, 8)
    T = int(cu[-1])
    r = _rng(12)
    for causal in (True, False):
        whole_o, whole_l = att.attn_fwd(q, k, v, cu, 0.3, causal)
        for trial in range(6):
            ncut = int(r.integers(1, 9))
            cuts = np.unique(np.concatenate([[0, T], r.integers(1, T, ncut)]))
            qa, qb = sorted(r.integers(0, T + 1, 2)) if trial % 2 else (0, T)
            if qa == qb:
                qb = min(T, qa + 1)
            outs, lses = [], []
            for a, b in zip(cuts[:-1], cuts[1:]):
                o, l = att.attn_fwd(q, k, v, cu, 0.3, causal, q_range=(qa, qb),
                                    kv_range=(int(a), int(b)))
                outs.append(o)
                lses.append(l)
            mo, ml = mrg.lse_merge(outs, lses)
            np.testing.assert_allclose(mo, whole_o[qa:qb], atol=1e-12)
            np.testing.assert_allclose(ml, whole_l[:, qa:qb], atol=1e-12)


def pin_merge_identity_and_neutral(att, mrg, prm):
    r = _rng(13)
    o = r.standard_normal((7, 3, 4))
    l = r.standard_normal((3, 7))
    l[1, 2] = -np.inf
    o[2, 1] = 0.0
    mo, ml = mrg.lse_merge([o], [l])
    np.testing.assert_allclose(mo, o, atol=1e-14)
    np.testing.assert_array_equal(np.isinf(ml), np.isinf(l))
    np.testing.assert_allclose(ml[np.isfinite(l)], l[np.isfinite(l)], atol=1e-14)
    mo2, ml2 = mrg.lse_merge([o, np.zeros_like(o)], [l, np.full_like(l, -np.inf)])
    np.testing.assert_allclose(mo2, mo, atol=1e-14)
    np.testing.assert_array_equal(ml2, ml)


def pin_empty_partial_rows(att, mrg, prm):
    """A key chunk entirely after a causal query's position gives lse=-inf, out=0."""
    cu, q, k, v, _ = _rand(14, [10, 10], 2, 1, 4)
    o, l = att.attn_fwd(q, k, v, cu, 0.5, True, q_range=(0, 10), kv_range=(5, 15))
    assert np.all(np.isneginf(l[:, :5])) and np.all(o[:5] == 0)
    assert np.all(np.isfinite(l[:, 5:]))
    o2, l2 = att.attn_fwd(q, k, v, cu, 0.5, True, q_range=(10, 20), kv_range=(0, 10))
    assert np.all(np.isneginf(l2)) and np.all(o2 == 0)


# --------------------------------------------------------------------------- backward


def _loss(att, q, k, v, dout, cu, scale, causal):
    out, _ = att.attn_fwd(q, k, v, cu, scale, causal)
    return float((out * dout).sum())


def pin_finite_differences(att, mrg, prm):
    """Central differences (h = 1e-6, float64) of L = sum(dOut * out)."""
    lens = [7, 13]
    cu, q, k, v, dout = _rand(15, lens, 2, 1, 8)
    h = 1e-6
    for causal in (True, False):
        dq, dk, dv = att.attn_bwd(q, k, v, dout, cu, 0.4, causal)
        for name, X, G in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(X)
            it = np.nditer(X, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                old = X[idx]
                X[idx] = old + h
                fp = _loss(att, q, k, v, dout, cu, 0.4, causal)
                X[idx] = old - h
                fm = _loss(att, q, k, v, dout, cu, 0.4, causal)
                X[idx] = old
                num[idx] = (fp - fm) / (2 * h)
            rel = np.linalg.norm(num - G) / np.linalg.norm(num)
            assert rel < 1e-6, (name, causal, rel)


def pin_autograd_library(att, mrg, prm):
    """Gradients equal torch autograd through SDPA (float64, packed mask, GQA)."""
    F = torch.nn.functional
    lens = [5, 12, 1, 8]
    cu, q, k, v, dout = _rand(16, lens, 4, 2, 8)
    for causal in (True, False):
        dq, dk, dv = att.attn_bwd(q, k, v, dout, cu, 0.3, causal)
        Q, K, V, M = _sdpa_masked(q, k, v, cu, 0.3, causal, 2)
        Q, K, V = (x.clone().requires_grad_(True) for x in (Q, K, V))
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=M, scale=0.3, enable_gqa=True)
        (o * torch.from_numpy(dout).permute(1, 0, 2)[None]).sum().backward()
        for mine, X in ((dq, Q), (dk, K), (dv, V)):
            np.testing.assert_allclose(mine, X.grad[0].permute(1, 0, 2).numpy(), atol=1e-11)


def pin_gradient_invariants(att, mrg, prm):
    """Constant V -> dQ = dK = 0; constant keys per doc -> dQ = 0
    (sum_j dS_tj = 0); sum of dK over each document = 0."""
    lens = [6, 1, 9]
    cu, q, k, v, dout = _rand(17, lens, 4, 2, 8)
    v2 = v.copy()
    v2[:] = v[0:1]
    dq, dk, _ = att.attn_bwd(q, k, v2, dout, cu, 0.3, True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    k2 = k.copy()
    for b in range(len(lens)):
        k2[cu[b]:cu[b + 1]] = k[cu[b]]
    dq2, _, _ = att.attn_bwd(q, k2, v, dout, cu, 0.3, True)
    assert np.abs(dq2).max() < 1e-12
    _, dk3, _ = att.attn_bwd(q, k, v, dout, cu, 0.3, True)
    for b in range(len(lens)):
        assert np.abs(dk3[cu[b]:cu[b + 1]].sum(0)).max() < 1e-12


def pin_bwd_rows_variants(att, mrg, prm):
    """Sampled dQ rows and dK/dV key rows equal the whole-stream backward."""
    lens = [9, 1, 15, 6]
    cu, q, k, v, dout = _rand(18, lens, 4, 2, 8)
    dq, dk, dv = att.attn_bwd(q, k, v, dout, cu, 0.3, True)
    rows = np.array([0, 4, 9, 10, 24, 30])
    np.testing.assert_allclose(att.attn_bwd_dq_rows(q, k, v, dout, cu, 0.3, True, rows),
                               dq[rows], atol=1e-13)
    keys = np.array([2, 9, 12, 25, 30])
    for g in range(2):
        dk2, dv2 = att.attn_bwd_dkv_rows(q, k, v, dout, cu, 0.3, True, keys, g)
        np.testing.assert_allclose(dk2, dk[keys, g], atol=1e-13)
        np.testing.assert_allclose(dv2, dv[keys, g], atol=1e-13)


def _chunks(T, n_cuts, r):
    cuts = np.unique(np.concatenate([[0, T], r.integers(1, T, n_cuts)]))
    return [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]


def pin_bwd_blocks_sum_to_whole(att, mrg, prm):
    """Ring backward: the block contributions of any (query chunking x key
    chunking), cuts through documents included, add up to the whole-stream
    gradients (which finite differences and autograd pin)."""
    lens = [6, 1, 11, 0, 9]
    cu, q, k, v, dout = _rand(19, lens, 4, 2, 8)
    T = int(cu[-1])
    r = _rng(20)
    for causal in (True, False):
        dq, dk, dv = att.attn_bwd(q, k, v, dout, cu, 0.35, causal)
        for nq, nk in ((0, 0), (2, 3), (5, 1)):
            sq, sk, sv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
            for qa, qb in _chunks(T, nq, r):
                for ka, kb in _chunks(T, nk, r):
                    bq, bk, bv = att.attn_bwd_block(q, k, v, dout, cu, 0.35, causal, (qa, qb),
                                                    (ka, kb))
                    sq[qa:qb] += bq
                    sk[ka:kb] += bk
                    sv[ka:kb] += bv
            for a, b in ((sq, dq), (sk, dk), (sv, dv)):
                np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def pin_bwd_block_autograd(att, mrg, prm):
    """One block's contributions equal torch autograd (float64) of
    L = sum(dOut * out) with every score outside the block, and every value
    row's use outside it, held constant (detached): only the block's terms
    then carry gradient, and the probabilities stay those of the full row."""
    lens = [7, 12, 5]
    Hq, Hkv, d = 4, 2, 8
    cu, q, k, v, dout = _rand(21, lens, Hq, Hkv, d)
    T = int(cu[-1])
    scale = 0.3
    doc = np.searchsorted(cu, np.arange(T), side="right") - 1
    for causal in (True, False):
        for (qa, qb), (ka, kb) in (((3, 20), (5, 15)), ((0, T), (10, 24)), ((9, 24), (0, 9))):
            Q, K, V = (torch.from_numpy(x).clone().requires_grad_(True) for x in (q, k, v))
            Ke = K.repeat_interleave(Hq // Hkv, dim=1)            # [T, Hq, d]
            Ve = V.repeat_interleave(Hq // Hkv, dim=1)
            t = torch.arange(T)
            same = torch.from_numpy(doc[:, None] == doc[None, :])
            allowed = same & (t[None, :] <= t[:, None]) if causal else same
            blk = (((t >= qa) & (t < qb))[:, None] & ((t >= ka) & (t < kb))[None, :])
            live = torch.einsum("thd,jhd->htj", Q, Ke) * scale
            dead = torch.einsum("thd,jhd->htj", Q.detach(), Ke.detach()) * scale
            S = torch.where(blk[None], live, dead).masked_fill(~allowed[None], float("-inf"))
            P = torch.softmax(S, dim=-1)                          # [Hq, T, T]
            Pb = torch.where(blk[None], P, torch.zeros_like(P))
            out = (torch.einsum("htj,jhd->thd", Pb, Ve)
                   + torch.einsum("htj,jhd->thd", P - Pb, Ve.detach()))
            (out * torch.from_numpy(dout)).sum().backward()
            bq, bk, bv = att.attn_bwd_block(q, k, v, dout, cu, scale, causal, (qa, qb), (ka, kb))
            np.testing.assert_allclose(bq, Q.grad[qa:qb].numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(bk, K.grad[ka:kb].numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(bv, V.grad[ka:kb].numpy(), rtol=0, atol=1e-12)
            # nothing outside the block moves
            assert float(Q.grad[:qa].abs().sum() + Q.grad[qb:].abs().sum()) == 0.0
            assert float(K.grad[:ka].abs().sum() + K.grad[kb:].abs().sum()) == 0.0


def pin_bwd_block_empty(att, mrg, prm):
    """Causal block whose keys all come after its queries: all zeros."""
    lens = [10, 10]
    cu, q, k, v, dout = _rand(22, lens, 2, 1, 4)
    bq, bk, bv = att.attn_bwd_block(q, k, v, dout, cu, 0.5, True, (0, 8), (8, 20))
    assert not bq.any() and not bk.any() and not bv.any()
    assert bq.shape == (8, 2, 4) and bk.shape == (12, 1, 4)


# --------------------------------------------------------------------------- permutation


def pin_permutation(att, mrg, prm):
    T, H, d = 6, 8, 3
    x = np.arange(T * H * d).reshape(T, H, d)
    for P in (1, 2, 4, 8):
        y = prm.seq2head(x, P)
        assert y.shape == (P, T, H // P, d)
        np.testing.assert_array_equal(prm.head2seq(y, P), x)
    y = prm.seq2head(x, 4)          # h = 2
    # hand-checked positions: head 5 of token 3 is group 2, local head 1
    np.testing.assert_array_equal(y[2, 3, 1], x[3, 5])
    np.testing.assert_array_equal(y[0, 5, 0], x[5, 0])
    np.testing.assert_array_equal(y[3, 0, 1], x[0, 7])
    np.testing.assert_array_equal(prm.seq2head(x, 1)[0], x)
    np.testing.assert_array_equal(prm.seq2head(x, 8)[:, :, 0], x.transpose(1, 0, 2))


def pin_permutation_groups(att, mrg, prm):
    """BASP subgroup all-to-all: B = 1 is the plain permutation with P = K;
    round trip; hand-checked positions; each group's output is made of its
    own sequence's rows only (changing another sequence leaves it alone)."""
    L, H, d = 5, 6, 2
    x = np.arange(3 * L * H * d).reshape(3 * L, H, d)
    np.testing.assert_array_equal(prm.seq2head_groups(x[:L], 1, 3)[0], prm.seq2head(x[:L], 3))
    for B, K in ((1, 2), (3, 1), (3, 2), (3, 3), (3, 6)):
        y = prm.seq2head_groups(x, B, K)
        assert y.shape == (B, K, 3 * L // B, H // K, d)
        np.testing.assert_array_equal(prm.head2seq_groups(y, B, K), x)
    y = prm.seq2head_groups(x, 3, 2)     # h = 3
    # token 4 of sequence 2 is row 14; its head 4 is group 1, local head 1
    np.testing.assert_array_equal(y[2, 1, 4, 1], x[14, 4])
    np.testing.assert_array_equal(y[1, 0, 0, 2], x[5, 2])
    np.testing.assert_array_equal(y[0, 1, 3, 0], x[3, 3])
    x2 = x.copy()
    x2[L:2 * L] += 1000                  # sequence 1 only
    y2 = prm.seq2head_groups(x2, 3, 2)
    np.testing.assert_array_equal(y2[0], y[0])
    np.testing.assert_array_equal(y2[2], y[2])
    assert (y2[1] != y[1]).all()


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
