"""Document-masked (varlen) attention, forward and backward, in float64.

Definition followed (no tiling, no online softmax):

* Scaled dot-product attention, softmax(Q K^T / sqrt(d_k)) V, one head at a
  time, heads concatenated: BASP, Sec. II-A "Scaled Dot-Product Attention"
  and "Multi-Head Attention"; HSAP, Sec. 2.2.1 (Q, K, V in R^{N x H x d}).
* Packed documents: attention only within each segment, addressed by
  cumulative lengths ``cu_seqlens``; tokens of different documents never
  attend to each other (HSAP, Sec. 2.1 "Sequence Packing", the
  cross-contamination problem; NSP, Sec. 2.2 "Sequence Packing").
* Causal: query t of a document sees the keys of its own document at
  positions <= t (top-left aligned self-attention).  ``causal=False`` sees
  the whole document.
* Grouped-query heads (the pages never mention GQA; reading): query head h
  uses key/value head h // (Hq // Hkv).
* Partial blocks of ring-style InterSP (HSAP, Sec. 2.2.1 and Sec. 3.2
  "Partition attention computation blocks"): restrict queries to a global
  range [qa, qb) and keys to [ka, kb); a query with no allowed key gets
  lse = -inf and out = 0 (the pages are silent; this makes the merge of any
  key chunking exact).
* lse is the natural-log log-sum-exp of the *scaled* scores, laid out
  [Hq, rows]; out is [rows, Hq, d].

Backward: the analytic gradients of L = sum(dOut * out) for the definition
above (the attention the backward pass recomputes, NSP Sec. 2.3):
  delta_t = <dOut_t, out_t>, dP_tj = <dOut_t, v_j>, dS_tj = p_tj (dP_tj - delta_t),
  dV_j = sum_t p_tj dOut_t, dQ_t = scale sum_j dS_tj k_j, dK_j = scale sum_t dS_tj q_t,
with dK/dV summed over the query heads of each key/value group.

Score matrices are materialised one block of query rows at a time; every
row always sees its full key set, so the blocking changes nothing but memory.
"""
from __future__ import annotations

import numpy as np

_BLOCK_ELEMS = 1 << 25      # max float64 scores materialised at once (256 MB)


def doc_index(cu: np.ndarray, t):
    """Document containing global token t (zero-length documents never do)."""
    return np.searchsorted(cu, t, side="right") - 1


def allowed_interval(t: int, cu, causal: bool, kv_range=None):
    """Keys [lo, hi) that query t may attend to (empty when hi <= lo)."""
    cu = np.asarray(cu, dtype=np.int64)
    b = int(doc_index(cu, t))
    lo, hi = int(cu[b]), (t + 1 if causal else int(cu[b + 1]))
    if kv_range is not None:
        lo, hi = max(lo, kv_range[0]), min(hi, kv_range[1])
    return lo, max(lo, hi)


def _rows_per_block(G: int, nk: int) -> int:
    return int(max(1, min(1024, _BLOCK_ELEMS // (G * max(nk, 1)))))


def _docs_of_rows(rows: np.ndarray, cu: np.ndarray):
    """Yield (doc b, positions into rows) for every document holding rows."""
    docs = doc_index(cu, rows)
    for b in np.unique(docs):
        yield int(b), np.nonzero(docs == b)[0]


def _block(qg, kg, rows, keys, scale, causal, kv_lo, kv_hi):
    """Scores, mask, lse and probabilities of one row block of one kv group.

    qg [nb, G, d] are the query heads of the group, kg [nk, d] the keys
    ``keys`` (global ids) of the document.  Returns p [nb, G, nk] (zero where
    masked) and lse [nb, G] (-inf for rows with no allowed key).
    """
    nb, G, d = qg.shape
    x = scale * (qg.reshape(nb * G, d) @ kg.T).reshape(nb, G, -1)
    allowed = np.broadcast_to((keys >= kv_lo) & (keys < kv_hi), (nb, len(keys)))
    if causal:
        allowed = allowed & (keys[None, :] <= rows[:, None])
    x = np.where(allowed[:, None, :], x, -np.inf)
    m = x.max(axis=-1) if x.shape[-1] else np.full((nb, G), -np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    with np.errstate(divide="ignore"):      # log(0) only on rows masked to -inf
        lse = np.where(empty, -np.inf, m_safe + np.log(np.exp(x - m_safe[..., None]).sum(-1)))
    lse_safe = np.where(empty, 0.0, lse)
    p = np.where(empty[..., None], 0.0, np.exp(x - lse_safe[..., None]))
    return p, lse


def attn_fwd_rows(q, k, v, cu_seqlens, scale, causal=True, rows=None, kv_range=None):
    """out [n, Hq, d] and lse [Hq, n] for the global query ids ``rows``."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), Hq, v.shape[2]))
    lse = np.full((Hq, len(rows)), -np.inf)
    ka, kb = (0, k.shape[0]) if kv_range is None else kv_range
    for b, pos in _docs_of_rows(rows, cu):
        kv_lo, kv_hi = max(int(cu[b]), ka), min(int(cu[b + 1]), kb)
        if kv_hi <= kv_lo:
            continue
        keys = np.arange(kv_lo, kv_hi)
        nb = _rows_per_block(G, len(keys))
        for s in range(0, len(pos), nb):
            pb = pos[s:s + nb]
            rb = rows[pb]
            for g in range(Hkv):
                hs = slice(g * G, (g + 1) * G)
                p, l = _block(q[rb, hs, :], k[keys, g, :], rb, keys, scale, causal,
                              kv_lo, kv_hi)
                nbr = len(pb)
                out[pb, hs, :] = (p.reshape(nbr * G, -1) @ v[keys, g, :]).reshape(nbr, G, -1)
                lse[hs, pb] = l.T
    return out, lse


def attn_fwd(q, k, v, cu_seqlens, scale, causal=True, q_range=None, kv_range=None):
    """Whole stream (or the partial block q_range x kv_range, global ids)."""
    qa, qb = (0, q.shape[0]) if q_range is None else q_range
    return attn_fwd_rows(q, k, v, cu_seqlens, scale, causal, np.arange(qa, qb), kv_range)


def attn_probs(q, k, cu_seqlens, scale, causal, h):
    """Dense [T, T] attention probabilities of query head h (tiny T only)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, _ = q.shape
    g = h // (Hq // k.shape[1])
    P = np.zeros((T, T))
    for t in range(T):
        lo, hi = allowed_interval(t, cu, causal)
        x = scale * (k[lo:hi, g, :] @ q[t, h, :])
        e = np.exp(x - x.max())
        P[t, lo:hi] = e / e.sum()
    return P


def attn_bwd(q, k, v, dout, cu_seqlens, scale, causal=True):
    """dq [T,Hq,d], dk [T,Hkv,d], dv [T,Hkv,d] of L = sum(dout * out)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dv = np.zeros_like(v, dtype=np.float64)
    for b in range(len(cu) - 1):
        lo, hi = int(cu[b]), int(cu[b + 1])
        if hi <= lo:
            continue
        keys = np.arange(lo, hi)
        nb = _rows_per_block(G, len(keys))
        for s in range(lo, hi, nb):
            rb = np.arange(s, min(s + nb, hi))
            n = len(rb)
            for g in range(Hkv):
                hs = slice(g * G, (g + 1) * G)
                qg, kg, vg, dog = q[rb, hs, :], k[keys, g, :], v[keys, g, :], dout[rb, hs, :]
                p, _ = _block(qg, kg, rb, keys, scale, causal, lo, hi)
                pf = p.reshape(n * G, -1)
                o = (pf @ vg).reshape(n, G, -1)
                delta = (dog * o).sum(-1)                                     # [n, G]
                dP = (dog.reshape(n * G, -1) @ vg.T).reshape(n, G, -1)        # [n, G, nk]
                dS = p * (dP - delta[..., None])
                dSf = dS.reshape(n * G, -1)
                dv[keys, g, :] += pf.T @ dog.reshape(n * G, -1)
                dk[keys, g, :] += scale * (dSf.T @ qg.reshape(n * G, -1))
                dq[rb, hs, :] = scale * (dSf @ kg).reshape(n, G, -1)
    return dq, dk, dv


def attn_bwd_dq_rows(q, k, v, dout, cu_seqlens, scale, causal, rows):
    """dQ [n, Hq, d] for the global query ids ``rows`` only."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    rows = np.asarray(rows, dtype=np.int64)
    dq = np.zeros((len(rows), Hq, d))
    for b, pos in _docs_of_rows(rows, cu):
        lo, hi = int(cu[b]), int(cu[b + 1])
        keys = np.arange(lo, hi)
        nb = _rows_per_block(G, len(keys))
        for s in range(0, len(pos), nb):
            pb = pos[s:s + nb]
            rb = rows[pb]
            n = len(pb)
            for g in range(Hkv):
                hs = slice(g * G, (g + 1) * G)
                qg, kg, vg, dog = q[rb, hs, :], k[keys, g, :], v[keys, g, :], dout[rb, hs, :]
                p, _ = _block(qg, kg, rb, keys, scale, causal, lo, hi)
                o = (p.reshape(n * G, -1) @ vg).reshape(n, G, -1)
                delta = (dog * o).sum(-1)
                dP = (dog.reshape(n * G, -1) @ vg.T).reshape(n, G, -1)
                dS = p * (dP - delta[..., None])
                dq[pb, hs, :] = scale * (dS.reshape(n * G, -1) @ kg).reshape(n, G, -1)
    return dq


def attn_bwd_dkv_rows(q, k, v, dout, cu_seqlens, scale, causal, key_rows, g):
    """dK, dV [n, d] of key/value head g for the global key ids ``key_rows``.

    Every query that can see one of the keys contributes; its probabilities
    are normalised over its full key set, as in the definition.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    hs = slice(g * G, (g + 1) * G)
    key_rows = np.asarray(key_rows, dtype=np.int64)
    dk = np.zeros((len(key_rows), d))
    dv = np.zeros((len(key_rows), v.shape[2]))
    for b, kpos in _docs_of_rows(key_rows, cu):
        lo, hi = int(cu[b]), int(cu[b + 1])
        keys = np.arange(lo, hi)
        sel = key_rows[kpos] - lo                      # sampled keys, doc-relative
        first_q = int(key_rows[kpos].min()) if causal else lo
        nb = _rows_per_block(G, len(keys))
        for s in range(first_q, hi, nb):
            rb = np.arange(s, min(s + nb, hi))
            n = len(rb)
            qg, dog = q[rb, hs, :], dout[rb, hs, :]
            kg, vg = k[keys, g, :], v[keys, g, :]
            p, _ = _block(qg, kg, rb, keys, scale, causal, lo, hi)
            o = (p.reshape(n * G, -1) @ vg).reshape(n, G, -1)
            delta = (dog * o).sum(-1)
            ps = p[:, :, sel]                                                  # [n, G, m]
            dPs = (dog.reshape(n * G, -1) @ vg[sel].T).reshape(n, G, -1)
            dSs = ps * (dPs - delta[..., None])
            dv[kpos] += ps.reshape(n * G, -1).T @ dog.reshape(n * G, -1)
            dk[kpos] += scale * (dSs.reshape(n * G, -1).T @ qg.reshape(n * G, -1))
    return dk, dv


def attn_bwd_block(q, k, v, dout, cu_seqlens, scale, causal, q_range, kv_range):
    """Gradient contributions of one ring block: queries [qa, qb) against keys
    [ka, kb) (global ids), for the backward of a ring-style InterSP step
    (HSAP Sec. 2.2.1: the KV blocks circulate, each rank's queries meet every
    block once; HSAP Sec. 3.2 blocks A1-A5).

    The probabilities are those of the whole row (normalised over the row's
    full key set, i.e. by the row's global lse) and delta_t = <dOut_t, out_t>
    uses the row's full output; only the sums are restricted to the block:
      dq[t - qa] = scale sum_{j in block} dS_tj k_j,
      dk[j - ka] = scale sum_{t in block, h in grp(g)} dS_tj q_t,
      dv[j - ka] = sum_{t in block, h in grp(g)} p_tj dOut_t.
    Summing the blocks of any (query chunking x key chunking) gives
    ``attn_bwd``.  Returns dq [qb - qa, Hq, d], dk / dv [kb - ka, Hkv, d].
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    qa, qb = q_range
    ka, kb = kv_range
    dq = np.zeros((qb - qa, Hq, d))
    dk = np.zeros((kb - ka, Hkv, d))
    dv = np.zeros((kb - ka, Hkv, v.shape[2]))
    rows = np.arange(qa, qb)
    for b, pos in _docs_of_rows(rows, cu):
        lo, hi = int(cu[b]), int(cu[b + 1])
        keys = np.arange(lo, hi)                        # the row's full key set
        sel = (keys >= ka) & (keys < kb)                # the block's keys
        if not sel.any():
            continue
        nb = _rows_per_block(G, len(keys))
        for s in range(0, len(pos), nb):
            rb = rows[pos[s:s + nb]]
            n = len(rb)
            for g in range(Hkv):
                hs = slice(g * G, (g + 1) * G)
                qg, kg, vg, dog = q[rb, hs, :], k[keys, g, :], v[keys, g, :], dout[rb, hs, :]
                p, _ = _block(qg, kg, rb, keys, scale, causal, lo, hi)
                o = (p.reshape(n * G, -1) @ vg).reshape(n, G, -1)
                delta = (dog * o).sum(-1)                                     # [n, G]
                ps = p[:, :, sel]                                             # block columns
                dPs = (dog.reshape(n * G, -1) @ vg[sel].T).reshape(n, G, -1)
                dSs = (ps * (dPs - delta[..., None])).reshape(n * G, -1)
                kj = keys[sel] - ka
                dq[rb - qa, hs, :] += scale * (dSs @ kg[sel]).reshape(n, G, -1)
                dk[kj, g, :] += scale * (dSs.T @ qg.reshape(n * G, -1))
                dv[kj, g, :] += ps.reshape(n * G, -1).T @ dog.reshape(n * G, -1)
    return dq, dk, dv
