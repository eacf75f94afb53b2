"""Shared helpers of the GPU parity tests: device copies of seeded
workloads, oracle caching, sampled rows and the comparison metrics.

Tolerances (stated for bf16 inputs with float32 accumulation):
out max-abs <= 2e-2, lse max-abs <= 1e-3, gradient relative L2 <= 1e-2 per
tensor.  float32 inputs are held to a tighter internal bar (out 1e-4, lse
1e-5), the plainest reading of true float32 arithmetic.
"""
from __future__ import annotations

import time

import numpy as np
import torch

import oracle
from variable_length_sequence_gb300.workloads import Workload, make_workload

TOL_OUT, TOL_LSE, TOL_GRAD = 2e-2, 1e-3, 1e-2
TOL_OUT_F32, TOL_LSE_F32 = 1e-4, 1e-5
# Internal per-(row, head) bar for gradients: the error of one row's d-vector
# against TOL_ROW x (its own norm + the tensor's RMS row norm).  The kernels'
# own roundings (P and dS to bf16, the result to bf16: 2^-9 relative each)
# leave a row at a few 1e-3 of that; a row computed from the wrong keys,
# rows or heads is off by about its whole norm.
TOL_ROW = 5e-2

_WL_CACHE: dict = {}


def workload(cid: int, shuffle: bool = False) -> Workload:
    key = (cid, shuffle)
    if key not in _WL_CACHE:
        t = time.time()
        _WL_CACHE[key] = make_workload(cid, shuffle=shuffle)
        print(f"[workload C{cid}{' shuffled' if shuffle else ''}: {time.time() - t:.1f}s]")
    return _WL_CACHE[key]


def to_dev(w: Workload) -> dict:
    d = {n: getattr(w, n).cuda() for n in ("q", "k", "v")}
    if w.dout is not None:
        d["dout"] = w.dout.cuda()
    d["cu"] = torch.from_numpy(w.cu_seqlens).cuda()
    return d


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def max_abs(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    fa, fb = np.isfinite(a), np.isfinite(b)
    assert np.array_equal(fa, fb), "non-finite pattern differs"
    assert np.array_equal(a[~fa], b[~fb]), "infinities differ"
    return float(np.abs(a[fa] - b[fb]).max()) if fa.any() else 0.0


def rel_l2(a, b_ref) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b_ref, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_rows_close(got, ref, label: str = ""):
    """Every (row, head) d-vector of a gradient [rows, heads, d] within TOL_ROW
    of the reference, relative to its own norm plus the RMS row norm."""
    g, r = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.linalg.norm(g - r, axis=-1)
    nrm = np.linalg.norm(r, axis=-1)
    rms = float(np.sqrt(np.mean(nrm ** 2)))
    worst = err / (nrm + rms)
    i = np.unravel_index(int(np.argmax(worst)), worst.shape)
    print(f"[{label}] worst row {i}: {float(worst[i]):.3e} of (norm + rms) (tol {TOL_ROW})")
    assert float(worst[i]) <= TOL_ROW, f"{label}: row {i} error {float(worst[i])}"


def sample_rows(cu: np.ndarray, n_random: int, seed: int, extra=()) -> np.ndarray:
    """First and last row of every non-empty document plus seeded random rows."""
    cu = np.asarray(cu, np.int64)
    T = int(cu[-1])
    rows = set(int(x) for x in extra if 0 <= x < T)
    for b in range(len(cu) - 1):
        if cu[b + 1] > cu[b]:
            rows.add(int(cu[b]))
            rows.add(int(cu[b + 1] - 1))
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, T, n_random))
    return np.array(sorted(rows), dtype=np.int64)


def oracle_inputs(w: Workload):
    return tuple(w.f64(n) for n in ("q", "k", "v")) + ((w.f64("dout"),) if w.dout is not None
                                                       else (None,))


def timed(label: str, fn, *a, **k):
    t = time.time()
    r = fn(*a, **k)
    print(f"[{label}: {time.time() - t:.1f}s]")
    return r


def assert_fwd_close(out_gpu, lse_gpu, out_ref, lse_ref, f32: bool = False, label: str = ""):
    tol_o, tol_l = (TOL_OUT_F32, TOL_LSE_F32) if f32 else (TOL_OUT, TOL_LSE)
    eo = max_abs(out_gpu, out_ref)
    el = max_abs(lse_gpu, lse_ref)
    print(f"[{label}] out max-abs {eo:.3e} (tol {tol_o}), lse max-abs {el:.3e} (tol {tol_l})")
    assert eo <= tol_o, f"{label}: out max-abs {eo} > {tol_o}"
    assert el <= tol_l, f"{label}: lse max-abs {el} > {tol_l}"
