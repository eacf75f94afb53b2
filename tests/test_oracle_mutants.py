"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that at least one pin fails for each: the pins have teeth.  The real oracle
files are never modified; each mutant is compiled from the source text with
one replacement applied."""
import importlib.util
import os
import types

import pytest

import oracle.attention as att
import oracle.merge as mrg
import oracle.permute as prm
from oracle_pins import ALL_PINS

ORACLE_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")

MUTANTS = [
    # (file, original text, planted mistake, why it is plausible)
    ("attention.py", "keys[None, :] <= rows[:, None]", "keys[None, :] < rows[:, None]",
     "causal off by one (query misses itself)"),
    ("attention.py", "hs = slice(g * G, (g + 1) * G)\n                p, l",
     "hs = slice(g, Hq, Hkv)\n                p, l", "strided instead of contiguous GQA groups"),
    ("attention.py", "x = scale * (qg", "x = (qg", "scale dropped"),
    ("attention.py", "kv_lo, kv_hi = max(int(cu[b]), ka)", "kv_lo, kv_hi = max(0, ka)",
     "document start ignored (cross-contamination)"),
    ("attention.py", "lse = np.where(empty, -np.inf, m_safe + np.log(",
     "lse = np.where(empty, -np.inf, np.log(", "max not added back into lse"),
    ("attention.py", "dS = p * (dP - delta[..., None])\n                dSf",
     "dS = p * dP\n                dSf", "delta term dropped in dS"),
    ("attention.py", "dk[keys, g, :] += scale * (dSf.T", "dk[keys, g, :] += (dSf.T",
     "scale dropped in dK"),
    ("attention.py", "dv[keys, g, :] += pf.T @ dog", "dv[keys, g, :] += pf.T @ dog[::-1]",
     "wrong rows of dOut in dV"),
    ("attention.py", "p, _ = _block(qg, kg, rb, keys, scale, causal, lo, hi)\n"
     "                o = (p.reshape(n * G, -1) @ vg).reshape(n, G, -1)\n"
     "                delta = (dog * o).sum(-1)                                     # [n, G]\n"
     "                ps",
     "p, _ = _block(qg, kg, rb, keys, scale, causal, max(lo, ka), min(hi, kb))\n"
     "                o = (p.reshape(n * G, -1) @ vg).reshape(n, G, -1)\n"
     "                delta = (dog * o).sum(-1)                                     # [n, G]\n"
     "                ps",
     "ring block backward normalised over the block's keys only"),
    ("attention.py", "dk[kj, g, :] += scale * (dSs.T", "dk[kj, g, :] += (dSs.T",
     "scale dropped in the block dK"),
    ("attention.py", "kj = keys[sel] - ka", "kj = keys[sel] - lo",
     "block keys offset by the document start instead of the block start"),
    ("merge.py", "np.exp(L - np.where(empty, 0.0, lse))", "np.exp(L - np.where(empty, 0.0, m))",
     "weights not normalised by the merged lse"),
    ("merge.py", "m_safe + np.log(", "np.log(", "max not added back into merged lse"),
    ("permute.py", "out[g, t, j, :] = x[t, g * h + j, :]", "out[g, t, j, :] = x[t, j * P + g, :]",
     "strided head groups"),
    ("permute.py", "out[b, g, t, j, :] = x[b * L + t, g * h + j, :]",
     "out[b, g, t, j, :] = x[g * L + t, b * h + j, :]", "subgroup exchange across sequences"),
    ("permute.py", "out[b, g, t, j, :] = x[b * L + t, g * h + j, :]",
     "out[b, g, t, j, :] = x[t * B + b, g * h + j, :]", "sequences interleaved by token"),
]


def _load_mutant(fname, old, new):
    mods = {"attention.py": att, "merge.py": mrg, "permute.py": prm}
    with open(os.path.join(ORACLE_DIR, fname)) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found in {fname}: {old!r}"
    mutated = types.ModuleType("mutant_" + fname[:-3])
    exec(compile(src.replace(old, new, 1), f"<mutant {fname}>", "exec"), mutated.__dict__)
    out = dict(mods)
    out[fname] = mutated
    return out["attention.py"], out["merge.py"], out["permute.py"]


@pytest.mark.parametrize("fname,old,new,why", MUTANTS, ids=[m[3] for m in MUTANTS])
def test_mutant_is_caught(fname, old, new, why):
    a, m, p = _load_mutant(fname, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(a, m, p)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches: {why}"
