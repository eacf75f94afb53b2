"""Seeded synthetic workloads for the varlen attention hot path.

This module holds only input generation (document lengths, random tensors,
``cu_seqlens``); it contains none of the attention, merge or permutation
arithmetic.  It is the one module that both the CUDA path's callers (tests,
``bench.py``) and the fp64 oracle's callers use, so that the two sides see the
same bits.

Workload shapes follow the pages' long-tailed length mixes:

* NSP (Nested Sequence Parallelism), Sec. 2.2 "Sequence Packing":
  packed batches under a token budget, most documents short, a few very long
  (Sec. 3, Fig. 2), maximum contexts of 192K and 384K tokens (Sec. 6, setup).
* HSAP, Sec. 2.1 "Sequence Packing": packed hybrid-context documents
  addressed by cumulative lengths (``cu_len``).
* DCP (Training Variable Long Sequences with Data-Centric Parallel), Sec. 4.1:
  a short-dominated synthetic length distribution.

Recipe (the pages give no generator; this is the plainest reading of them):

* seed ``1000 + config number``; draw order: lengths, Q, K, V, dOut;
* lognormal lengths: ``round(exp(N(ln median, sigma^2)))``, clipped, drawn
  until the token budget is filled, the last document truncated to fill
  (it may then be shorter than the clip minimum);
* long documents of configs 3 and 4 are placed first (``shuffle=True`` moves
  them to a seeded random position instead);
* Q/K/V/dOut iid N(0, 1), drawn in float32 and rounded to bfloat16
  (round-to-nearest-even) for the bf16 configs.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


@dataclass(frozen=True)
class Config:
    cid: int
    name: str
    T: int
    Hq: int
    Hkv: int
    d: int
    dtype: str              # "f32" or "bf16"
    bwd: bool
    fixed_lengths: tuple = ()
    long_doc: int = 0       # one document of this length placed first (0: none)
    median: float = 0.0     # lognormal median of the other documents
    sigma: float = 0.0
    clip: tuple = (1, 1)
    uniform: tuple = ()     # (lo, hi) inclusive integer uniform lengths
    shards: int = 1         # ring-style contiguous shards (chunked mode)
    permute_groups: int = 0  # seq->head permutation groups (0: none)
    causal: bool = True


CONFIGS = {
    1: Config(1, "fp32_4docs_381tok_h4_d64_fwd", 381, 4, 4, 64, "f32", False,
              fixed_lengths=(17, 64, 100, 200)),
    2: Config(2, "bf16_32k_lognormal1024_h32kv4_d128", 32768, 32, 4, 128, "bf16", True,
              median=1024.0, sigma=1.2, clip=(64, 16384)),
    3: Config(3, "bf16_128k_ring8_long64k_h32kv4_d128", 131072, 32, 4, 128, "bf16", False,
              long_doc=65536, median=2048.0, sigma=1.2, clip=(128, 32768),
              shards=8, permute_groups=8),
    4: Config(4, "bf16_384k_long256k_h32kv4_d128", 393216, 32, 4, 128, "bf16", True,
              long_doc=262144, median=2048.0, sigma=1.2, clip=(128, 16384)),
    5: Config(5, "bf16_64k_uniform32to256_h32kv4_d128", 65536, 32, 4, 128, "bf16", True,
              uniform=(32, 256)),
}


def seed_of(cid: int) -> int:
    return 1000 + cid


def draw_lengths(cfg: Config, rng: np.random.Generator, shuffle: bool = False) -> list:
    """Document lengths summing exactly to cfg.T (see module docstring)."""
    if cfg.fixed_lengths:
        lens = list(cfg.fixed_lengths)
        assert sum(lens) == cfg.T
        return lens
    lens = []
    total = 0
    if cfg.long_doc:
        lens.append(cfg.long_doc)
        total = cfg.long_doc
    while total < cfg.T:
        if cfg.uniform:
            L = int(rng.integers(cfg.uniform[0], cfg.uniform[1] + 1))
        else:
            L = int(round(float(np.exp(rng.normal(np.log(cfg.median), cfg.sigma)))))
            L = min(max(L, cfg.clip[0]), cfg.clip[1])
        L = min(L, cfg.T - total)
        lens.append(L)
        total += L
    if shuffle and cfg.long_doc:
        pos = int(rng.integers(0, len(lens)))
        lens.insert(pos, lens.pop(0))
    return lens


def cu_from_lengths(lens) -> np.ndarray:
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return cu


def _normal(rng: np.random.Generator, shape, dtype: str) -> torch.Tensor:
    x = torch.from_numpy(rng.standard_normal(size=shape, dtype=np.float32))
    return x.to(torch.bfloat16) if dtype == "bf16" else x


@dataclass
class Workload:
    cfg: Config
    lengths: list
    cu_seqlens: np.ndarray          # int32 [ndoc+1]
    q: torch.Tensor                 # CPU [T, Hq, d]  (bf16 or f32)
    k: torch.Tensor                 # CPU [T, Hkv, d]
    v: torch.Tensor
    dout: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def ndoc(self) -> int:
        return len(self.lengths)

    def f64(self, name: str) -> np.ndarray:
        """The (already rounded) tensor as float64 numpy, for the oracle."""
        return getattr(self, name).to(torch.float64).numpy()


def make_workload(cid: int, shuffle: bool = False, with_dout: Optional[bool] = None,
                  seed: Optional[int] = None) -> Workload:
    cfg = CONFIGS[cid]
    rng = np.random.default_rng(seed_of(cid) if seed is None else seed)
    lens = draw_lengths(cfg, rng, shuffle=shuffle)
    T = cfg.T
    q = _normal(rng, (T, cfg.Hq, cfg.d), cfg.dtype)
    k = _normal(rng, (T, cfg.Hkv, cfg.d), cfg.dtype)
    v = _normal(rng, (T, cfg.Hkv, cfg.d), cfg.dtype)
    want_dout = cfg.bwd if with_dout is None else with_dout
    dout = _normal(rng, (T, cfg.Hq, cfg.d), cfg.dtype) if want_dout else None
    return Workload(cfg, lens, cu_from_lengths(lens), q, k, v, dout)


def make_workload_device(cid: int, device, seed: Optional[int] = None) -> Workload:
    """Config `cid` with its seeded lengths (the same draw as make_workload)
    and its tensors drawn on `device` by torch's seeded generator: the same
    shapes and N(0, 1) values rounded to bf16, generated in milliseconds
    instead of minutes for the large configs.  Not the same numbers as
    make_workload (the benchmark needs the distribution, not the bits)."""
    cfg = CONFIGS[cid]
    s = seed_of(cid) if seed is None else seed
    lens = draw_lengths(cfg, np.random.default_rng(s))
    gen = torch.Generator(device=device)
    gen.manual_seed(s)
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    T = cfg.T

    def draw(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dt)
    q = draw((T, cfg.Hq, cfg.d))
    k = draw((T, cfg.Hkv, cfg.d))
    v = draw((T, cfg.Hkv, cfg.d))
    dout = draw((T, cfg.Hq, cfg.d)) if cfg.bwd else None
    return Workload(cfg, lens, cu_from_lengths(lens), q, k, v, dout)


def make_custom(lengths, Hq: int, Hkv: int, d: int, dtype: str = "bf16", seed: int = 0,
                with_dout: bool = True) -> Workload:
    """A small seeded workload with explicit document lengths (edge cases)."""
    lens = [int(x) for x in lengths]
    T = int(sum(lens))
    cfg = Config(0, f"custom_T{T}_h{Hq}kv{Hkv}_d{d}", T, Hq, Hkv, d, dtype, with_dout)
    rng = np.random.default_rng(seed)
    q = _normal(rng, (T, Hq, d), dtype)
    k = _normal(rng, (T, Hkv, d), dtype)
    v = _normal(rng, (T, Hkv, d), dtype)
    dout = _normal(rng, (T, Hq, d), dtype) if with_dout else None
    return Workload(cfg, lens, cu_from_lengths(lens), q, k, v, dout)


def make_growing(lengths, Hq: int, Hkv: int, d: int, seed: int = 0, gain: float = 8.0,
                 ramp: float = 4.0, with_dout: bool = True) -> Workload:
    """make_custom's bf16 draws with one component overwritten so that scores
    rise along every document: component 0 of every query is ``gain`` and
    component 0 of key j is ``ramp * (j - start of j's document) / 128``.
    Against later keys of its document a query's scores then climb by about
    gain * ramp / sqrt(d) per 128 keys (at the usual scale 1/sqrt(d)), on top
    of the N(0, 1) noise of the other components, so a row's running maximum
    keeps growing as key tiles are visited in order: inputs that drive the
    online softmax's rescaling of a running output."""
    w = make_custom(lengths, Hq, Hkv, d, dtype="bf16", seed=seed, with_dout=with_dout)
    cu = w.cu_seqlens.astype(np.int64)
    pos = np.arange(w.T, dtype=np.int64) - np.repeat(cu[:-1], np.diff(cu))
    q = w.q.float()
    k = w.k.float()
    q[:, :, 0] = gain
    k[:, :, 0] = torch.from_numpy((ramp * pos / 128.0).astype(np.float32))[:, None]
    w.q = q.to(torch.bfloat16)
    w.k = k.to(torch.bfloat16)
    w.extra.update(gain=gain, ramp=ramp)
    return w


def shard_bounds(T: int, shards: int) -> list:
    """Contiguous equal shards [start, end) of the packed stream (ring SP)."""
    assert T % shards == 0
    n = T // shards
    return [(i * n, (i + 1) * n) for i in range(shards)]
