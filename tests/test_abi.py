"""The C-ABI library builds, loads without a GPU, exports every function
include/nsp.h declares, and rejects bad arguments on the host before any
CUDA call (only the *_validate entry points and host helpers run here)."""
import ctypes as C
import os

import numpy as np
import pytest

from variable_length_sequence_gb300 import build as nsp_build
from variable_length_sequence_gb300 import nsp


@pytest.fixture(scope="module")
def lib():
    nsp_build.build()
    return nsp.load()


def test_exports_every_header_function(lib):
    names = nsp.header_functions()
    assert "nsp_attn_fwd" in names and "nsp_seq2head_permute" in names
    for n in names:
        assert hasattr(lib, n), f"libnsp.so does not export {n}"
    assert set(names) >= set(nsp._SIGNATURES), "binding names a function the header lacks"


def test_status_strings(lib):
    for st in range(7):
        assert nsp.status_str(st).startswith("NSP_")
    assert nsp.status_str(99) == "NSP_ERR_UNKNOWN"
    assert b"sm_103a" in lib.nsp_version()


A = 1 << 20          # fake, 16-byte aligned "device" addresses: never dereferenced


def fwd_args(**kw):
    a = dict(q=A, k=A + 4096, v=A + 8192, cu=A + 12288, ndoc=3, q_start=0, q_len=300,
             kv_start=0, kv_len=300, Hq=32, Hkv=4, d=128, causal=1, io=nsp.NSP_BF16,
             out=A + 16384, out_dtype=nsp.NSP_BF16, ws=A + 32768,
             ws_bytes=nsp.nsp_attn_fwd_workspace_size(300, 300, 32, 4, 128))
    a.update(kw)
    return a


def call_fwd_validate(lib, a):
    return lib.nsp_attn_fwd_validate(a["q"], a["k"], a["v"], a["cu"], a["ndoc"], a["q_start"],
                                     a["q_len"], a["kv_start"], a["kv_len"], a["Hq"], a["Hkv"],
                                     a["d"], a["causal"], a["io"], a["out"], a["out_dtype"],
                                     a["ws"], a["ws_bytes"])


@pytest.mark.parametrize("kw,expect", [
    ({}, nsp.NSP_OK),
    ({"Hq": 30}, nsp.NSP_ERR_INVALID),                 # Hq % Hkv != 0
    ({"Hkv": 0}, nsp.NSP_ERR_INVALID),
    ({"ndoc": 0}, nsp.NSP_ERR_INVALID),
    ({"d": 96}, nsp.NSP_ERR_UNSUPPORTED),
    ({"causal": 2}, nsp.NSP_ERR_INVALID),
    ({"io": 7}, nsp.NSP_ERR_INVALID),
    ({"out_dtype": nsp.NSP_F32}, nsp.NSP_OK),          # float32 partials
    ({"io": nsp.NSP_F32, "out_dtype": nsp.NSP_BF16}, nsp.NSP_ERR_INVALID),
    ({"q_len": -1}, nsp.NSP_ERR_INVALID),
    ({"q": A + 8}, nsp.NSP_ERR_ALIGN),
    ({"cu": A + 4}, nsp.NSP_ERR_ALIGN),
    ({"out": A + 16384 + 16}, nsp.NSP_ERR_ALIGN),       # bf16 out: 32-byte vectors
    ({"out": A + 16384 + 16, "out_dtype": nsp.NSP_F32}, nsp.NSP_OK),
    ({"q": 0}, nsp.NSP_ERR_INVALID),
    ({"ws": 0}, nsp.NSP_ERR_WORKSPACE),
    ({"ws_bytes": 100}, nsp.NSP_ERR_WORKSPACE),
    ({"q_len": 0, "kv_len": 0, "ws_bytes": 4096}, nsp.NSP_OK),
])
def test_fwd_validation(lib, kw, expect):
    assert call_fwd_validate(lib, fwd_args(**kw)) == expect


def test_bwd_validation(lib):
    ws = nsp.nsp_attn_bwd_workspace_size(1000, 32, 4, 128, nsp.NSP_BF16)
    # only the CUDA-core path (here: float32 inputs) needs a float32 dq accumulator
    ws32 = nsp.nsp_attn_bwd_workspace_size(1000, 32, 4, 128, nsp.NSP_F32)
    assert ws32 >= ws + 1000 * 32 * 128 * 4
    ptrs = [A + 4096 * i for i in range(10)]
    ok = lib.nsp_attn_bwd_validate(*ptrs[:7], 5, 1000, 32, 4, 128, 1, nsp.NSP_BF16,
                                   *ptrs[7:10], A + (1 << 16), ws)
    assert ok == nsp.NSP_OK
    assert lib.nsp_attn_bwd_validate(*ptrs[:7], 5, 1000, 32, 4, 128, 1, nsp.NSP_BF16,
                                     *ptrs[7:10], A + (1 << 16), ws - 1) == nsp.NSP_ERR_WORKSPACE
    bad = list(ptrs)
    bad[5] = A + 4                                 # lse misaligned
    assert lib.nsp_attn_bwd_validate(*bad[:7], 5, 1000, 32, 4, 128, 1, nsp.NSP_BF16,
                                     *bad[7:10], A + (1 << 16), ws) == nsp.NSP_ERR_ALIGN
    for i in (7, 8, 9):                            # bf16 dq / dk / dv: 32-byte vectors
        bad = list(ptrs)
        bad[i] += 16
        assert lib.nsp_attn_bwd_validate(*bad[:7], 5, 1000, 32, 4, 128, 1, nsp.NSP_BF16,
                                         *bad[7:10], A + (1 << 16), ws) == nsp.NSP_ERR_ALIGN
        assert lib.nsp_attn_bwd_validate(*bad[:7], 5, 1000, 32, 4, 128, 1, nsp.NSP_F32,
                                         *bad[7:10], A + (1 << 16), ws32) == nsp.NSP_OK


def test_merge_and_permute_validation(lib):
    outs = (C.c_void_p * 2)(A, A + 4096)
    lses = (C.c_void_p * 2)(A + 8192, A + 12288)
    v = lib.nsp_lse_merge_validate
    assert v(C.cast(outs, C.c_void_p), C.cast(lses, C.c_void_p), 2, 16, 4, 128, A + 65536,
             nsp.NSP_BF16, A + 131072) == nsp.NSP_OK
    assert v(C.cast(outs, C.c_void_p), C.cast(lses, C.c_void_p), 0, 16, 4, 128, A + 65536,
             nsp.NSP_BF16, None) == nsp.NSP_ERR_INVALID
    assert v(C.cast(outs, C.c_void_p), C.cast(lses, C.c_void_p), 65, 16, 4, 128, A + 65536,
             nsp.NSP_BF16, None) == nsp.NSP_ERR_INVALID
    p = lib.nsp_seq2head_permute_validate
    assert p(A, A + (1 << 24), 1024, 32, 128, 8, 2) == nsp.NSP_OK
    assert p(A, A + (1 << 24), 1024, 32, 128, 5, 2) == nsp.NSP_ERR_INVALID   # H % P
    assert p(A, A + (1 << 24), 1024, 32, 128, 8, 3) == nsp.NSP_ERR_INVALID   # elem size
    assert p(A, A + 1024, 1024, 32, 128, 8, 2) == nsp.NSP_ERR_INVALID        # overlap
    assert p(A + 2, A + (1 << 24), 1024, 32, 128, 8, 2) == nsp.NSP_ERR_ALIGN


def test_attn_pairs_counts_allowed_pairs(lib):
    cu = np.array([0, 3, 3, 7, 8], dtype=np.int32)       # lengths 3, 0, 4, 1
    brute_c = sum(1 for b in range(4) for t in range(cu[b], cu[b + 1])
                  for j in range(cu[b], t + 1))
    brute_n = sum(int(cu[b + 1] - cu[b]) ** 2 for b in range(4))
    assert nsp.nsp_attn_pairs(cu, True) == brute_c == 6 + 10 + 1
    assert nsp.nsp_attn_pairs(cu, False) == brute_n == 9 + 16 + 1
    with pytest.raises(nsp.NspError):
        nsp.nsp_attn_pairs(np.array([0, 5, 3], dtype=np.int32))


@pytest.mark.parametrize("causal", [True, False])
def test_ds_cache_size_matches_enumeration(lib, causal):
    """nsp_attn_bwd_ds_cache_size = Hq x (128-row query tile, 128-key tile)
    pairs holding at least one visible (query, key) pair x 32768 bytes, by
    enumerating the pairs of ragged streams (empty and one-token documents,
    documents that end inside and on tile edges); the batched form sums the
    pairs of every block, tiles aligned to the block's own starts."""
    rng = np.random.default_rng(41)
    cases = [[1], [128], [129], [0, 5, 0, 260, 0, 1], [300, 77, 150], [33] * 20,
             [127, 1, 128, 256, 3]]
    cases += [list(rng.integers(0, 400, rng.integers(1, 9))) for _ in range(6)]
    for lens in cases:
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        doc = np.repeat(np.arange(len(lens)), lens)
        nt = (T + 127) // 128
        pairs = 0
        for i in range(nt):
            for j in range(nt):
                t = np.arange(i * 128, min(T, i * 128 + 128))
                s = np.arange(j * 128, min(T, j * 128 + 128))
                vis = doc[t][:, None] == doc[s][None, :]
                if causal:
                    vis &= s[None, :] <= t[:, None]
                pairs += bool(vis.any())
        assert nsp.nsp_attn_bwd_ds_cache_size(cu, 6, causal) == 6 * pairs * 32768, lens
    # a table of blocks: every block's tiles aligned to its own q_start and kv_start
    lens = [300, 77, 1, 150, 400]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    doc = np.repeat(np.arange(len(lens)), lens)
    ranges = [(0, T, 0, T), (4, 300, 100, 500), (320, 11, 0, 330), (500, 428, 700, 228),
              (0, 0, 0, 10), (128, 256, 128, 256)]
    total = 0
    for qa, ql, ka, kl in ranges:
        for i0 in range(qa, qa + ql, 128):
            for j0 in range(ka, ka + kl, 128):
                t = np.arange(i0, min(qa + ql, i0 + 128))
                s_ = np.arange(j0, min(ka + kl, j0 + 128))
                vis = doc[t][:, None] == doc[s_][None, :]
                if causal:
                    vis &= s_[None, :] <= t[:, None]
                total += bool(vis.any())
    assert nsp.nsp_attn_bwd_blocks_ds_cache_size(cu, ranges, 6, causal) == 6 * total * 32768
    assert nsp.nsp_attn_bwd_blocks_ds_cache_size(cu, [(0, 10, T - 5, 10)], 6, causal) == 0
    assert nsp.nsp_attn_bwd_ds_cache_size(np.array([0, 5, 3], dtype=np.int32), 4) == 0
    assert nsp.nsp_attn_bwd_ds_cache_size(np.array([1, 5], dtype=np.int32), 4) == 0
    assert nsp.nsp_attn_bwd_ds_cache_size(np.array([0, 5], dtype=np.int32), 0) == 0


def test_accumulate_rejects_on_host(lib):
    """nsp_attn_fwd_accumulate: lse_acc is required and 16-byte aligned, and
    the scale must be positive; all three are refused before any launch."""
    ws = nsp.nsp_attn_fwd_workspace_size(300, 300, 32, 4, 128)
    f = lib.nsp_attn_fwd_accumulate

    def call(lse, scale=0.088, acc=A + 16384):
        return f(A, A + 4096, A + 8192, A + 12288, 3, 0, 300, 0, 300, 32, 4, 128, scale, 1,
                 nsp.NSP_BF16, acc, lse, A + 32768, ws, None)
    assert call(None) == nsp.NSP_ERR_INVALID
    assert call(A + (1 << 16) + 4) == nsp.NSP_ERR_ALIGN
    assert call(A + (1 << 16), scale=0.0) == nsp.NSP_ERR_INVALID
    assert call(A + (1 << 16), acc=A + 16388) == nsp.NSP_ERR_ALIGN


def test_noalloc_rejects_on_host_like_fwd(lib):
    """nsp_attn_fwd_noalloc returns the same codes as nsp_attn_fwd for
    out-of-range sizes and scales (all refused before any CUDA call), and
    NSP_ERR_WORKSPACE for problems whose scheduler state exceeds its static
    scratch."""
    def noalloc(q_len, scale=0.088):
        return lib.nsp_attn_fwd_noalloc(A, A, A, A, 1, 0, q_len, 0, q_len, 8, 2, 128, scale, 1,
                                        nsp.NSP_BF16, A, nsp.NSP_BF16, None, None, None)

    def fwd(q_len):
        return lib.nsp_attn_fwd(A, A, A, A, 1, 0, q_len, 0, q_len, 8, 2, 128, 0.088, 1,
                                nsp.NSP_BF16, A, nsp.NSP_BF16, None, A, 1 << 40, None)
    for q_len in (1 << 31, (1 << 62) + 5):
        assert noalloc(q_len) == fwd(q_len) == nsp.NSP_ERR_UNSUPPORTED
    assert noalloc(-1) == fwd(-1) == nsp.NSP_ERR_INVALID
    assert noalloc(1 << 24) == nsp.NSP_ERR_WORKSPACE          # 16M tokens: beyond 1 MiB
    assert noalloc(1000, scale=0.0) == nsp.NSP_ERR_INVALID


def test_fwd_blocks_rejects_on_host(lib):
    """nsp_attn_fwd_blocks: block count, ranges inside [0, T), required and
    aligned outputs, and outputs that share bytes are refused before any
    launch."""
    T, Hq, d = 1000, 4, 128
    row = Hq * d * 4

    def call(blocks, accumulate=0, nb=None):
        arr = nsp._block_array(blocks)
        ws = nsp.nsp_attn_fwd_blocks_workspace_size(blocks, Hq, 2, d) if blocks else 0
        return lib.nsp_attn_fwd_blocks(A, A, A, A, 2, T, len(blocks) if nb is None else nb,
                                       C.cast(arr, C.c_void_p), Hq, 2, d, 0.088, 1, nsp.NSP_BF16,
                                       accumulate, A, max(ws, 1 << 20), None)

    class P:                       # a fake device pointer the binding passes through
        def __init__(self, addr):
            self.addr = addr

        def data_ptr(self):
            return self.addr

        def is_contiguous(self):
            return True
    out0, out1 = P(A), P(A + 200 * row)
    ok = [(0, 100, 0, 100, out0, None), (100, 100, 0, 200, out1, None)]
    assert nsp.nsp_attn_fwd_blocks_workspace_size(ok, Hq, 2, d) > 0
    assert call(ok, nb=0) == nsp.NSP_ERR_INVALID
    assert call(ok, nb=65) == nsp.NSP_ERR_INVALID
    assert call([(0, 100, 950, 100, out0, None)]) == nsp.NSP_ERR_INVALID      # keys past T
    assert call([(-1, 10, 0, 10, out0, None)]) == nsp.NSP_ERR_INVALID
    assert call([(0, 100, 0, 100, out0, None)], accumulate=1) == nsp.NSP_ERR_INVALID  # lse needed
    assert call([(0, 100, 0, 100, P(A + 4), None)]) == nsp.NSP_ERR_ALIGN
    overlapping = [(0, 100, 0, 100, out0, None), (100, 100, 0, 200, P(A + 50 * row), None)]
    assert call(overlapping) == nsp.NSP_ERR_INVALID


def test_bwd_blocks_rejects_on_host(lib):
    """nsp_attn_bwd_blocks: tensor-core shapes only (bf16, d = 64 or 128),
    q_start a multiple of 4, ranges inside [0, T), a workspace large enough;
    refused before any launch."""
    T = 1000

    def call(ranges, io=nsp.NSP_BF16, d=128, nr=None, ws=1 << 26):
        arr = nsp._range_array(ranges)
        return lib.nsp_attn_bwd_blocks(A, A, A, A, A, A, A, 2, T, len(ranges) if nr is None else nr,
                                       C.cast(arr, C.c_void_p), 8, 2, d, 0.088, 1, io, A, A, A,
                                       A, ws, None)
    ok = [(0, 500, 0, 500), (500, 500, 0, 1000)]
    assert nsp.nsp_attn_bwd_blocks_workspace_size(T, ok, 8, 2, 128) > 0
    assert call(ok, io=nsp.NSP_F32) == nsp.NSP_ERR_UNSUPPORTED
    assert call(ok, d=96) == nsp.NSP_ERR_UNSUPPORTED               # head dimension 64 or 128
    assert call([(2, 10, 0, 10)]) == nsp.NSP_ERR_UNSUPPORTED       # q_start not a multiple of 4
    assert call([(0, 10, 995, 10)]) == nsp.NSP_ERR_INVALID         # keys past T
    assert call(ok, nr=0) == nsp.NSP_ERR_INVALID
    assert call(ok, ws=16) == nsp.NSP_ERR_WORKSPACE


def test_wait_timeout_setter(lib):
    """The bound of device waits: a process-wide setting, default restored by
    a negative value; each call returns the previous bound."""
    prev = nsp.nsp_set_wait_timeout_cycles(777)
    try:
        assert nsp.nsp_set_wait_timeout_cycles(-5) == 777
        assert nsp.nsp_set_wait_timeout_cycles(prev) == 4000000000
    finally:
        nsp.nsp_set_wait_timeout_cycles(prev)


def _brute_cost(cu, qa, qb, ka, kb, causal):
    """Allowed pairs and 128 x 128 tiles holding one, by enumeration."""
    cu = np.asarray(cu, np.int64)
    doc = np.searchsorted(cu, np.arange(cu[-1]), side="right") - 1
    pairs, tiles = 0, set()
    for t in range(qa, qb):
        for j in range(ka, kb):
            if doc[t] == doc[j] and (not causal or j <= t):
                pairs += 1
                tiles.add(((t - qa) // 128, (j - ka) // 128))
    return pairs, len(tiles)


@pytest.mark.parametrize("causal", [True, False])
def test_attn_cost_matches_enumeration(lib, causal):
    r = np.random.default_rng(3)
    lens = [1, 300, 0, 45, 129, 7, 260, 2]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    ranges = [(0, T, 0, T), (100, 500, 0, 300), (300, 700, 350, T), (0, 128, 500, T)]
    for _ in range(4):
        a, b = sorted(r.integers(0, T + 1, 2))
        c, e = sorted(r.integers(0, T + 1, 2))
        ranges.append((int(a), int(b), int(c), int(e)))
    for qa, qb, ka, kb in ranges:
        c = nsp.nsp_attn_cost(cu, 32, 4, 128, causal, nsp.NSP_BF16, qa, qb - qa, ka, kb - ka)
        pairs, tiles = _brute_cost(cu, qa, qb, ka, kb, causal)
        assert c["pairs"] == pairs and c["tiles"] == tiles, (qa, qb, ka, kb)
        assert c["fwd_flop"] == 4 * 128 * 32 * pairs and c["bwd_flop"] == 10 * 128 * 32 * pairs
    whole = nsp.nsp_attn_cost(cu, 32, 4, 128, causal)
    assert whole["pairs"] == nsp.nsp_attn_pairs(cu, causal)
    # compulsory bytes of the whole stream, bf16: q/out/dout/dq 32 heads, k/v/dk/dv 4 heads
    row_q, row_kv, lse = T * 32 * 128 * 2, T * 4 * 128 * 2, T * 32 * 4
    assert whole["fwd_bytes"] == 2 * row_q + 2 * row_kv + lse
    assert whole["bwd_bytes"] == 4 * row_q + 4 * row_kv + lse
    with pytest.raises(nsp.NspError):
        nsp.nsp_attn_cost(cu, 32, 4, 128, causal, nsp.NSP_BF16, 10, T)   # past the stream


def test_batch_merge_and_headgroups_reject_on_host(lib):
    """nsp_lse_merge_batch, nsp_attn_fwd_headgroups, nsp_attn_bwd_headgroups:
    bad segment counts, head groups that do not divide Hq and misaligned
    pointers are refused before any launch."""
    outs = (C.c_void_p * 3)(A, A + 4096, A + 8192)
    lses = (C.c_void_p * 3)(A + 12288, A + 16384, A + 20480)
    dst = (C.c_void_p * 2)(A + 65536, A + 131072)

    def merge(nseg, counts, o=outs):
        c = (C.c_int32 * len(counts))(*counts)
        return lib.nsp_lse_merge_batch(nseg, C.cast(c, C.c_void_p), C.cast(o, C.c_void_p),
                                       C.cast(lses, C.c_void_p), 16, 4, 128,
                                       C.cast(dst, C.c_void_p), nsp.NSP_BF16, None, None)
    assert merge(0, [1]) == nsp.NSP_ERR_INVALID
    assert merge(2, [1, 0]) == nsp.NSP_ERR_INVALID
    assert merge(17, [1] * 17) == nsp.NSP_ERR_INVALID
    bad = (C.c_void_p * 3)(A, A + 4100, A + 8192)                # second partial misaligned
    assert merge(2, [1, 2], bad) == nsp.NSP_ERR_ALIGN
    a = fwd_args()
    ws = a["ws_bytes"]
    for P in (0, 3, 64):
        assert lib.nsp_attn_fwd_headgroups(a["q"], a["k"], a["v"], a["cu"], 3, 300, 32, 4, 128, P,
                                           0.088, 1, nsp.NSP_BF16, a["out"], nsp.NSP_BF16, None,
                                           a["ws"], ws, None) == nsp.NSP_ERR_INVALID
    wsb = nsp.nsp_attn_bwd_workspace_size(300, 32, 4, 128, nsp.NSP_BF16)
    ptrs = [A + 4096 * i for i in range(10)]
    assert lib.nsp_attn_bwd_headgroups(*ptrs[:7], 3, 300, 32, 4, 128, 5, 0.088, 1, nsp.NSP_BF16,
                                       *ptrs[7:10], A + (1 << 16), wsb, None) == nsp.NSP_ERR_INVALID


def test_plain_c_program_links_and_calls(lib, tmp_path):
    """The header is plain C and the library links into a C program with no
    torch or Python: a host-only call (nsp_attn_cost) from C gives the pairs
    an enumeration gives."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_nsp.c"
    src.write_text(r'''
#include <stdio.h>
#include "nsp.h"
int main(void) {
  const int32_t cu[4] = {0, 3, 3, 7};          /* lengths 3, 0, 4 */
  nsp_attn_cost_t c;
  int32_t st = nsp_attn_cost(cu, 3, 0, 7, 0, 7, 8, 2, 64, 1, NSP_BF16, &c);
  printf("%d %.0f %.0f %s\n", st, c.pairs, c.tiles, nsp_version());
  return st;
}
''')
    exe = tmp_path / "use_nsp"
    libdir = os.path.dirname(nsp.LIB_PATH)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-I", os.path.dirname(nsp.HEADER), str(src),
                        "-o", str(exe), f"-L{libdir}", "-l:libnsp.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    st, pairs, tiles, version = out.stdout.split(maxsplit=3)
    assert (int(st), int(pairs), int(tiles)) == (nsp.NSP_OK, 6 + 10, 1)
    assert "sm_103a" in version


def test_binding_arity_matches_header(lib):
    """Every ctypes signature in the binding has as many arguments as the
    header's declaration of that function (a shifted argument would pass
    the wrong pointer)."""
    import re
    with open(nsp.HEADER) as f:
        src = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    decls = {}
    for m in re.finditer(r"\b(nsp_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src):
        params = m.group(2).strip()
        decls[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    for name, (_, args) in nsp._SIGNATURES.items():
        assert name in decls, name
        assert len(args) == decls[name], (name, len(args), decls[name])
