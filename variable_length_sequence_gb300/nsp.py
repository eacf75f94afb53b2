"""Thin Python binding of ``libnsp.so`` (C ABI declared in ``include/nsp.h``).

Argument marshalling only: every function named like the C entry point takes
torch tensors (or raw integers) and passes their data pointers, sizes and the
current CUDA stream to the library.  All computation happens in the
library's kernels; there is no Python or CPU fallback, and loading fails
loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libnsp.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "nsp.h")

NSP_OK, NSP_ERR_INVALID, NSP_ERR_UNSUPPORTED, NSP_ERR_WORKSPACE = 0, 1, 2, 3
NSP_ERR_CUDA, NSP_ERR_TIMEOUT, NSP_ERR_ALIGN = 4, 5, 6
NSP_F32, NSP_BF16 = 0, 1

_lib: Optional[C.CDLL] = None

_vp, _i32, _i64, _f32, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t

_SIGNATURES = {
    "nsp_status_str": (C.c_char_p, [_i32]),
    "nsp_version": (C.c_char_p, []),
    "nsp_kernel_launches": (_i64, []),
    "nsp_set_wait_timeout_cycles": (_i64, [_i64]),
    "nsp_path_launches": (_i64, [_i32]),
    "nsp_attn_fwd_workspace_size": (_sz, [_i64, _i64, _i32, _i32, _i32]),
    "nsp_attn_fwd": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _i32, _i32, _i32,
                            _f32, _i32, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
    "nsp_attn_fwd_accumulate": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _i32,
                                       _i32, _i32, _f32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "nsp_attn_fwd_headgroups": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                       _f32, _i32, _i32, _vp, _i32, _vp, _vp, _sz, _vp]),
    "nsp_attn_fwd_blocks_workspace_size": (_sz, [_i32, _vp, _i32, _i32, _i32]),
    "nsp_attn_fwd_blocks": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _vp, _i32, _i32, _i32, _f32,
                                   _i32, _i32, _i32, _vp, _sz, _vp]),
    "nsp_attn_bwd_blocks_workspace_size": (_sz, [_i64, _i32, _vp, _i32, _i32, _i32]),
    "nsp_attn_bwd_blocks": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _vp, _i32,
                                   _i32, _i32, _f32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "nsp_attn_fwd_validate": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _i32,
                                     _i32, _i32, _i32, _i32, _vp, _i32, _vp, _sz]),
    "nsp_attn_fwd_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64, _i64, _i32,
                                    _i32, _i32, _f32, _i32, _i32, _vp, _i32, _vp, _vp, _vp]),
    "nsp_attn_bwd_workspace_size": (_sz, [_i64, _i32, _i32, _i32, _i32]),
    "nsp_attn_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                            _f32, _i32, _i32, _vp, _vp, _vp, _vp, _sz, _vp]),
    "nsp_attn_bwd_validate": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                     _i32, _i32, _i32, _vp, _vp, _vp, _vp, _sz]),
    "nsp_attn_bwd_headgroups": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                       _i32, _i32, _f32, _i32, _i32, _vp, _vp, _vp, _vp, _sz,
                                       _vp]),
    "nsp_attn_bwd_accumulate_workspace_size": (_sz, [_i64, _i64, _i32, _i32, _i32, _i32]),
    "nsp_attn_bwd_accumulate": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i64,
                                       _i64, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _vp, _vp,
                                       _vp, _sz, _vp]),
    "nsp_lse_merge": (_i32, [_vp, _vp, _i32, _i64, _i32, _i32, _vp, _i32, _vp, _vp]),
    "nsp_lse_merge_batch": (_i32, [_i32, _vp, _vp, _vp, _i64, _i32, _i32, _vp, _i32, _vp, _vp]),
    "nsp_lse_merge_validate": (_i32, [_vp, _vp, _i32, _i64, _i32, _i32, _vp, _i32, _vp]),
    "nsp_seq2head_permute": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _i32, _i32, _vp]),
    "nsp_seq2head_permute_validate": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _i32]),
    "nsp_seq2head_permute_groups": (_i32, [_vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _i32,
                                           _vp]),
    "nsp_status_query": (_i32, [_vp, _vp]),
    "nsp_attn_bwd_ds_cache_size": (_sz, [_vp, _i32, _i32, _i32]),
    "nsp_attn_bwd_blocks_ds_cache_size": (_sz, [_vp, _i32, _i32, _vp, _i32, _i32]),
    "nsp_bwd_ds_cache_used": (_i32, [_vp, C.POINTER(C.c_int32), _vp]),
    "nsp_attn_pairs": (_i32, [_vp, _i32, _i32, C.POINTER(C.c_double)]),
    "nsp_attn_cost": (_i32, [_vp, _i32, _i64, _i64, _i64, _i64, _i32, _i32, _i32, _i32, _i32,
                             _vp]),
}


class Block(C.Structure):
    """nsp_block_t: one (query range, key range) block of a batched forward."""
    _fields_ = [("q_start", C.c_int64), ("q_len", C.c_int64), ("kv_start", C.c_int64),
                ("kv_len", C.c_int64), ("out", C.c_void_p), ("lse", C.c_void_p)]


class Range(C.Structure):
    """nsp_range_t: one (query range, key range) block of a batched backward."""
    _fields_ = [("q_start", C.c_int64), ("q_len", C.c_int64), ("kv_start", C.c_int64),
                ("kv_len", C.c_int64)]


class AttnCost(C.Structure):
    """nsp_attn_cost_t."""
    _fields_ = [(n, C.c_double) for n in ("pairs", "fwd_flop", "bwd_flop", "tiles",
                                           "fwd_bytes", "bwd_bytes")]


class NspError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_str(status)} ({status})")


def header_functions() -> list:
    """Names of the functions declared in include/nsp.h."""
    with open(HEADER) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nsp_[a-z0-9_]+)\s*\(", src)))


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libnsp.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = C.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load().nsp_status_str(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libnsp takes contiguous tensors only")
    return t.data_ptr() or None


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return NSP_BF16
    if t.dtype == torch.float32:
        return NSP_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(fn: str, st: int) -> int:
    if st != NSP_OK:
        raise NspError(fn, st)
    return st


# ----------------------------------------------------------------------------- raw entry points

def nsp_attn_fwd_workspace_size(q_len: int, kv_len: int, Hq: int, Hkv: int, d: int) -> int:
    return int(load().nsp_attn_fwd_workspace_size(q_len, kv_len, Hq, Hkv, d))


def _block_array(blocks):
    """blocks: sequence of (q_start, q_len, kv_start, kv_len, out, lse)."""
    arr = (Block * len(blocks))()
    for i, (qs, ql, ks, kl, out, lse) in enumerate(blocks):
        arr[i] = Block(int(qs), int(ql), int(ks), int(kl), _ptr(out), _ptr(lse))
    return arr


def nsp_attn_fwd_blocks_workspace_size(blocks, Hq: int, Hkv: int, d: int) -> int:
    arr = _block_array(blocks)
    return int(load().nsp_attn_fwd_blocks_workspace_size(len(blocks), C.cast(arr, C.c_void_p),
                                                         int(Hq), int(Hkv), int(d)))


def nsp_attn_fwd_blocks(q, k, v, cu_seqlens, ndoc, T, blocks, Hq, Hkv, d, scale, causal,
                        accumulate, workspace, stream=None) -> int:
    arr = _block_array(blocks)
    st = load().nsp_attn_fwd_blocks(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(ndoc),
                                    int(T), len(blocks), C.cast(arr, C.c_void_p), int(Hq),
                                    int(Hkv), int(d), float(scale), int(bool(causal)), _dtype(q),
                                    int(bool(accumulate)), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    return _check("nsp_attn_fwd_blocks", st)


def _range_array(ranges):
    arr = (Range * len(ranges))()
    for i, (qs, ql, ks, kl) in enumerate(ranges):
        arr[i] = Range(int(qs), int(ql), int(ks), int(kl))
    return arr


def nsp_attn_bwd_blocks_workspace_size(T: int, ranges, Hq: int, Hkv: int, d: int) -> int:
    arr = _range_array(ranges)
    return int(load().nsp_attn_bwd_blocks_workspace_size(int(T), len(ranges),
                                                         C.cast(arr, C.c_void_p), int(Hq),
                                                         int(Hkv), int(d)))


def nsp_attn_bwd_blocks(q, k, v, out, dout, lse, cu_seqlens, ndoc, T, ranges, Hq, Hkv, d, scale,
                        causal, dq_acc, dk_acc, dv_acc, workspace, stream=None) -> int:
    arr = _range_array(ranges)
    st = load().nsp_attn_bwd_blocks(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                    _ptr(cu_seqlens), int(ndoc), int(T), len(ranges),
                                    C.cast(arr, C.c_void_p), int(Hq), int(Hkv), int(d),
                                    float(scale), int(bool(causal)), _dtype(q), _ptr(dq_acc),
                                    _ptr(dk_acc), _ptr(dv_acc), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    return _check("nsp_attn_bwd_blocks", st)


def nsp_attn_bwd_workspace_size(T: int, Hq: int, Hkv: int, d: int, io_dtype: int = NSP_BF16) -> int:
    return int(load().nsp_attn_bwd_workspace_size(T, Hq, Hkv, d, int(io_dtype)))


def nsp_attn_fwd(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start, kv_len, Hq, Hkv, d,
                 scale, causal, out, lse, workspace, stream=None) -> int:
    st = load().nsp_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(ndoc),
                             int(q_start), int(q_len), int(kv_start), int(kv_len), int(Hq),
                             int(Hkv), int(d), float(scale), int(bool(causal)), _dtype(q),
                             _ptr(out), _dtype(out), _ptr(lse), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    return _check("nsp_attn_fwd", st)


def nsp_attn_fwd_accumulate(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start, kv_len, Hq,
                            Hkv, d, scale, causal, acc, lse_acc, workspace, stream=None) -> int:
    st = load().nsp_attn_fwd_accumulate(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(ndoc),
                                        int(q_start), int(q_len), int(kv_start), int(kv_len),
                                        int(Hq), int(Hkv), int(d), float(scale),
                                        int(bool(causal)), _dtype(q), _ptr(acc), _ptr(lse_acc),
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    return _check("nsp_attn_fwd_accumulate", st)


def nsp_attn_fwd_headgroups(q, k, v, cu_seqlens, ndoc, T, Hq, Hkv, d, P, scale, causal, out, lse,
                            workspace, stream=None) -> int:
    st = load().nsp_attn_fwd_headgroups(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(ndoc),
                                        int(T), int(Hq), int(Hkv), int(d), int(P), float(scale),
                                        int(bool(causal)), _dtype(q), _ptr(out), _dtype(out),
                                        _ptr(lse), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    return _check("nsp_attn_fwd_headgroups", st)


def nsp_attn_fwd_noalloc(q, k, v, cu_seqlens, ndoc, q_start, q_len, kv_start, kv_len, Hq, Hkv,
                         d, scale, causal, out, lse, device_status=None, stream=None) -> int:
    """nsp_attn_fwd for callers that cannot allocate: no workspace argument
    (the library's static device scratch is used; see include/nsp.h)."""
    st = load().nsp_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), int(ndoc),
                                     int(q_start), int(q_len), int(kv_start), int(kv_len),
                                     int(Hq), int(Hkv), int(d), float(scale), int(bool(causal)),
                                     _dtype(q), _ptr(out), _dtype(out), _ptr(lse),
                                     _ptr(device_status), _stream(stream))
    return _check("nsp_attn_fwd_noalloc", st)


def nsp_attn_bwd(q, k, v, out, dout, lse, cu_seqlens, ndoc, T, Hq, Hkv, d, scale, causal,
                 dq, dk, dv, workspace, stream=None) -> int:
    st = load().nsp_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                             _ptr(cu_seqlens), int(ndoc), int(T), int(Hq), int(Hkv), int(d),
                             float(scale), int(bool(causal)), _dtype(q), _ptr(dq), _ptr(dk),
                             _ptr(dv), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    return _check("nsp_attn_bwd", st)


def nsp_attn_bwd_headgroups(q, k, v, out, dout, lse, cu_seqlens, ndoc, T, Hq, Hkv, d, P, scale,
                            causal, dq, dk, dv, workspace, stream=None) -> int:
    st = load().nsp_attn_bwd_headgroups(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout),
                                        _ptr(lse), _ptr(cu_seqlens), int(ndoc), int(T), int(Hq),
                                        int(Hkv), int(d), int(P), float(scale),
                                        int(bool(causal)), _dtype(q), _ptr(dq), _ptr(dk),
                                        _ptr(dv), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    return _check("nsp_attn_bwd_headgroups", st)


def nsp_attn_bwd_accumulate_workspace_size(q_len: int, kv_len: int, Hq: int, Hkv: int, d: int,
                                           io_dtype: int = NSP_BF16) -> int:
    return int(load().nsp_attn_bwd_accumulate_workspace_size(q_len, kv_len, Hq, Hkv, d,
                                                             int(io_dtype)))


def nsp_attn_bwd_accumulate(q, k, v, out, dout, lse, cu_seqlens, ndoc, q_start, q_len, kv_start,
                            kv_len, Hq, Hkv, d, scale, causal, dq_acc, dk_acc, dv_acc, workspace,
                            stream=None) -> int:
    st = load().nsp_attn_bwd_accumulate(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(cu_seqlens),
        int(ndoc), int(q_start), int(q_len), int(kv_start), int(kv_len), int(Hq), int(Hkv),
        int(d), float(scale), int(bool(causal)), _dtype(q), _ptr(dq_acc), _ptr(dk_acc),
        _ptr(dv_acc), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream))
    return _check("nsp_attn_bwd_accumulate", st)


def nsp_lse_merge(outs: Sequence[torch.Tensor], lses: Sequence[torch.Tensor], out, lse,
                  stream=None) -> int:
    n = len(outs)
    T, H, d = outs[0].shape
    po = (C.c_void_p * n)(*[_ptr(o) for o in outs])
    pl = (C.c_void_p * n)(*[_ptr(l) for l in lses])
    st = load().nsp_lse_merge(C.cast(po, C.c_void_p), C.cast(pl, C.c_void_p), n, T, H, d,
                              _ptr(out), _dtype(out), _ptr(lse), _stream(stream))
    return _check("nsp_lse_merge", st)


def nsp_lse_merge_batch(segments, outs_merged, lses_merged=None, stream=None) -> int:
    """segments: list of (outs, lses) partial lists; outs_merged / lses_merged:
    one tensor per segment (lses_merged entries may be None)."""
    nseg = len(segments)
    if len({o.dtype for o in outs_merged}) != 1:
        raise ValueError("nsp_lse_merge_batch: every merged output must have the same dtype")
    counts = (C.c_int32 * nseg)(*[len(o) for o, _ in segments])
    po = [_ptr(o) for os_, _ in segments for o in os_]
    pl = [_ptr(l) for _, ls in segments for l in ls]
    T, H, d = segments[0][0][0].shape
    a_o = (C.c_void_p * len(po))(*po)
    a_l = (C.c_void_p * len(pl))(*pl)
    a_d = (C.c_void_p * nseg)(*[_ptr(o) for o in outs_merged])
    a_dl = None
    if lses_merged is not None:
        a_dl = C.cast((C.c_void_p * nseg)(*[_ptr(l) if l is not None else None
                                             for l in lses_merged]), C.c_void_p)
    st = load().nsp_lse_merge_batch(nseg, C.cast(counts, C.c_void_p), C.cast(a_o, C.c_void_p),
                                    C.cast(a_l, C.c_void_p), T, H, d, C.cast(a_d, C.c_void_p),
                                    _dtype(outs_merged[0]), a_dl, _stream(stream))
    return _check("nsp_lse_merge_batch", st)


def nsp_seq2head_permute(inp, out, T, H, d, P, inverse=False, stream=None) -> int:
    st = load().nsp_seq2head_permute(_ptr(inp), _ptr(out), int(T), int(H), int(d), int(P),
                                     inp.element_size(), int(bool(inverse)), _stream(stream))
    return _check("nsp_seq2head_permute", st)


def nsp_seq2head_permute_groups(inp, out, B, L, H, d, K, inverse=False, stream=None) -> int:
    st = load().nsp_seq2head_permute_groups(_ptr(inp), _ptr(out), int(B), int(L), int(H), int(d),
                                            int(K), inp.element_size(), int(bool(inverse)),
                                            _stream(stream))
    return _check("nsp_seq2head_permute_groups", st)


def nsp_kernel_launches() -> int:
    return int(load().nsp_kernel_launches())


def nsp_path_launches(tensor_core: bool) -> int:
    """Attention kernels launched so far on the tensor-core (True) or the
    CUDA-core (False) path."""
    return int(load().nsp_path_launches(int(bool(tensor_core))))


def nsp_set_wait_timeout_cycles(cycles: int) -> int:
    """Bound of the kernels' device waits in GPU cycles (< 0: the default);
    returns the previous bound."""
    return int(load().nsp_set_wait_timeout_cycles(int(cycles)))


def nsp_status_query(workspace, stream=None) -> int:
    return int(load().nsp_status_query(_ptr(workspace), _stream(stream)))


def nsp_attn_bwd_ds_cache_size(cu_seqlens_host, Hq, causal=True) -> int:
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    return int(load().nsp_attn_bwd_ds_cache_size(cu.ctypes.data, len(cu) - 1, int(Hq),
                                                 int(bool(causal))))


def nsp_attn_bwd_blocks_ds_cache_size(cu_seqlens_host, ranges, Hq, causal=True) -> int:
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    arr = _range_array(ranges)
    return int(load().nsp_attn_bwd_blocks_ds_cache_size(cu.ctypes.data, len(cu) - 1, len(ranges),
                                                        C.cast(arr, C.c_void_p), int(Hq),
                                                        int(bool(causal))))


def nsp_bwd_ds_cache_used(workspace, stream=None) -> bool:
    used = C.c_int32(0)
    _check("nsp_bwd_ds_cache_used",
           load().nsp_bwd_ds_cache_used(_ptr(workspace), C.byref(used), _stream(stream)))
    return bool(used.value)


def bwd_workspace(T, Hq, Hkv, d, device, io_dtype=NSP_BF16, ds_cache_bytes=0):
    """A backward workspace; ds_cache_bytes > 0 appends a dS cache of that
    size (nsp_attn_bwd_ds_cache_size gives the size that holds every tile)."""
    base = nsp_attn_bwd_workspace_size(T, Hq, Hkv, d, io_dtype)
    if ds_cache_bytes > 0:
        base = (base + 1023) // 1024 * 1024 + int(ds_cache_bytes)
    return torch.empty(base, dtype=torch.uint8, device=device)


def nsp_attn_pairs(cu_seqlens_host, causal=True) -> float:
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    out = C.c_double(0.0)
    st = load().nsp_attn_pairs(cu.ctypes.data, len(cu) - 1, int(bool(causal)), C.byref(out))
    _check("nsp_attn_pairs", st)
    return out.value


def nsp_attn_cost(cu_seqlens_host, Hq, Hkv, d, causal=True, io_dtype=NSP_BF16, q_start=0,
                  q_len=None, kv_start=0, kv_len=None) -> dict:
    """Cost of one attention call (whole stream by default) as a dict."""
    import numpy as np
    cu = np.ascontiguousarray(np.asarray(cu_seqlens_host, dtype=np.int32))
    T = int(cu[-1])
    q_len = T - q_start if q_len is None else q_len
    kv_len = T - kv_start if kv_len is None else kv_len
    c = AttnCost()
    st = load().nsp_attn_cost(cu.ctypes.data, len(cu) - 1, int(q_start), int(q_len),
                              int(kv_start), int(kv_len), int(Hq), int(Hkv), int(d),
                              int(bool(causal)), int(io_dtype), C.cast(C.pointer(c), C.c_void_p))
    _check("nsp_attn_cost", st)
    return {n: getattr(c, n) for n, _ in AttnCost._fields_}


# ----------------------------------------------------------------------------- conveniences

def attn_fwd(q, k, v, cu_seqlens, scale=None, causal=True, out_dtype=None, q_start=0,
             kv_start=0, workspace=None, stream=None):
    """Allocate out/lse/workspace with torch and call nsp_attn_fwd.

    q [q_len, Hq, d], k/v [kv_len, Hkv, d] on the GPU, cu_seqlens int32 on the GPU.
    """
    q_len, Hq, d = q.shape
    kv_len, Hkv, _ = k.shape
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty((q_len, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, q_len), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(nsp_attn_fwd_workspace_size(q_len, kv_len, Hq, Hkv, d),
                                dtype=torch.uint8, device=q.device)
    nsp_attn_fwd(q, k, v, cu_seqlens, cu_seqlens.numel() - 1, q_start, q_len, kv_start, kv_len,
                 Hq, Hkv, d, scale, causal, out, lse, workspace, stream)
    return out, lse


def attn_fwd_headgroups(qg, k, v, cu_seqlens, scale=None, causal=True, out_dtype=None,
                        workspace=None, stream=None):
    """Forward on q in the head-group-major layout qg [P, T, Hq/P, d]; returns
    out in the same layout and lse [Hq, T]."""
    P, T, hpg, d = qg.shape
    Hq, Hkv = P * hpg, k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    out = torch.empty(qg.shape, dtype=out_dtype or qg.dtype, device=qg.device)
    lse = torch.empty((Hq, T), dtype=torch.float32, device=qg.device)
    if workspace is None:
        workspace = torch.empty(nsp_attn_fwd_workspace_size(T, T, Hq, Hkv, d), dtype=torch.uint8,
                                device=qg.device)
    nsp_attn_fwd_headgroups(qg, k, v, cu_seqlens, cu_seqlens.numel() - 1, T, Hq, Hkv, d, P, scale,
                            causal, out, lse, workspace, stream)
    return out, lse


def attn_bwd_headgroups(qg, k, v, outg, doutg, lse, cu_seqlens, scale=None, causal=True,
                        workspace=None, stream=None):
    """Backward with q, out, dout (and the returned dq) in [P, T, Hq/P, d]."""
    P, T, hpg, d = qg.shape
    Hq, Hkv = P * hpg, k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(qg), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(nsp_attn_bwd_workspace_size(T, Hq, Hkv, d, _dtype(qg)),
                                dtype=torch.uint8, device=qg.device)
    nsp_attn_bwd_headgroups(qg, k, v, outg, doutg, lse, cu_seqlens, cu_seqlens.numel() - 1, T,
                            Hq, Hkv, d, P, scale, causal, dq, dk, dv, workspace, stream)
    return dq, dk, dv


def ring_accumulate_init(q_len, Hq, d, device):
    """A fresh ring accumulator: acc = 0 [q_len, Hq, d] float32, lse_acc = -inf [Hq, q_len]."""
    acc = torch.zeros((q_len, Hq, d), dtype=torch.float32, device=device)
    lse = torch.full((Hq, q_len), float("-inf"), dtype=torch.float32, device=device)
    return acc, lse


def attn_fwd_accumulate(q, k, v, cu_seqlens, acc, lse_acc, scale=None, causal=True, q_start=0,
                        kv_start=0, workspace=None, stream=None):
    """Merge the block (q rows from q_start) x (keys from kv_start) into acc/lse_acc in place."""
    q_len, Hq, d = q.shape
    kv_len, Hkv, _ = k.shape
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nsp_attn_fwd_workspace_size(q_len, kv_len, Hq, Hkv, d),
                                dtype=torch.uint8, device=q.device)
    nsp_attn_fwd_accumulate(q, k, v, cu_seqlens, cu_seqlens.numel() - 1, q_start, q_len,
                            kv_start, kv_len, Hq, Hkv, d, scale, causal, acc, lse_acc,
                            workspace, stream)
    return acc, lse_acc


def attn_fwd_blocks(q, k, v, cu_seqlens, blocks, scale=None, causal=True, accumulate=False,
                    workspace=None, stream=None):
    """Batched blocks of the whole stream q [T, Hq, d], k/v [T, Hkv, d]:
    blocks = [(q_start, q_len, kv_start, kv_len, out, lse), ...] with float32
    out [q_len, Hq, d] and lse [Hq, q_len] written (accumulate=False) or
    merged into (accumulate=True)."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nsp_attn_fwd_blocks_workspace_size(blocks, Hq, Hkv, d),
                                dtype=torch.uint8, device=q.device)
    nsp_attn_fwd_blocks(q, k, v, cu_seqlens, cu_seqlens.numel() - 1, T, blocks, Hq, Hkv, d, scale,
                        causal, accumulate, workspace, stream)


def attn_bwd_blocks(q, k, v, out, dout, lse, cu_seqlens, ranges, dq_acc, dk_acc, dv_acc,
                    scale=None, causal=True, workspace=None, stream=None, ds_cache_bytes=0):
    """Add the backward contributions of blocks [(q_start, q_len, kv_start,
    kv_len), ...] of the whole stream into float32 dq_acc [T, Hq, d] and
    dk_acc / dv_acc [T, Hkv, d] (lse [Hq, T], the rows' final lse).  A new
    workspace gets ds_cache_bytes of dS cache appended."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        n = nsp_attn_bwd_blocks_workspace_size(T, ranges, Hq, Hkv, d)
        if ds_cache_bytes > 0:
            n = (n + 1023) // 1024 * 1024 + int(ds_cache_bytes)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    nsp_attn_bwd_blocks(q, k, v, out, dout, lse, cu_seqlens, cu_seqlens.numel() - 1, T, ranges,
                        Hq, Hkv, d, scale, causal, dq_acc, dk_acc, dv_acc, workspace, stream)


def attn_bwd(q, k, v, out, dout, lse, cu_seqlens, scale=None, causal=True, workspace=None,
             stream=None):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if workspace is None:
        workspace = torch.empty(nsp_attn_bwd_workspace_size(T, Hq, Hkv, d, _dtype(q)),
                                dtype=torch.uint8, device=q.device)
    nsp_attn_bwd(q, k, v, out, dout, lse, cu_seqlens, cu_seqlens.numel() - 1, T, Hq, Hkv, d,
                 scale, causal, dq, dk, dv, workspace, stream)
    return dq, dk, dv


def attn_bwd_accumulate(q, k, v, out, dout, lse, cu_seqlens, dq_acc, dk_acc, dv_acc, scale=None,
                        causal=True, q_start=0, kv_start=0, workspace=None, stream=None):
    """Add the block (q rows from q_start) x (keys from kv_start) into the
    float32 gradient accumulators in place."""
    q_len, Hq, d = q.shape
    kv_len, Hkv, _ = k.shape
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(nsp_attn_bwd_accumulate_workspace_size(q_len, kv_len, Hq, Hkv, d,
                                                                       _dtype(q)),
                                dtype=torch.uint8, device=q.device)
    nsp_attn_bwd_accumulate(q, k, v, out, dout, lse, cu_seqlens, cu_seqlens.numel() - 1, q_start,
                            q_len, kv_start, kv_len, Hq, Hkv, d, scale, causal, dq_acc, dk_acc,
                            dv_acc, workspace, stream)
    return dq_acc, dk_acc, dv_acc


def lse_merge(outs, lses, out_dtype=torch.float32, stream=None):
    T, H, d = outs[0].shape
    out = torch.empty((T, H, d), dtype=out_dtype, device=outs[0].device)
    lse = torch.empty((H, T), dtype=torch.float32, device=outs[0].device)
    nsp_lse_merge(outs, lses, out, lse, stream)
    return out, lse


def seq2head(x, P, stream=None):
    T, H, d = x.shape
    out = torch.empty((P, T, H // P, d), dtype=x.dtype, device=x.device)
    nsp_seq2head_permute(x, out, T, H, d, P, False, stream)
    return out


def seq2head_groups(x, B, K, stream=None):
    """[B L, H, d] -> [B, K, L, H / K, d]: the receive side of B independent
    K-way (batch-aware subgroup) all-to-alls."""
    BL, H, d = x.shape
    L = BL // B
    out = torch.empty((B, K, L, H // K, d), dtype=x.dtype, device=x.device)
    nsp_seq2head_permute_groups(x, out, B, L, H, d, K, False, stream)
    return out


def head2seq_groups(y, stream=None):
    B, K, L, h, d = y.shape
    out = torch.empty((B * L, K * h, d), dtype=y.dtype, device=y.device)
    nsp_seq2head_permute_groups(y, out, B, L, K * h, d, K, True, stream)
    return out


def head2seq(y, stream=None):
    P, T, h, d = y.shape
    out = torch.empty((T, P * h, d), dtype=y.dtype, device=y.device)
    nsp_seq2head_permute(y, out, T, P * h, d, P, True, stream)
    return out
