"""Float64 CPU oracle for split-KV decode attention (ctypes wrapper of oracle.c).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package. It shares no code with
the CUDA path and never calls it.

The arithmetic lives in ``oracle.c`` (plain C, float64); this module only
compiles it with gcc, marshals arrays and returns numpy float64 results.
Inputs are the raw bit patterns the GPU path also reads: bf16 tensors are
passed as their 16-bit words, fp8 KV as its bytes, and the C side converts
them exactly to float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math: IEEE order)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(
                ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                 "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


class OracleProblem(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim_qk", "head_dim_v", "is_mla",
        "ckv_dim", "kpe_dim", "paged", "page_size", "cache_len", "max_pages_per_seq",
        "num_pages", "kv_fp8", "sparse_block_size", "max_sparse_blocks", "q_len",
        "sparse_batch", "sparse_heads", "kv_groups", "fp8_mma")]


class OracleInputs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_pe", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("kv_num_blks", ctypes.c_void_p), ("kv_idx", ctypes.c_void_p), ("scale", ctypes.c_double),
        ("k_scale_shift", ctypes.c_void_p), ("v_scale_shift", ctypes.c_void_p),
        ("kv_full_num_blks", ctypes.c_void_p), ("kv_full_idx", ctypes.c_void_p),
        ("softcap", ctypes.c_double),
        ("spec_mask", ctypes.c_void_p),
        ("mask_sink", ctypes.c_void_p), ("mask_window", ctypes.c_void_p),
        ("alibi_slopes", ctypes.c_void_p),
        ("p8_bound", ctypes.c_void_p),
    ]


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_double.restype = ctypes.c_double
        L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.oracle_f16_round.restype = ctypes.c_double
        L.oracle_f16_round.argtypes = [ctypes.c_double]
        L.oracle_softmax_attend.restype = None
        L.oracle_softmax_attend.argtypes = [ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_merge.restype = None
        L.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_merge_rows.restype = None
        L.oracle_merge_rows.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_decode.restype = ctypes.c_int
        L.oracle_decode.argtypes = [ctypes.POINTER(OracleProblem), ctypes.POINTER(OracleInputs),
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        L.oracle_split.restype = ctypes.c_int
        L.oracle_split.argtypes = [ctypes.POINTER(OracleProblem), ctypes.POINTER(OracleInputs),
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int]
        _lib = L
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


# ---------------------------------------------------------------- marshalling

def _host(t):
    """A contiguous CPU tensor (or None)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(np.ascontiguousarray(t))
    return t.detach().to("cpu").contiguous()


def _bits(t):
    """bf16 -> its uint16 words; fp8 -> its bytes; int32/float32 unchanged."""
    t = _host(t)
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8)
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(bits)


def e4m3_to_double(byte: int) -> float:
    return lib().oracle_e4m3_to_double(byte)


def e4m3_encode(x: float) -> int:
    """float32 -> e4m3fn code byte, round to nearest even, saturating to +-448."""
    return lib().oracle_e4m3_encode(float(x))


def f16_round(x: float) -> float:
    """The nearest binary16 value (ties to even), as a float."""
    return lib().oracle_f16_round(float(x))


def softmax_attend(s, v):
    """Core over an explicit list: s [n] float64, v [n][dv] float64 -> (out [dv], lse)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    n = s.shape[0]
    dv = v.shape[1] if v.ndim == 2 else 0
    out = np.zeros(max(dv, 1), dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().oracle_softmax_attend(n, s.ctypes.data, v.ctypes.data if n else None, dv,
                                out.ctypes.data, lse.ctypes.data)
    return out[:dv], float(lse[0])


def merge(o, lse):
    """LSE merge. o [..., S, dv], lse [..., S] (float64-convertible) -> (out [..., dv], lse [...])."""
    o = np.ascontiguousarray(np.asarray(o, dtype=np.float64))
    lse = np.ascontiguousarray(np.asarray(lse, dtype=np.float64))
    S, dv = o.shape[-2], o.shape[-1]
    lead = o.shape[:-2]
    rows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (dv,), dtype=np.float64)
    lo = np.zeros(lead, dtype=np.float64)
    lib().oracle_merge_rows(rows, S, dv, o.ctypes.data, lse.ctypes.data, out.ctypes.data,
                            lo.ctypes.data)
    return out, lo


class _Prepared:
    """Keeps the marshalled host tensors alive while the C call runs."""

    def __init__(self, prob: dict, tensors: dict, scale: float, softcap: float = 0.0):
        p = OracleProblem()
        for name, _ in OracleProblem._fields_:
            setattr(p, name, int(prob.get(name, 0)))
        self.problem = p
        self.keep = {k: _bits(v) for k, v in tensors.items()}
        for k in ("block_table", "seq_lens", "kv_num_blks", "kv_idx", "k_scale_shift", "v_scale_shift",
                  "kv_full_num_blks", "kv_full_idx", "spec_mask", "mask_sink", "mask_window"):
            if self.keep.get(k) is not None:
                self.keep[k] = self.keep[k].to(torch.int32).contiguous()
        for k in ("k_scale", "v_scale", "alibi_slopes"):
            if self.keep.get(k) is not None:
                self.keep[k] = self.keep[k].to(torch.float32).contiguous()
        i = OracleInputs()
        for k in ("q", "q_pe", "k", "v", "k_scale", "v_scale", "block_table", "seq_lens",
                  "kv_num_blks", "kv_idx", "k_scale_shift", "v_scale_shift", "kv_full_num_blks",
                  "kv_full_idx", "spec_mask", "mask_sink", "mask_window", "alibi_slopes"):
            setattr(i, k, _ptr(self.keep.get(k)))
        i.scale = float(scale)
        i.softcap = float(softcap)
        self.inputs = i


def problem_from(work) -> dict:
    """Oracle problem dict from a workload description (see the package's workloads module)."""
    w = work
    return dict(
        batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
        head_dim_qk=w.head_dim_qk, head_dim_v=w.head_dim_v, is_mla=int(w.is_mla),
        ckv_dim=w.ckv_dim, kpe_dim=w.kpe_dim, paged=int(w.paged), page_size=w.page_size,
        cache_len=w.cache_len, max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages,
        kv_fp8=3 if getattr(w, "kv_int4_groups", 0) else
        ((2 if getattr(w, "kv_token_scale", False) else 1) if w.kv_fp8 else 0),
        kv_groups=getattr(w, "kv_int4_groups", 0),
        sparse_block_size=w.sparse_block_size,
        max_sparse_blocks=w.max_sparse_blocks, q_len=getattr(w, "q_len", 1),
        sparse_batch=getattr(w, "sparse_batch", 0), sparse_heads=getattr(w, "sparse_heads", 0),
        fp8_mma=int(getattr(w, "fp8_mma", False)))


def decode(prob: dict, tensors: dict, scale: float, num_threads: int | None = None,
           softcap: float = 0.0):
    """Full decode attention -> (out [B][HQ][Dv], lse [B][HQ]) in float64; with
    several query tokens (q_len = Q > 1) out [B][HQ][Q][Dv] and lse [B][HQ][Q]."""
    prep = _Prepared(prob, tensors, scale, softcap)
    p = prep.problem
    lead = (p.batch, p.num_q_heads) + ((p.q_len,) if p.q_len > 1 else ())
    out = np.zeros(lead + (p.head_dim_v,), dtype=np.float64)
    lse = np.zeros(lead, dtype=np.float64)
    st = lib().oracle_decode(ctypes.byref(p), ctypes.byref(prep.inputs), out.ctypes.data,
                             lse.ctypes.data, num_threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle_decode failed with status {st}")
    return out, lse


def decode_p8_bound(prob: dict, tensors: dict, scale: float, num_threads: int | None = None,
                    softcap: float = 0.0):
    """decode() of an fp8_mma problem, with the rounding bound of its weights:
    (out, lse, bound), bound shaped like out."""
    prep = _Prepared(prob, tensors, scale, softcap)
    p = prep.problem
    lead = (p.batch, p.num_q_heads) + ((p.q_len,) if p.q_len > 1 else ())
    out = np.zeros(lead + (p.head_dim_v,), dtype=np.float64)
    lse = np.zeros(lead, dtype=np.float64)
    bound = np.zeros(lead + (p.head_dim_v,), dtype=np.float64)
    prep.inputs.p8_bound = bound.ctypes.data
    st = lib().oracle_decode(ctypes.byref(p), ctypes.byref(prep.inputs), out.ctypes.data,
                             lse.ctypes.data, num_threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle_decode failed with status {st}")
    return out, lse, bound


def split(prob: dict, tensors: dict, scale: float, chunk_bounds, num_threads: int | None = None):
    """Per-chunk results over list-index boundaries -> (o [B][HQ][C][Dv], lse [B][HQ][C]);
    with several query tokens (q_len = Q > 1) o [B][HQ][Q][C][Dv], lse [B][HQ][Q][C]."""
    prep = _Prepared(prob, tensors, scale)
    p = prep.problem
    bounds = np.ascontiguousarray(np.asarray(chunk_bounds, dtype=np.int64))
    C = bounds.shape[0] - 1
    lead = (p.batch, p.num_q_heads) + ((p.q_len,) if p.q_len > 1 else ())
    o = np.zeros(lead + (C, p.head_dim_v), dtype=np.float64)
    lse = np.zeros(lead + (C,), dtype=np.float64)
    st = lib().oracle_split(ctypes.byref(p), ctypes.byref(prep.inputs), C, bounds.ctypes.data,
                            o.ctypes.data, lse.ctypes.data, num_threads or default_threads())
    if st != 0:
        raise ValueError(f"oracle_split failed with status {st}")
    return o, lse
