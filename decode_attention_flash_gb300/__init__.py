"""GB300 split-KV decode attention: Python binding of libdecode_attn.so.

The functions here carry the names of the C ABI in ``include/decode_attn.h``
and only marshal arguments (torch tensors -> device pointers, dicts -> C
structs, status codes -> exceptions). Every step of the computation runs in
the library's CUDA kernels; there is no fallback: importing this package
fails loudly when the compiled library is missing.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

from . import _build

__all__ = [
    "DecodeAttnError", "Problem", "Args", "PlanInfo", "load", "decode_attn_create",
    "decode_attn_plan", "decode_attn_plan_ex", "decode_attn_get_plan", "decode_attn_plan_info",
    "decode_attn_run", "decode_attn_run_noalloc", "decode_attn_merge", "decode_attn_get_error",
    "decode_attn_get_error_noalloc", "decode_attn_destroy",
    "decode_attn_status_string", "DecodeAttention", "DA_KV_CONTIGUOUS", "DA_KV_PAGED",
    "DA_DTYPE_BF16", "DA_DTYPE_FP8_E4M3", "DA_DTYPE_FP8_E4M3_TOKEN_SCALE", "DA_DTYPE_INT4_GROUPS",
]

DA_OK, DA_ERR_INVALID_ARG, DA_ERR_UNSUPPORTED, DA_ERR_CUDA = 0, 1, 2, 3
DA_ERR_WORKSPACE, DA_ERR_NOT_PLANNED, DA_ERR_DEVICE = 4, 5, 6
DA_KV_CONTIGUOUS, DA_KV_PAGED = 0, 1
DA_DTYPE_BF16, DA_DTYPE_FP8_E4M3, DA_DTYPE_FP8_E4M3_TOKEN_SCALE, DA_DTYPE_INT4_GROUPS = 0, 1, 2, 3
DA_DEVERR_PAGE_INDEX, DA_DEVERR_SPARSE_INDEX, DA_DEVERR_SEQ_LEN, DA_DEVERR_TIMEOUT = 1, 2, 4, 8


class DecodeAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {decode_attn_status_string(status)} (status {status})")


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim_qk", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32), ("is_mla", ctypes.c_int32), ("ckv_dim", ctypes.c_int32),
        ("kpe_dim", ctypes.c_int32), ("kv_layout", ctypes.c_int), ("page_size", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("sparse_block_size", ctypes.c_int32), ("max_sparse_blocks", ctypes.c_int32),
        ("q_len", ctypes.c_int32), ("sparse_batch", ctypes.c_int32),
        ("sparse_heads", ctypes.c_int32), ("kv_groups", ctypes.c_int32),
        ("fp8_mma", ctypes.c_int32),
    ]


class Args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("q_pe", ctypes.c_void_p), ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("kv_num_blks", ctypes.c_void_p), ("kv_idx", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("k_scale_shift", ctypes.c_void_p), ("v_scale_shift", ctypes.c_void_p),
        ("kv_full_num_blks", ctypes.c_void_p), ("kv_full_idx", ctypes.c_void_p),
        ("softcap", ctypes.c_float), ("spec_mask", ctypes.c_void_p),
        ("mask_sink", ctypes.c_void_p), ("mask_window", ctypes.c_void_p),
        ("alibi_slopes", ctypes.c_void_p),
    ]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "kv_tile", "chunk_tokens", "num_splits", "num_units", "rows_per_unit", "grid_x", "grid_y",
        "grid_z", "ctas_per_sm", "writes_final")] + [
        ("counters_offset", ctypes.c_int64), ("partial_o_offset", ctypes.c_int64), ("partial_lse_offset", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def load(build_if_missing: bool = False):
    """Loads libdecode_attn.so (building it first only when asked)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise ImportError(
                f"{_build.LIB} is missing: build it with `python -c \"import __graft_entry__ as g; "
                "g.build()\"` (there is no non-CUDA fallback)")
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    vp, i32, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int
    sig = {
        "decode_attn_create": (st, [ctypes.POINTER(Problem), ctypes.c_int, ctypes.POINTER(vp)]),
        "decode_attn_plan": (st, [vp, vp, i32, ctypes.POINTER(ctypes.c_size_t)]),
        "decode_attn_plan_ex": (st, [vp, vp, vp, i32, ctypes.POINTER(ctypes.c_size_t)]),
        "decode_attn_get_plan": (st, [vp, ctypes.POINTER(PlanInfo)]),
        "decode_attn_plan_info": (st, [ctypes.POINTER(Problem), i32, vp, i32,
                                       ctypes.POINTER(PlanInfo)]),
        "decode_attn_run": (st, [vp, ctypes.POINTER(Args), vp, ctypes.c_size_t, vp]),
        "decode_attn_merge": (st, [vp, vp, vp, i32, i32, i32, vp, vp, vp]),
        "decode_attn_run_noalloc": (st, [vp, ctypes.POINTER(Args), vp]),
        "decode_attn_get_error": (st, [vp, vp, vp, ctypes.POINTER(ctypes.c_uint32)]),
        "decode_attn_get_error_noalloc": (st, [vp, vp, ctypes.POINTER(ctypes.c_uint32)]),
        "decode_attn_destroy": (None, [vp]),
        "decode_attn_status_string": (ctypes.c_char_p, [st]),
        # test hooks (include/decode_attn_testing.h)
        "decode_attn_test_fill_smem": (st, [ctypes.c_uint32, i32, vp]),
        "decode_attn_test_set_stall": (st, [vp, ctypes.c_uint32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int, what: str):
    if status != DA_OK:
        raise DecodeAttnError(status, what)


def _ptr(t):
    """Device pointer of a tensor argument. The library reads every tensor as
    row-major device memory through the bare pointer, so host tensors and
    strided views are refused here instead of being read as something else."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_cuda:
            raise ValueError("tensor arguments must be in device memory (got a host tensor)")
        if not t.is_contiguous():
            raise ValueError("tensor arguments must be contiguous (row-major, last index fastest)")
        return ctypes.c_void_p(t.data_ptr())
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_problem(**kw) -> Problem:
    p = Problem()
    for name, _ in Problem._fields_:
        setattr(p, name, int(kw.get(name, 0)))
    return p


def _host_i32(t):
    if t is None:
        return None, None
    h = torch.as_tensor(t, dtype=torch.int32).to("cpu").contiguous()
    return h, ctypes.c_void_p(h.data_ptr())


# ---------------------------------------------------------------- the C ABI, by name

def decode_attn_status_string(status: int) -> str:
    return load().decode_attn_status_string(int(status)).decode()


def decode_attn_create(problem: Problem, device: int = 0):
    ctx = ctypes.c_void_p()
    _check(load().decode_attn_create(ctypes.byref(problem), int(device), ctypes.byref(ctx)),
           "decode_attn_create")
    return ctx


def decode_attn_plan(ctx, seq_lens_host=None, num_splits_override: int = 0) -> int:
    return decode_attn_plan_ex(ctx, seq_lens_host, None, num_splits_override)


def decode_attn_plan_ex(ctx, seq_lens_host=None, kv_num_blks_host=None,
                        num_splits_override: int = 0) -> int:
    sl, slp = _host_i32(seq_lens_host)
    nb, nbp = _host_i32(kv_num_blks_host)
    ws = ctypes.c_size_t()
    _check(load().decode_attn_plan_ex(ctx, slp, nbp, int(num_splits_override), ctypes.byref(ws)),
           "decode_attn_plan")
    return ws.value


def decode_attn_get_plan(ctx) -> dict:
    info = PlanInfo()
    _check(load().decode_attn_get_plan(ctx, ctypes.byref(info)), "decode_attn_get_plan")
    return info.as_dict()


def decode_attn_plan_info(problem: Problem, num_sms: int, seq_lens_host=None,
                          num_splits_override: int = 0) -> dict:
    sl, slp = _host_i32(seq_lens_host)
    info = PlanInfo()
    _check(load().decode_attn_plan_info(ctypes.byref(problem), int(num_sms), slp,
                                        int(num_splits_override), ctypes.byref(info)),
           "decode_attn_plan_info")
    return info.as_dict()


def make_args(tensors: dict, scale: float, out, lse=None, softcap: float = 0.0) -> Args:
    a = Args()
    for k in ("q", "q_pe", "k", "v", "k_scale", "v_scale", "block_table", "seq_lens",
              "kv_num_blks", "kv_idx"):
        a.__setattr__(k, _ptr(tensors.get(k)))
    a.scale = float(scale)
    a.out = _ptr(out)
    a.lse = _ptr(lse)
    a.k_scale_shift = _ptr(tensors.get("k_scale_shift"))
    a.v_scale_shift = _ptr(tensors.get("v_scale_shift"))
    a.kv_full_num_blks = _ptr(tensors.get("kv_full_num_blks"))
    a.kv_full_idx = _ptr(tensors.get("kv_full_idx"))
    a.softcap = float(softcap)
    a.spec_mask = _ptr(tensors.get("spec_mask"))
    # flex-style mods, per query head: the sink/window mask_mod and ALiBi slopes
    a.mask_sink = _ptr(tensors.get("mask_sink"))
    a.mask_window = _ptr(tensors.get("mask_window"))
    a.alibi_slopes = _ptr(tensors.get("alibi_slopes"))
    return a


def decode_attn_run(ctx, args: Args, workspace: torch.Tensor, stream=None):
    _check(load().decode_attn_run(ctx, ctypes.byref(args), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
           "decode_attn_run")


def decode_attn_run_noalloc(ctx, args: Args, stream=None):
    """decode_attn_run without a workspace: the library's static device scratch
    (32 MiB per device) is used instead, for callers that cannot allocate."""
    _check(load().decode_attn_run_noalloc(ctx, ctypes.byref(args), _stream(stream)),
           "decode_attn_run_noalloc")


def decode_attn_merge(ctx, o_part, lse_part, num_splits: int, rows: int, dv: int, out, lse=None,
                      stream=None):
    _check(load().decode_attn_merge(ctx, _ptr(o_part), _ptr(lse_part), int(num_splits), int(rows),
                                    int(dv), _ptr(out), _ptr(lse), _stream(stream)),
           "decode_attn_merge")


def decode_attn_get_error(ctx, workspace: torch.Tensor, stream=None) -> int:
    flags = ctypes.c_uint32()
    st = load().decode_attn_get_error(ctx, _ptr(workspace), _stream(stream), ctypes.byref(flags))
    if st not in (DA_OK, DA_ERR_DEVICE):
        raise DecodeAttnError(st, "decode_attn_get_error")
    return flags.value


def decode_attn_get_error_noalloc(ctx, stream=None) -> int:
    flags = ctypes.c_uint32()
    st = load().decode_attn_get_error_noalloc(ctx, _stream(stream), ctypes.byref(flags))
    if st not in (DA_OK, DA_ERR_DEVICE):
        raise DecodeAttnError(st, "decode_attn_get_error_noalloc")
    return flags.value


def decode_attn_destroy(ctx):
    if ctx:
        load().decode_attn_destroy(ctx)


# ---------------------------------------------------------------- convenience wrapper

class DecodeAttention:
    """One problem shape: create + plan once, run many times.

    The workspace is a zeroed uint8 tensor allocated here with torch (the
    library itself never allocates device memory).
    """

    def __init__(self, device=0, seq_lens_host=None, kv_num_blks_host=None,
                 num_splits_override=0, **problem):
        load()
        self.problem = make_problem(**problem)
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        self.ctx = decode_attn_create(self.problem, self.device.index or 0)
        self.replan(seq_lens_host, kv_num_blks_host, num_splits_override)

    def replan(self, seq_lens_host=None, kv_num_blks_host=None, num_splits_override=0):
        ws = decode_attn_plan_ex(self.ctx, seq_lens_host, kv_num_blks_host, num_splits_override)
        self.plan = decode_attn_get_plan(self.ctx)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=self.device)

    def run(self, tensors: dict, scale: float, out=None, lse=None, stream=None, softcap=0.0):
        p = self.problem
        lead = (p.batch, p.num_q_heads) + ((p.q_len,) if p.q_len > 1 else ())
        if out is None:
            out = torch.empty(lead + (p.head_dim_v,), dtype=torch.bfloat16, device=self.device)
        # the library writes through raw pointers: refuse buffers of the wrong size
        # or type here rather than let it write past them
        if out.dtype != torch.bfloat16 or out.numel() != math.prod(lead) * p.head_dim_v:
            raise ValueError(f"out must be bf16 with {lead + (p.head_dim_v,)} elements")
        if lse is not None and (lse.dtype != torch.float32 or lse.numel() != math.prod(lead)):
            raise ValueError(f"lse must be float32 with {lead} elements")
        decode_attn_run(self.ctx, make_args(tensors, scale, out, lse, softcap), self.workspace, stream)
        return out

    def errors(self, stream=None) -> int:
        return decode_attn_get_error(self.ctx, self.workspace, stream)

    def close(self):
        decode_attn_destroy(self.ctx)
        self.ctx = None

    def __del__(self):
        try:
            if getattr(self, "ctx", None):
                self.close()
        except Exception:
            pass


def problem_kwargs(work) -> dict:
    """Problem fields for a workload description (see ``workloads``)."""
    w = work
    return dict(batch=w.batch, num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                head_dim_qk=w.head_dim_qk, head_dim_v=w.head_dim_v, is_mla=int(w.is_mla),
                ckv_dim=w.ckv_dim, kpe_dim=w.kpe_dim,
                kv_layout=DA_KV_PAGED if w.paged else DA_KV_CONTIGUOUS,
                page_size=w.page_size, max_seq_len=w.max_seq_len,
                max_pages_per_seq=w.max_pages_per_seq, num_pages=w.num_pages,
                q_dtype=DA_DTYPE_BF16,
                kv_dtype=DA_DTYPE_INT4_GROUPS if getattr(w, "kv_int4_groups", 0) else
                ((DA_DTYPE_FP8_E4M3_TOKEN_SCALE if getattr(w, "kv_token_scale", False)
                  else DA_DTYPE_FP8_E4M3) if w.kv_fp8 else DA_DTYPE_BF16),
                kv_groups=getattr(w, "kv_int4_groups", 0),
                sparse_block_size=w.sparse_block_size, max_sparse_blocks=w.max_sparse_blocks,
                q_len=getattr(w, "q_len", 1), sparse_batch=getattr(w, "sparse_batch", 0),
                sparse_heads=getattr(w, "sparse_heads", 0), fp8_mma=int(getattr(w, "fp8_mma", False)))
