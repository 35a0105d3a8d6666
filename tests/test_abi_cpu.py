"""CPU-side checks of the C-ABI library: it loads, exports every entry point the
header declares, and its host-only planner covers every position exactly once."""

import ctypes
import math
import os
import re
import subprocess

import pytest
import torch

import decode_attention_flash_gb300 as da
from decode_attention_flash_gb300 import _build
from decode_attention_flash_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return da.load(build_if_missing=True)


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
            name = m.group(1)
            if name not in ("defined",) and not name.startswith("__"):
                names.add(name)
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("decode_attn_create", "decode_attn_plan", "decode_attn_run",
                     "decode_attn_merge", "decode_attn_get_error", "decode_attn_destroy",
                     "decode_attn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for s in range(7):
        assert da.decode_attn_status_string(s)
    assert "unknown" in da.decode_attn_status_string(99)


def test_merge_rejects_bad_arguments(lib):
    st = lib.decode_attn_merge(None, None, None, 1, 1, 128, None, None, None)
    assert st == da.DA_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(buf, ctypes.c_void_p)
    assert lib.decode_attn_merge(None, p, p, 0, 1, 128, p, None, None) == da.DA_ERR_INVALID_ARG
    assert lib.decode_attn_merge(None, p, p, 2, 1, 130, p, None, None) == da.DA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_create_without_a_device_reports_cuda_error(lib):
    w = W.config(1, shape_only=True)
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_create(da.make_problem(**da.problem_kwargs(w)), 0)
    assert e.value.status == da.DA_ERR_CUDA


def test_create_validates_the_problem(lib):
    bad = dict(batch=1, num_q_heads=8, num_kv_heads=3, head_dim_qk=128, head_dim_v=128,
               max_seq_len=64)
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_create(da.make_problem(**bad), 0)
    assert e.value.status == da.DA_ERR_INVALID_ARG
    bad = dict(batch=1, num_q_heads=8, num_kv_heads=1, head_dim_qk=64, head_dim_v=64,
               max_seq_len=64)
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_create(da.make_problem(**bad), 0)
    assert e.value.status == da.DA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ planner (host logic)

def _problem(w):
    return da.make_problem(**da.problem_kwargs(w))


def _check_cover(plan, lengths, align):
    """Every position of every unit is in exactly one split, splits are tile-aligned."""
    chunk, S = plan["chunk_tokens"], plan["num_splits"]
    assert chunk % align == 0 and chunk > 0
    for n in lengths:
        covered = 0
        prev_hi = 0
        for s in range(S):
            lo, hi = s * chunk, min((s + 1) * chunk, n)
            if hi <= lo:
                continue
            assert lo == prev_hi  # contiguous, no overlap, no gap
            covered += hi - lo
            prev_hi = hi
        assert covered == n


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_planner_covers_every_position_once(lib, cfg):
    w = W.config(cfg, shape_only=True)
    plan = da.decode_attn_plan_info(_problem(w), 152, w.tensors["seq_lens"], w.num_splits)
    lens = [int(x) for x in w.tensors["seq_lens"]]
    _check_cover(plan, lens, plan["kv_tile"])
    # MLA runs each split on a cluster of two CTAs
    assert plan["grid_x"] == plan["num_splits"] * (2 if w.is_mla else 1)
    assert plan["grid_z"] == w.batch
    if cfg == 1:
        assert plan["num_splits"] == 4 and plan["chunk_tokens"] == 128
    else:
        # enough CTAs with work to fill every SM, and splits within the fused merge's limit
        busy = sum(math.ceil(n / plan["chunk_tokens"]) for n in lens) * plan["grid_y"]
        busy *= 2 if w.is_mla else 1  # CTAs per split
        assert busy >= 152
        assert 1 <= plan["num_splits"] <= 256


def test_planner_sparse_splits_whole_blocks(lib):
    w = W.config(4, shape_only=True)
    plan = da.decode_attn_plan_info(_problem(w), 152, None, 0)
    assert plan["chunk_tokens"] % w.sparse_block_size == 0
    # with the real list lengths the splits cover the 36 listed blocks
    nb = w.tensors["kv_num_blks"].contiguous()
    lengths = [int(x) * w.sparse_block_size for x in nb.flatten()]
    _check_cover(plan, lengths, w.sparse_block_size)


def test_planner_override_and_workspace_layout(lib):
    w = W.make_gqa(batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[1000, 5], cache_len=1024,
                   seed=1)
    for S in (1, 2, 3, 7, 16):
        plan = da.decode_attn_plan_info(_problem(w), 152, w.tensors["seq_lens"], S)
        assert plan["num_splits"] <= S
        _check_cover(plan, [1000, 5], 64)
        assert plan["counters_offset"] == 256
        if plan["num_splits"] == 1:
            assert plan["writes_final"] == 1
            assert plan["workspace_bytes"] == 512
        else:
            units, rows = 4, 4
            need_o = units * plan["num_splits"] * rows * 128 * 4
            assert plan["partial_lse_offset"] - plan["partial_o_offset"] >= need_o
            assert plan["workspace_bytes"] - plan["partial_lse_offset"] >= units * plan[
                "num_splits"] * rows * 4
            assert plan["partial_o_offset"] % 256 == 0 and plan["partial_lse_offset"] % 256 == 0


def test_planner_without_host_lengths_assumes_full_rows(lib):
    w = W.config(2, shape_only=True)
    p1 = da.decode_attn_plan_info(_problem(w), 152, None, 0)
    _check_cover(p1, [w.max_seq_len] * w.batch, 64)
