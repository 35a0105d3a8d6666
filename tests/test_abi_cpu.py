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


def _gqa_schedule(ctas, unit_tiles):
    """The persistent GQA kernel's schedule, as its comments define it: the units'
    tiles laid end to end are cut into `ctas` equal ranges [floor(c*T/C),
    floor((c+1)*T/C)); returns per-unit lists of (cta, first tile, last tile)."""
    T = sum(unit_tiles)
    bounds = [c * T // ctas for c in range(ctas + 1)]
    segs = []
    start = 0
    for t in unit_tiles:
        seg = []
        for c in range(ctas):
            lo, hi = max(bounds[c], start), min(bounds[c + 1], start + t)
            if hi > lo:
                seg.append((c, lo - start, hi - start))
        segs.append(seg)
        start += t
    return segs, bounds


def _check_gqa_plan(plan, unit_tiles, num_sms=152):
    C = plan["grid_x"]
    assert plan["grid_y"] == plan["grid_z"] == 1
    assert 1 <= C <= max(sum(unit_tiles), 1)
    assert C <= num_sms * plan["ctas_per_sm"] or plan["num_splits"] > 0
    segs, bounds = _gqa_schedule(C, unit_tiles)
    # every tile of every unit is in exactly one segment, segments are contiguous
    for t, seg in zip(unit_tiles, segs):
        pos = 0
        for _, lo, hi in seg:
            assert lo == pos
            pos = hi
        assert pos == t
        # the device finds a unit's segments from its first and last tile: c_first..c_last
        if seg:
            assert [c for c, _, _ in seg] == list(range(seg[0][0], seg[-1][0] + 1))
    # balance: every CTA streams floor or ceil of T/C tiles
    sizes = [bounds[c + 1] - bounds[c] for c in range(C)]
    assert max(sizes) - min(sizes) <= 1
    # the workspace holds a partial slot for every (unit + cta), and per unit its
    # counter plus the counters of a two-level merge (groups of ceil(sqrt(pieces))
    # pieces, pieces <= CTAs: at most ceil(sqrt(C)) + 1 groups)
    U, G = plan["num_units"], plan["rows_per_unit"]
    assert plan["counters_offset"] == 256
    assert plan["partial_o_offset"] - plan["counters_offset"] >= U * (1 + math.isqrt(C - 1) + 2) * 4
    assert plan["partial_lse_offset"] - plan["partial_o_offset"] >= (U + C) * G * 128 * 4
    assert plan["workspace_bytes"] - plan["partial_lse_offset"] >= (U + C) * G * 4


def _check_mla_plan(plan, row_tiles, num_sms=152):
    """Persistent MLA grid: one cluster of two CTAs per pair of SMs (never more
    clusters than tiles); the rows' tiles are cut into one range per cluster,
    exactly as for the GQA CTAs, with a partial slot per (row + cluster)."""
    assert plan["grid_x"] % 2 == 0 and plan["grid_y"] == plan["grid_z"] == 1
    C = plan["grid_x"] // 2
    assert C == min(num_sms * plan["ctas_per_sm"] // 2, max(sum(row_tiles), 1))
    segs, bounds = _gqa_schedule(C, row_tiles)
    for t, seg in zip(row_tiles, segs):
        pos = 0
        for _, lo, hi in seg:
            assert lo == pos
            pos = hi
        assert pos == t
        if seg:
            assert [c for c, _, _ in seg] == list(range(seg[0][0], seg[-1][0] + 1))
    sizes = [bounds[c + 1] - bounds[c] for c in range(C)]
    assert max(sizes) - min(sizes) <= 1
    U = plan["num_units"]
    assert plan["counters_offset"] == 256
    assert plan["partial_o_offset"] - plan["counters_offset"] >= U * 2 * 4
    assert plan["partial_lse_offset"] - plan["partial_o_offset"] >= (U + C) * 128 * 512 * 4
    assert plan["workspace_bytes"] - plan["partial_lse_offset"] >= (U + C) * 2 * 128 * 4


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 6, 7, 8])
def test_planner_covers_every_position_once(lib, cfg):
    w = W.config(cfg, shape_only=True)
    nb = w.tensors.get("kv_num_blks")
    plan = da.decode_attn_plan_info(_problem(w), 152, w.tensors["seq_lens"], w.num_splits)
    lens = [int(x) for x in w.tensors["seq_lens"]]
    if w.is_mla:
        _check_mla_plan(plan, [math.ceil(n / 64) for n in lens])
        return
    if w.sparse_block_size:
        tiles = [int(x) * (w.sparse_block_size // 64) for x in w.tensors["kv_num_blks"].flatten()]
        tiles = [256 * 2] * len(tiles)  # plan_info assumes full lists without host counts
    else:
        tiles = [math.ceil(n / 64) for n in lens for _ in range(w.num_kv_heads)]
    _check_gqa_plan(plan, tiles)
    if cfg == 1:
        assert plan["grid_x"] == 4  # the forced 4 splits of the one unit
    else:
        assert plan["grid_x"] == min(152 * plan["ctas_per_sm"], sum(tiles))


def test_planner_sparse_with_list_lengths(lib):
    """With the host list lengths the grid covers exactly the listed blocks."""
    w = W.config(4, shape_only=True)
    tiles = [int(x) * 2 for x in w.tensors["kv_num_blks"].flatten()]
    plan = da.decode_attn_plan_info(_problem(w), 152, None, 0)
    _check_gqa_plan(plan, [512] * len(tiles))
    # the schedule of the real lists: balanced and gap-free
    segs, bounds = _gqa_schedule(min(304, sum(tiles)), tiles)
    assert sum(hi - lo for seg in segs for _, lo, hi in seg) == sum(tiles)


def test_planner_override_and_workspace_layout(lib):
    w = W.make_gqa(batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[1000, 5], cache_len=1024,
                   seed=1)
    tiles = [16, 16, 1, 1]
    for S in (1, 2, 3, 7, 16):
        plan = da.decode_attn_plan_info(_problem(w), 152, w.tensors["seq_lens"], S)
        _check_gqa_plan(plan, tiles)
        assert plan["grid_x"] == min(S * 4, sum(tiles))


def test_planner_without_host_lengths_assumes_full_rows(lib):
    w = W.config(2, shape_only=True)
    p1 = da.decode_attn_plan_info(_problem(w), 152, None, 0)
    _check_gqa_plan(p1, [w.max_seq_len // 64] * (w.batch * w.num_kv_heads))


def test_several_query_tokens_per_row(lib):
    """q_len > 1: the G x q_len rows of a kv head are one unit (rows_per_unit), at
    most 16 of them; MLA takes up to 16 query tokens, one unit each."""
    w = W.config(6, shape_only=True)
    assert w.q_len == 4 and w.tensors["q"].shape == (32, 32, 4, 128)
    plan = da.decode_attn_plan_info(_problem(w), 152, w.tensors["seq_lens"], 0)
    assert plan["rows_per_unit"] == 16 and plan["num_units"] == 256
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim_qk=128, head_dim_v=128,
                max_seq_len=64)
    for q_len, status in ((0, da.DA_OK), (1, da.DA_OK), (4, da.DA_OK), (5, da.DA_ERR_UNSUPPORTED),
                          (-1, da.DA_ERR_INVALID_ARG)):
        prob = da.make_problem(**base, q_len=q_len)
        if status == da.DA_OK:
            info = da.decode_attn_plan_info(prob, 152)
            assert info["rows_per_unit"] == 4 * max(q_len, 1)
        else:
            with pytest.raises(da.DecodeAttnError) as e:
                da.decode_attn_plan_info(prob, 152)
            assert e.value.status == status
    # several query tokens over block-sparse tables are planned like the dense case
    sparse = dict(base, sparse_block_size=64, max_sparse_blocks=1, q_len=2)
    assert da.decode_attn_plan_info(da.make_problem(**sparse), 152)["rows_per_unit"] == 8
    # MLA: a unit per (row, query token); token t of Q sees seq_len - Q + 1 + t positions
    m = W.config(5, shape_only=True)
    lens = m.tensors["seq_lens"]
    for q_len in (2, 4, 16):
        info = da.decode_attn_plan_info(da.make_problem(**dict(da.problem_kwargs(m), q_len=q_len)), 152,
                                        lens, 0)
        assert info["num_units"] == m.batch * q_len and info["rows_per_unit"] == 128
        tiles = sum(-(-max(int(n) - (q_len - 1 - t), 0) // 64) for n in lens.tolist() for t in range(q_len))
        assert info["grid_x"] == 2 * min(76, tiles)
    with pytest.raises(da.DecodeAttnError) as e:
        da.decode_attn_plan_info(da.make_problem(**dict(da.problem_kwargs(m), q_len=17)), 152)
    assert e.value.status == da.DA_ERR_UNSUPPORTED


def test_broadcast_block_mask_extents_are_validated(lib):
    """sparse_batch / sparse_heads: 0 (the problem's own) or a positive extent."""
    base = dict(batch=4, num_q_heads=8, num_kv_heads=2, head_dim_qk=128, head_dim_v=128,
                max_seq_len=256, sparse_block_size=64, max_sparse_blocks=4)
    for sb, sh in ((0, 0), (1, 1), (1, 2), (4, 1), (3, 5)):
        da.decode_attn_plan_info(da.make_problem(**base, sparse_batch=sb, sparse_heads=sh), 152)
    for sb, sh in ((-1, 0), (0, -2)):
        with pytest.raises(da.DecodeAttnError) as e:
            da.decode_attn_plan_info(da.make_problem(**base, sparse_batch=sb, sparse_heads=sh), 152)
        assert e.value.status == da.DA_ERR_INVALID_ARG


def test_int4_groups_are_validated(lib):
    """int4 rows: 4 or 8 groups run; 1 and 2 are the format's but unsupported
    (rows not a multiple of 16 bytes); anything else is invalid."""
    base = dict(batch=2, num_q_heads=8, num_kv_heads=2, head_dim_qk=128, head_dim_v=128,
                max_seq_len=256, kv_dtype=da.DA_DTYPE_INT4_GROUPS)
    for g in (4, 8):
        da.decode_attn_plan_info(da.make_problem(**base, kv_groups=g), 152)
    for g, status in ((1, da.DA_ERR_UNSUPPORTED), (2, da.DA_ERR_UNSUPPORTED),
                      (3, da.DA_ERR_INVALID_ARG), (0, da.DA_ERR_INVALID_ARG),
                      (16, da.DA_ERR_INVALID_ARG)):
        with pytest.raises(da.DecodeAttnError) as e:
            da.decode_attn_plan_info(da.make_problem(**base, kv_groups=g), 152)
        assert e.value.status == status
    # contiguous rows travel as 128-byte lines: L a multiple of 8 (4 groups) or 4 (8 groups)
    for g, L, ok in ((4, 260, False), (4, 264, True), (8, 260, True), (8, 262, False)):
        prob = da.make_problem(**dict(base, max_seq_len=L), kv_groups=g)
        if ok:
            da.decode_attn_plan_info(prob, 152)
        else:
            with pytest.raises(da.DecodeAttnError) as e:
                da.decode_attn_plan_info(prob, 152)
            assert e.value.status == da.DA_ERR_UNSUPPORTED


def test_binding_refuses_host_tensors_as_device_arguments():
    # the library reads every tensor through a bare device pointer: a host
    # tensor must be refused by the binding, not passed on as an address
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="device memory"):
        da.make_args({"q": q}, 0.1, None, None)
    assert da.make_args({}, 0.1, None, None).q is None
