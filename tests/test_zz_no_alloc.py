"""decode_attn_run_noalloc: the entry point for callers that cannot allocate
device memory (it runs on the library's static device scratch instead of a
caller workspace). Checked through the C ABI against decode_attn_run on the
same inputs, within the parity tolerances, on two calls in a row -- the
second call finds the scratch as the first one left it.

This file is named so pytest collects it last."""

import ctypes

import pytest
import torch

import decode_attention_flash_gb300 as da
from decode_attention_flash_gb300 import workloads as W
from helpers import BF16_ATOL, BF16_RTOL, LSE_ATOL

pytestmark = pytest.mark.gpu


def _case():
    return W.make_gqa(name="noalloc", batch=6, num_q_heads=32, num_kv_heads=8,
                      seq_lens=[1500, 1, 700, 4000, 33, 2048], layout="paged", page_size=16,
                      seed=31)


def _run(lib, ctx, w, t, noalloc):
    dev = t["q"].device
    out = torch.full((w.batch, w.num_q_heads, w.head_dim_v), 3.0, dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.batch, w.num_q_heads), 3.0, dtype=torch.float32, device=dev)
    args = da.make_args(t, w.scale, out, lse)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        st = lib.decode_attn_run_noalloc(ctx, ctypes.byref(args), stream)
    else:
        ws = torch.zeros(da.decode_attn_get_plan(ctx)["workspace_bytes"], dtype=torch.uint8,
                         device=dev)
        st = lib.decode_attn_run(ctx, ctypes.byref(args), ctypes.c_void_p(ws.data_ptr()),
                                 ws.numel(), stream)
    assert st == da.DA_OK, da.decode_attn_status_string(st)
    torch.cuda.synchronize()
    return out.double().cpu(), lse.double().cpu()


def test_noalloc_matches_workspace_entry_point_twice():
    lib = da.load()
    w = _case()
    t = w.to("cuda")
    ctx = da.decode_attn_create(da.make_problem(**da.problem_kwargs(w)), 0)
    try:
        da.decode_attn_plan(ctx, w.tensors["seq_lens"], 0)
        assert da.decode_attn_get_plan(ctx)["num_splits"] > 1  # the partials go through scratch
        ref_out, ref_lse = _run(lib, ctx, w, t, noalloc=False)
        for _ in range(2):
            out, lse = _run(lib, ctx, w, t, noalloc=True)
            err = float((out - ref_out).abs().max())
            rel = err / max(float(ref_out.abs().max()), 1e-6)
            assert err <= BF16_ATOL and rel <= BF16_RTOL, (err, rel)
            assert float((lse - ref_lse).abs().max()) <= LSE_ATOL
    finally:
        da.decode_attn_destroy(ctx)


def test_noalloc_back_to_back_shapes_are_bitwise_the_workspace_entry_point():
    """An MLA problem (its counters are per row and value half) and a second GQA
    shape with another unit count, run back to back on the shared static array:
    the same kernel on the same plan as decode_attn_run, so the same bits."""
    lib = da.load()
    cases = [
        W.make_mla(name="noalloc_mla", batch=5, seq_lens=[700, 0, 64, 3000, 129], seed=33),
        W.make_gqa(name="noalloc_gqa2", batch=9, num_q_heads=16, num_kv_heads=4,
                   seq_lens=[90, 2500, 1, 640, 0, 1800, 77, 4096, 333], layout="paged",
                   page_size=32, seed=34),
    ]
    for w in cases + cases:  # each shape twice, alternating
        t = w.to("cuda")
        ctx = da.decode_attn_create(da.make_problem(**da.problem_kwargs(w)), 0)
        try:
            da.decode_attn_plan(ctx, w.tensors["seq_lens"], 0)
            ref_out, ref_lse = _run(lib, ctx, w, t, noalloc=False)
            out, lse = _run(lib, ctx, w, t, noalloc=True)
            assert torch.equal(out, ref_out), w.name
            assert torch.equal(lse.nan_to_num(neginf=-1e30), ref_lse.nan_to_num(neginf=-1e30)), w.name
        finally:
            da.decode_attn_destroy(ctx)


def test_noalloc_refuses_a_plan_beyond_the_static_scratch():
    lib = da.load()
    # 256 (b, kv head) units x 64 splits x 8 heads x 128 dims x 4 B of partials > 32 MiB
    w = W.make_gqa(name="big", batch=32, num_q_heads=64, num_kv_heads=8, seq_lens=[8192] * 32,
                   cache_len=8192, seed=32, shape_only=True)
    ctx = da.decode_attn_create(da.make_problem(**da.problem_kwargs(w)), 0)
    try:
        da.decode_attn_plan(ctx, None, 64)
        assert da.decode_attn_get_plan(ctx)["workspace_bytes"] > (32 << 20)
        args = da.make_args({}, w.scale, None, None)
        st = lib.decode_attn_run_noalloc(ctx, ctypes.byref(args),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == da.DA_ERR_WORKSPACE
    finally:
        da.decode_attn_destroy(ctx)


def test_noalloc_error_word_reports_a_bad_page():
    # a block-table entry outside the pool: the page is skipped on the device and
    # its bit waits in the static array's error word until read (and cleared)
    lib = da.load()
    w = _case()
    bt = w.tensors["block_table"].clone()
    bt[0, 3] = w.num_pages + 5
    w.tensors["block_table"] = bt
    dev = torch.device("cuda", 0)
    t = w.to(dev)
    ctx = da.decode_attn_create(da.make_problem(**da.problem_kwargs(w)), 0)
    try:
        da.decode_attn_plan(ctx, w.tensors["seq_lens"], 0)
        assert da.decode_attn_get_error_noalloc(ctx) == 0  # what earlier calls left is read out here
        _run(lib, ctx, w, t, noalloc=True)
        assert da.decode_attn_get_error_noalloc(ctx) & da.DA_DEVERR_PAGE_INDEX
        assert da.decode_attn_get_error_noalloc(ctx) == 0  # cleared by the read
        w.tensors["block_table"][0, 3] = bt[0, 2]  # a valid page again
        _run(lib, ctx, w, w.to(dev), noalloc=True)
        assert da.decode_attn_get_error_noalloc(ctx) == 0
    finally:
        da.decode_attn_destroy(ctx)
