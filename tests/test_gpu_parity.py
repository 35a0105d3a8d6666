"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded inputs, plus the bit-exact gather checks and device error flags.

Tolerances (floating point): bf16 outputs max-abs 2e-2 and rel 1e-2
(rel = max|gpu - oracle| / max(max|oracle|, 1e-6)), LSE within 1e-3 absolute,
fp8 KV within 3e-2 against the oracle on the same dequantised values.
"""

import numpy as np
import pytest
import torch

import decode_attention_flash_gb300 as da
from decode_attention_flash_gb300 import workloads as W
from helpers import assert_parity, reference, run_gpu

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ small cases, several tiles + ragged tails

def test_tiny_config_four_splits():
    w = W.config(1)
    out, lse, flags, eng = run_gpu(w)
    assert eng.plan["num_splits"] == 4 and flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="config 1")


@pytest.mark.parametrize("splits", [0, 1, 2, 5])
@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
def test_paged_ragged(splits, page_size):
    lens = [1, 17, 64, 65, 700, 1000, 0, 333]
    w = W.make_gqa(name="paged", batch=8, num_q_heads=32, num_kv_heads=8, seq_lens=lens,
                   layout="paged", page_size=page_size, seed=100 + page_size)
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"paged P={page_size} S={splits}")


@pytest.mark.parametrize("pieces", [9, 10, 16, 31])
def test_unit_cut_into_many_pieces_merges_in_two_levels(pieces):
    # one unit over `pieces` CTAs: groups of ceil(sqrt(pieces)) pieces are merged
    # first (the last group may be short), then the groups; repeated calls give
    # the same bits (every counter is back at zero after a call)
    w = W.make_gqa(name="many", batch=1, num_q_heads=8, num_kv_heads=1, seq_lens=[64 * pieces - 17],
                   layout="paged", page_size=16, seed=300 + pieces)
    out, lse, flags, eng = run_gpu(w, num_splits_override=pieces)
    assert flags == 0 and eng.plan["grid_x"] == pieces
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"{pieces} pieces")
    out2, lse2, flags2, _ = run_gpu(w, engine=eng)  # same workspace: counters reused
    assert flags2 == 0 and torch.equal(out2, out) and torch.equal(lse2, lse)


@pytest.mark.parametrize("group", [1, 2, 4, 8, 16])
def test_contiguous_group_sizes(group):
    hkv = 2
    w = W.make_gqa(name="contig", batch=3, num_q_heads=group * hkv, num_kv_heads=hkv,
                   seq_lens=[257, 1, 900], cache_len=1000, seed=200 + group)
    out, lse, flags, _ = run_gpu(w, num_splits_override=3)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"G={group}")


@pytest.mark.parametrize("kind", ["paged", "contiguous", "sparse", "query_tokens", "int4", "mla"])
@pytest.mark.parametrize("splits", [0, 3])
def test_every_row_empty(kind, splits):
    """No row has a position, so the tile sequence is empty and no CTA streams:
    every output row must still be written (zeros, LSE -inf; the buffers start
    poisoned) and no error bit set."""
    if kind == "mla":
        w = W.make_mla(name="mla_empty", batch=3, seq_lens=[0, 0, 0], seed=61)
    elif kind == "sparse":
        w = W.make_gqa(name="sp_empty", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[512, 300],
                       cache_len=512, sparse_block_size=128, kv_num_blks=[[0, 0], [0, 0]],
                       kv_idx=[[[0] * 4] * 2] * 2, seed=62)
    else:
        w = W.make_gqa(name=f"{kind}_empty", batch=5, num_q_heads=16, num_kv_heads=4, seq_lens=[0] * 5,
                       layout="contiguous" if kind == "contiguous" else "paged", page_size=16,
                       cache_len=256 if kind == "contiguous" else None,
                       q_len=3 if kind == "query_tokens" else 1,
                       kv_int4_groups=4 if kind == "int4" else 0, seed=63)
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    assert torch.all(out == 0), f"{kind}: empty rows must be zero"
    assert torch.all(lse == -float("inf")), f"{kind}: empty rows must have LSE -inf"
    ref_out, ref_lse = reference(w)
    assert np.all(ref_out == 0) and np.all(ref_lse == -np.inf)


def test_lse_pointer_may_be_null():
    w = W.make_gqa(name="nolse", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[300, 40],
                   cache_len=300, seed=5)
    out, _, flags, _ = run_gpu(w, num_splits_override=2, with_lse=False)
    ref_out, _ = reference(w)
    assert_parity(out, None, ref_out, None, what="lse=NULL")


def test_plan_without_host_lengths():
    w = W.make_gqa(name="nohost", batch=4, num_q_heads=16, num_kv_heads=4, layout="paged",
                   seq_lens=[100, 2000, 3, 1500], seed=6)
    out, lse, flags, eng = run_gpu(w, seq_lens_host=False, num_splits_override=0)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="plan without host lengths")


def test_fp8_small():
    w = W.make_gqa(name="fp8", batch=2, num_q_heads=16, num_kv_heads=2, seq_lens=[3000, 77],
                   cache_len=3000, kv_fp8=True, seed=8)
    for S in (0, 1, 4):
        out, lse, flags, _ = run_gpu(w, num_splits_override=S)
        assert flags == 0
        ref_out, ref_lse = reference(w)
        assert_parity(out, lse, ref_out, ref_lse, fp8=True, what=f"fp8 S={S}")


def test_fp8_paged():
    w = W.make_gqa(name="fp8p", batch=3, num_q_heads=24, num_kv_heads=3, seq_lens=[500, 16, 95],
                   layout="paged", page_size=16, kv_fp8=True, seed=9)
    out, lse, flags, _ = run_gpu(w, num_splits_override=2)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, fp8=True, what="fp8 paged")


def _sparse(seed=10, lens=(4096, 4000), block=128):
    g = torch.Generator().manual_seed(seed)
    num, idx = W.sparse_lists(2, 4, 4096, block, keep_random=5, keep_last=2, g=g, max_blocks=12)
    return W.make_gqa(name="sparse", batch=2, num_q_heads=16, num_kv_heads=4, seq_lens=list(lens),
                      cache_len=4096, sparse_block_size=block, kv_num_blks=num, kv_idx=idx,
                      seed=seed)


@pytest.mark.parametrize("splits", [0, 1, 3])
def test_sparse_small(splits):
    w = _sparse()
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"sparse S={splits}")


def test_sparse_block_64_and_empty_lists():
    g = torch.Generator().manual_seed(11)
    num, idx = W.sparse_lists(2, 2, 1024, 64, keep_random=3, keep_last=1, g=g, max_blocks=8)
    num[1, 0] = 0  # an empty list: out 0, lse -inf
    w = W.make_gqa(name="sparse64", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[1024, 1000],
                   cache_len=1024, sparse_block_size=64, kv_num_blks=num, kv_idx=idx, seed=11)
    out, lse, flags, _ = run_gpu(w, num_splits_override=2)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="sparse 64")
    assert torch.all(out[1, :4] == 0) and torch.all(lse[1, :4] == -float("inf"))


def test_split_count_invariance():
    w = W.make_gqa(name="inv", batch=2, num_q_heads=8, num_kv_heads=1, seq_lens=[4000, 2500],
                   cache_len=4000, seed=12)
    outs = [run_gpu(w, num_splits_override=s)[0].double() for s in (1, 2, 7, 16)]
    for o in outs[1:]:
        assert float((o - outs[0]).abs().max()) < 5e-3


# ------------------------------------------------------------------ bit-exact gathers

def test_paged_equals_contiguous_on_depaged_cache_bitwise():
    w = W.make_gqa(name="pg", batch=4, num_q_heads=16, num_kv_heads=4,
                   seq_lens=[1000, 64, 1, 513], layout="paged", page_size=16, seed=13)
    t = w.tensors
    L = w.max_pages_per_seq * w.page_size
    pages = t["block_table"].long()
    k = t["k"][pages].permute(0, 2, 1, 3, 4).reshape(w.batch, w.num_kv_heads, L, 128)
    v = t["v"][pages].permute(0, 2, 1, 3, 4).reshape(w.batch, w.num_kv_heads, L, 128)
    c = W.Workload(name="depaged", batch=w.batch, num_q_heads=16, num_kv_heads=4, head_dim_qk=128,
                   head_dim_v=128, scale=w.scale, cache_len=L,
                   tensors=dict(q=t["q"], k=k.contiguous(), v=v.contiguous(), seq_lens=t["seq_lens"]))
    for S in (1, 3):
        op, lp, _, _ = run_gpu(w, num_splits_override=S)
        oc, lc, _, _ = run_gpu(c, num_splits_override=S)
        assert torch.equal(op.view(torch.int16), oc.view(torch.int16))
        assert torch.equal(lp, lc)


def test_sparse_equals_contiguous_on_compacted_blocks_bitwise():
    w = _sparse(seed=14, lens=(4096, 4096))
    t = w.tensors
    G, SBS = w.group, w.sparse_block_size
    rows_k, rows_v, lens = [], [], []
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            blocks = t["kv_idx"][b, h, :int(t["kv_num_blks"][b, h])].long()
            pos = (blocks[:, None] * SBS + torch.arange(SBS)).reshape(-1)
            rows_k.append(t["k"][b, h, pos])
            rows_v.append(t["v"][b, h, pos])
            lens.append(pos.numel())
    L = max(lens)
    BH = w.batch * w.num_kv_heads
    k = torch.zeros((BH, 1, L, 128), dtype=torch.bfloat16)
    v = torch.zeros((BH, 1, L, 128), dtype=torch.bfloat16)
    for i in range(BH):
        k[i, 0, :lens[i]] = rows_k[i]
        v[i, 0, :lens[i]] = rows_v[i]
    c = W.Workload(name="compact", batch=BH, num_q_heads=G, num_kv_heads=1, head_dim_qk=128,
                   head_dim_v=128, scale=w.scale, cache_len=L,
                   tensors=dict(q=t["q"].reshape(BH, G, 128).contiguous(), k=k, v=v,
                                seq_lens=torch.tensor(lens, dtype=torch.int32)))
    S = 4  # 7 listed blocks: 256-position splits in both problems
    os_, ls_, _, es = run_gpu(w, num_splits_override=S)
    oc, lc, _, ec = run_gpu(c, num_splits_override=S)
    assert es.plan["chunk_tokens"] == ec.plan["chunk_tokens"]
    assert torch.equal(os_.reshape(BH, G, 128).view(torch.int16), oc.view(torch.int16))
    assert torch.equal(ls_.reshape(BH, G), lc)


@pytest.mark.parametrize("splits", [1, 4])
def test_single_token_rows_return_the_value_row_bitwise(splits):
    w = W.make_gqa(name="one", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[1, 1, 1],
                   layout="paged", page_size=16, seed=15)
    out, lse, _, _ = run_gpu(w, num_splits_override=splits)
    t = w.tensors
    for b in range(3):
        page = int(t["block_table"][b, 0])
        for hq in range(8):
            assert torch.equal(out[b, hq].view(torch.int16), t["v"][page, hq // 4, 0].view(torch.int16))


# ------------------------------------------------------------------ device error flags (host-made faults)

def test_bad_page_index_sets_flag_and_is_skipped():
    w = W.make_gqa(name="badpage", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[100, 50],
                   layout="paged", page_size=16, seed=16)
    bt = w.tensors["block_table"].clone()
    bt[0, 1] = w.num_pages + 5
    bt[1, 0] = -3
    w.tensors["block_table"] = bt
    out, lse, flags, _ = run_gpu(w, num_splits_override=1)
    assert flags & da.DA_DEVERR_PAGE_INDEX
    assert torch.all(torch.isfinite(out.float()))


def test_seq_len_over_capacity_sets_flag():
    w = W.make_gqa(name="badlen", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[100, 50],
                   cache_len=128, seed=17, poison=False)
    eng = da.DecodeAttention(device=0, num_splits_override=2, **da.problem_kwargs(w))
    w.tensors["seq_lens"] = torch.tensor([5000, -4], dtype=torch.int32)
    out, lse, flags, _ = run_gpu(w, engine=eng)
    assert flags & da.DA_DEVERR_SEQ_LEN
    assert torch.all(out[1] == 0) and torch.all(lse[1] == -float("inf"))


def test_bad_sparse_index_sets_flag():
    w = _sparse(seed=18)
    idx = w.tensors["kv_idx"].clone()
    idx[0, 0, 0] = 10_000
    w.tensors["kv_idx"] = idx
    out, lse, flags, _ = run_gpu(w, num_splits_override=1)
    assert flags & da.DA_DEVERR_SPARSE_INDEX
    assert torch.all(torch.isfinite(out.float()))


def test_workspace_too_small_is_rejected():
    w = W.make_gqa(name="ws", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[1000, 50],
                   cache_len=1000, seed=19)
    eng = da.DecodeAttention(device=0, num_splits_override=4, **da.problem_kwargs(w))
    eng.workspace = eng.workspace[:64]
    with pytest.raises(da.DecodeAttnError) as e:
        eng.run(w.to("cuda"), w.scale)
    assert e.value.status == da.DA_ERR_WORKSPACE


# ------------------------------------------------------------------ standalone merge

def test_standalone_merge_matches_oracle_merge():
    import oracle
    g = torch.Generator().manual_seed(20)
    rows, S, dv = 300, 9, 512
    o = torch.randn((rows, S, dv), generator=g)
    lse = torch.randn((rows, S), generator=g) * 3
    lse[::7, 2] = -float("inf")
    lse[5] = -float("inf")  # a row with every split empty
    o[::7, 2] = float("nan")  # never read
    dev = torch.device("cuda", 0)
    out = torch.empty((rows, dv), dtype=torch.bfloat16, device=dev)
    lo = torch.empty((rows,), dtype=torch.float32, device=dev)
    da.decode_attn_merge(None, o.to(dev), lse.to(dev), S, rows, dv, out, lo)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge(o.double().numpy(), lse.double().numpy())
    assert_parity(out.cpu(), lo.cpu(), ref_o, ref_l, what="merge")


# ------------------------------------------------------------------ MLA latent decode (cluster-pair tcgen05 kernel)

@pytest.mark.parametrize("splits", [1, 2, 3])
def test_mla_small(splits):
    w = W.make_mla(name="mla", batch=4, seq_lens=[100, 64, 1000, 1], seed=40 + splits)
    out, lse, flags, eng = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"MLA S={splits}")


@pytest.mark.parametrize("scale", [-0.07, 0.0])
def test_mla_negative_and_zero_scale(scale):
    # a negative scale turns the running maximum into a minimum of the raw
    # scores; a zero scale gives uniform weights over exactly the valid tokens
    w = W.make_mla(name="mla_scale", batch=3, seq_lens=[130, 1, 777], scale=scale, seed=48)
    out, lse, flags, eng = run_gpu(w, num_splits_override=2)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"MLA scale={scale}")


@pytest.mark.parametrize("scale", [-0.09, 0.0])
def test_gqa_negative_and_zero_scale(scale):
    w = W.make_gqa(name="gqa_scale", batch=3, num_q_heads=16, num_kv_heads=4, seq_lens=[130, 1, 777],
                   layout="paged", page_size=16, scale=scale, seed=49)
    out, lse, flags, _ = run_gpu(w, num_splits_override=2)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"GQA scale={scale}")


def test_mla_empty_row_and_auto_plan():
    w = W.make_mla(name="mla0", batch=3, seq_lens=[0, 2500, 700], seed=45)
    out, lse, flags, eng = run_gpu(w)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="MLA auto plan")
    assert torch.all(out[0] == 0) and torch.all(lse[0] == -float("inf"))


def test_mla_single_token_returns_the_latent_row_bitwise():
    w = W.make_mla(name="mla1", batch=2, seq_lens=[1, 1], seed=46)
    out, lse, _, _ = run_gpu(w, num_splits_override=1)
    t = w.tensors
    for b in range(2):
        page = int(t["block_table"][b, 0])
        row = t["k"][page, 0]
        for h in range(128):
            assert torch.equal(out[b, h].view(torch.int16), row.view(torch.int16))


def test_mla_bad_page_sets_flag():
    w = W.make_mla(name="mla2", batch=2, seq_lens=[300, 200], seed=47)
    bt = w.tensors["block_table"].clone()
    bt[0, 1] = -1
    w.tensors["block_table"] = bt
    out, lse, flags, _ = run_gpu(w, num_splits_override=2)
    assert flags & da.DA_DEVERR_PAGE_INDEX
    assert torch.all(torch.isfinite(out.float()))


@pytest.mark.parametrize("q_len,tree", [(2, False), (3, False), (4, True), (16, False), (5, True)])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_mla_several_query_tokens(q_len, tree, splits):
    # Query token t of q_len sees the positions n <= N_b - q_len + t (or those its
    # draft-tree word selects among the last q_len): rows shorter than q_len
    # leave their first tokens without a position (out 0, LSE -inf); the cut
    # falls inside a page, on a page boundary and in the first page.
    lens = [1, 2, 64, 65, 700, 0, 130, 17]
    w = W.make_mla(name="mla_q", batch=8, seq_lens=lens, seed=500 + q_len, q_len=q_len, tree_mask=tree)
    out, lse, flags, eng = run_gpu(w, num_splits_override=splits)
    assert flags == 0 and out.shape == (8, 128, q_len, 512) and lse.shape == (8, 128, q_len)
    assert eng.plan["num_units"] == 8 * q_len
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"MLA q_len={q_len} tree={tree} S={splits}")


@pytest.mark.parametrize("splits", [1, 3])
def test_mla_non_finite_valid_keys_reach_the_sum_as_they_are(splits):
    # The two CTAs of a pair each hold half of every score and exchange their
    # halves in a narrowed float encoding that keeps NaN and the infinities.
    # NaN in a latent key element of row 0 (the first value half's dimensions)
    # turns all 128 heads of row 0 into NaN; +inf in a rope element of row 1
    # (the second half's rope columns) turns the heads whose q_pe component is
    # positive into NaN (inf - inf) and gives that token weight 0 in the others;
    # row 2 is untouched.
    w = W.make_mla(name="mla_nf", batch=3, seq_lens=[300, 200, 130], seed=49)
    t = w.tensors
    k, v, bt = t["k"].clone(), t["v"].clone(), t["block_table"]
    k[int(bt[0, 1]), 5, 7] = float("nan")
    v[int(bt[1, 2]), 10, 40] = float("inf")
    t["k"], t["v"] = k, v
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    got, gl = out.double().numpy(), lse.double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref_out))
    assert np.array_equal(np.isnan(gl), np.isnan(ref_lse))
    assert np.isnan(ref_out[0]).all() and 0 < np.isnan(ref_out[1]).all(-1).sum() < 128
    fin = ~np.isnan(ref_out)
    assert np.max(np.abs(got[fin] - ref_out[fin])) <= 2e-2
    lfin = ~np.isnan(ref_lse)
    assert np.max(np.abs(gl[lfin] - ref_lse[lfin])) <= 1e-3


@pytest.mark.parametrize("where", ["key", "query"])
@pytest.mark.parametrize("splits", [1, 3])
def test_gqa_nan_input_reaches_exactly_the_rows_that_read_it(where, splits):
    # A NaN in a valid key of kv head 0 of row 0 poisons the G query heads of
    # that group (every one of them weighs the token); a NaN in one query
    # element poisons that head alone. The others stay within tolerance.
    w = W.make_gqa(name="gqa_nan", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[300, 200, 130],
                   layout="paged", page_size=16, seed=50)
    t = w.tensors
    if where == "key":
        k = t["k"].clone()
        k[int(t["block_table"][0, 1]), 0, 5, 7] = float("nan")
        t["k"] = k
    else:
        q = t["q"].clone()
        q[1, 6, 3] = float("nan")
        t["q"] = q
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    got, gl = out.double().numpy(), lse.double().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref_out))
    assert np.array_equal(np.isnan(gl), np.isnan(ref_lse))
    assert np.isnan(ref_lse).sum() == (4 if where == "key" else 1)
    fin = ~np.isnan(ref_out)
    assert np.max(np.abs(got[fin] - ref_out[fin])) <= 2e-2
    lfin = ~np.isnan(ref_lse)
    assert np.max(np.abs(gl[lfin] - ref_lse[lfin])) <= 1e-3


# ------------------------------------------------------------------ several query tokens per row (causal)

@pytest.mark.parametrize("q_len,group,layout", [(2, 4, "paged"), (3, 2, "contiguous"),
                                                (4, 4, "paged"), (2, 8, "contiguous"),
                                                (16, 1, "paged"), (5, 3, "paged")])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_several_query_tokens_causal(q_len, group, layout, splits):
    # rows shorter than q_len leave their first query tokens without a position
    # (out 0, LSE -inf); the causal cut falls inside a tile, on a tile boundary
    # (64, 65) and inside a page
    lens = [1, 2, 17, 64, 65, 700, 0, 333]
    w = W.make_gqa(name="spec", batch=8, num_q_heads=2 * group, num_kv_heads=2, seq_lens=lens,
                   layout=layout, page_size=16, q_len=q_len, seed=400 + 10 * q_len + group)
    out, lse, flags, eng = run_gpu(w, num_splits_override=splits)
    assert flags == 0 and eng.plan["rows_per_unit"] == group * q_len
    assert out.shape == (8, 2 * group, q_len, 128)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"q_len={q_len} G={group} {layout} S={splits}")


def test_several_query_tokens_fp8():
    w = W.make_gqa(name="spec8", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[900, 3, 130],
                   cache_len=900, kv_fp8=True, q_len=4, seed=431)
    for S in (0, 2):
        out, lse, flags, _ = run_gpu(w, num_splits_override=S)
        assert flags == 0
        ref_out, ref_lse = reference(w)
        assert_parity(out, lse, ref_out, ref_lse, fp8=True, what=f"fp8 q_len=4 S={S}")


# ------------------------------------------------------------------ e4m3 with a per-token scale and shift

@pytest.mark.parametrize("layout,splits", [("contiguous", 0), ("contiguous", 3), ("paged", 0),
                                           ("paged", 2)])
def test_fp8_per_token_scale_shift(layout, splits):
    lens = [3000, 77, 1, 640] if layout == "contiguous" else [1000, 16, 95, 0]
    w = W.make_gqa(name="fp8tok", batch=4, num_q_heads=16, num_kv_heads=2, seq_lens=lens,
                   layout=layout, page_size=16, cache_len=3000 if layout == "contiguous" else None,
                   kv_fp8=True, kv_token_scale=True, seed=440 + splits)
    out, lse, flags, eng = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, fp8=True, what=f"fp8/token {layout} S={splits}")


def test_fp8_per_token_scale_shift_two_n_tiles_and_several_queries():
    # 12 query heads per kv head and 2 query tokens: 24 rows -> capped at 16, so use
    # 16 heads x 1 token (two n-tiles) and 4 heads x 3 tokens (12 rows)
    for hq, hkv, q_len in ((32, 2, 1), (8, 2, 3)):
        w = W.make_gqa(name="fp8tok2", batch=2, num_q_heads=hq, num_kv_heads=hkv,
                       seq_lens=[700, 5], cache_len=700, kv_fp8=True, kv_token_scale=True,
                       q_len=q_len, seed=450 + hq)
        out, lse, flags, _ = run_gpu(w, num_splits_override=2)
        assert flags == 0
        ref_out, ref_lse = reference(w)
        assert_parity(out, lse, ref_out, ref_lse, fp8=True, what=f"fp8/token hq={hq} q_len={q_len}")


def test_binding_refuses_output_buffers_of_the_wrong_size():
    # the library writes through raw pointers: the binding checks out / lse first
    w = W.make_gqa(name="shape", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[70, 5],
                   cache_len=72, q_len=2, seed=460)
    dev = torch.device("cuda", 0)
    eng = da.DecodeAttention(device=0, seq_lens_host=w.tensors["seq_lens"], **da.problem_kwargs(w))
    t = w.to(dev)
    with pytest.raises(ValueError):
        eng.run(t, w.scale, out=torch.empty((2, 8, 128), dtype=torch.bfloat16, device=dev))
    with pytest.raises(ValueError):
        eng.run(t, w.scale, lse=torch.empty((2, 8), dtype=torch.float32, device=dev))
    out = eng.run(t, w.scale)
    torch.cuda.synchronize()
    assert out.shape == (2, 8, 2, 128) and eng.errors() == 0
    eng.close()


# ------------------------------------------------------------------ the flex block mask's full-block table

def _split_lists(w):
    """The same kept blocks as two tables: the first half of each list stays in
    KV_NUM_BLKS / KV_IDX, the rest moves to FULL_KV_NUM_BLKS / FULL_KV_IDX."""
    nb, idx = w.tensors["kv_num_blks"], w.tensors["kv_idx"]
    keep = (nb // 2).to(torch.int32)
    part, full = torch.zeros_like(idx), torch.zeros_like(idx)
    for b in range(idx.shape[0]):
        for h in range(idx.shape[1]):
            k, n = int(keep[b, h]), int(nb[b, h])
            part[b, h, :k] = idx[b, h, :k]
            full[b, h, :n - k] = idx[b, h, k:n]
    return dict(w.tensors, kv_num_blks=keep, kv_idx=part, kv_full_num_blks=(nb - keep).to(torch.int32),
                kv_full_idx=full)


@pytest.mark.parametrize("splits", [0, 3])
def test_full_block_table(splits):
    w = _sparse()
    whole = dict(w.tensors)
    w.tensors = _split_lists(w)
    nb_total = whole["kv_num_blks"]  # the planner's host counts: both tables summed
    eng = da.DecodeAttention(device=0, seq_lens_host=w.tensors["seq_lens"], kv_num_blks_host=nb_total,
                             num_splits_override=splits, **da.problem_kwargs(w))
    out, lse, flags, _ = run_gpu(w, engine=eng)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"full table S={splits}")
    # the same tiles in the same order as one list: bit-identical on the GPU
    w.tensors = whole
    out1, lse1, flags1, _ = run_gpu(w, engine=eng)
    assert flags1 == 0 and torch.equal(out1, out) and torch.equal(lse1, lse)
    eng.close()


def test_bad_full_table_index_sets_flag():
    w = _sparse()
    t = _split_lists(w)
    t["kv_full_idx"] = t["kv_full_idx"].clone()
    t["kv_full_idx"][0, 0, 0] = 10 ** 6
    assert int(t["kv_full_num_blks"][0, 0]) > 0
    w.tensors = t
    out, lse, flags, _ = run_gpu(w)
    assert flags & da.DA_DEVERR_SPARSE_INDEX
    assert torch.all(torch.isfinite(out.float()))


# ------------------------------------------------------------------ tanh soft-capping of the scores

@pytest.mark.parametrize("softcap", [0.7, 5.0])
@pytest.mark.parametrize("kind", ["paged", "fp8", "fp8token", "spec", "sparse"])
def test_softcap(kind, softcap):
    if kind == "paged":
        w = W.make_gqa(name="cap", batch=4, num_q_heads=16, num_kv_heads=2,
                       seq_lens=[1000, 17, 1, 300], page_size=16, seed=470)
    elif kind == "fp8":
        w = W.make_gqa(name="cap8", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[900, 40],
                       cache_len=900, kv_fp8=True, seed=471)
    elif kind == "fp8token":
        w = W.make_gqa(name="cap8t", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[640, 90],
                       cache_len=640, kv_fp8=True, kv_token_scale=True, seed=472)
    elif kind == "spec":
        w = W.make_gqa(name="capq", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[500, 2, 65],
                       layout="paged", page_size=16, q_len=3, seed=473)
    else:
        w = _sparse(seed=474)
    fp8 = bool(w.kv_fp8)
    ref_out, ref_lse = reference(w, softcap=softcap)
    plain_out, _ = reference(w)
    # the cap changes the answer: a test that ignored it would fail
    assert float(np.abs(ref_out - plain_out).max()) > 0.05
    for S in (0, 3):
        out, lse, flags, _ = run_gpu(w, num_splits_override=S, softcap=softcap)
        assert flags == 0
        assert_parity(out, lse, ref_out, ref_lse, fp8=fp8, what=f"softcap {softcap} {kind} S={S}")


def test_softcap_zero_is_bitwise_the_uncapped_path():
    w = W.make_gqa(name="cap0", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[333, 70],
                   page_size=16, seed=475)
    out0, lse0, _, eng = run_gpu(w)
    out1, lse1, _, _ = run_gpu(w, engine=eng, softcap=0.0)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
    eng.close()


def test_softcap_rejected_when_negative_and_for_mla():
    w = W.make_gqa(name="capbad", batch=1, num_q_heads=8, num_kv_heads=2, seq_lens=[64],
                   cache_len=64, seed=476)
    with pytest.raises(da.DecodeAttnError):
        run_gpu(w, softcap=-1.0)
    with pytest.raises(da.DecodeAttnError):
        run_gpu(w, softcap=float("nan"))
    m = W.make_mla(name="mlacap", batch=1, seq_lens=[100], seed=477)
    with pytest.raises(da.DecodeAttnError):
        run_gpu(m, softcap=1.0)


# ------------------------------------------------------------------ draft-tree masks (speculative decoding)

@pytest.mark.parametrize("q_len,group,layout", [(4, 4, "paged"), (5, 3, "contiguous"),
                                                (16, 1, "paged"), (8, 2, "contiguous")])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_tree_mask(q_len, group, layout, splits):
    lens = [1, 3, 17, 64, 65, 700, 0, 333]
    w = W.make_gqa(name="tree", batch=8, num_q_heads=2 * group, num_kv_heads=2, seq_lens=lens,
                   layout=layout, page_size=16, q_len=q_len, tree_mask=True,
                   seed=480 + 10 * q_len + group)
    out, lse, flags, eng = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"tree q_len={q_len} G={group} {layout} S={splits}")


def test_tree_mask_fp8_and_per_token_fp8():
    for tok in (False, True):
        w = W.make_gqa(name="tree8", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[900, 3, 130],
                       cache_len=900, kv_fp8=True, kv_token_scale=tok, q_len=4, tree_mask=True,
                       seed=490 + tok)
        for S in (0, 2):
            out, lse, flags, _ = run_gpu(w, num_splits_override=S)
            assert flags == 0
            ref_out, ref_lse = reference(w)
            assert_parity(out, lse, ref_out, ref_lse, fp8=True, what=f"tree fp8 tok={tok} S={S}")


def test_tree_mask_lower_triangle_is_bitwise_causal():
    Q = 6
    w = W.make_gqa(name="tri", batch=4, num_q_heads=12, num_kv_heads=6, seq_lens=[5, 600, 64, 97],
                   page_size=16, q_len=Q, seed=495)
    out0, lse0, _, eng = run_gpu(w)
    tri = torch.tensor([(2 << t) - 1 for t in range(Q)], dtype=torch.int32).repeat(4, 1)
    w.tensors = dict(w.tensors, spec_mask=tri.contiguous())
    out1, lse1, flags, _ = run_gpu(w, engine=eng)
    assert flags == 0 and torch.equal(out0, out1) and torch.equal(lse0, lse1)
    # and a different tree changes the answer
    w.tensors["spec_mask"] = W.draft_tree_mask(4, Q, W._gen(5))
    out2, _, _, _ = run_gpu(w, engine=eng)
    assert not torch.equal(out0, out2)
    eng.close()


# ------------------------------------------------------------------ block masks broadcast over rows / heads

@pytest.mark.parametrize("shape", [(1, 1), (1, 4), (5, 1), (2, 2), (2, 16)])
@pytest.mark.parametrize("splits", [0, 3])
def test_broadcast_block_mask(shape, splits):
    # (2, 16): tables with a row per query head (SPARSE_HQ = HQ); the flex
    # decode template reads them at the kv head (off_hkv % SPARSE_HQ), so kv
    # head h reads row h and the rows of the other query heads are not read
    SZ, SH = shape
    B, HKV, L, blk = 5, 4, 2048, 128
    g = torch.Generator().manual_seed(500 + 10 * SZ + SH)
    nb = torch.randint(0, 9, (SZ, SH), generator=g, dtype=torch.int32)
    idx = torch.stack([torch.stack([torch.randperm(L // blk, generator=g)[:8] for _ in range(SH)])
                       for _ in range(SZ)]).to(torch.int32)
    w = W.make_gqa(name="bcast", batch=B, num_q_heads=16, num_kv_heads=HKV,
                   seq_lens=[2048, 1000, 64, 0, 1500], cache_len=L, sparse_block_size=blk,
                   kv_num_blks=nb, kv_idx=idx, sparse_shape=shape, seed=501)
    eng = da.DecodeAttention(device=0, seq_lens_host=w.tensors["seq_lens"], kv_num_blks_host=nb,
                             num_splits_override=splits, **da.problem_kwargs(w))
    out, lse, flags, _ = run_gpu(w, engine=eng)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"broadcast {shape} S={splits}")
    # the written-out tables give the same bits
    rows, heads = torch.arange(B) % SZ, torch.arange(HKV) % SH
    full = W.make_gqa(name="bcast_full", batch=B, num_q_heads=16, num_kv_heads=HKV,
                      seq_lens=[2048, 1000, 64, 0, 1500], cache_len=L, sparse_block_size=blk,
                      kv_num_blks=nb[rows][:, heads], kv_idx=idx[rows][:, heads], seed=501)
    out2, lse2, flags2, _ = run_gpu(full, num_splits_override=splits)
    if splits:
        assert flags2 == 0 and torch.equal(out, out2) and torch.equal(lse, lse2)
    eng.close()


# ------------------------------------------------------------------ int4 group-wise K/V

@pytest.mark.parametrize("groups", [4, 8])
@pytest.mark.parametrize("layout,page", [("contiguous", 0), ("paged", 16), ("paged", 32),
                                         ("paged", 128)])
@pytest.mark.parametrize("splits", [0, 3])
def test_int4_groups(groups, layout, page, splits):
    lens = [1000, 17, 1, 300, 0, 64]
    w = W.make_gqa(name="i4", batch=6, num_q_heads=16, num_kv_heads=2, seq_lens=lens,
                   layout=layout, page_size=page or 16, cache_len=1024 if layout == "contiguous" else None,
                   kv_int4_groups=groups, seed=510 + groups + page + splits)
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"int4 g={groups} {layout}/{page} S={splits}")


@pytest.mark.parametrize("group", [1, 4, 8, 16])
def test_int4_group_sizes_and_two_n_tiles(group):
    w = W.make_gqa(name="i4g", batch=3, num_q_heads=2 * group, num_kv_heads=2, seq_lens=[700, 65, 5],
                   cache_len=704, kv_int4_groups=4, seed=530 + group)
    out, lse, flags, _ = run_gpu(w, num_splits_override=2)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"int4 G={group}")


def test_int4_with_query_tokens_tree_softcap_and_sparse():
    w = W.make_gqa(name="i4q", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[500, 2, 65],
                   layout="paged", page_size=16, q_len=3, tree_mask=True, kv_int4_groups=8, seed=540)
    out, lse, flags, _ = run_gpu(w, num_splits_override=3, softcap=4.0)
    assert flags == 0
    ref_out, ref_lse = reference(w, softcap=4.0)
    assert_parity(out, lse, ref_out, ref_lse, what="int4 q_len=3 tree softcap")
    s = W.make_gqa(name="i4s", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[4096, 4000],
                   cache_len=4096, sparse_block_size=128, kv_num_blks=[[5, 3], [0, 8]],
                   kv_idx=[[[0, 3, 7, 9, 31, 0, 0, 0], [1, 2, 30, 0, 0, 0, 0, 0]],
                           [[0] * 8, [4, 5, 6, 10, 11, 12, 29, 31]]],
                   kv_int4_groups=4, seed=541)
    for S in (0, 2):
        out, lse, flags, _ = run_gpu(s, num_splits_override=S)
        assert flags == 0
        ref_out, ref_lse = reference(s)
        assert_parity(out, lse, ref_out, ref_lse, what=f"int4 sparse S={S}")


# ------------------------------------------------------------------ large batches of short rows

def test_mla_batch_larger_than_the_block():
    # 400 rows: the prologue walks the batch in chunks of the block's 384
    # threads, carrying the tile offset from one chunk to the next
    g = torch.Generator().manual_seed(71)
    lens = torch.randint(0, 300, (400,), generator=g).tolist()
    lens[5] = lens[399] = 0
    w = W.make_mla(name="mla_big", batch=400, seq_lens=lens, seed=72)
    out, lse, flags, _ = run_gpu(w)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="MLA B=400")


def test_gqa_thousands_of_units():
    # 1000 rows x 8 kv heads: each prologue thread scans ~42 units
    g = torch.Generator().manual_seed(74)
    lens = torch.randint(0, 200, (1000,), generator=g).tolist()
    w = W.make_gqa(name="gqa_big", batch=1000, num_q_heads=32, num_kv_heads=8, seq_lens=lens,
                   layout="paged", page_size=16, seed=73)
    out, lse, flags, _ = run_gpu(w)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="GQA B=1000")


# ------------------------------------------------------------------ query range of the f16 operand paths

def _scaled_q(w, factor):
    w.tensors["q"] = (w.tensors["q"].float() * factor).to(torch.bfloat16)
    return w


@pytest.mark.parametrize("factor", [1e5, 1e-6])
@pytest.mark.parametrize("kind", ["e4m3", "e4m3_token", "int4", "e4m3_g16"])
def test_f16_operand_paths_take_any_bf16_query(kind, factor):
    """e4m3 and int4 keys meet Q in f16, whose range is far narrower than bf16's:
    q ~ N(0,1) x 1e5 has elements beyond f16's largest finite value, and
    q ~ N(0,1) x 1e-6 lies in f16's subnormals. The query rows of a kv head are
    scaled by an exact power of two before the f16 rounding and the score
    factor takes it back, so both must match the oracle. For the large queries the scores reach
    ~1e5: the LSE is then checked against a relative bound on top of the
    absolute 1e-3 -- for e4m3 keys (decoded exactly) that of the fp32 score
    arithmetic, 1e-5 |lse| (about 2^-17, a few roundings of a 128-term dot
    product); for int4 keys, whose dequantised value code * scale + shift is
    rounded to f16 (a relative 2^-11 per element), the bound of that rounding
    on any score of the row, 2^-11 * scale * sum_d |q_d| * max |k|, with max |k|
    at most 15 |scale| + |shift| over the cache's coefficient words."""
    kw = dict(kv_fp8=True)
    if kind == "e4m3_token":
        kw = dict(kv_fp8=True, kv_token_scale=True)
    elif kind == "int4":
        kw = dict(kv_int4_groups=4)
    hkv, g = (2, 16) if kind == "e4m3_g16" else (2, 8)
    layout = "paged" if kind == "int4" else "contiguous"
    w = W.make_gqa(name=f"qrange_{kind}", batch=3, num_q_heads=g * hkv, num_kv_heads=hkv,
                   seq_lens=[2000, 129, 1], layout=layout, page_size=16,
                   cache_len=2048 if layout == "contiguous" else None, seed=560, **kw)
    _scaled_q(w, factor)
    for S in (0, 3):
        out, lse, flags, _ = run_gpu(w, num_splits_override=S)
        assert flags == 0
        ref_out, ref_lse = reference(w)
        assert_parity(out, None, ref_out, None, fp8=True, what=f"{kind} x{factor} S={S}")
        lg = lse.double().numpy()
        assert np.all(np.isfinite(lg))
        bound = 1e-3 + 1e-5 * np.abs(ref_lse)
        if kind == "int4":
            # (the spare pages are NaN-poisoned: they hold no key of any row)
            coef = w.tensors["k"][..., :4].reshape(-1).numpy().view(np.float16).astype(np.float64)
            kmax = 15 * np.nanmax(np.abs(coef[0::2])) + np.nanmax(np.abs(coef[1::2]))
            q1 = w.tensors["q"].double().abs().sum(-1).numpy()
            bound = bound + 2.0 ** -11 * w.scale * q1 * kmax
        assert np.all(np.abs(lg - ref_lse) <= bound), f"{kind} x{factor} LSE"


# ------------------------------------------------------------------ flex-style mask_mod / score_mod

def _mods(w, window=True, sink=True, alibi=True, seed=0):
    g = torch.Generator().manual_seed(900 + seed)
    HQ = w.num_q_heads
    if window:
        # per query head: a window of 1..300 positions, or none (-1) for some heads
        win = torch.randint(1, 300, (HQ,), generator=g, dtype=torch.int32)
        win[torch.randint(0, HQ, (max(1, HQ // 4),), generator=g)] = -1
        w.tensors["mask_window"] = win
        if sink:
            w.tensors["mask_sink"] = torch.randint(0, 8, (HQ,), generator=g, dtype=torch.int32)
    if alibi:
        w.tensors["alibi_slopes"] = (torch.rand(HQ, generator=g) * 0.2 - 0.05).to(torch.float32)
    return w


@pytest.mark.parametrize("kind", ["paged", "contiguous_g16", "sparse_full", "query_tokens",
                                  "fp8", "fp8token", "int4", "window_only", "alibi_only"])
@pytest.mark.parametrize("splits", [0, 3])
def test_flex_mods_per_query_head(kind, splits):
    """A sink/window mask_mod and ALiBi slopes that differ between the query heads
    of one kv head's group (some heads with no window at all), against the oracle."""
    lens = [700, 1, 65, 333]
    fp8 = kind in ("fp8", "fp8token")
    if kind == "contiguous_g16":
        w = W.make_gqa(name=kind, batch=4, num_q_heads=32, num_kv_heads=2, seq_lens=lens,
                       cache_len=700, seed=910)
    elif kind == "sparse_full":
        # each list's last two blocks (the row's tail) move to the full-block table,
        # which the mask_mod does not touch
        w = _sparse(seed=911)
        num, idx = w.tensors["kv_num_blks"], w.tensors["kv_idx"]
        assert int(num.min()) == int(num.max()) == 7
        w.tensors["kv_num_blks"] = (num - 2).contiguous()
        w.tensors["kv_full_num_blks"] = torch.full_like(num, 2)
        w.tensors["kv_full_idx"] = torch.cat([idx[..., 5:], idx[..., :5]], -1).contiguous()
    elif kind == "query_tokens":
        w = W.make_gqa(name=kind, batch=4, num_q_heads=8, num_kv_heads=2, seq_lens=lens,
                       layout="paged", page_size=16, q_len=3, seed=912)
    else:
        kw = {"fp8": dict(kv_fp8=True), "fp8token": dict(kv_fp8=True, kv_token_scale=True),
              "int4": dict(kv_int4_groups=4)}.get(kind, {})
        w = W.make_gqa(name=kind, batch=4, num_q_heads=32, num_kv_heads=8, seq_lens=lens,
                       layout="paged", page_size=16, seed=913, **kw)
    _mods(w, window=kind != "alibi_only", alibi=kind != "window_only", seed=splits)
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, fp8=fp8 or kind == "int4", what=f"mods {kind} S={splits}")


def test_flex_mods_that_change_nothing_are_bitwise_the_plain_path():
    w = W.make_gqa(name="noop_mods", batch=3, num_q_heads=16, num_kv_heads=4, seq_lens=[900, 17, 300],
                   layout="paged", page_size=16, seed=914)
    base_out, base_lse, _, eng = run_gpu(w, num_splits_override=2)
    w.tensors["mask_window"] = torch.full((16,), 5000, dtype=torch.int32)
    w.tensors["alibi_slopes"] = torch.zeros(16, dtype=torch.float32)
    out, lse, flags, _ = run_gpu(w, engine=eng)
    assert flags == 0 and torch.equal(out, base_out) and torch.equal(lse, base_lse)


def test_flex_mods_refused_for_mla_and_alibi_with_softcap():
    m = W.make_mla(name="mla_mods", batch=1, seq_lens=[64], seed=915)
    m.tensors["mask_window"] = torch.full((128,), 8, dtype=torch.int32)
    with pytest.raises(da.DecodeAttnError) as e:
        run_gpu(m)
    assert e.value.status == da.DA_ERR_UNSUPPORTED
    w = W.make_gqa(name="alibi_cap", batch=1, num_q_heads=8, num_kv_heads=2, seq_lens=[100],
                   cache_len=100, seed=916)
    w.tensors["alibi_slopes"] = torch.full((8,), 0.1, dtype=torch.float32)
    with pytest.raises(da.DecodeAttnError) as e:
        run_gpu(w, softcap=5.0)
    assert e.value.status == da.DA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ e4m3 tensor-core arithmetic (fp8_mma)

def _assert_p8(out, lse, w, what):
    """Parity of the fp8_mma path: the oracle quantises the queries exactly as the
    kernel does, so the LSE keeps its 1e-3; the weights that meet V are rounded to
    e4m3 by both, the kernel against its running maximum and the oracle against the
    row's, so the outputs may differ by twice the weights' rounding bound, plus the
    bf16 rounding of the output (2^-8 relative) and fp32 slack."""
    import oracle
    ref_out, ref_lse, bound = oracle.decode_p8_bound(oracle.problem_from(w), w.tensors, w.scale)
    got = out.double().numpy()
    assert np.all(np.isfinite(got)), what
    excess = np.abs(got - ref_out) - (2 * bound + 2.0 ** -8 * np.abs(ref_out) + 1e-4)
    assert np.all(excess <= 0), f"{what}: worst excess {excess.max():.3e}"
    fin = np.isfinite(ref_lse)
    lg = lse.double().numpy()
    assert np.array_equal(np.isfinite(lg), fin), what
    if fin.any():
        assert np.max(np.abs(lg[fin] - ref_lse[fin])) <= 1e-3, what
    return float(np.max(np.abs(got - ref_out)))


@pytest.mark.parametrize("kind", ["contiguous", "paged", "g16", "query_tokens", "softcap", "mods",
                                  "sparse"])
@pytest.mark.parametrize("splits", [0, 3])
def test_fp8_mma(kind, splits):
    lens = [3000, 1, 77, 700]
    if kind == "g16":
        w = W.make_gqa(name=kind, batch=4, num_q_heads=32, num_kv_heads=2, seq_lens=lens,
                       cache_len=3000, kv_fp8=True, seed=950)
    elif kind == "query_tokens":
        w = W.make_gqa(name=kind, batch=4, num_q_heads=16, num_kv_heads=4, seq_lens=lens,
                       layout="paged", page_size=16, q_len=3, kv_fp8=True, seed=951)
    elif kind == "sparse":
        g = torch.Generator().manual_seed(952)
        num, idx = W.sparse_lists(2, 4, 4096, 128, keep_random=5, keep_last=2, g=g, max_blocks=12)
        w = W.make_gqa(name=kind, batch=2, num_q_heads=16, num_kv_heads=4, seq_lens=[4096, 4000],
                       cache_len=4096, sparse_block_size=128, kv_num_blks=num, kv_idx=idx,
                       kv_fp8=True, seed=953)
    else:
        w = W.make_gqa(name=kind, batch=4, num_q_heads=32, num_kv_heads=4, seq_lens=lens,
                       layout="paged" if kind != "contiguous" else "contiguous", page_size=16,
                       cache_len=3000 if kind == "contiguous" else None, kv_fp8=True, seed=954)
    if kind == "mods":
        w.tensors["mask_window"] = torch.tensor([100, -1, 5, 2000] * 8, dtype=torch.int32)
        w.tensors["alibi_slopes"] = torch.linspace(-0.02, 0.05, 32, dtype=torch.float32)
    w.fp8_mma = True
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits, softcap=30.0 if kind == "softcap" else 0.0)
    assert flags == 0
    if kind == "softcap":
        import oracle
        ref_out, ref_lse, bound = oracle.decode_p8_bound(oracle.problem_from(w), w.tensors, w.scale,
                                                         softcap=30.0)
        got = out.double().numpy()
        assert np.all(np.abs(got - ref_out) <= 2 * bound + 2.0 ** -8 * np.abs(ref_out) + 1e-4)
        assert np.max(np.abs(lse.double().numpy() - ref_lse)) <= 1e-3
    else:
        _assert_p8(out, lse, w, f"fp8_mma {kind} S={splits}")


def test_fp8_mma_full_size_long_context():
    w = W.config(3)
    w.fp8_mma = True
    out, lse, flags, _ = run_gpu(w)
    assert flags == 0
    err = _assert_p8(out, lse, w, "fp8_mma config 3 shapes")
    assert err <= 3e-2  # the fp8 tolerance holds at this length (the weights' errors average out)


def test_fp8_mma_refused_for_other_caches():
    w = W.make_gqa(name="bf16_mma", batch=1, num_q_heads=8, num_kv_heads=2, seq_lens=[100],
                   cache_len=100, seed=955)
    w.fp8_mma = True
    with pytest.raises(da.DecodeAttnError) as e:
        run_gpu(w)
    assert e.value.status == da.DA_ERR_UNSUPPORTED


@pytest.mark.parametrize("q_len,tree", [(2, False), (4, False), (3, True)])
@pytest.mark.parametrize("splits", [0, 3])
def test_several_query_tokens_on_block_sparse_rows(q_len, tree, splits):
    g = torch.Generator().manual_seed(960 + q_len)
    num, idx = W.sparse_lists(3, 2, 4096, 128, keep_random=6, keep_last=2, g=g, max_blocks=12)
    w = W.make_gqa(name="sparse_q", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[4096, 4000, 3970],
                   cache_len=4096, sparse_block_size=128, kv_num_blks=num, kv_idx=idx, q_len=q_len,
                   tree_mask=tree, seed=961 + q_len)
    out, lse, flags, _ = run_gpu(w, num_splits_override=splits)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what=f"sparse q_len={q_len} tree={tree} S={splits}")
