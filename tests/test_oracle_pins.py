"""Pins for the float64 oracle: it is checked against things other than itself.

* format definitions (bf16 and OCP E4M3, every code, against torch's casts and
  the fixtures in tests/golden/);
* closed forms (one key, equal values, q = 0, two keys) and the shift
  invariance of softmax;
* exact brute force (50-digit decimal) on tiny inputs in every cache layout;
* invariants the definition fixes: split-then-merge equals unsplit, masked
  or unlisted KV has no effect, paged equals contiguous on the de-paged cache,
  sparse equals dense on the compacted cache, MLA equals GQA with
  k = [ckv; kpe] and v = ckv.
"""

import itertools
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from decode_attention_flash_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ------------------------------------------------------------------ decoders

def test_bf16_decoder_every_code():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_double(c & 0xFFFF) for c in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7f and 0xff
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(np.abs(got)) == 448.0


def test_f16_decoder_every_code():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.float16).double().numpy()
    got = np.array([oracle.f16_to_double(c & 0xFFFF) for c in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_decoder_golden_codes():
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code, value in rows:
        got = oracle.e4m3_to_double(int(code, 16))
        if value == "nan":
            assert math.isnan(got)
        else:
            assert got == float(value) and math.copysign(1, got) == math.copysign(1, float(value))


# ------------------------------------------------------------------ core closed forms

def test_core_single_key_returns_value_and_score():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((1, 7))
    out, lse = oracle.softmax_attend(np.array([0.37]), v)
    assert np.array_equal(out, v[0])
    assert lse == 0.37


def test_core_empty_list():
    out, lse = oracle.softmax_attend(np.zeros(0), np.zeros((0, 5)))
    assert np.all(out == 0) and lse == -math.inf


def test_core_equal_values_return_that_value():
    rng = np.random.default_rng(2)
    s = rng.standard_normal(50) * 4
    v = np.tile(rng.standard_normal(9), (50, 1))
    out, _ = oracle.softmax_attend(s, v)
    assert rel_err(out, v[0]) < 1e-14


def test_core_shift_invariance():
    rng = np.random.default_rng(3)
    s = rng.standard_normal(100) * 3
    v = rng.standard_normal((100, 16))
    out0, lse0 = oracle.softmax_attend(s, v)
    for c in (-700.0, -3.5, 0.25, 50.0, 900.0):
        out1, lse1 = oracle.softmax_attend(s + c, v)
        assert rel_err(out1, out0) < 1e-12
        assert abs(lse1 - (lse0 + c)) < 1e-12 * max(1.0, abs(c))


def test_core_uniform_scores_give_mean_and_log_count():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((37, 5))
    out, lse = oracle.softmax_attend(np.zeros(37), v)
    assert rel_err(out, v.mean(axis=0)) < 1e-13
    assert abs(lse - math.log(37)) < 1e-14


def test_core_two_keys_closed_form():
    s0, s1 = 0.3, -1.7
    v = np.array([[1.0, -2.0, 0.5], [3.0, 4.0, -1.0]])
    out, lse = oracle.softmax_attend(np.array([s0, s1]), v)
    sig = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    assert rel_err(out, sig * v[0] + (1 - sig) * v[1]) < 1e-15
    assert abs(lse - math.log(math.exp(s0) + math.exp(s1))) < 1e-15


def test_core_ordering_of_scores_does_not_matter():
    rng = np.random.default_rng(5)
    s = rng.standard_normal(64)
    v = rng.standard_normal((64, 8))
    perm = rng.permutation(64)
    a, la = oracle.softmax_attend(s, v)
    b, lb = oracle.softmax_attend(s[perm], v[perm])
    assert rel_err(a, b) < 1e-14 and abs(la - lb) < 1e-14


def test_core_a_dominant_score_selects_its_value():
    # softmax with one score far above the rest is (numerically) a one-hot
    v = np.array([[1.0, 2.0], [5.0, -7.0], [0.0, 3.0]])
    out, lse = oracle.softmax_attend(np.array([0.0, 800.0, 1.0]), v)
    assert np.array_equal(out, v[1]) and lse == 800.0


# ------------------------------------------------------------------ merge closed forms

def test_merge_single_split_is_identity():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((1, 12))
    out, lse = oracle.merge(o, np.array([1.25]))
    assert np.array_equal(out, o[0]) and lse == 1.25


def test_merge_ignores_empty_splits_and_handles_all_empty():
    rng = np.random.default_rng(7)
    o = rng.standard_normal((3, 4))
    o[1] = np.nan  # an empty split's O is never read
    out, lse = oracle.merge(o, np.array([0.5, -math.inf, 0.5]))
    assert rel_err(out, (o[0] + o[2]) / 2) < 1e-15
    assert abs(lse - (0.5 + math.log(2))) < 1e-15
    out, lse = oracle.merge(o, np.full(3, -math.inf))
    assert np.all(out == 0) and lse == -math.inf


def test_merge_two_splits_closed_form():
    o = np.array([[1.0, 0.0], [0.0, 1.0]])
    a, b = 0.7, -0.4
    out, lse = oracle.merge(o, np.array([a, b]))
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    assert rel_err(out, [wa, 1 - wa]) < 1e-15
    assert abs(lse - math.log(math.exp(a) + math.exp(b))) < 1e-15


# ------------------------------------------------------------------ golden: two keys

def test_golden_two_keys_decode():
    rows = {}
    with open(os.path.join(GOLDEN, "two_keys.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                name, *vals = ln.split()
                rows[name] = [float(x) for x in vals]
    q = torch.tensor([[rows["q"]]], dtype=torch.bfloat16)  # [1][1][2]
    k = torch.tensor([[[rows["k0"], rows["k1"]]]], dtype=torch.bfloat16)  # [1][1][2][2]
    v = torch.tensor([[[rows["v0"], rows["v1"]]]], dtype=torch.bfloat16)
    prob = dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim_qk=2, head_dim_v=2,
                cache_len=2)
    out, lse = oracle.decode(prob, dict(q=q, k=k, v=v, seq_lens=torch.tensor([2])), 1.0)
    s0 = sum(a * b for a, b in zip(rows["q"], rows["k0"]))
    s1 = sum(a * b for a, b in zip(rows["q"], rows["k1"]))
    sig = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = [sig * a + (1 - sig) * b for a, b in zip(rows["v0"], rows["v1"])]
    assert rel_err(out[0, 0], expect) < 1e-15
    assert abs(lse[0, 0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-15


# ------------------------------------------------------------------ brute force (exact decimal)

def _dec(x) -> Decimal:
    return Decimal(float(x))


def _token_dequant(codes, words):
    """e4m3 * scale + shift with the per-row words split by torch (fp16 views)."""
    w = words.to(torch.int32)
    scale = (w & 0xFFFF).to(torch.int16).view(torch.float16).double()
    shift = ((w >> 16) & 0xFFFF).to(torch.int16).view(torch.float16).double()
    return codes.double() * scale.unsqueeze(-1) + shift.unsqueeze(-1)


def _int4_dequant(words, groups):
    """int32 rows [groups coefficient words | D/8 data words] -> float64 [.., D],
    decoded with numpy bit operations: code of element 8w + i = bits 4i.. of
    data word w, times its group's fp16 scale, plus its fp16 shift."""
    u = words.numpy().astype(np.int64) & 0xFFFFFFFF
    data = u[..., groups:]
    codes = (data[..., :, None] >> (4 * np.arange(8))) & 0xF
    codes = codes.reshape(*data.shape[:-1], -1).astype(np.float64)
    D = codes.shape[-1]
    coef = u[..., :groups]
    scale = (coef & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    shift = (coef >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    scale = np.repeat(scale, D // groups, axis=-1)
    shift = np.repeat(shift, D // groups, axis=-1)
    return torch.from_numpy(codes * scale + shift)


def _dec_tanh(x: Decimal) -> Decimal:
    e = (2 * x).exp()
    return (e - 1) / (e + 1)


def brute_force(w: W.Workload, softcap: float = 0.0):
    """Independent 50-digit evaluation straight from the cache layouts."""
    getcontext().prec = 50
    t = w.tensors
    B, HQ, HKV = w.batch, w.num_q_heads, w.num_kv_heads
    G = HQ // HKV
    q = t["q"].double()
    if w.kv_int4_groups:
        k = _int4_dequant(t["k"], w.kv_int4_groups)
        v = _int4_dequant(t["v"], w.kv_int4_groups)
    elif w.kv_fp8 and w.kv_token_scale:
        k = _token_dequant(t["k"], t["k_scale_shift"])
        v = _token_dequant(t["v"], t["v_scale_shift"])
    elif w.kv_fp8:
        k = t["k"].double() * t["k_scale"].double().view(1, -1, 1, 1)
        v = t["v"].double() * t["v_scale"].double().view(1, -1, 1, 1)
    else:
        k, v = t["k"].double(), t["v"].double()
    Q = w.q_len
    out = np.zeros((B, HQ, Q, w.head_dim_v))
    lse = np.zeros((B, HQ, Q))
    for b, hq, tq in itertools.product(range(B), range(HQ), range(Q)):
        n_b = int(t["seq_lens"][b])
        h = hq // G
        full = set()  # positions of the full-block table: no mask_mod there (flex)
        if w.sparse_block_size:
            pos = []
            lists = [(t["kv_num_blks"], t["kv_idx"], False)]
            if "kv_full_num_blks" in t:
                lists.append((t["kv_full_num_blks"], t["kv_full_idx"], True))
            zb, zh = b % (w.sparse_batch or B), h % (w.sparse_heads or HKV)
            for nums, idx, is_full in lists:
                for j in range(int(nums[zb, zh])):
                    blk = int(idx[zb, zh, j])
                    ns = [blk * w.sparse_block_size + i for i in range(w.sparse_block_size)
                          if blk * w.sparse_block_size + i < n_b]
                    pos += ns
                    if is_full:
                        full |= set(ns)
        else:
            pos = list(range(n_b))
        q_pos = n_b - Q + tq  # the query token's own position
        if "mask_window" in t:
            # sink/window mask_mod of query head hq: keep n < sink, or n within the
            # last `window` positions up to the query's (window < 0: no window)
            win = int(t["mask_window"][hq])
            sink = int(t["mask_sink"][hq]) if "mask_sink" in t else 0
            pos = [n for n in pos if n in full or n < sink or win < 0 or n > q_pos - win]
        # query token tq of Q is the row's position n_b - Q + tq: it sees n <= that,
        # or, with a draft-tree mask, the older positions and the new ones its row marks
        if "spec_mask" in t:
            words = t["spec_mask"][b, tq].tolist()
            pos = [n for n in pos if n < n_b - Q or
                   (words[(n - n_b + Q) // 32] >> ((n - n_b + Q) % 32)) & 1]
        else:
            pos = [n for n in pos if n <= n_b - Q + tq]
        keys, vals = [], []
        for n in pos:
            if w.is_mla:
                page = int(t["block_table"][b, n // w.page_size])
                ckv = t["k"][page, n % w.page_size].double()
                kpe = t["v"][page, n % w.page_size].double()
                keys.append(torch.cat([ckv, kpe]))
                vals.append(ckv)
            elif w.paged:
                page = int(t["block_table"][b, n // w.page_size])
                keys.append(k[page, h, n % w.page_size])
                vals.append(v[page, h, n % w.page_size])
            else:
                keys.append(k[b, h, n])
                vals.append(v[b, h, n])
        qi = (b, hq, tq) if Q > 1 else (b, hq)
        qv = torch.cat([q[qi], t["q_pe"][qi].double()]) if w.is_mla else q[qi]
        if not pos:
            lse[b, hq, tq] = -math.inf
            continue
        s = [_dec(w.scale) * sum(_dec(a) * _dec(c) for a, c in zip(qv.tolist(), kk.tolist()))
             for kk in keys]
        if softcap > 0:
            cap = _dec(softcap)
            s = [cap * _dec_tanh(x / cap) for x in s]
        if "alibi_slopes" in t:  # ALiBi score_mod: slope of the head times (n - q_pos)
            slope = _dec(t["alibi_slopes"][hq])
            s = [x + slope * (n - q_pos) for x, n in zip(s, pos)]
        m = max(s)
        e = [(x - m).exp() for x in s]
        den = sum(e)
        for d in range(w.head_dim_v):
            out[b, hq, tq, d] = float(sum(ei * _dec(vv[d]) for ei, vv in zip(e, vals)) / den)
        lse[b, hq, tq] = float(m + den.ln())
    if Q == 1:
        return out[:, :, 0], lse[:, :, 0]
    return out, lse


def _tiny_cases():
    cases = []
    cases.append(W.make_gqa(name="contig", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=4,
                            seq_lens=[5, 1], cache_len=6, seed=11, scale=0.7))
    cases.append(W.make_gqa(name="paged", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=4,
                            seq_lens=[6, 3], layout="paged", page_size=2, seed=12, scale=0.6))
    cases.append(W.make_gqa(name="fp8", batch=1, num_q_heads=2, num_kv_heads=2, head_dim=4,
                            seq_lens=[6], cache_len=6, kv_fp8=True, seed=13, scale=0.5))
    cases.append(W.make_gqa(name="fp8_token", batch=2, num_q_heads=2, num_kv_heads=1, head_dim=4,
                            seq_lens=[6, 3], layout="paged", page_size=2, kv_fp8=True,
                            kv_token_scale=True, seed=19, scale=0.5))
    num = torch.tensor([[2, 1]], dtype=torch.int32)
    idx = torch.tensor([[[2, 0, 0], [1, 0, 0]]], dtype=torch.int32)
    cases.append(W.make_gqa(name="sparse", batch=1, num_q_heads=4, num_kv_heads=2, head_dim=4,
                            seq_lens=[5], cache_len=6, sparse_block_size=2, kv_num_blks=num,
                            kv_idx=idx, seed=14, scale=0.8))
    full = W.make_gqa(name="sparse_full", batch=1, num_q_heads=4, num_kv_heads=2, head_dim=4,
                      seq_lens=[7], cache_len=8, sparse_block_size=2,
                      kv_num_blks=torch.tensor([[1, 0]]), kv_idx=torch.tensor([[[3, 0, 0], [0, 0, 0]]]),
                      seed=20, scale=0.8, poison=False)
    full.tensors["kv_full_num_blks"] = torch.tensor([[1, 2]], dtype=torch.int32)
    full.tensors["kv_full_idx"] = torch.tensor([[[0, 0, 0], [2, 1, 0]]], dtype=torch.int32)
    cases.append(full)
    cases.append(W.make_mla(name="mla", batch=2, num_q_heads=3, ckv_dim=4, kpe_dim=2,
                            seq_lens=[4, 2], page_size=2, seed=15, scale=0.9))
    # several query tokens on the latent cache: causal, with a row shorter than
    # q_len, and a draft-token tree
    cases.append(W.make_mla(name="mla_causal_q3", batch=2, num_q_heads=3, ckv_dim=4, kpe_dim=2,
                            seq_lens=[5, 2], page_size=2, seed=30, scale=0.8, q_len=3))
    cases.append(W.make_mla(name="mla_tree_q4", batch=2, num_q_heads=2, ckv_dim=4, kpe_dim=2,
                            seq_lens=[7, 4], page_size=2, seed=31, scale=0.7, q_len=4,
                            tree_mask=True))
    cases.append(W.make_gqa(name="empty_row", batch=2, num_q_heads=2, num_kv_heads=1,
                            head_dim=3, seq_lens=[0, 2], cache_len=2, seed=16, scale=1.0))
    # several query tokens per row, causal over the new tokens; the second row is
    # shorter than q_len, so its first query token sees no position at all
    cases.append(W.make_gqa(name="causal_q3", batch=2, num_q_heads=4, num_kv_heads=2,
                            head_dim=4, seq_lens=[5, 2], cache_len=6, seed=17, scale=0.7,
                            q_len=3))
    cases.append(W.make_gqa(name="causal_q2_paged", batch=2, num_q_heads=2, num_kv_heads=1,
                            head_dim=4, seq_lens=[5, 3], layout="paged", page_size=2, seed=18,
                            scale=0.6, q_len=2))
    # one block table broadcast over every row and kv head, and one per kv head
    # broadcast over the rows (flex's SPARSE_Z / SPARSE_HQ extents)
    cases.append(W.make_gqa(name="sparse_bcast_1x1", batch=3, num_q_heads=4, num_kv_heads=2,
                            head_dim=4, seq_lens=[7, 3, 8], cache_len=8, sparse_block_size=2,
                            kv_num_blks=[2], kv_idx=[[3, 1, 0]], sparse_shape=(1, 1), seed=21,
                            scale=0.8))
    cases.append(W.make_gqa(name="sparse_bcast_1xH", batch=2, num_q_heads=4, num_kv_heads=2,
                            head_dim=4, seq_lens=[8, 5], cache_len=8, sparse_block_size=2,
                            kv_num_blks=[1, 3], kv_idx=[[2, 0, 0], [0, 2, 3]], sparse_shape=(1, 2),
                            seed=22, scale=0.7))
    # int4 group-wise rows (2 and 4 groups), contiguous and paged
    cases.append(W.make_gqa(name="int4_g2", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                            seq_lens=[6, 2], cache_len=6, kv_int4_groups=2, seed=23, scale=0.6))
    cases.append(W.make_gqa(name="int4_g4_paged", batch=2, num_q_heads=2, num_kv_heads=1,
                            head_dim=32, seq_lens=[5, 3], layout="paged", page_size=2,
                            kv_int4_groups=4, seed=24, scale=0.5))
    # a draft-token tree over the new tokens; the second row is shorter than q_len
    cases.append(W.make_gqa(name="tree_q5", batch=2, num_q_heads=4, num_kv_heads=2,
                            head_dim=4, seq_lens=[8, 3], cache_len=8, seed=19, scale=0.8,
                            q_len=5, tree_mask=True))
    cases.append(W.make_gqa(name="tree_q4_paged", batch=2, num_q_heads=2, num_kv_heads=1,
                            head_dim=4, seq_lens=[6, 4], layout="paged", page_size=2, seed=20,
                            scale=0.7, q_len=4, tree_mask=True))
    # several query tokens over a block-sparse row: the causal mask on the listed blocks
    cases.append(W.make_gqa(name="sparse_q3", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=4,
                            seq_lens=[8, 5], cache_len=8, sparse_block_size=2,
                            kv_num_blks=[[3, 1], [2, 2]], kv_idx=[[[3, 0, 1], [2, 0, 0]], [[2, 1, 0], [0, 2, 0]]],
                            seed=29, scale=0.7, q_len=3))
    # flex-style mods: a per-query-head sink/window mask (heads of one group with
    # different windows, one without a window) and ALiBi slopes
    mw = W.make_gqa(name="sink_window", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=4,
                    seq_lens=[7, 3], cache_len=8, seed=25, scale=0.8)
    mw.tensors["mask_window"] = torch.tensor([2, -1, 1, 3], dtype=torch.int32)
    mw.tensors["mask_sink"] = torch.tensor([1, 0, 2, 0], dtype=torch.int32)
    cases.append(mw)
    al = W.make_gqa(name="alibi_paged", batch=2, num_q_heads=4, num_kv_heads=1, head_dim=4,
                    seq_lens=[6, 4], layout="paged", page_size=2, seed=26, scale=0.7)
    al.tensors["alibi_slopes"] = torch.tensor([0.5, 0.25, -0.125, 0.0], dtype=torch.float32)
    cases.append(al)
    # the full-block table takes the score_mod but not the mask_mod
    sf = W.make_gqa(name="window_full_blocks", batch=1, num_q_heads=4, num_kv_heads=2, head_dim=4,
                    seq_lens=[8], cache_len=8, sparse_block_size=2,
                    kv_num_blks=torch.tensor([[2, 1]]), kv_idx=torch.tensor([[[3, 0, 0], [2, 0, 0]]]),
                    seed=27, scale=0.6, poison=False)
    sf.tensors["kv_full_num_blks"] = torch.tensor([[1, 1]], dtype=torch.int32)
    sf.tensors["kv_full_idx"] = torch.tensor([[[1, 0, 0], [0, 0, 0]]], dtype=torch.int32)
    sf.tensors["mask_window"] = torch.tensor([1, 3, 2, 0], dtype=torch.int32)
    sf.tensors["alibi_slopes"] = torch.tensor([0.3, -0.2, 0.1, 0.05], dtype=torch.float32)
    cases.append(sf)
    # several query tokens: the window moves with each token's position
    mq = W.make_gqa(name="window_alibi_q3", batch=2, num_q_heads=2, num_kv_heads=1, head_dim=4,
                    seq_lens=[7, 4], cache_len=8, seed=28, scale=0.7, q_len=3)
    mq.tensors["mask_window"] = torch.tensor([2, 4], dtype=torch.int32)
    mq.tensors["alibi_slopes"] = torch.tensor([0.2, 0.4], dtype=torch.float32)
    cases.append(mq)
    return cases


@pytest.mark.parametrize("w", _tiny_cases(), ids=lambda w: w.name)
def test_brute_force_tiny(w):
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=2)
    bo, bl = brute_force(w)
    assert np.all(np.isfinite(out))
    fin = np.isfinite(bl)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.all(lse[~fin] == -math.inf)
    assert np.max(np.abs(out - bo)) < 1e-12
    assert np.max(np.abs(lse[fin] - bl[fin])) < 1e-12


# ------------------------------------------------------------------ invariants at moderate size

def test_query_token_t_equals_a_single_token_decode_over_its_prefix():
    # token t of q_len new tokens is position N_b - q_len + t: the same as one
    # query over the first N_b - q_len + 1 + t positions (a shorter row)
    Q = 4
    lens = [70, 3, 129, 1]
    w = W.make_gqa(name="spec", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=32,
                   seq_lens=lens, layout="paged", page_size=16, seed=41, q_len=Q)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=2)
    assert out.shape == (4, 8, Q, 32) and lse.shape == (4, 8, Q)
    for t in range(Q):
        one = dict(w.tensors)
        one["q"] = w.tensors["q"][:, :, t].contiguous()
        one["seq_lens"] = torch.clamp(torch.tensor(lens) - Q + 1 + t, min=0).to(torch.int32)
        prob = dict(oracle.problem_from(w), q_len=1)
        o1, l1 = oracle.decode(prob, one, w.scale, num_threads=2)
        assert np.array_equal(o1, out[:, :, t]) and np.array_equal(l1, lse[:, :, t])
    # rows shorter than q_len: their first tokens see nothing
    assert np.all(lse[3, :, :Q - 1] == -math.inf) and np.all(out[3, :, :Q - 1] == 0)
    assert np.all(lse[1, :, 0] == -math.inf) and np.all(np.isfinite(lse[1, :, 1:]))


def _with_mask(w, rows):
    """The workload with every row's draft mask set to ``rows`` (one int per token)."""
    m = torch.tensor(rows, dtype=torch.int64).view(1, -1, 1).expand(w.batch, -1, -1)
    return dict(w.tensors, spec_mask=m.to(torch.int32).contiguous())


def _pack_int4(codes, scales, shifts):
    """Hand-packed int4 rows: codes [.., D] (0..15), per-group fp16-exact scales
    and shifts [.., G] -> int32 rows in the group-wise layout."""
    G, D = scales.shape[-1], codes.shape[-1]
    words = []
    for gi in range(G):
        sb = int(np.array([scales[gi]], dtype=np.float16).view(np.uint16)[0])
        hb = int(np.array([shifts[gi]], dtype=np.float16).view(np.uint16)[0])
        words.append(sb | (hb << 16))
    for wi in range(D // 8):
        words.append(sum(int(codes[8 * wi + i]) << (4 * i) for i in range(8)))
    return [x - (1 << 32) if x >= (1 << 31) else x for x in words]


def test_int4_every_code_through_a_single_key():
    # one key: out is that key's value row exactly, code * scale + shift of
    # its group, for all sixteen codes in every nibble position and group
    D, G = 64, 4
    codes = np.array([(7 * d + d // 8) % 16 for d in range(D)])
    scales = np.array([0.5, 0.25, 2.0, 0.125])
    shifts = np.array([-3.0, 1.5, -0.75, 4.0])
    row = _pack_int4(codes, scales, shifts)
    k = torch.tensor([[[_pack_int4(codes[::-1].copy(), scales, shifts)]]], dtype=torch.int32)
    v = torch.tensor([[[row]]], dtype=torch.int32)
    q = torch.ones((1, 1, D), dtype=torch.bfloat16)
    prob = dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim_qk=D, head_dim_v=D,
                cache_len=1, kv_fp8=3, kv_groups=G)
    out, lse = oracle.decode(prob, dict(q=q, k=k, v=v, seq_lens=torch.tensor([1])), 0.1)
    want = codes * np.repeat(scales, D // G) + np.repeat(shifts, D // G)
    assert np.array_equal(out[0, 0], want)
    kvals = codes[::-1] * np.repeat(scales, D // G) + np.repeat(shifts, D // G)
    assert abs(lse[0, 0] - 0.1 * kvals.sum()) < 1e-12


@pytest.mark.parametrize("groups", [1, 2, 4, 8])
def test_int4_equals_bf16_on_the_same_values(groups):
    # scales 2^-k and small shifts make every code * scale + shift exact in
    # bf16: the int4 oracle on the packed rows and the bf16 oracle on the
    # values give the same bits
    D = 64
    g = torch.Generator().manual_seed(60 + groups)
    B, HKV, L = 2, 2, 9
    codes = torch.randint(0, 16, (B, HKV, L, D), generator=g).numpy()
    scales = 2.0 ** -torch.randint(0, 4, (B, HKV, L, groups), generator=g).numpy()
    shifts = torch.randint(-8, 8, (B, HKV, L, groups), generator=g).numpy() / 4.0
    packed = [[[_pack_int4(codes[b, h, n], scales[b, h, n], shifts[b, h, n]) for n in range(L)]
               for h in range(HKV)] for b in range(B)]
    vals = codes * np.repeat(scales, D // groups, -1) + np.repeat(shifts, D // groups, -1)
    w = W.make_gqa(name="i4", batch=B, num_q_heads=4, num_kv_heads=HKV, head_dim=D,
                   seq_lens=[9, 4], cache_len=L, seed=61)
    vb = torch.from_numpy(vals).to(torch.bfloat16)
    assert np.array_equal(vb.double().numpy(), vals)
    dense = dict(w.tensors, k=vb, v=torch.flip(vb, dims=[-1]).contiguous())
    o1, l1 = oracle.decode(oracle.problem_from(w), dense, w.scale, num_threads=2)
    pk = torch.tensor(packed, dtype=torch.int32)
    pv = torch.tensor([[[_pack_int4(codes[b, h, n][::-1].copy(),
                                    scales[b, h, n][::-1].copy(), shifts[b, h, n][::-1].copy())
                         for n in range(L)] for h in range(HKV)] for b in range(B)],
                      dtype=torch.int32)
    prob = dict(oracle.problem_from(w), kv_fp8=3, kv_groups=groups)
    o2, l2 = oracle.decode(prob, dict(w.tensors, k=pk, v=pv), w.scale, num_threads=2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("shape", [(1, 1), (1, 2), (3, 1), (2, 2), (2, 8)])
def test_broadcast_block_mask_equals_the_expanded_tables(shape):
    # tables of extents (SZ, SH) read at (b % SZ, h % SH): the same result as
    # tables written out for every (b, kv head); SH = 8 = HQ is the flex
    # template's per-query-head extent, still read at the kv head h
    SZ, SH = shape
    B, HKV, L, blk = 6, 4, 256, 32
    g = torch.Generator().manual_seed(50 + SZ * 10 + SH)
    nb = torch.randint(0, 5, (SZ, SH), generator=g, dtype=torch.int32)
    idx = torch.stack([torch.stack([torch.randperm(L // blk, generator=g)[:5] for _ in range(SH)])
                       for _ in range(SZ)]).to(torch.int32)
    lens = [256, 200, 31, 0, 129, 64]
    w = W.make_gqa(name="bc", batch=B, num_q_heads=8, num_kv_heads=HKV, head_dim=16, seq_lens=lens,
                   cache_len=L, sparse_block_size=blk, kv_num_blks=nb, kv_idx=idx,
                   sparse_shape=shape, seed=51, poison=False)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=2)
    rows = torch.arange(B) % SZ
    heads = torch.arange(HKV) % SH
    full = dict(w.tensors, kv_num_blks=nb[rows][:, heads].contiguous(),
                kv_idx=idx[rows][:, heads].contiguous())
    prob = dict(oracle.problem_from(w), sparse_batch=0, sparse_heads=0)
    o2, l2 = oracle.decode(prob, full, w.scale, num_threads=2)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2)


def test_tree_mask_lower_triangle_is_the_causal_mask():
    Q = 5
    w = W.make_gqa(name="tri", batch=3, num_q_heads=6, num_kv_heads=2, head_dim=16,
                   seq_lens=[40, 3, 17], layout="paged", page_size=4, seed=42, q_len=Q)
    causal = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=2)
    tri = oracle.decode(oracle.problem_from(w), _with_mask(w, [(2 << t) - 1 for t in range(Q)]),
                        w.scale, num_threads=2)
    assert np.array_equal(causal[0], tri[0]) and np.array_equal(causal[1], tri[1])
    # the reversed bit order (the upper triangle) is a different mask
    up = oracle.decode(oracle.problem_from(w),
                       _with_mask(w, [((1 << Q) - 1) ^ ((1 << t) - 1) for t in range(Q)]),
                       w.scale, num_threads=2)
    assert not np.array_equal(causal[0], up[0])


def test_tree_mask_of_all_ones_sees_the_whole_row():
    Q = 3
    lens = [33, 2, 9]
    w = W.make_gqa(name="ones", batch=3, num_q_heads=4, num_kv_heads=1, head_dim=16,
                   seq_lens=lens, cache_len=33, seed=43, q_len=Q)
    out, lse = oracle.decode(oracle.problem_from(w), _with_mask(w, [(1 << Q) - 1] * Q),
                             w.scale, num_threads=2)
    for t in range(Q):
        one = dict(w.tensors, q=w.tensors["q"][:, :, t].contiguous())
        o1, l1 = oracle.decode(dict(oracle.problem_from(w), q_len=1), one, w.scale, num_threads=2)
        assert np.array_equal(o1, out[:, :, t]) and np.array_equal(l1, lse[:, :, t])


def test_tree_mask_each_token_alone_returns_its_value_row():
    # a row made only of the new tokens, each seeing itself alone: one key each,
    # so out is that position's value row and lse its score
    Q = 6
    w = W.make_gqa(name="self", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8,
                   seq_lens=[Q, Q], cache_len=Q, seed=44, scale=0.9, q_len=Q)
    out, lse = oracle.decode(oracle.problem_from(w), _with_mask(w, [1 << t for t in range(Q)]),
                             w.scale, num_threads=2)
    k, v, q = (w.tensors[x].double() for x in ("k", "v", "q"))
    for b, hq, t in itertools.product(range(2), range(4), range(Q)):
        h = hq // 2
        assert np.array_equal(out[b, hq, t], v[b, h, t].numpy())
        assert abs(lse[b, hq, t] - w.scale * float(q[b, hq, t] @ k[b, h, t])) < 1e-12


def _gqa_case(layout="contiguous", seed=21, **kw):
    args = dict(batch=3, num_q_heads=8, num_kv_heads=2, head_dim=32, seq_lens=[70, 1, 129],
                layout=layout, page_size=16, seed=seed)
    args.update(kw)
    return W.make_gqa(**args)


def test_split_then_merge_equals_unsplit():
    w = _gqa_case(seq_lens=[70, 0, 129])
    prob = oracle.problem_from(w)
    out, lse = oracle.decode(prob, w.tensors, w.scale)
    rng = np.random.default_rng(8)
    for _ in range(6):
        cuts = np.sort(rng.integers(0, 140, size=rng.integers(1, 7)))
        bounds = np.concatenate([[0], cuts, [140]])  # repeated cuts give empty chunks
        o_s, l_s = oracle.split(prob, w.tensors, w.scale, bounds)
        mo, ml = oracle.merge(o_s, l_s)
        assert np.max(np.abs(mo - out)) <= 1e-12 * max(1.0, np.max(np.abs(out)))
        fin = np.isfinite(lse)
        assert np.array_equal(np.isfinite(ml), fin)
        assert np.max(np.abs(ml[fin] - lse[fin])) < 1e-12


def test_values_past_sequence_end_have_no_effect():
    w = _gqa_case(poison=False)
    prob = oracle.problem_from(w)
    out, lse = oracle.decode(prob, w.tensors, w.scale)
    t = dict(w.tensors)
    k, v = t["k"].clone(), t["v"].clone()
    for b, n in enumerate(t["seq_lens"].tolist()):
        k[b, :, n:] = 3.0e38
        v[b, :, n:] = -1.0e38
    t.update(k=k, v=v)
    out2, lse2 = oracle.decode(prob, t, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_paged_equals_contiguous_on_depaged_cache():
    w = _gqa_case(layout="paged", page_size=16, poison=False)
    t = w.tensors
    out_p, lse_p = oracle.decode(oracle.problem_from(w), t, w.scale)
    L = w.max_pages_per_seq * w.page_size
    # de-page with torch indexing: token n of row b is page table[b][n // P], slot n % P
    pages = t["block_table"].long()  # [B][max_pages]
    k = t["k"][pages].permute(0, 2, 1, 3, 4).reshape(w.batch, w.num_kv_heads, L, w.head_dim_qk)
    v = t["v"][pages].permute(0, 2, 1, 3, 4).reshape(w.batch, w.num_kv_heads, L, w.head_dim_v)
    c = W.Workload(name="depaged", batch=w.batch, num_q_heads=w.num_q_heads,
                   num_kv_heads=w.num_kv_heads, head_dim_qk=w.head_dim_qk,
                   head_dim_v=w.head_dim_v, scale=w.scale, cache_len=L)
    out_c, lse_c = oracle.decode(oracle.problem_from(c), dict(q=t["q"], k=k.contiguous(),
                                 v=v.contiguous(), seq_lens=t["seq_lens"]), w.scale)
    assert np.array_equal(out_p, out_c) and np.array_equal(lse_p, lse_c)


def _sparse_case(seed=31, poison=True):
    g = torch.Generator().manual_seed(seed)
    num, idx = W.sparse_lists(2, 2, 1024, 64, keep_random=3, keep_last=2, g=g, max_blocks=16)
    return W.make_gqa(name="sparse", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                      seq_lens=[1000, 1024], cache_len=1024, sparse_block_size=64,
                      kv_num_blks=num, kv_idx=idx, seed=seed, poison=poison)


def test_sparse_equals_dense_on_compacted_cache():
    w = _sparse_case(poison=True)
    t = w.tensors
    out_s, lse_s = oracle.decode(oracle.problem_from(w), t, w.scale)
    assert np.all(np.isfinite(out_s))  # NaN-poisoned unlisted blocks never reached
    # compact each (b, h) list into its own dense row, then attend densely
    rows_k, rows_v, lens = [], [], []
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            blocks = t["kv_idx"][b, h, :int(t["kv_num_blks"][b, h])].long()
            pos = (blocks[:, None] * 64 + torch.arange(64)).reshape(-1)
            pos = pos[pos < int(t["seq_lens"][b])]
            rows_k.append(t["k"][b, h, pos])
            rows_v.append(t["v"][b, h, pos])
            lens.append(pos.numel())
    L = max(lens)
    BH = w.batch * w.num_kv_heads
    k = torch.zeros((BH, 1, L, 16), dtype=torch.bfloat16)
    v = torch.zeros((BH, 1, L, 16), dtype=torch.bfloat16)
    for i in range(BH):
        k[i, 0, :lens[i]] = rows_k[i]
        v[i, 0, :lens[i]] = rows_v[i]
    # one dense "batch row" per (b, kv head), holding that head's G query heads
    G = w.group
    q = t["q"].reshape(BH, G, 16)
    dense = dict(batch=BH, num_q_heads=G, num_kv_heads=1, head_dim_qk=16, head_dim_v=16,
                 cache_len=L)
    out_d, lse_d = oracle.decode(dense, dict(q=q, k=k, v=v, seq_lens=torch.tensor(lens)), w.scale)
    assert np.array_equal(out_s.reshape(BH, G, 16), out_d)
    assert np.array_equal(lse_s.reshape(BH, G), lse_d)


def test_unlisted_sparse_blocks_have_no_effect():
    w = _sparse_case(poison=False)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    t = dict(w.tensors)
    k, v = t["k"].clone(), t["v"].clone()
    for b in range(w.batch):
        for h in range(w.num_kv_heads):
            keep = torch.zeros(16, dtype=torch.bool)
            keep[t["kv_idx"][b, h, :int(t["kv_num_blks"][b, h])].long()] = True
            mask = keep.repeat_interleave(64) & (torch.arange(1024) < int(t["seq_lens"][b]))
            k[b, h, ~mask] = 1.0e30
            v[b, h, ~mask] = -5.0e30
    t.update(k=k, v=v)
    out2, lse2 = oracle.decode(oracle.problem_from(w), t, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_mla_equals_gqa_with_concatenated_keys():
    w = W.make_mla(batch=3, num_q_heads=16, ckv_dim=32, kpe_dim=8, seq_lens=[100, 7, 64],
                   page_size=16, seed=41)
    t = w.tensors
    out_m, lse_m = oracle.decode(oracle.problem_from(w), t, w.scale)
    # the same problem as GQA with one kv head: k = [ckv ; kpe], v = ckv, q = [q_nope ; q_pe]
    q = torch.cat([t["q"], t["q_pe"]], dim=-1)
    k = torch.cat([t["k"], t["v"]], dim=-1).unsqueeze(1)  # [pages][1][P][40]
    v = t["k"].unsqueeze(1)
    prob = dict(batch=3, num_q_heads=16, num_kv_heads=1, head_dim_qk=40, head_dim_v=32,
                paged=1, page_size=16, max_pages_per_seq=w.max_pages_per_seq,
                num_pages=w.num_pages)
    out_g, lse_g = oracle.decode(prob, dict(q=q, k=k.contiguous(), v=v.contiguous(),
                                            block_table=t["block_table"], seq_lens=t["seq_lens"]),
                                 w.scale)
    assert np.array_equal(out_m, out_g) and np.array_equal(lse_m, lse_g)


def test_fp8_dequant_equals_bf16_path_on_dequantised_values():
    w = _gqa_case(kv_fp8=True, poison=False, seq_lens=[33, 2, 64], head_dim=16)
    t = w.tensors
    out8, lse8 = oracle.decode(oracle.problem_from(w), t, w.scale)
    # the dequantised cache, formed by torch, is not always exact in bf16, so compare
    # against a float64 evaluation of the same values (numpy, per row)
    kd = t["k"].double() * t["k_scale"].double().view(1, -1, 1, 1)
    vd = t["v"].double() * t["v_scale"].double().view(1, -1, 1, 1)
    q = t["q"].double()
    for b in range(w.batch):
        n = int(t["seq_lens"][b])
        for hq in range(w.num_q_heads):
            h = hq // w.group
            s = w.scale * (kd[b, h, :n] @ q[b, hq]).numpy()
            o, l = oracle.softmax_attend(s, vd[b, h, :n].numpy())
            assert np.max(np.abs(o - out8[b, hq])) < 1e-12
            assert abs(l - lse8[b, hq]) < 1e-12


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_fp8_per_token_scale_shift_equals_float64_on_dequantised_values(layout):
    # value = e4m3 * scale[row] + shift[row]: against a numpy evaluation of the
    # same dequantised rows, gathered through the table independently
    w = _gqa_case(layout=layout, kv_fp8=True, kv_token_scale=True, poison=False,
                  seq_lens=[33, 2, 64], head_dim=16, seed=27)
    t = w.tensors
    assert oracle.problem_from(w)["kv_fp8"] == 2
    out8, lse8 = oracle.decode(oracle.problem_from(w), t, w.scale)
    kd = _token_dequant(t["k"], t["k_scale_shift"])
    vd = _token_dequant(t["v"], t["v_scale_shift"])
    q = t["q"].double()
    for b in range(w.batch):
        n = int(t["seq_lens"][b])
        for hq in range(w.num_q_heads):
            h = hq // w.group
            if layout == "paged":
                rows = [(int(t["block_table"][b, i // w.page_size]), i % w.page_size) for i in range(n)]
                kk = torch.stack([kd[pg, h, r] for pg, r in rows]) if rows else kd[0, h, :0]
                vv = torch.stack([vd[pg, h, r] for pg, r in rows]) if rows else vd[0, h, :0]
            else:
                kk, vv = kd[b, h, :n], vd[b, h, :n]
            s_ = w.scale * (kk @ q[b, hq]).numpy()
            o, l = oracle.softmax_attend(s_, vv.numpy())
            assert np.max(np.abs(o - out8[b, hq])) < 1e-12
            assert abs(l - lse8[b, hq]) < 1e-12


def test_fp8_per_token_shift_alone_moves_scores_by_q_sum():
    # the same codes and scales with every key shift 0, then every key shift c:
    # each score of a row grows by c * sum_d q[d], so the softmax is unchanged
    # and the LSE grows by scale * c * sum(q)
    w = _gqa_case(kv_fp8=True, kv_token_scale=True, poison=False, seq_lens=[40, 9, 1],
                  head_dim=16, seed=28)
    words = w.tensors["k_scale_shift"] & 0xFFFF  # the scales, shift 0
    c = torch.tensor(0.375, dtype=torch.float16)  # exact in fp16 and float64
    t0, t1 = dict(w.tensors), dict(w.tensors)
    t0["k_scale_shift"] = words
    t1["k_scale_shift"] = words | (int(c.view(torch.int16)) << 16)
    out0, lse0 = oracle.decode(oracle.problem_from(w), t0, w.scale)
    out1, lse1 = oracle.decode(oracle.problem_from(w), t1, w.scale)
    qsum = w.tensors["q"].double().sum(-1).numpy()  # [B][HQ]
    assert np.max(np.abs(out1 - out0)) < 1e-12
    assert np.max(np.abs(lse1 - lse0 - w.scale * 0.375 * qsum)) < 1e-9


def test_full_block_table_equals_appending_its_blocks_to_the_first():
    # without a mask_mod, the flex block mask's FULL_KV tables are attended like
    # the KV tables: the same result as one list holding both, in that order
    w = _sparse_case(poison=False)
    t = dict(w.tensors)
    nb, idx = t["kv_num_blks"], t["kv_idx"]
    keep = (nb // 2).to(torch.int32)  # first half of each list stays, the rest moves
    full_n = (nb - keep).to(torch.int32)
    full_idx = torch.zeros_like(idx)
    part_idx = torch.zeros_like(idx)
    for b in range(idx.shape[0]):
        for h in range(idx.shape[1]):
            k, n = int(keep[b, h]), int(nb[b, h])
            part_idx[b, h, :k] = idx[b, h, :k]
            full_idx[b, h, :n - k] = idx[b, h, k:n]
    split = dict(t, kv_num_blks=keep, kv_idx=part_idx, kv_full_num_blks=full_n, kv_full_idx=full_idx)
    o1, l1 = oracle.decode(oracle.problem_from(w), t, w.scale, num_threads=2)
    o2, l2 = oracle.decode(oracle.problem_from(w), split, w.scale, num_threads=2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # a bad full-list entry is an index error, like a bad first-list entry
    assert int(full_n[0, 0]) > 0
    bad = dict(split, kv_full_idx=full_idx.clone())
    bad["kv_full_idx"][0, 0, 0] = 10 ** 6
    with pytest.raises(ValueError):
        oracle.decode(oracle.problem_from(w), bad, w.scale)


@pytest.mark.parametrize("softcap", [0.5, 3.0])
def test_softcap_brute_force(softcap):
    # tanh soft-capping of the scaled score, against 50-digit exp-based tanh
    w = W.make_gqa(name="cap", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=4,
                   seq_lens=[5, 2], cache_len=6, seed=21, scale=1.7)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=2,
                             softcap=softcap)
    bo, bl = brute_force(w, softcap=softcap)
    assert np.max(np.abs(out - bo)) < 1e-12 and np.max(np.abs(lse - bl)) < 1e-12


def test_softcap_limits():
    w = _gqa_case(seed=22)
    o0, l0 = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    # a cap far above every score changes them by O(s^3 / cap^2): nothing at 1e-9
    o1, l1 = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, softcap=1e6)
    assert np.max(np.abs(o1 - o0)) < 1e-9 and np.max(np.abs(l1 - l0)) < 1e-9
    # a tiny cap flattens every score to about +-cap: weights within e^(2 cap) of
    # each other, so the output is the plain mean of the values within that ratio
    cap = 1e-6
    o2, l2 = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, softcap=cap)
    t = w.tensors
    for b in range(w.batch):
        n = int(t["seq_lens"][b])
        for hq in range(w.num_q_heads):
            h = hq // w.group
            mean = t["v"][b, h, :n].double().mean(0).numpy()
            assert np.max(np.abs(o2[b, hq] - mean)) < 1e-5
            assert abs(l2[b, hq] - math.log(n)) < 1e-5


def test_bad_page_index_is_reported():
    w = _gqa_case(layout="paged")
    t = dict(w.tensors)
    bt = t["block_table"].clone()
    bt[0, 0] = w.num_pages  # out of the pool
    t["block_table"] = bt
    with pytest.raises(ValueError):
        oracle.decode(oracle.problem_from(w), t, w.scale)


def test_threads_do_not_change_results():
    w = _gqa_case(layout="paged")
    a = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=1)
    b = oracle.decode(oracle.problem_from(w), w.tensors, w.scale, num_threads=7)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_int4_row_from_hand_encoded_words():
    # tests/golden/int4_row.txt: coefficient and data words written out by
    # hand; with one key the oracle's output row is that value row exactly
    words, probes = None, []
    with open(os.path.join(GOLDEN, "int4_row.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("words"):
                words = [int(x, 16) for x in line.split()[1:]]
            else:
                i, v = line.split()
                probes.append((int(i), float(v)))
    assert words is not None and len(words) == 4 + 64 // 8 and len(probes) == 16
    row = [x - (1 << 32) if x >= (1 << 31) else x for x in words]
    zero_key = [0] * 4 + [0] * 8  # scale 0, shift 0, codes 0: a zero key
    k = torch.tensor([[[zero_key]]], dtype=torch.int32)
    v = torch.tensor([[[row]]], dtype=torch.int32)
    q = torch.ones((1, 1, 64), dtype=torch.bfloat16)
    prob = dict(batch=1, num_q_heads=1, num_kv_heads=1, head_dim_qk=64, head_dim_v=64,
                cache_len=1, kv_fp8=3, kv_groups=4)
    out, lse = oracle.decode(prob, dict(q=q, k=k, v=v, seq_lens=torch.tensor([1])), 0.1)
    for i, want in probes:
        assert out[0, 0, i] == want, (i, out[0, 0, i], want)
    assert lse[0, 0] == 0.0  # one key with score 0


# ------------------------------------------------------------------ flex-style mask_mod / score_mod

def _mods_case(seed=41, **kw):
    return W.make_gqa(name="mods", batch=3, num_q_heads=8, num_kv_heads=2, seq_lens=[300, 41, 1],
                      cache_len=300, seed=seed, **kw)


def test_window_wider_than_the_row_and_zero_slopes_change_nothing():
    w = _mods_case()
    base = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    t = dict(w.tensors)
    t["mask_window"] = torch.full((8,), 400, dtype=torch.int32)
    t["alibi_slopes"] = torch.zeros(8, dtype=torch.float32)
    out = oracle.decode(oracle.problem_from(w), t, w.scale)
    assert np.array_equal(out[0], base[0]) and np.array_equal(out[1], base[1])


def test_sink_alone_equals_a_decode_over_the_first_positions():
    # window 0 keeps no recent position: only the sink's first positions remain,
    # i.e. the same as a row of length `sink`
    w = _mods_case(seed=42)
    t = dict(w.tensors)
    t["mask_window"] = torch.zeros(8, dtype=torch.int32)
    t["mask_sink"] = torch.full((8,), 20, dtype=torch.int32)
    out, lse = oracle.decode(oracle.problem_from(w), t, w.scale)
    short = dict(w.tensors)
    short["seq_lens"] = torch.minimum(w.tensors["seq_lens"], torch.tensor(20, dtype=torch.int32))
    ref_out, ref_lse = oracle.decode(oracle.problem_from(w), short, w.scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def test_window_equals_a_decode_over_the_last_positions():
    # a window of W (no sink) keeps the last W positions: the same scores as a
    # cache holding only them (the row's tail moved to the front)
    w = _mods_case(seed=43)
    Wn = 17
    t = dict(w.tensors)
    t["mask_window"] = torch.full((8,), Wn, dtype=torch.int32)
    out, lse = oracle.decode(oracle.problem_from(w), t, w.scale)
    tail = dict(w.tensors)
    k, v = w.tensors["k"].clone(), w.tensors["v"].clone()
    lens = w.tensors["seq_lens"].clone()
    for b, n in enumerate(w.tensors["seq_lens"].tolist()):
        lo = max(0, n - Wn)
        k[b, :, :n - lo] = w.tensors["k"][b, :, lo:n]
        v[b, :, :n - lo] = w.tensors["v"][b, :, lo:n]
        lens[b] = n - lo
    tail.update(k=k, v=v, seq_lens=lens)
    ref_out, ref_lse = oracle.decode(oracle.problem_from(w), tail, w.scale)
    assert np.max(np.abs(out - ref_out)) < 1e-12 and np.max(np.abs(lse - ref_lse)) < 1e-12


def test_alibi_two_keys_closed_form():
    # two keys at positions 0 and 1, query at position 1: scores s0 - slope and s1
    w = W.make_gqa(name="alibi2", batch=1, num_q_heads=1, num_kv_heads=1, head_dim=4,
                   seq_lens=[2], cache_len=2, seed=44, scale=0.5)
    w.tensors["alibi_slopes"] = torch.tensor([0.75], dtype=torch.float32)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    q = w.tensors["q"][0, 0].double()
    k = w.tensors["k"][0, 0].double()
    v = w.tensors["v"][0, 0].double()
    s0 = float(w.scale * (q @ k[0])) - 0.75
    s1 = float(w.scale * (q @ k[1]))
    sig = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = sig * v[0].numpy() + (1 - sig) * v[1].numpy()
    assert np.max(np.abs(out[0, 0] - expect)) < 1e-14
    assert abs(lse[0, 0] - math.log(math.exp(s0) + math.exp(s1))) < 1e-14


def test_mask_mod_skips_the_full_block_table():
    # with every position in the full table, a mask that would drop them all
    # changes nothing (flex applies no mask_mod to full blocks)
    w = W.make_gqa(name="fullonly", batch=1, num_q_heads=2, num_kv_heads=1, seq_lens=[256],
                   cache_len=256, sparse_block_size=64, kv_num_blks=torch.tensor([[0]]),
                   kv_idx=torch.zeros((1, 1, 4), dtype=torch.int32), seed=45, poison=False)
    w.tensors["kv_full_num_blks"] = torch.tensor([[4]], dtype=torch.int32)
    w.tensors["kv_full_idx"] = torch.tensor([[[0, 1, 2, 3]]], dtype=torch.int32)
    base = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    t = dict(w.tensors)
    t["mask_window"] = torch.zeros(2, dtype=torch.int32)
    out = oracle.decode(oracle.problem_from(w), t, w.scale)
    assert np.array_equal(out[0], base[0]) and np.array_equal(out[1], base[1])


def test_softcap_with_alibi_is_refused():
    w = _mods_case(seed=46)
    t = dict(w.tensors)
    t["alibi_slopes"] = torch.full((8,), 0.1, dtype=torch.float32)
    with pytest.raises(ValueError):
        oracle.decode(oracle.problem_from(w), t, w.scale, softcap=5.0)


# ------------------------------------------------------------------ e4m3 tensor-core arithmetic (fp8_mma)

def test_e4m3_encoder_matches_torch_rounding():
    # every e4m3 value, every midpoint between neighbours (ties to even), and
    # random floats in range, against torch's float32 -> float8_e4m3fn cast
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    fin = vals[torch.isfinite(vals)].unique()
    mids = (fin[1:] + fin[:-1]) / 2
    g = torch.Generator().manual_seed(61)
    rnd = (torch.rand(20000, generator=g) * 2 - 1) * 448 * torch.rand(20000, generator=g) ** 6
    xs = torch.cat([fin, mids, rnd, -rnd]).float()
    want = xs.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle.e4m3_encode(x) for x in xs.tolist()]
    assert got == want
    # saturation and NaN, from the format (448 is the largest finite value)
    assert oracle.e4m3_encode(449.0) == 0x7E and oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE and oracle.e4m3_encode(float("nan")) == 0x7F


def test_f16_rounding_matches_numpy():
    g = np.random.default_rng(62)
    xs = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-9, 5, 20000),
                         np.float16(np.arange(1, 2000, dtype=np.float16)).astype(np.float64) * 1.000244140625])
    for x in xs[:5000].tolist() + xs[20000:].tolist():
        assert oracle.f16_round(x) == float(np.float16(x))


def _mma_case(seed, lens=(257, 1, 40), exact_q=False, G=4, paged=False):
    w = W.make_gqa(name="fp8mma", batch=len(lens), num_q_heads=2 * G, num_kv_heads=2,
                   seq_lens=list(lens), cache_len=None if paged else max(lens), kv_fp8=True,
                   layout="paged" if paged else "contiguous", page_size=16, seed=seed)
    w.fp8_mma = True
    if exact_q:
        # query rows of e4m3 values times a power of two, each holding 448 * 2^j:
        # the quantisation is then exact (scale 2^j, codes the values themselves)
        g = torch.Generator().manual_seed(seed + 1)
        codes = torch.randint(0, 256, w.tensors["q"].shape, generator=g, dtype=torch.int32)
        v = codes.to(torch.uint8).view(torch.float8_e4m3fn).float()
        v = torch.where(torch.isfinite(v), v, torch.zeros_like(v))
        v[..., 0] = 448.0
        j = torch.randint(-8, 3, w.tensors["q"].shape[:-1] + (1,), generator=g).float()
        w.tensors["q"] = (v * torch.exp2(j)).to(torch.bfloat16)
    return w


def test_fp8_mma_single_key_returns_the_value_row_and_exact_queries_keep_their_scores():
    w = _mma_case(63, lens=(1, 1, 1), exact_q=True)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    plain = oracle.problem_from(w)
    plain["fp8_mma"] = 0
    ref_out, ref_lse = oracle.decode(plain, w.tensors, w.scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def test_fp8_mma_equal_scores_give_the_mean():
    # q = 0: every weight is 1 (exact in e4m3 after the 2^8 scaling): the mean of the values
    w = _mma_case(64, lens=(300, 17, 2))
    w.tensors["q"] = torch.zeros_like(w.tensors["q"])
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    plain = oracle.problem_from(w)
    plain["fp8_mma"] = 0
    ref_out, ref_lse = oracle.decode(plain, w.tensors, w.scale)
    assert np.array_equal(out, ref_out) and np.array_equal(lse, ref_lse)


def test_fp8_mma_weight_rounding_stays_within_the_reported_bound():
    # with exactly representable queries, the only difference from exact weights is
    # the rounding of the weights, which the bound covers (one side rounds)
    w = _mma_case(65, lens=(1000, 64, 3), exact_q=True)
    out, lse, bound = oracle.decode_p8_bound(oracle.problem_from(w), w.tensors, w.scale)
    plain = oracle.problem_from(w)
    plain["fp8_mma"] = 0
    ref_out, ref_lse = oracle.decode(plain, w.tensors, w.scale)
    assert np.array_equal(lse, ref_lse)
    assert np.all(np.abs(out - ref_out) <= bound * (1 + 1e-12))
    assert np.max(np.abs(out - ref_out)) > 0  # the rounding did act


def test_fp8_mma_brute_force():
    """50-digit evaluation with the roundings done by torch's own casts:
    the query in fp32 steps (amax, 448 / amax, q * inv, e4m3 cast, amax / 448),
    the weights through float16 then float8_e4m3fn."""
    getcontext().prec = 50
    w = _mma_case(66, lens=(9, 2, 5), G=2)
    w.tensors["q"] = (w.tensors["q"].float() * 37.0).to(torch.bfloat16)
    out, lse = oracle.decode(oracle.problem_from(w), w.tensors, w.scale)
    t = w.tensors
    k = t["k"].double() * t["k_scale"].double().view(1, -1, 1, 1)
    v = t["v"].double() * t["v_scale"].double().view(1, -1, 1, 1)
    for b in range(w.batch):
        for hq in range(w.num_q_heads):
            h = hq // (w.num_q_heads // w.num_kv_heads)
            q = t["q"][b, hq].float()
            amax = q.abs().max()
            inv = torch.tensor(448.0, dtype=torch.float32) / amax
            codes = (q * inv).clamp(-448, 448).to(torch.float8_e4m3fn).float().double()
            sq = float(amax / torch.tensor(448.0, dtype=torch.float32))
            qt = [_dec(c) * _dec(sq) for c in codes.tolist()]
            n = int(t["seq_lens"][b])
            s = [_dec(w.scale) * sum(a * _dec(c) for a, c in zip(qt, k[b, h, j].tolist())) for j in range(n)]
            m = max(s)
            p = [(x - m).exp() for x in s]
            l = sum(p)
            wts = []
            for pj in p:
                y = torch.tensor(float(256 * pj), dtype=torch.float64).to(torch.float16).float()
                wts.append(_dec(float(y.to(torch.float8_e4m3fn).float())) / 256)
            for d in range(w.head_dim_v):
                ref = float(sum(wj * _dec(v[b, h, j, d]) for j, wj in enumerate(wts)) / l)
                assert abs(out[b, hq, d] - ref) < 1e-12
            assert abs(lse[b, hq] - float(m + l.ln())) < 1e-12
