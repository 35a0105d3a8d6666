"""Seeded synthetic inputs for decode attention (shared by tests, bench and smoke).

This module only draws random numbers and lays them out in the cache formats
the library reads; it holds none of the attention arithmetic. Everything is
generated on the CPU with a seeded ``torch.Generator`` so the CUDA path and
the float64 oracle see bit-identical inputs.

Layouts (row-major, last index fastest):
  q            bf16 [B][HQ][D]          query head hq reads kv head hq // G
               (q_len > 1: [B][HQ][q_len][D], the row's last q_len tokens)
  k, v         contiguous bf16|e4m3 [B][HKV][L][D]
               paged      bf16      [num_pages][HKV][page_size][D]
  MLA          q_nope [B][HQ][512], q_pe [B][HQ][64],
               ckv [num_pages][page_size][512], kpe [num_pages][page_size][64]
  block_table  int32 [B][max_pages_per_seq]
  seq_lens     int32 [B]
  kv_num_blks  int32 [B][HKV],  kv_idx int32 [B][HKV][max_sparse_blocks]
  k_scale, v_scale  fp32 [HKV] (fp8 KV with per-kv-head scales)
  k_scale_shift, v_scale_shift  int32, one word per cache row (fp8 KV with
               per-token scales): fp16 scale in the low half, fp16 shift in
               the high half; contiguous [B][HKV][L], paged [pages][HKV][P]

Conventions of the synthetic data:
  * paged pools hold sum_b ceil(N_b / page_size) pages plus 64 spare pages;
    one seeded permutation of the page ids is handed out in consecutive
    runs to rows b = 0..B-1; unused block-table slots are 0;
  * spare pages, the slots past N_b in a row's last page, and unlisted
    sparse blocks are filled with NaN, so any read of them shows up in the
    output;
  * fp8 KV is quantised per kv head with scale = amax / 448 and a
    round-to-nearest-even saturating cast to float8_e4m3fn; with per-token
    scales each cache row gets shift = (max + min) / 2 and scale =
    (max - min) / 2 / 448, both rounded to fp16, then the same cast of
    (x - shift) / scale.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

SPARE_PAGES = 64
E4M3_MAX = 448.0


@dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim_qk: int
    head_dim_v: int
    scale: float
    is_mla: bool = False
    ckv_dim: int = 0
    kpe_dim: int = 0
    paged: bool = False
    page_size: int = 0
    cache_len: int = 0
    max_pages_per_seq: int = 0
    num_pages: int = 0
    kv_fp8: bool = False
    sparse_block_size: int = 0
    max_sparse_blocks: int = 0
    num_splits: int = 0  # 0: planner decides
    q_len: int = 1       # query tokens per row
    sparse_batch: int = 0  # block mask extents (batch, kv heads), broadcast by
    sparse_heads: int = 0  # modulo; 0 = the problem's
    kv_token_scale: bool = False  # fp8 KV with a per-token fp16 scale and shift
    fp8_mma: bool = False         # e4m3 tensor-core QK / PV (Q and the PV weights rounded to e4m3)
    kv_int4_groups: int = 0       # int4 group-wise KV: the number of groups per row
    tensors: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_seq_len(self) -> int:
        return self.max_pages_per_seq * self.page_size if self.paged else self.cache_len

    def to(self, device) -> dict:
        """The tensors moved to ``device`` (non-blocking from pinned memory when possible)."""
        return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.tensors.items()}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _lengths(batch: int, lo: int, hi: int, g) -> torch.Tensor:
    """Per-row lengths drawn uniformly from the integers lo..hi (inclusive)."""
    return torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int32)


def _page_pool(seq_lens: torch.Tensor, page_size: int, g, spare: int = SPARE_PAGES):
    """Block table from one seeded permutation of a shared page pool."""
    pages_per_row = [(int(n) + page_size - 1) // page_size for n in seq_lens.tolist()]
    num_pages = sum(pages_per_row) + spare
    max_pages = max(max(pages_per_row, default=0), 1)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    table = torch.zeros((len(pages_per_row), max_pages), dtype=torch.int32)
    used = torch.zeros(num_pages, dtype=torch.bool)
    off = 0
    for b, np_ in enumerate(pages_per_row):
        table[b, :np_] = perm[off:off + np_]
        used[perm[off:off + np_].long()] = True
        off += np_
    return table, num_pages, max_pages, used


def _poison_paged(cache: torch.Tensor, table, seq_lens, page_size, used, head_axis: bool):
    """NaN into spare pages and into the slots past N_b of each row's last page."""
    nan = float("nan")
    cache[~used] = nan
    for b, n in enumerate(seq_lens.tolist()):
        if n % page_size:
            last = int(table[b, n // page_size])
            if head_axis:
                cache[last, :, n % page_size:] = nan
            else:
                cache[last, n % page_size:] = nan


def quantize_e4m3_per_token(x: torch.Tensor):
    """Per cache row (last axis = D) asymmetric e4m3: fp16 shift = (max + min) / 2,
    fp16 scale = (max - min) / 2 / 448 (1 for a constant row), RNE saturating
    cast of (x - shift) / scale. NaN rows stay NaN. Returns (codes, scale_shift
    int32 words: scale bits low, shift bits high)."""
    finite = torch.nan_to_num(x, nan=0.0)
    mx, mn = finite.amax(dim=-1), finite.amin(dim=-1)
    shift = ((mx + mn) / 2).to(torch.float16)
    scale = ((mx - mn) / 2 / E4M3_MAX).to(torch.float16)
    scale = torch.where(scale > 0, scale, torch.ones_like(scale))
    y = ((finite - shift.float().unsqueeze(-1)) / scale.float().unsqueeze(-1))
    y = y.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    y = y.view(torch.uint8).masked_fill(torch.isnan(x), 0x7F).view(torch.float8_e4m3fn)
    words = (scale.view(torch.int16).to(torch.int32) & 0xFFFF) | (
        shift.view(torch.int16).to(torch.int32) << 16)
    return y.contiguous(), words.contiguous()


def quantize_int4_groups(x: torch.Tensor, groups: int):
    """Int4 group-wise asymmetric rows (last axis = D): per group fp16 shift =
    min and fp16 scale = (max - min) / 15 (1 for a constant group), codes
    round((x - shift) / scale) clamped to 0..15. Returns int32 rows of
    ``groups`` coefficient words (scale bits low, shift bits high) followed by
    D / 8 words of eight codes, element 8w + i in bits 4i.. of word w. Rows
    holding NaN get NaN coefficients."""
    D = x.shape[-1]
    if x.dim() > 1 and x.shape[0] > 1 and x.numel() > (1 << 24):  # in slices, to bound memory
        n = max(1, (1 << 24) // (x.numel() // x.shape[0]))
        return torch.cat([quantize_int4_groups(x[i:i + n], groups)
                          for i in range(0, x.shape[0], n)]).contiguous()
    finite = torch.nan_to_num(x, nan=0.0)
    xg = finite.reshape(*x.shape[:-1], groups, D // groups)
    mx, mn = xg.amax(dim=-1), xg.amin(dim=-1)
    shift = mn.to(torch.float16)
    scale = ((mx - mn) / 15).to(torch.float16)
    scale = torch.where(scale > 0, scale, torch.ones_like(scale))
    codes = torch.round((xg - shift.float().unsqueeze(-1)) / scale.float().unsqueeze(-1))
    codes = codes.clamp(0, 15).to(torch.int64).reshape(*x.shape[:-1], D // 8, 8)
    data = (codes << (4 * torch.arange(8, dtype=torch.int64))).sum(dim=-1)
    nanrow = torch.isnan(x).any(dim=-1, keepdim=True)
    sbits = scale.view(torch.int16).to(torch.int64) & 0xFFFF
    hbits = shift.view(torch.int16).to(torch.int64) & 0xFFFF
    coef = torch.where(nanrow, torch.full_like(sbits, 0x7E007E00), sbits | (hbits << 16))
    words = torch.cat([coef, data], dim=-1)
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words)
    return words.to(torch.int32).contiguous()


def quantize_e4m3(x: torch.Tensor, head_axis: int):
    """Per-kv-head e4m3 quantisation: scale_h = amax_h / 448, RNE saturating cast."""
    dims = [d for d in range(x.dim()) if d != head_axis]
    amax = x.abs().amax(dim=dims).to(torch.float32)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    shape = [1] * x.dim()
    shape[head_axis] = -1
    y = (x / scale.view(shape)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return y, scale.contiguous()


def make_gqa(*, name="gqa", batch, num_q_heads, num_kv_heads, head_dim=128, seq_lens,
             layout="contiguous", page_size=16, cache_len=None, kv_fp8=False,
             sparse_block_size=0, kv_num_blks=None, kv_idx=None, scale=None, seed=0,
             num_splits=0, poison=True, shape_only=False, q_len=1,
             kv_token_scale=False, tree_mask=False, sparse_shape=None,
             kv_int4_groups=0) -> Workload:
    """A GQA decode workload. ``seq_lens`` is a list/tensor of per-row lengths;
    ``q_len`` > 1 gives each row that many query tokens (its last positions);
    ``tree_mask`` adds a random draft-token tree over them (``spec_mask``).
    ``kv_int4_groups`` > 0 stores K/V as int4 group-wise rows with that many
    groups (``quantize_int4_groups``).
    ``sparse_shape`` = (SZ, SH): the block tables' batch and head extents when
    the mask is broadcast (row b, kv head h read table (b % SZ, h % SH)).

    ``shape_only`` skips drawing the K/V caches (lengths, tables and lists are
    drawn exactly as in the full workload)."""
    g = _gen(seed)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)
    B, HQ, HKV, D = batch, num_q_heads, num_kv_heads, head_dim
    assert seq_lens.numel() == B and HQ % HKV == 0
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q = _randn_bf16((B, HQ, D) if q_len <= 1 else (B, HQ, q_len, D), g)
    w = Workload(name=name, batch=B, num_q_heads=HQ, num_kv_heads=HKV, head_dim_qk=D,
                 head_dim_v=D, scale=float(torch.tensor(scale, dtype=torch.float32)),
                 kv_fp8=kv_fp8, num_splits=num_splits, q_len=max(1, q_len),
                 kv_token_scale=bool(kv_fp8 and kv_token_scale), kv_int4_groups=kv_int4_groups)
    assert not (kv_fp8 and kv_int4_groups)
    t = {"q": q, "seq_lens": seq_lens}
    if tree_mask and q_len > 1:
        t["spec_mask"] = draft_tree_mask(B, q_len, _gen(seed + 7919))
    if layout == "paged":
        table, num_pages, max_pages, used = _page_pool(seq_lens, page_size, g)
        w.paged, w.page_size, w.num_pages, w.max_pages_per_seq = True, page_size, num_pages, max_pages
        t["block_table"] = table
        if shape_only:
            w.tensors = t
            return w
        k = torch.randn((num_pages, HKV, page_size, D), generator=g, dtype=torch.float32)
        v = torch.randn((num_pages, HKV, page_size, D), generator=g, dtype=torch.float32)
        if poison:
            _poison_paged(k, table, seq_lens, page_size, used, True)
            _poison_paged(v, table, seq_lens, page_size, used, True)
        head_axis = 1
    else:
        L = int(cache_len if cache_len is not None else max(int(seq_lens.max()), 1))
        w.cache_len = L
        if shape_only:
            if sparse_block_size:
                w.sparse_block_size = sparse_block_size
                SZ, SH = sparse_shape if sparse_shape else (B, HKV)
                if sparse_shape:
                    w.sparse_batch, w.sparse_heads = SZ, SH
                t["kv_num_blks"] = torch.as_tensor(kv_num_blks, dtype=torch.int32).reshape(SZ, SH)
                t["kv_idx"] = torch.as_tensor(kv_idx, dtype=torch.int32).reshape(SZ, SH, -1)
                w.max_sparse_blocks = t["kv_idx"].shape[-1]
            w.tensors = t
            return w
        k = torch.randn((B, HKV, L, D), generator=g, dtype=torch.float32)
        v = torch.randn((B, HKV, L, D), generator=g, dtype=torch.float32)
        w.cache_len = L
        head_axis = 1
        if poison and sparse_block_size == 0:
            for b, n in enumerate(seq_lens.tolist()):
                k[b, :, n:] = float("nan")
                v[b, :, n:] = float("nan")
    if sparse_block_size:
        assert layout != "paged", "block-sparse decode reads a contiguous cache"
        SZ, SH = sparse_shape if sparse_shape else (B, HKV)
        if sparse_shape:
            w.sparse_batch, w.sparse_heads = SZ, SH
        kv_num_blks = torch.as_tensor(kv_num_blks, dtype=torch.int32).reshape(SZ, SH)
        kv_idx = torch.as_tensor(kv_idx, dtype=torch.int32).reshape(SZ, SH, -1)
        w.sparse_block_size, w.max_sparse_blocks = sparse_block_size, kv_idx.shape[-1]
        t["kv_num_blks"], t["kv_idx"] = kv_num_blks.contiguous(), kv_idx.contiguous()
        if poison:
            nblocks = (w.cache_len + sparse_block_size - 1) // sparse_block_size
            for b in range(B):
                for h in range(HKV):
                    keep = torch.zeros(nblocks, dtype=torch.bool)
                    zb, zh = b % SZ, h % SH
                    keep[kv_idx[zb, zh, :int(kv_num_blks[zb, zh])].long()] = True
                    mask = keep.repeat_interleave(sparse_block_size)[:w.cache_len]
                    mask &= torch.arange(w.cache_len) < int(seq_lens[b])
                    k[b, h, ~mask] = float("nan")
                    v[b, h, ~mask] = float("nan")
    if kv_int4_groups:
        t.update(k=quantize_int4_groups(k, kv_int4_groups), v=quantize_int4_groups(v, kv_int4_groups))
    elif kv_fp8 and kv_token_scale:
        kq, kss = quantize_e4m3_per_token(k)
        vq, vss = quantize_e4m3_per_token(v)
        t.update(k=kq, v=vq, k_scale_shift=kss, v_scale_shift=vss)
    elif kv_fp8:
        # quantise the finite values; NaN poison stays NaN (e4m3fn has NaN)
        kf = torch.nan_to_num(k, nan=0.0)
        vf = torch.nan_to_num(v, nan=0.0)
        kq, ks = quantize_e4m3(kf, head_axis)
        vq, vs = quantize_e4m3(vf, head_axis)
        # 0x7f is the e4m3fn NaN code
        kq = kq.view(torch.uint8).masked_fill(torch.isnan(k), 0x7F).view(torch.float8_e4m3fn)
        vq = vq.view(torch.uint8).masked_fill(torch.isnan(v), 0x7F).view(torch.float8_e4m3fn)
        t.update(k=kq.contiguous(), v=vq.contiguous(), k_scale=ks, v_scale=vs)
    else:
        t.update(k=k.to(torch.bfloat16).contiguous(), v=v.to(torch.bfloat16).contiguous())
    w.tensors = t
    return w


def draft_tree_mask(batch, q_len, g):
    """Packed masks of a random tree of ``q_len`` draft tokens per row, as int32
    words ``[batch][q_len][ceil(q_len / 32)]``: token j hangs under a parent
    drawn from the earlier tokens (or under the verified prefix), and its row
    has bit i set for itself and each of its ancestors i."""
    words = (q_len + 31) // 32
    bits = np.zeros((batch, q_len, words), dtype=np.uint32)
    for b in range(batch):
        parent = [-1] + [int(torch.randint(-1, j, (1,), generator=g)) for j in range(1, q_len)]
        for j in range(q_len):
            i = j
            while i >= 0:
                bits[b, j, i // 32] |= np.uint32(1) << np.uint32(i % 32)
                i = parent[i]
    return torch.from_numpy(bits.view(np.int32)).contiguous()


def sparse_lists(batch, num_kv_heads, cache_len, block_size, keep_random, keep_last, g,
                 max_blocks=None):
    """Per (b, kv head): ``keep_random`` distinct blocks drawn from the leading
    blocks plus the last ``keep_last`` blocks, sorted; padded with 0."""
    nblocks = (cache_len + block_size - 1) // block_size
    max_blocks = max_blocks or nblocks
    num = torch.zeros((batch, num_kv_heads), dtype=torch.int32)
    idx = torch.zeros((batch, num_kv_heads, max_blocks), dtype=torch.int32)
    head = nblocks - keep_last
    for b in range(batch):
        for h in range(num_kv_heads):
            pick = torch.randperm(head, generator=g)[:keep_random]
            blocks = torch.cat([pick, torch.arange(head, nblocks)]).sort().values
            num[b, h] = blocks.numel()
            idx[b, h, :blocks.numel()] = blocks.to(torch.int32)
    return num, idx


def make_mla(*, name="mla", batch, num_q_heads=128, ckv_dim=512, kpe_dim=64, seq_lens,
             page_size=64, scale=None, seed=0, num_splits=0, poison=True,
             shape_only=False, q_len=1, tree_mask=False) -> Workload:
    """An MLA decode workload over a paged latent cache; ``q_len`` > 1 gives
    each row that many query tokens (its last positions, q_nope
    [B][HQ][q_len][ckv], q_pe [B][HQ][q_len][kpe]); ``tree_mask`` adds a random
    draft-token tree over them (``spec_mask``)."""
    g = _gen(seed)
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)
    B, HQ = batch, num_q_heads
    scale = 1.0 / math.sqrt(192.0) if scale is None else scale
    lead = (B, HQ) if q_len <= 1 else (B, HQ, q_len)
    q_nope = _randn_bf16(lead + (ckv_dim,), g)
    q_pe = _randn_bf16(lead + (kpe_dim,), g)
    table, num_pages, max_pages, used = _page_pool(seq_lens, page_size, g)
    w = Workload(name=name, batch=B, num_q_heads=HQ, num_kv_heads=1,
                 head_dim_qk=ckv_dim + kpe_dim, head_dim_v=ckv_dim,
                 scale=float(torch.tensor(scale, dtype=torch.float32)), is_mla=True,
                 ckv_dim=ckv_dim, kpe_dim=kpe_dim, paged=True, page_size=page_size,
                 max_pages_per_seq=max_pages, num_pages=num_pages, num_splits=num_splits,
                 q_len=max(1, q_len))
    extra = {}
    if tree_mask and q_len > 1:
        extra["spec_mask"] = draft_tree_mask(B, q_len, _gen(seed + 7919))
    if shape_only:
        w.tensors = {"q": q_nope, "q_pe": q_pe, "block_table": table, "seq_lens": seq_lens, **extra}
        return w
    ckv = torch.randn((num_pages, page_size, ckv_dim), generator=g, dtype=torch.float32)
    kpe = torch.randn((num_pages, page_size, kpe_dim), generator=g, dtype=torch.float32)
    if poison:
        _poison_paged(ckv, table, seq_lens, page_size, used, False)
        _poison_paged(kpe, table, seq_lens, page_size, used, False)
    w.tensors = {"q": q_nope, "q_pe": q_pe, "k": ckv.to(torch.bfloat16).contiguous(),
                 "v": kpe.to(torch.bfloat16).contiguous(), "block_table": table,
                 "seq_lens": seq_lens, **extra}
    return w


# ------------------------------------------------------------------ the workloads
# 1-5 are the five decode configurations; 6 is the multi-token query extension
# (speculative decoding) on the paged GQA shapes; 7 is config 3 with e4m3 K/V
# scaled per token (fp16 scale and shift per cache row).

CONFIG_NAMES = {
    1: "tiny GQA decode (B1 HQ8 HKV1 D128, contiguous L512, 4 splits)",
    2: "paged GQA decode (B32 HQ32 HKV8 D128, N_b~U[1024,8192], page 16)",
    3: "long-context fp8 KV (B1 HQ64 HKV8 D128, contiguous L131072, e4m3)",
    4: "block-sparse decode (B8 HQ32 HKV8 D128, L32768, 36 of 256 blocks of 128)",
    5: "MLA latent decode (B64 HQ128, ckv512+kpe64, N_b~U[2048,8192], page 64)",
    6: "speculative paged GQA decode (B32 HQ32 HKV8 D128, 4 query tokens, N_b~U[1024,8192], page 16)",
    7: "long-context fp8 KV, per-token scale+shift (B1 HQ64 HKV8 D128, contiguous L131072, e4m3)",
    8: "paged GQA decode, int4 group-wise KV (B32 HQ32 HKV8 D128, 4 groups of 32, N_b~U[1024,8192], page 16)",
}


def config(i: int, shape_only: bool = False, seed: int | None = None, q_len: int = 1) -> Workload:
    """The decode workloads (CONFIG_NAMES); ``shape_only`` skips drawing the K/V caches.
    ``seed`` replaces the workload's own seed (1000 + i): another draw of the same
    recipe (lengths, tables, values). ``q_len`` gives the MLA workload (5) several
    query tokens per row."""
    own_seed = seed is None
    seed = 1000 + i if seed is None else seed
    so = dict(shape_only=shape_only)
    if i == 1:
        return make_gqa(name="tiny_gqa", batch=1, num_q_heads=8, num_kv_heads=1,
                        seq_lens=[512], cache_len=512, seed=seed, num_splits=4, **so)
    if i == 2:
        g = _gen(seed + 500)
        lens = _lengths(32, 1024, 8192, g)
        return make_gqa(name="paged_gqa", batch=32, num_q_heads=32, num_kv_heads=8,
                        seq_lens=lens, layout="paged", page_size=16, seed=seed, **so)
    if i == 3:
        return make_gqa(name="fp8_long", batch=1, num_q_heads=64, num_kv_heads=8,
                        seq_lens=[131072], cache_len=131072, kv_fp8=True, seed=seed, **so)
    if i == 4:
        g = _gen(seed + 500)
        num, idx = sparse_lists(8, 8, 32768, 128, keep_random=32, keep_last=4, g=g,
                                max_blocks=256)
        return make_gqa(name="block_sparse", batch=8, num_q_heads=32, num_kv_heads=8,
                        seq_lens=[32768] * 8, cache_len=32768, sparse_block_size=128,
                        kv_num_blks=num, kv_idx=idx, seed=seed, **so)
    if i == 5:
        g = _gen(seed + 500)
        lens = _lengths(64, 2048, 8192, g)
        return make_mla(name="mla", batch=64, seq_lens=lens, seed=seed, q_len=q_len, **so)
    if i == 6:
        g = _gen(seed + 500)
        lens = _lengths(32, 1024, 8192, g)
        return make_gqa(name="spec_paged_gqa", batch=32, num_q_heads=32, num_kv_heads=8,
                        seq_lens=lens, layout="paged", page_size=16, seed=seed, q_len=4, **so)
    if i == 7:
        return make_gqa(name="fp8_token_long", batch=1, num_q_heads=64, num_kv_heads=8,
                        seq_lens=[131072], cache_len=131072, kv_fp8=True, kv_token_scale=True,
                        seed=seed, **so)
    if i == 8:
        g = _gen((1002 if own_seed else seed) + 500)  # the lengths of the bf16 paged workload (2)
        lens = _lengths(32, 1024, 8192, g)
        return make_gqa(name="int4_paged_gqa", batch=32, num_q_heads=32, num_kv_heads=8,
                        seq_lens=lens, layout="paged", page_size=16, seed=seed, kv_int4_groups=4,
                        **so)
    raise ValueError(f"no workload {i}")
