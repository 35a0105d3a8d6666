"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare against the float64 oracle."""

import numpy as np
import torch

import decode_attention_flash_gb300 as da
import oracle

BF16_ATOL, BF16_RTOL, LSE_ATOL, FP8_TOL = 2e-2, 1e-2, 1e-3, 3e-2


def run_gpu(w, num_splits_override=None, with_lse=True, seq_lens_host=True, engine=None,
            softcap=0.0):
    dev = torch.device("cuda", 0)
    if engine is None:
        nb = w.tensors.get("kv_num_blks") if w.sparse_block_size else None
        engine = da.DecodeAttention(
            device=0, seq_lens_host=w.tensors["seq_lens"] if seq_lens_host else None,
            kv_num_blks_host=nb,
            num_splits_override=w.num_splits if num_splits_override is None else num_splits_override,
            **da.problem_kwargs(w))
    t = w.to(dev)
    lead = (w.batch, w.num_q_heads) + ((w.q_len,) if w.q_len > 1 else ())
    lse = torch.full(lead, 12345.0, dtype=torch.float32, device=dev) if with_lse else None
    out = torch.full(lead + (w.head_dim_v,), 777.0, dtype=torch.bfloat16, device=dev)
    engine.run(t, w.scale, out=out, lse=lse, softcap=softcap)
    torch.cuda.synchronize()
    flags = engine.errors()
    return out.cpu(), (lse.cpu() if lse is not None else None), flags, engine


def reference(w, rows=None, softcap=0.0):
    """Oracle output; `rows` (list of batch rows) restricts it to a subset."""
    if rows is None:
        return oracle.decode(oracle.problem_from(w), w.tensors, w.scale, softcap=softcap)
    t = dict(w.tensors)
    idx = torch.tensor(rows, dtype=torch.long)
    t["q"] = t["q"][idx].contiguous()
    if "q_pe" in t:
        t["q_pe"] = t["q_pe"][idx].contiguous()
    t["seq_lens"] = t["seq_lens"][idx].contiguous()
    if "block_table" in t:
        t["block_table"] = t["block_table"][idx].contiguous()
    if not w.paged:
        t["k"] = t["k"][idx].contiguous()
        t["v"] = t["v"][idx].contiguous()
    if "kv_num_blks" in t:
        t["kv_num_blks"] = t["kv_num_blks"][idx].contiguous()
        t["kv_idx"] = t["kv_idx"][idx].contiguous()
    prob = oracle.problem_from(w)
    prob["batch"] = len(rows)
    return oracle.decode(prob, t, w.scale)


def assert_parity(out, lse, ref_out, ref_lse, fp8=False, what=""):
    got = out.double().numpy()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - ref_out))) if got.size else 0.0
    rel = err / max(float(np.max(np.abs(ref_out))) if got.size else 0.0, 1e-6)
    atol, rtol = (FP8_TOL, FP8_TOL) if fp8 else (BF16_ATOL, BF16_RTOL)
    assert err <= atol and rel <= rtol, f"{what}: max-abs {err:.3e}, rel {rel:.3e}"
    if lse is not None:
        lg = lse.double().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lg), fin), f"{what}: LSE finiteness differs"
        assert np.all(lg[~fin] == -np.inf), f"{what}: empty rows must have LSE -inf"
        if fin.any():
            lerr = float(np.max(np.abs(lg[fin] - ref_lse[fin])))
            assert lerr <= LSE_ATOL, f"{what}: LSE max-abs {lerr:.3e}"
    return err, rel
