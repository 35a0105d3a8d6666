"""The timeout path of the GQA kernel, without faulting or hanging the GPU: the
test hook decode_attn_test_set_stall makes the first pipeline wait of one
consumer warp per CTA wait on a barrier that nothing arrives on, with a short
limit. The kernel must then give up its other bounded waits, wait for every
copy it issued, report DA_DEVERR_TIMEOUT through decode_attn_get_error (which
also clears the counters an aborted call may leave), and the next call on the
same workspace must match the oracle."""

import ctypes

import pytest
import torch

import decode_attention_flash_gb300 as da
from decode_attention_flash_gb300 import workloads as W
from helpers import assert_parity, reference, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("splits", [1, 3])
def test_stalled_wait_reports_timeout_then_the_context_recovers(splits):
    lib = da.load()
    w = W.make_gqa(name="stall", batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[300, 70],
                   layout="paged", page_size=16, seed=91)
    eng = da.DecodeAttention(device=0, seq_lens_host=w.tensors["seq_lens"],
                             num_splits_override=splits, **da.problem_kwargs(w))
    t = w.to("cuda")
    assert lib.decode_attn_test_set_stall(eng.ctx, 200_000) == da.DA_OK  # 0.2 ms
    out = torch.zeros((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device="cuda")
    eng.run(t, w.scale, out=out)
    torch.cuda.synchronize()
    assert eng.errors() & da.DA_DEVERR_TIMEOUT
    # the stall was for one call only; the workspace's error word and counters are clean
    got, lse, flags, _ = run_gpu(w, engine=eng)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(got, lse, ref_out, ref_lse, what=f"after a timeout, S={splits}")


def test_stall_hook_refuses_bad_arguments():
    lib = da.load()
    w = W.make_mla(name="mla_stall", batch=1, seq_lens=[64], seed=92)
    eng = da.DecodeAttention(device=0, **da.problem_kwargs(w))
    assert lib.decode_attn_test_set_stall(eng.ctx, 1000) == da.DA_ERR_INVALID_ARG  # MLA
    assert lib.decode_attn_test_set_stall(None, 1000) == da.DA_ERR_INVALID_ARG
