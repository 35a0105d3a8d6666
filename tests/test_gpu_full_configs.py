"""Parity at the workloads' full sizes (the five decode configurations and the
speculative-decoding one), in the launch configuration the
benchmark times (the planner's own split choice from the host lengths), against
the float64 oracle on every output row."""

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


def test_full_size_mla_config():
    w = W.config(5)
    out, lse, flags, eng = run_gpu(w)
    assert flags == 0
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="config 5")


def test_full_size_mla_config_with_four_query_tokens():
    # the MLA workload with 4 query tokens per row (causal over each row's last
    # 4 positions), every output row against the oracle
    w = W.config(5, q_len=4)
    out, lse, flags, eng = run_gpu(w)
    assert flags == 0 and out.shape == (64, 128, 4, 512)
    ref_out, ref_lse = reference(w)
    assert_parity(out, lse, ref_out, ref_lse, what="config 5, q_len 4")
