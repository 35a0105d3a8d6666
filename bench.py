"""Benchmark: split-KV decode attention on GB300 through the C ABI.

One step = one decode call (split kernel + LSE merge) over the whole batch of
the workload, K/V cache resident in HBM. Default workload: paged GQA decode
(B=32, HQ=32, HKV=8, D=128, N_b ~ U[1024, 8192], page 16). The metric is the
achieved KV-cache bandwidth (algorithmic KV bytes / time, GB/s), with us per
call and the fraction of measured HBM peak alongside.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..8] [--impl reference]
                  [--tree-mask] [--softcap C]

Configs 1-5 are the five decode workloads; 6 is the speculative-decoding one
(the paged GQA shapes with 4 query tokens per row, causal over the new tokens,
or a random draft-token tree with --tree-mask); 7 is config 3 with e4m3 K/V
scaled per token (fp16 scale and shift per row); 8 is config 2 with int4
group-wise K/V (4 groups of 32 elements per row).

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
units are independent, no collective on the data path); rank 0 prints one
JSON line with the whole-job aggregate (bytes of all ranks / max rank time).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from decode_attention_flash_gb300 import workloads as W  # noqa: E402

DEFAULT_CONFIG = 2
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(
            d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = {
    "gqa_split_kernel": ["gqa_split.cuh", "gqa_split.cu", "gqa_kind_bf16.cu", "gqa_kind_e4m3.cu",
                         "gqa_kind_e4m3_token.cu", "gqa_kind_int4.cu", "gqa_kind_e4m3_mma.cu", "ptx.cuh",
                         "internal.h"],
    "mla_split_kernel": ["mla_split.cu", "ptx.cuh", "internal.h"],
}


def kernel_hash(kernel: str) -> str:
    """Hash of the sources of a kernel: traffic figures are only valid for it."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "decode_attention_flash_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, cfg: int, args=None):
    """DRAM read+write bytes per launch from the committed ncu summary, or None
    when the kernel's sources changed since that capture or the run is another
    workload than the captured one (another seed, query-token count, mask,
    soft cap or arithmetic)."""
    if args is not None and (args.seed is not None or args.q_len > 1 or args.tree_mask or args.softcap
                             or args.fp8_mma or args.splits):
        return None
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"config{cfg}")
    if not rec or rec.get("kernel") != kernel or rec.get("source_hash") != kernel_hash(kernel):
        return None
    return rec["dram_bytes_per_launch"]


def algorithmic_bytes(w) -> dict:
    """The method's own bytes per call: kept KV + Q + O (+ LSE)."""
    t = w.tensors
    if w.sparse_block_size:
        nb = t["kv_num_blks"].long()
        positions = 0
        for b in range(w.batch):
            n_b = int(t["seq_lens"][b])
            for h in range(w.num_kv_heads):
                zb, zh = b % (w.sparse_batch or w.batch), h % (w.sparse_heads or w.num_kv_heads)
                blocks = t["kv_idx"][zb, zh, :int(nb[zb, zh])].long()
                positions += int(torch.clamp(n_b - blocks * w.sparse_block_size, 0,
                                             w.sparse_block_size).sum())
        kv_tokens_heads = positions
    else:
        kv_tokens_heads = int(t["seq_lens"].long().sum()) * (1 if w.is_mla else w.num_kv_heads)
    elt = 1 if w.kv_fp8 else 2
    Q = getattr(w, "q_len", 1)  # query tokens per row (their causal triangle is not subtracted)
    if w.is_mla:
        kv = kv_tokens_heads * (w.ckv_dim + w.kpe_dim) * 2
        q = w.batch * w.num_q_heads * Q * (w.ckv_dim + w.kpe_dim) * 2
        flops = kv_tokens_heads * w.num_q_heads * Q * (2 * (w.ckv_dim + w.kpe_dim) + 2 * w.ckv_dim)
    else:
        kv = kv_tokens_heads * (w.head_dim_qk + w.head_dim_v) * elt
        if getattr(w, "kv_int4_groups", 0):  # int32 rows: groups coefficient words + D / 8 data words
            kv = kv_tokens_heads * 2 * (w.kv_int4_groups + w.head_dim_qk // 8) * 4
        if getattr(w, "kv_token_scale", False):
            kv += kv_tokens_heads * 2 * 4  # the K and V scale words of every row
        q = w.batch * w.num_q_heads * Q * w.head_dim_qk * 2
        flops = kv_tokens_heads * w.group * Q * 2 * (w.head_dim_qk + w.head_dim_v)
    o = w.batch * w.num_q_heads * Q * (w.head_dim_v * 2 + 4)
    return {"kv": kv, "q": q, "o": o, "total": kv + q + o, "flops": flops}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names[1:], f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    rank, world = int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_name(cfg, args):
    name = W.CONFIG_NAMES[cfg]
    if args.tree_mask:
        name += ", draft-tree mask"
    if args.softcap:
        name += f", tanh soft cap {args.softcap:g}"
    if args.seed is not None:
        name += f", seed {args.seed}"
    if args.fp8_mma:
        name += ", e4m3 tensor-core QK/PV (fp8_mma)"
    if args.q_len > 1:
        name += f", {args.q_len} query tokens per row"
    return name


def timed_oracle(w, rows, threads, softcap=0.0):
    """The float64 oracle on a subset of batch rows; returns (seconds, fraction of KV)."""
    import oracle
    t0 = time.perf_counter()
    sub = _subset(w, rows)
    oracle.decode(oracle.problem_from(sub), sub.tensors, sub.scale, num_threads=threads,
                  softcap=softcap)
    dt = time.perf_counter() - t0
    frac = algorithmic_bytes(sub)["kv"] / max(algorithmic_bytes(w)["kv"], 1)
    return dt, frac


def _subset(w, rows):
    import copy
    t = dict(w.tensors)
    idx = torch.tensor(rows, dtype=torch.long)
    for k in ("q", "q_pe", "seq_lens", "block_table", "kv_num_blks", "kv_idx", "spec_mask"):
        if k in t:
            t[k] = t[k][idx].contiguous()
    if not w.paged:
        for k in ("k_scale_shift", "v_scale_shift"):
            if k in t:
                t[k] = t[k][idx].contiguous()
        # row selection through a byte view: CPU indexing of float8 tensors is
        # missing in some PyTorch releases
        for k in ("k", "v"):
            x = t[k]
            t[k] = (x.view(torch.uint8)[idx].contiguous().view(x.dtype)
                    if x.dtype == torch.float8_e4m3fn else x[idx].contiguous())
    s = copy.copy(w)
    s.batch = len(rows)
    s.tensors = t
    return s


def pick_oracle_rows(w, target_s=1.0, threads=1):
    """Batch rows of the workload sized for ~target_s seconds of oracle time."""
    rows = [0]
    timed_oracle(w, rows, threads)  # first call also loads the library
    dt, _ = timed_oracle(w, rows, threads)
    per_row = max(dt, 1e-4)
    n = max(1, min(w.batch, int(target_s / per_row)))
    return list(range(n))


def run_reference(args, w, cfg):
    """The oracle, as it stands, on the host cores: each step a bounded sample."""
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    import oracle
    threads = oracle.default_threads()
    rows = pick_oracle_rows(w, target_s=2.0, threads=threads)
    for _ in range(args.warmup):
        timed_oracle(w, rows, threads, args.softcap)
    times = []
    frac = 1.0
    for _ in range(args.steps):
        dt, frac = timed_oracle(w, rows, threads, args.softcap)
        times.append(dt)
    ab = algorithmic_bytes(w)
    mean = statistics.mean(times)
    value = ab["kv"] * frac / mean / 1e9
    line = {
        "impl": "reference", "metric": "decode attention KV GB/s & % of GB300 HBM peak; \u00b5s per decode call", "value": value,
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(cfg, args), "sample_rows": len(rows)},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"batch rows 0..{len(rows) - 1} of {w.batch}, all heads"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, cfg):
    import decode_attention_flash_gb300 as da
    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, tf_peak, tf_sus, peak_kind = measured_peaks()
    nb = w.tensors.get("kv_num_blks") if w.sparse_block_size else None
    eng = da.DecodeAttention(device=local, seq_lens_host=w.tensors["seq_lens"], kv_num_blks_host=nb,
                             num_splits_override=args.splits if args.splits else w.num_splits,
                             **da.problem_kwargs(w))
    plan = eng.plan
    t = w.to(dev)
    lead = (w.batch, w.num_q_heads) + ((w.q_len,) if w.q_len > 1 else ())
    out = torch.empty(lead + (w.head_dim_v,), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(lead, dtype=torch.float32, device=dev)
    a = da.make_args(t, w.scale, out, lse, softcap=args.softcap)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        da.decode_attn_run(eng.ctx, a, eng.workspace, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if eng.errors() != 0:
        raise RuntimeError("device error flags set during warm-up")

    # ---------------- device-timed region (one kernel launch per call), L2 flushed between steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for i in range(args.steps):
            flush.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    call_ms = [e[0].elapsed_time(e[1]) for e in ev]
    mean_call = max_over_ranks(statistics.mean(call_ms), world)
    mean_split = mean_call  # the split kernel (with its fused merge) is the whole call
    launches_per_step = 1

    ab = algorithmic_bytes(w)
    value = world * ab["kv"] / (mean_call * 1e-3) / 1e9
    pct_hbm = ab["total"] / (mean_call * 1e-3) / 1e9 / hbm_peak
    split_gbs = ab["total"] / (mean_split * 1e-3) / 1e9

    # ---------------- end to end through the public API with host buffers
    # A step's inputs sit in one pinned host buffer and its outputs in one
    # device buffer (1 KiB-aligned views), so each step makes one copy in and
    # one copy out; the tensors handed to the API are views of them.
    def packed(tensors, device=None, pin=False):
        offs, off = {}, 0
        for k, v in tensors.items():
            offs[k] = off
            off += (v.numel() * v.element_size() + 1023) // 1024 * 1024
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = {k: buf[o:o + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                 for (k, v), o in zip(tensors.items(), offs.values())}
        return buf, views

    in_names = [k for k in ("q", "q_pe", "seq_lens", "block_table", "kv_num_blks", "kv_idx",
                            "spec_mask") if k in w.tensors]
    h_in, h_views = packed({k: w.tensors[k] for k in in_names}, pin=True)
    for k in in_names:
        h_views[k].copy_(w.tensors[k])
    d_in, d_views = packed({k: w.tensors[k] for k in in_names}, device=dev)
    t_e2e = dict(t)
    t_e2e.update(d_views)
    d_res, d_res_views = packed({"out": out, "lse": lse}, device=dev)
    h_res = torch.empty_like(d_res, device="cpu").pin_memory()
    h2d = sum(w.tensors[k].numel() * w.tensors[k].element_size() for k in in_names)
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    # the call's arguments point at the same buffers every step: built once,
    # as a caller of the C ABI would (the checked wrapper runs once first)
    eng.run(t_e2e, w.scale, out=d_res_views["out"], lse=d_res_views["lse"], stream=stream,
            softcap=args.softcap)
    a_e2e = da.make_args(t_e2e, w.scale, d_res_views["out"], d_res_views["lse"], softcap=args.softcap)
    e2e_ms = []
    for i in range(args.steps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        d_in.copy_(h_in, non_blocking=True)
        da.decode_attn_run(eng.ctx, a_e2e, eng.workspace, stream)
        h_res.copy_(d_res, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= 3:
            e2e_ms.append(e0.elapsed_time(e1))
    mean_e2e = max_over_ranks(statistics.mean(e2e_ms), world)
    e2e_value = world * ab["kv"] / (mean_e2e * 1e-3) / 1e9
    if eng.errors() != 0:
        raise RuntimeError("device error flags set during the timed region")

    # ---------------- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.default_threads()
        rows = pick_oracle_rows(w, target_s=10.0, threads=threads)
        # a sample the oracle finishes quickly is evaluated again until about a
        # second of wall time has gone by (the mean is reported)
        dts = []
        while not dts or (sum(dts) < 1.0 and len(dts) < 100):
            dt, frac = timed_oracle(w, rows, threads)
            dts.append(dt)
        dt = statistics.mean(dts)
        cpu = {"value": ab["kv"] * frac / dt / 1e9, "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"batch rows 0..{len(rows) - 1} of {w.batch} ({frac:.3f} of the KV bytes), "
                         f"mean of {len(dts)} runs of {dt:.2f} s wall"}
        # the same oracle on one core, over its own bounded sample (~3 s)
        rows1 = pick_oracle_rows(w, target_s=3.0, threads=1)
        dt1, frac1 = timed_oracle(w, rows1, 1)
        cpu["single_core"] = {"value": ab["kv"] * frac1 / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"batch rows 0..{len(rows1) - 1} of {w.batch} "
                                        f"({frac1:.3f} of the KV bytes), {dt1:.2f} s wall"}

    kname = "mla_split_kernel" if w.is_mla else "gqa_split_kernel"
    if w.is_mla:
        # MLA sits near the ridge: report the tensor side of its roofline too
        tflops = ab["flops"] / (mean_split * 1e-3) / 1e12
    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": "decode attention KV GB/s & % of GB300 HBM peak; \u00b5s per decode call",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_call, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4" if w.kv_int4_groups else ("f8e4m3" if w.kv_fp8 else "bf16"),
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, args), "us_per_call": mean_call * 1e3,
                       "pct_hbm_peak_kv_q_o": pct_hbm, "hbm_peak_gbs": hbm_peak,
                       "peak_source": peak_kind, "l2": "512 MiB buffer written between steps",
                       "plan": {k: plan[k] for k in ("chunk_tokens", "num_splits", "grid_x",
                                                     "grid_y", "grid_z", "ctas_per_sm")},
                       "algorithmic_bytes": ab["total"], "kv_bytes": ab["kv"],
                       "us_min": min(call_ms) * 1e3, "us_max": max(call_ms) * 1e3},
            "roofline": {"bound": "hbm", "achieved": split_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": split_gbs / hbm_peak,
                         "traffic": recorded_traffic(kname, cfg, args),
                         "kernel": kname, "kernel_us": mean_split * 1e3,
                         "peak_source": f"of {peak_kind} ({'MEASURED_PEAKS.json hbm_gbs' if peak_kind == 'measured' else 'fallback'})"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "us_per_call": mean_e2e * 1e3},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if w.is_mla:
            line["roofline_tensor"] = {"bound": "tensor", "achieved": tflops, "peak": tf_peak,
                                       "unit": "TFLOP/s", "frac": tflops / tf_peak,
                                       "flops_per_launch": ab["flops"]}
        print(json.dumps(line), flush=True)
    eng.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--splits", type=int, default=0, help="num_splits_override (0 = planner)")
    ap.add_argument("--tree-mask", action="store_true",
                    help="several-token configs: a random draft-token tree instead of the causal mask")
    ap.add_argument("--softcap", type=float, default=0.0,
                    help="tanh soft cap c of the scaled scores, s -> c tanh(s / c) (0 = off)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=None,
                    help="another draw of the workload's recipe (default: its own seed, 1000 + config)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="the MLA configuration: query tokens per row (speculative decoding, causal "
                         "over the row's last q_len positions)")
    ap.add_argument("--fp8-mma", action="store_true",
                    help="e4m3 K/V configurations: QK and PV on e4m3 tensor cores (queries and "
                         "weights rounded to e4m3)")
    args = ap.parse_args()
    if args.q_len > 1 and args.config != 5:
        raise SystemExit("--q-len applies to the MLA configuration (5); config 6 is the GQA one")
    w = W.config(args.config, seed=args.seed, q_len=args.q_len)
    if args.fp8_mma:
        if not w.kv_fp8 or w.kv_token_scale:
            raise SystemExit("--fp8-mma needs a configuration with e4m3 K/V and per-head scales")
        w.fp8_mma = True
    if args.tree_mask:
        if w.q_len < 2:
            raise SystemExit("--tree-mask needs a configuration with several query tokens")
        w.tensors["spec_mask"] = W.draft_tree_mask(w.batch, w.q_len,
                                                   torch.Generator().manual_seed(1234))
    if args.impl == "reference":
        run_reference(args, w, args.config)
    else:
        run_ours(args, w, args.config)


if __name__ == "__main__":
    main()
