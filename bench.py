"""Benchmark of the sparse MLA forward on GB300.

Default workload: the causal ramp-padded prefill (s_q=8192, s_kv=8192, h_q=64,
d_qk=d_v=512, topk width 1152, row i holds min(i+1, 1027) valid indices, padded with -1),
run WITHOUT topk_length -- the kernel derives each row's length itself.  One step = one call
of the whole forward on that batch.  The metric is valid-token TFLOP/s,
2*h_q*valid*(d_qk+d_v) summed over rows, divided by the device time of the call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config ramp|full|scattered|decode|tiny|bwd]
                  [--impl ours|reference]

--config bwd times the backward instead (sparse_mla_bwd on s_q=4096, s_kv=32768, h_q=64,
d_qk=576, topk=2048, all valid): one step = one backward call given the forward's out / lse,
metric = 2*h_q*valid*(3*d_qk + 2*d_v) FLOPs (S and dP recomputed, dQ, dK, dV) per second.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own batch of the same shape (weak
scaling, no collective on the data path); the time is the max over ranks.
--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "sparse-MLA fwd ms/call & valid-token TFLOP/s; % of GB300 bf16 tensor peak"
METRIC_BWD = "sparse-MLA bwd ms/call & valid-token TFLOP/s; % of GB300 bf16 tensor peak"
UNIT = "TFLOP/s"
# FlashMLA PR #196 "Numbers" (B200, not GB300): ramp-padded, no topk_length, 1.144 ms for
# 1.0337 TFLOP of valid-token work -> 903.6 TFLOP/s.  Context only.
PAGES_B200_TFLOPS = {("ramp", False): 1.0337e12 / 1.144e-3 / 1e12,
                     ("ramp", True): 1.0337e12 / 1.101e-3 / 1e12}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=["ramp", "full", "scattered", "decode", "decode_b2", "decode_b8", "tiny",
                                         "bwd"],
                    default="ramp")
    ap.add_argument("--n-split", default="auto",
                    help="split-KV ranges per row: 'auto' (split only when items < SMs) or an integer")
    ap.add_argument("--with-len", action="store_true", help="pass topk_length in the timed steps")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-chunks", type=int, default=16, help="row chunks of the host-buffer end-to-end leg")
    ap.add_argument("--skip-cpu", action="store_true", help="no CPU-oracle baseline leg")
    ap.add_argument("--skip-e2e", action="store_true", help="no host-buffer end-to-end leg")
    ap.add_argument("--skip-decode", action="store_true", help="no decode fixed-vs-dynamic leg")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--shard", choices=["replicas", "rows"], default="replicas",
                    help="multi-GPU: every rank runs its own batch (replicas, weak scaling) or its "
                         "contiguous rows of one batch (rows, strong scaling; flat workloads only)")
    return ap.parse_args()


def make_workload(name, with_len):
    if name == "ramp":
        return W.ramp(with_len=with_len)
    if name == "full":
        return W.full()
    if name == "scattered":
        return W.scattered()
    if name == "decode":
        return W.decode(dynamic=True)
    if name == "decode_b2":
        return W.decode_fixed(n_req=2)
    if name == "decode_b8":
        return W.decode_fixed(n_req=8)
    if name == "bwd":
        return W.bwd_prefill()
    return W.tiny(with_len=with_len, with_sink=True)


def describe(w, name):
    q = w["q"]
    s_q, h_q, d_qk = q.shape
    topk = w["indices"].reshape(s_q, -1).shape[1]
    text = {
        "ramp": f"causal ramp-padded prefill s_q={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 "
                f"topk={topk} (row i: min(i+1,1027) valid, -1 padded)",
        "full": f"fully-valid prefill s_q={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 topk={topk}",
        "scattered": f"scattered-invalid prefill + sink s_q={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} "
                     f"d_v=512 topk={topk} p_invalid=0.3",
        "decode": f"paged decode B={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 topk={topk} "
                  f"topk_length=1024 INT_MAX suffix, 64-token pages",
        "decode_b2": f"small-batch paged decode B=2 x S_q=2 s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 "
                     f"topk={topk} all valid, 64-token pages",
        "decode_b8": f"small-batch paged decode B=8 x S_q=2 s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 "
                     f"topk={topk} all valid, 64-token pages",
        "tiny": f"tiny s_q={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} topk={topk}",
        "bwd": f"sparse backward s_q={s_q} s_kv={w['s_kv']} h_q={h_q} d_qk={d_qk} d_v=512 topk={topk} all valid",
    }[name]
    return text


def valid_flops(w, rows=None, backward=False):
    """Valid-token FLOPs: forward 2*h_q*(d_qk + d_v) per counted slot; backward
    2*h_q*(3*d_qk + 2*d_v) (S and dP recomputed, then dQ, dK and dV)."""
    idx = w["indices"].reshape(w["q"].shape[0], -1)
    tl = w["topk_length"]
    if rows is not None:
        idx = idx[rows]
        tl = None if tl is None else np.asarray(tl)[rows]
    counts = W.valid_slot_count(idx, w["s_kv"], tl)
    h_q, d_qk = w["q"].shape[1], w["q"].shape[2]
    per = (3 * d_qk + 2 * w["d_v"]) if backward else (d_qk + w["d_v"])
    return float(2.0 * h_q * counts.sum() * per)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash(kernel="fwd"):
    """Hash of the sources that define a kernel: the forward's file and PTX wrappers, plus the
    backward's own file for the backward (it is compiled in the forward's translation unit and
    uses its helpers)."""
    files = ["sparse_mla_attention_fwd_gb300/csrc/sparse_mla_fwd.cu",
             "sparse_mla_attention_fwd_gb300/csrc/smla_ptx.cuh"]
    if kernel == "bwd":
        files.append("sparse_mla_attention_fwd_gb300/csrc/sparse_mla_bwd.cuh")
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def profiled_counters(config_name):
    """Per-launch ncu counters (DRAM bytes read + written, L2 bytes to the SMs) for this
    workload's dominant kernel, from the machine-readable file beside the ncu summaries, if
    they were taken on the current kernel source; else an empty dict."""
    if not os.path.exists(TRAFFIC_FILE):
        return {}
    with open(TRAFFIC_FILE) as f:
        entry = json.load(f).get(config_name)
    kernel = "bwd" if config_name == "bwd" else "fwd"
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(kernel):
        return {}
    return entry


def algorithmic_bytes(w, backward=False):
    """Compulsory HBM bytes per call (inputs read once, outputs written once) and the L2 -> SM
    gather bytes (one d_qk row per counted slot)."""
    s_q, h_q, d_qk = w["q"].shape
    topk = w["indices"].reshape(s_q, -1).shape[1]
    counts = W.valid_slot_count(w["indices"], w["s_kv"], w["topk_length"])
    row = d_qk * 2
    gather = float(counts.sum()) * row
    hbm = s_q * h_q * d_qk * 2 + s_q * topk * 4       # Q and the index lists
    hbm += 0 if w["topk_length"] is None else s_q * 4
    if w.get("paged"):
        hbm += gather + w["block_table"].size * 4     # rows come from a pool far larger than L2
    else:
        hbm += w["kv"].shape[0] * row                 # the shared KV is read once
    if backward:
        # out, dout (bf16) and lse in; dq (fp32) and dkv (fp32) out
        hbm += s_q * h_q * w["d_v"] * 4 + s_q * h_q * 4 + s_q * h_q * d_qk * 4 + w["kv"].shape[0] * d_qk * 4
    else:
        # O (bf16), lse and max_logits (fp32) out
        hbm += s_q * h_q * w["d_v"] * 2 + s_q * h_q * 8
    return float(hbm), gather


def nearer_roof(tflops, hbm_gbs, peaks, src, traffic, kernel):
    """The roofline object for the roof the kernel is nearer to: the tensor roof (valid-token
    TFLOP/s against the measured burst bf16 peak) or the HBM roof (compulsory HBM bytes per call
    over the call time against the measured copy bandwidth).  The other roof's fraction is kept
    beside it.  The prefill shapes sit nearer the tensor roof; the paged decode, which reads
    every gathered row from HBM once, nearer the HBM roof."""
    tp = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hp = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    tensor = {"bound": "tensor", "achieved": tflops, "peak": tp, "unit": "TFLOP/s", "frac": tflops / tp,
              "peak_source": f"bf16_tflops burst ({src})"}
    hbm = {"bound": "hbm", "achieved": hbm_gbs, "peak": hp, "unit": "GB/s", "frac": hbm_gbs / hp,
           "peak_source": f"hbm_gbs copy ({src})"}
    near, far = (hbm, tensor) if hbm["frac"] > tensor["frac"] else (tensor, hbm)
    roof = dict(near)
    roof["traffic"] = traffic
    roof["kernel"] = kernel
    roof["other_roof"] = {k: far[k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    return roof


def bandwidth(w, config_name, ms, backward=False):
    """HBM and L2 GB/s of one call: algorithmic bytes and, where the ncu counters for the current
    kernel source are on file, measured bytes, each over the measured time per call."""
    hbm, gather = algorithmic_bytes(w, backward)
    c = profiled_counters(config_name)
    sec = ms * 1e-3
    dram = c.get("dram_bytes_per_launch")
    l2 = c.get("l2_to_sm_bytes_per_launch")
    return {"hbm_gbs": {"algorithmic": hbm / sec / 1e9, "measured": (dram / sec / 1e9) if dram else None,
                        "algorithmic_bytes": hbm, "measured_bytes": dram},
            "l2_gbs": {"algorithmic": gather / sec / 1e9, "measured": (l2 / sec / 1e9) if l2 else None,
                       "algorithmic_bytes": gather, "measured_bytes": l2},
            "counters_source": ("profiles/dram_traffic.json (ncu, current kernel source)" if c else
                                "no ncu counters on file for the current kernel source")}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, enabled=True):
        self.proc = None
        self.gpu = gpu_index
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, device=None):
    """Max of a float over every rank of the default process group: the job's time is its
    slowest rank's.  A no-op without an initialised group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, device=None):
    """Sum of a float over every rank (the units all ranks processed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_tflops(total_flops, total_ms):
    """Whole-job throughput: the work of all ranks over the slowest rank's time."""
    return total_flops / (total_ms * 1e-3) / 1e12


def run_reference(args, world, rank):
    """fp64 CPU oracle as the reference arm: each step is the oracle on a bounded sample of the
    workload's rows, spread over the batch."""
    if rank != 0:
        return
    import oracle

    w = make_workload(args.config, args.with_len)
    bwd = args.config == "bwd"
    if bwd:
        w["backward"], w["dout"] = True, W.dout_for(w)
    s_q = w["q"].shape[0]
    cores = len(os.sched_getaffinity(0))
    per_step = max(1, cores)
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        rows = rng.choice(s_q, size=min(per_step, s_q), replace=False)
        _oracle_call(oracle, w, rows)
    t_total, flops = 0.0, 0.0
    for _ in range(args.steps):
        rows = rng.choice(s_q, size=min(per_step, s_q), replace=False)
        t0 = time.perf_counter()
        _oracle_call(oracle, w, rows)
        t_total += time.perf_counter() - t0
        flops += valid_flops(w, rows, backward=bwd)
    value = flops / t_total / 1e12
    sample = f"{per_step} random rows per step of the {args.config} batch ({args.steps} steps)"
    line = {"impl": "reference", "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": describe(w, args.config), "topk_length": "passed" if w["topk_length"] is not None else "omitted"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _oracle_call(oracle, w, rows):
    if w.get("backward"):
        q = w["q"][rows]
        idx = w["indices"].reshape(w["q"].shape[0], -1)[rows]
        return oracle.sparse_mla_bwd(q, w["kv"], w["dout"][rows], idx, None, None, w["sm_scale"])
    if w.get("paged"):
        return oracle.sparse_mla_fwd_paged(w["q"], w["kv"], w["block_table"], w["indices"], w["page_block"],
                                           w.get("seqlens_k"), w["s_kv_per_req"], w["s_q_per_req"],
                                           w["topk_length"], w["attn_sink"], w["sm_scale"], w["d_v"], rows=rows)
    return oracle.sparse_mla_fwd(w["q"], w["kv"], w["indices"], w["topk_length"], w["attn_sink"],
                                 w["sm_scale"], w["d_v"], rows=rows)


def cpu_model():
    """The host CPU's model name (lscpu's "Model name", else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def cpu_baseline(w, name, budget_s=12.0):
    """The oracle as it stands, on a bounded row sample of the same workload."""
    import oracle

    s_q = w["q"].shape[0]
    cores = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(1)
    order = rng.permutation(s_q)
    done, t_total, flops, pos = 0, 0.0, 0.0, 0
    chunk = max(cores, 1)
    while t_total < budget_s and pos < s_q:
        rows = np.sort(order[pos:pos + chunk])
        pos += chunk
        t0 = time.perf_counter()
        _oracle_call(oracle, w, rows)
        t_total += time.perf_counter() - t0
        flops += valid_flops(w, rows, backward=bool(w.get("backward")))
        done += len(rows)
    return {"value": flops / t_total / 1e12, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
            "sample": f"{done} random rows of the {name} batch ({t_total:.1f} s of fp64 CPU work)"}


def shard_rows(w, rank, world):
    """This rank's contiguous rows of a flat workload (query rows are independent; the shared KV
    is whole on every rank)."""
    from sparse_mla_attention_fwd_gb300 import row_shard
    s_q = w["q"].shape[0]
    r0, r1 = row_shard(s_q, rank, world)
    out = dict(w)
    for k in ("q", "indices", "topk_length", "valid_counts"):
        if out.get(k) is not None:
            out[k] = np.ascontiguousarray(out[k][r0:r1])
    return out, (r0, r1)


def decode_fixed_vs_dynamic(smla, torch, dev, stream, flush, n=30):
    """The paged decode shape (256 requests, h_q 128, d_qk 576, 64-token pages, topk 2048) in its
    two forms, timed interleaved on the device: dynamic = the first 1024 slots valid, an INT_MAX
    suffix and topk_length = 1024; fixed = the same 1024 slots, a -1 suffix and no topk_length
    (FlashMLA PR #216, "Kernel performance" compares exactly these two runs).  The kernel derives
    the fixed run's length itself, so both should cost the same."""
    runs = {}
    for name, dyn in (("dynamic", True), ("fixed", False)):
        w = W.decode(dynamic=dyn)
        d = {}
        for k in ("q", "kv", "indices", "topk_length", "block_table"):
            a = w.get(k)
            if a is None:
                d[k] = None
                continue
            t = torch.from_numpy(np.ascontiguousarray(a))
            if a.dtype == np.uint16:
                t = t.view(torch.int16).view(torch.bfloat16)
            d[k] = t.to(dev)
        runs[name] = (w, d)
    w0 = runs["dynamic"][0]
    s_q, h_q = w0["q"].shape[:2]
    out = torch.empty((s_q, h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s_q, h_q), dtype=torch.float32, device=dev)
    mx = torch.empty_like(lse)

    def call(name):
        w, d = runs[name]
        smla.sparse_mla_fwd_paged(d["q"], d["kv"], d["block_table"], d["indices"], page_block=w["page_block"],
                                  s_kv_per_req=w["s_kv_per_req"], s_q_per_req=w["s_q_per_req"],
                                  topk_length=d["topk_length"], sm_scale=w["sm_scale"], out=out, lse=lse,
                                  max_logits=mx, stream=stream, n_split=1)

    for _ in range(3):
        call("dynamic")
        call("fixed")
    ms = {"dynamic": [], "fixed": []}
    for _ in range(n):
        for name in ("dynamic", "fixed"):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(name)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ms[name].append(a.elapsed_time(b))
    md, mf = float(np.median(ms["dynamic"])), float(np.median(ms["fixed"]))
    flops = valid_flops(w0)
    return {"workload": describe(w0, "decode"), "ms_dynamic": md, "ms_fixed": mf,
            "fixed_vs_dynamic_gap_pct": 100.0 * (mf - md) / md, "tflops_dynamic": flops / (md * 1e-3) / 1e12,
            "launches": 6 + 2 * n,
            "bandwidth": bandwidth(w0, "decode", md)}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch

    import sparse_mla_attention_fwd_gb300 as smla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    w = make_workload(args.config, args.with_len)
    if args.config == "bwd":
        return main_bwd(args, w, world, rank, local, dev, barrier)
    row_split = args.shard == "rows" and world > 1 and not w.get("paged")
    shard = None
    if row_split:
        w, shard = shard_rows(w, rank, world)
    s_q, h_q, d_qk = w["q"].shape
    flops = valid_flops(w)

    def host_tensor(a, pinned=True):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a)
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory() if pinned else t

    names = ["q", "kv", "indices", "topk_length", "attn_sink"]
    if w.get("paged"):
        names += ["block_table"]
    host = {k: host_tensor(w.get(k)) for k in names}
    devt = {k: (None if v is None else v.to(dev)) for k, v in host.items()}
    out = torch.empty((s_q, h_q, w["d_v"]), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((s_q, h_q), dtype=torch.float32, device=dev)
    mx = torch.empty((s_q, h_q), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    topk = w["indices"].reshape(s_q, -1).shape[1]
    n_split = smla.auto_splits(s_q, h_q, topk, dev) if args.n_split == "auto" else int(args.n_split)
    launches_per_call = 2 if n_split > 1 else 1   # split-KV adds the merge kernel

    def call(d, tl="auto"):
        t = d["topk_length"] if isinstance(tl, str) else tl
        if w.get("paged"):
            return smla.sparse_mla_fwd_paged(d["q"], d["kv"], d["block_table"], d["indices"],
                                             page_block=w["page_block"], s_kv_per_req=w["s_kv_per_req"],
                                             s_q_per_req=w["s_q_per_req"], topk_length=t,
                                             attn_sink=d["attn_sink"], sm_scale=w["sm_scale"],
                                             d_v=w["d_v"], out=out, lse=lse, max_logits=mx, stream=stream,
                                             n_split=n_split)
        return smla.sparse_mla_fwd(d["q"], d["kv"], d["indices"], t, d["attn_sink"], sm_scale=w["sm_scale"],
                                   d_v=w["d_v"], out=out, lse=lse, max_logits=mx, stream=stream, n_split=n_split)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > 129 MB L2

    def timed_steps(n, tl="auto"):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush.zero_()
            ev[i][0].record(stream)
            call(devt, tl)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]

    for _ in range(args.warmup):
        call(devt)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0.0)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    step_ms = timed_steps(args.steps)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    total_ms = max_over_ranks(float(np.sum(step_ms)), dev)
    ms_per_step = total_ms / args.steps
    job_flops = sum_over_ranks(flops, dev)      # replicas: every rank its own batch; rows: its slice
    value = job_tflops(job_flops * args.steps, total_ms)
    launches = args.steps * launches_per_call

    # the same rows with topk_length passed (padding-overhead check), non-paged ramp only: the
    # two forms alternate call by call, and the gap is taken between their medians
    extra = {}
    if args.config == "ramp":
        counts = torch.from_numpy(w["valid_counts"]).to(dev)
        no_len, with_len = [], []
        for _ in range(max(20, args.steps // 3)):
            no_len += timed_steps(1, tl=None)
            with_len += timed_steps(1, tl=counts)
        launches += (len(no_len) + len(with_len)) * launches_per_call
        ms_no_len, ms_len = float(np.median(no_len)), float(np.median(with_len))
        extra = {"ms_no_topk_length": ms_no_len, "ms_topk_length_passed": ms_len,
                 "padding_gap_pct": 100.0 * (ms_no_len - ms_len) / ms_len,
                 "padding_gap_how": f"medians of {len(no_len)} interleaved calls of each form",
                 "valid_token_tflop": flops / 1e12}

    # the decode shape's fixed-width run against its dynamic-length run (default run only)
    decode_leg = None
    if args.config == "ramp" and not args.skip_decode:
        decode_leg = decode_fixed_vs_dynamic(smla, torch, dev, stream, flush)
        launches += decode_leg["launches"]

    # end to end through the C ABI with host buffers: the host-buffer entry point copies each
    # row chunk's inputs in, runs the forward on it and copies its outputs out, with copies and
    # compute overlapped on three streams; all of it is inside the timed region
    e2e = None
    if not args.skip_e2e:
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        mx_h = torch.empty(mx.shape, dtype=mx.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = sum(t.numel() * t.element_size() for t in (out, lse, mx))
        copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        dev_buffers = dict(devt, out=out, lse=lse, max_logits=mx)
        e_ms = []

        def e2e_call():
            if w.get("paged"):
                # the paged form has no host-buffer entry: serial copies around the device call
                for k, v in host.items():
                    if v is not None:
                        devt[k].copy_(v, non_blocking=True)
                call(devt)
                out_h.copy_(out, non_blocking=True)
                lse_h.copy_(lse, non_blocking=True)
                mx_h.copy_(mx, non_blocking=True)
                return 1
            smla.sparse_mla_fwd_host(host["q"], host["kv"], host["indices"], host["topk_length"], host["attn_sink"],
                                     sm_scale=w["sm_scale"], d_v=w["d_v"], out=out_h, lse=lse_h, max_logits=mx_h,
                                     device=dev, dev_buffers=dev_buffers, n_chunks=args.e2e_chunks, stream=stream,
                                     copy_streams=copy_streams)
            return min(args.e2e_chunks, s_q)

        launches_e2e = 0
        for i in range(args.e2e_steps + 2):
            flush.zero_()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            launches_e2e += e2e_call()
            b.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                e_ms.append(a.elapsed_time(b))
        e2e_ms = max_over_ranks(float(np.mean(e_ms)), dev)
        e2e = {"value": job_tflops(job_flops, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms,
               "how": (f"sparse_mla_fwd_host: pinned host buffers, {args.e2e_chunks} row chunks, H2D / compute / "
                       "D2H overlapped on three streams" if not w.get("paged") else
                       "serial H2D, device call, D2H on one stream")}
        launches += launches_e2e * launches_per_call

    status = smla.sparse_mla_device_status()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    roof = nearer_roof(achieved, algorithmic_bytes(w)[0] / (ms_per_step * 1e-3) / 1e9, peaks, src,
                       profiled_counters(args.config).get("dram_bytes_per_launch"), "sparse_mla_fwd_kernel")
    base = PAGES_B200_TFLOPS.get((args.config, bool(args.with_len)))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if row_split else "weak", "vs_baseline": (value / base) if base else None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": describe(w, args.config),
                   "topk_length": "passed" if (args.with_len or w["topk_length"] is not None) else "omitted",
                   "l2": "flushed (256 MB write) between timed iterations", "n_split": n_split,
                   "pct_of_bf16_peak": 100.0 * achieved / peak,
                   "parallelism": (f"rows split over {world} GPUs (rank 0: rows {shard[0]}..{shard[1]})" if row_split
                                   else f"{world} replica(s), one batch per GPU"),
                   "vs_baseline_ref": "FlashMLA PR #196 B200 number (other hardware, context)" if base else None},
        "roofline": roof,
        "clocks": clocks,
        "gpu_launches": args.steps * launches_per_call,
        "gpu_launches_total": launches,
        "device_status": status,
    }
    line.update(extra)
    line["bandwidth"] = bandwidth(w, args.config, ms_per_step)
    if decode_leg is not None:
        line["decode_fixed_vs_dynamic"] = decode_leg
    if e2e is not None:
        line["e2e"] = e2e
    if not args.skip_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.config)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main_bwd(args, w, world, rank, local, dev, barrier):
    """The backward: each step is one sparse_mla_bwd call on the batch, given the forward's out
    and lse (computed once, outside the timed region)."""
    import torch

    import sparse_mla_attention_fwd_gb300 as smla

    w["backward"], w["dout"] = True, W.dout_for(w)
    s_q, h_q, d_qk = w["q"].shape
    s_kv = w["kv"].shape[0]
    flops = valid_flops(w, backward=True)
    stream = torch.cuda.current_stream(dev)

    def host_tensor(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.int16).view(torch.bfloat16)
        return t.pin_memory()

    host = {k: host_tensor(w[k]) for k in ("q", "kv", "indices", "dout")}
    d = {k: v.to(dev) for k, v in host.items()}
    out, lse, _ = smla.sparse_mla_fwd(d["q"], d["kv"], d["indices"], sm_scale=w["sm_scale"], stream=stream)
    host["out"], host["lse"] = out.cpu().pin_memory(), lse.cpu().pin_memory()
    d["out"], d["lse"] = out, lse
    dq = torch.empty((s_q, h_q, d_qk), dtype=torch.float32, device=dev)
    dkv = torch.empty((s_kv, d_qk), dtype=torch.float32, device=dev)

    def call():
        smla.sparse_mla_bwd(d["q"], d["kv"], d["out"], d["dout"], d["indices"], d["lse"], sm_scale=w["sm_scale"],
                            dq=dq, dkv=dkv, stream=stream)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    steps = max(3, min(args.steps, 30))          # a call is tens of ms: bound the timed work
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0.0)
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(np.sum(step_ms)), dev)
    ms_per_step = total_ms / steps
    job_flops = sum_over_ranks(flops, dev)
    value = job_tflops(job_flops * steps, total_ms)

    e2e = None
    if not args.skip_e2e:
        dq_h = torch.empty(dq.shape, dtype=dq.dtype).pin_memory()
        dkv_h = torch.empty(dkv.shape, dtype=dkv.dtype).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = dq.numel() * 4 + dkv.numel() * 4
        e_ms = []
        for i in range(4):
            flush.zero_()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k, v in host.items():
                d[k].copy_(v, non_blocking=True)
            call()
            dq_h.copy_(dq, non_blocking=True)
            dkv_h.copy_(dkv, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 1:
                e_ms.append(a.elapsed_time(b))
        e2e_ms = max_over_ranks(float(np.mean(e_ms)), dev)
        e2e = {"value": job_tflops(job_flops, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms}
    status = smla.sparse_mla_device_status()
    if rank != 0:
        return
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": describe(w, "bwd"), "topk_length": "omitted",
                   "l2": "flushed (256 MB write) between timed iterations",
                   "pct_of_bf16_peak": 100.0 * achieved / peak},
        "roofline": nearer_roof(achieved, algorithmic_bytes(w, backward=True)[0] / (ms_per_step * 1e-3) / 1e9,
                                peaks, src, profiled_counters("bwd").get("dram_bytes_per_launch"),
                                "sparse_mla_bwd_kernel"),
        "clocks": clocks, "gpu_launches": steps, "device_status": status,
    }
    line["bandwidth"] = bandwidth(w, "bwd", ms_per_step, backward=True)
    if e2e is not None:
        line["e2e"] = e2e
    if not args.skip_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, "bwd")
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
