"""Host-side arithmetic of bench.py, checked on CPU: the roofline object names the roof the
kernel is nearer to, and the algorithmic byte counts take every tensor of a call exactly once
(counted here from the arrays themselves)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402

PEAKS = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}


def test_nearer_roof_names_the_closer_roof():
    # 500 TFLOP/s is 25 % of the tensor roof; 4000 GB/s is 50 % of the HBM roof
    r = bench.nearer_roof(500.0, 4000.0, PEAKS, "test", 123, "k")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(0.5) and r["achieved"] == 4000.0 and r["peak"] == 8000.0
    assert r["other_roof"]["bound"] == "tensor" and r["other_roof"]["frac"] == pytest.approx(0.25)
    assert r["traffic"] == 123 and r["kernel"] == "k"
    r = bench.nearer_roof(1000.0, 800.0, PEAKS, "test", None, "k")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["frac"] == pytest.approx(0.5)
    assert r["other_roof"]["bound"] == "hbm" and r["other_roof"]["frac"] == pytest.approx(0.1)
    assert r["traffic"] is None


def _counted(w):
    """Counted slots of every row, by the definition: slot j counts iff j < L_t and
    0 <= idx < s_kv (L_t = topk when no topk_length is given)."""
    s_q = w["q"].shape[0]
    idx = np.asarray(w["indices"]).reshape(s_q, -1).astype(np.int64)
    topk = idx.shape[1]
    L = np.full(s_q, topk) if w["topk_length"] is None else np.clip(np.asarray(w["topk_length"]), 0, topk)
    j = np.arange(topk)[None, :]
    return ((j < L[:, None]) & (idx >= 0) & (idx < w["s_kv"])).sum()


@pytest.mark.parametrize("with_len", [False, True])
def test_forward_bytes_take_every_tensor_once(with_len):
    w = W.tiny(with_len=with_len)
    s_q, h_q, d_qk = w["q"].shape
    hbm, gather = bench.algorithmic_bytes(w)
    out_bytes = s_q * h_q * w["d_v"] * 2                   # O in bf16
    stats_bytes = 2 * s_q * h_q * 4                         # lse and max_logits in fp32
    expect = (np.asarray(w["q"]).nbytes + np.asarray(w["indices"]).nbytes + np.asarray(w["kv"]).nbytes
              + out_bytes + stats_bytes)
    if with_len:
        expect += np.asarray(w["topk_length"]).astype(np.int32).nbytes
    assert hbm == expect
    assert gather == _counted(w) * d_qk * 2


def test_backward_bytes_take_every_tensor_once():
    w = W.tiny()
    s_q, h_q, d_qk = w["q"].shape
    s_kv = w["kv"].shape[0]
    hbm, _ = bench.algorithmic_bytes(w, backward=True)
    ins = (np.asarray(w["q"]).nbytes + np.asarray(w["indices"]).nbytes + np.asarray(w["kv"]).nbytes
           + 2 * s_q * h_q * w["d_v"] * 2 + s_q * h_q * 4)     # + out, dout (bf16), lse
    outs = s_q * h_q * d_qk * 4 + s_kv * d_qk * 4              # dq, dkv (fp32)
    assert hbm == ins + outs


def test_paged_bytes_read_every_gathered_row():
    w = W.decode(n_req=4, s_kv=256, h_q=64, topk=128, n_valid=64, page_block=64)
    d_qk = w["q"].shape[2]
    hbm, gather = bench.algorithmic_bytes(w)
    s_q, h_q = w["q"].shape[0], w["q"].shape[1]
    expect = (np.asarray(w["q"]).nbytes + np.asarray(w["indices"]).nbytes
              + np.asarray(w["topk_length"]).astype(np.int32).nbytes + np.asarray(w["block_table"]).astype(np.int32).nbytes
              + gather + s_q * h_q * w["d_v"] * 2 + 2 * s_q * h_q * 4)
    assert gather == _counted(w) * d_qk * 2
    assert hbm == expect


def test_counters_are_used_only_for_the_kernel_source_they_were_taken_on(monkeypatch):
    entry = bench.profiled_counters("ramp")
    if entry:
        assert entry["kernel_source_hash"] == bench.kernel_source_hash("fwd")
        assert entry["dram_bytes_per_launch"] > 0
    # any other source: no counters, so the bench line reports traffic as unknown
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="fwd": "0" * 16)
    for name in ("ramp", "decode", "full", "scattered", "bwd"):
        assert bench.profiled_counters(name) == {}
    assert bench.profiled_counters("no_such_workload") == {}


def test_kernel_source_hash_covers_the_backward_file_only_for_the_backward():
    fwd, bwd = bench.kernel_source_hash("fwd"), bench.kernel_source_hash("bwd")
    assert len(fwd) == 16 and len(bwd) == 16 and fwd != bwd
    int(fwd, 16), int(bwd, 16)
