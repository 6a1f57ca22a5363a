"""GPU parity of the sparse MLA backward against the fp64 oracle (oracle/sparse_mla_bwd_oracle.c).

The CUDA forward produces out / lse, the CUDA backward the gradients; the oracle recomputes the
exact gradients of sum(dout * O) from q, kv and dout alone.  Acceptance:
  * bit-exact: dq is exactly 0 on rows without a counted slot, dkv exactly 0 on kv rows no
    counted slot selects;
  * elsewhere, per tensor, relative L2 error <= 1e-2 and max-abs error <= 3e-2 * max|ref|.
The tolerance follows from the arithmetic: P and sm_scale * dS enter the tensor-core products
as bf16 (unit roundoff 2^-9), D = <dout, out> uses the forward's bf16 out, and everything is
accumulated in fp32; independent rounding of that size leaves a relative L2 error of a few
2^-9 (~0.5 %).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_mla_attention_fwd_gb300 as smla
import workloads as W
from gpu_helpers import dev_tensor

REL_L2 = 1e-2
MAX_REL = 3e-2

pytestmark = pytest.mark.gpu


def _run(w, dout):
    q, kv, idx = dev_tensor(w["q"]), dev_tensor(w["kv"]), dev_tensor(w["indices"])
    tl, sink = dev_tensor(w["topk_length"]), dev_tensor(w["attn_sink"])
    out, lse, _ = smla.sparse_mla_fwd(q, kv, idx, tl, sink, sm_scale=w["sm_scale"])
    dq, dkv, ds = smla.sparse_mla_bwd(q, kv, out, dev_tensor(dout), idx, lse, tl, sink, sm_scale=w["sm_scale"])
    torch.cuda.synchronize()
    assert smla.sparse_mla_device_status(reset=True) == 0
    return dq.cpu().numpy(), dkv.cpu().numpy(), None if ds is None else ds.cpu().numpy()


def _close(got, ref, name):
    err = got.astype(np.float64) - ref
    scale = float(np.abs(ref).max())
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    assert rel <= REL_L2, f"{name}: relative L2 error {rel:.3e}"
    assert float(np.abs(err).max()) <= MAX_REL * max(scale, 1e-30), f"{name}: max-abs error {np.abs(err).max():.3e}"


def _counted(w):
    idx = w["indices"].reshape(w["indices"].shape[0], -1)
    s_kv = w["kv"].shape[0]
    ok = (idx >= 0) & (idx < s_kv)
    if w["topk_length"] is not None:
        ok &= np.arange(idx.shape[1])[None, :] < np.clip(w["topk_length"], 0, idx.shape[1])[:, None]
    return idx, ok


CASES = [
    # seed, s_q, s_kv, h_q, d_qk, topk, with_len, with_sink, dup
    (1, 64, 900, 64, 576, 200, True, True, True),
    (2, 40, 700, 128, 512, 130, False, False, False),
    (3, 24, 5000, 64, 576, 1024, False, True, False),
    (4, 32, 333, 64, 512, 64, True, True, True),
    (5, 16, 2000, 128, 576, 96, True, False, False),
    (6, 10, 50, 192, 576, 1, True, True, False),        # one slot per row, three head groups
    (7, 12, 3000, 256, 512, 2500, False, True, True),   # 40 blocks per row, four head groups
]


@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}_h{c[3]}_d{c[4]}_k{c[5]}" for c in CASES])
def test_bwd_matches_oracle(case):
    seed, s_q, s_kv, h_q, d_qk, topk, with_len, with_sink, dup = case
    w = W.random_case(seed, s_q, s_kv, h_q, d_qk, topk, with_len=with_len, with_sink=with_sink,
                      poison_suffix=with_len, dup=dup)
    dout = W.dout_for(w, salt=seed)
    dq, dkv, ds = _run(w, dout)
    rq, rkv, rs = oracle.sparse_mla_bwd(w["q"], w["kv"], dout, w["indices"], w["topk_length"], w["attn_sink"],
                                        w["sm_scale"])
    idx, ok = _counted(w)
    empty = ~ok.any(axis=1)
    assert empty.any() or s_q < 8
    assert np.all(dq[empty] == 0.0), "dq of rows without a counted slot must be exactly 0"
    untouched = np.ones(s_kv, bool)
    untouched[np.unique(idx[ok])] = False
    assert np.all(dkv[untouched] == 0.0), "dkv rows no slot selects must be exactly 0"
    _close(dq, rq, "dq")
    _close(dkv, rkv, "dkv")
    if with_sink:
        _close(ds, rs, "dsink")
    else:
        assert ds is None


def test_bwd_dq_is_deterministic_and_dkv_stable():
    w = W.random_case(6, 32, 800, 64, 576, 192, with_sink=True)
    dout = W.dout_for(w, salt=6)
    a = _run(w, dout)
    b = _run(w, dout)
    np.testing.assert_array_equal(a[0], b[0])          # dq: no atomics
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-4 * float(np.abs(a[1]).max()))


def test_bwd_full_size_sampled_rows_and_column_sums():
    """The backward on the bench shape (s_q 4096, s_kv 32768, h_q 64, d_qk 576, topk 2048) in the
    launch configuration bench.py times.  dq of a row depends on that row alone, so sampled rows
    are checked against the oracle one by one.  dkv is checked element by element on sampled kv
    rows (against the oracle over every query row that selects them) and, at every column,
    through a property that holds at any size: without a sink, sum_s dS_s = D (1 - sum_s p_s) = 0 for every (row, head), so the
    column sums of dkv are sum_{t,h} dO[t,h,d] on the value columns and 0 on the rope columns."""
    w = W.bwd_prefill()
    dout = W.dout_for(w)
    dq, dkv, ds = _run(w, dout)
    assert ds is None
    rows = np.array([0, 1, 777, 2048, 3001, 4095])
    idx = w["indices"].reshape(w["q"].shape[0], -1)
    rq, _, _ = oracle.sparse_mla_bwd(w["q"][rows], w["kv"], dout[rows], idx[rows], None, None, w["sm_scale"])
    _close(dq[rows], rq, "dq (sampled rows)")
    # dkv element by element on sampled kv rows: the oracle over every query row that selects
    # one of them gives those rows' complete gradient
    kv_rows = np.array([5, 12345, 20000, w["kv"].shape[0] - 1])
    sel = np.where(np.isin(idx, kv_rows).any(axis=1))[0]
    assert len(sel) > 100
    _, rkv, _ = oracle.sparse_mla_bwd(w["q"][sel], w["kv"], dout[sel], idx[sel], None, None, w["sm_scale"])
    _close(dkv[kv_rows], rkv[kv_rows], "dkv (sampled kv rows, every selecting row)")
    d_v = w["d_v"]
    ref = np.zeros(w["q"].shape[2])
    ref[:d_v] = oracle.bf16_bits_to_f64(dout).sum(axis=(0, 1))
    got = dkv.astype(np.float64).sum(axis=0)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    assert rel <= REL_L2, f"dkv column sums: relative L2 error {rel:.3e}"
