"""The host-buffer entry point (sparse_mla_fwd_host: inputs and outputs in pinned host memory,
copies pipelined over row chunks on their own streams) and the row-sharded forward
(sparse_mla_fwd_sharded).  Rows are independent, so every chunking and every sharding must give
the same bits as one device call on the whole batch; the device call itself is checked against
the oracle."""
import numpy as np
import pytest
import torch

import sparse_mla_attention_fwd_gb300 as smla
import workloads as W
from gpu_helpers import assert_parity, run_gpu, run_oracle, to_np

pytestmark = pytest.mark.gpu


def _host(a):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.pin_memory()


@pytest.mark.parametrize("n_chunks", [1, 3, 8, 64])
@pytest.mark.parametrize("with_len", [False, True])
def test_host_entry_equals_device_call(n_chunks, with_len):
    w = W.random_case(77, 37, 2000, 128, 576, 300, with_len=with_len, with_sink=True,
                      poison_suffix=with_len, dup=True)
    ref = run_gpu(w)
    out, lse, mx = smla.sparse_mla_fwd_host(_host(w["q"]), _host(w["kv"]), _host(w["indices"]),
                                            _host(w["topk_length"]), _host(w["attn_sink"]),
                                            sm_scale=w["sm_scale"], n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref[0].cpu().view(torch.int16))
    assert torch.equal(lse, ref[1].cpu()) and torch.equal(mx, ref[2].cpu())
    if n_chunks == 3:
        assert_parity(to_np(ref), run_oracle(w), f"device call len={with_len}")


def test_host_entry_with_an_empty_kv():
    # s_kv == 0: nothing to copy for kv, and every row is empty (O = 0, lse = +inf, max = -inf)
    w = W.random_case(80, 11, 40, 128, 576, 24, with_sink=True)
    w = dict(w, kv=w["kv"][:0])
    out, lse, mx = smla.sparse_mla_fwd_host(_host(w["q"]), _host(w["kv"]), _host(w["indices"]),
                                            attn_sink=_host(w["attn_sink"]), sm_scale=w["sm_scale"],
                                            n_chunks=4)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0) and torch.all(lse == float("inf")) and torch.all(mx == float("-inf"))


def test_host_entry_ramp_shape_in_chunks():
    # the benchmark's batch through the host entry, as bench.py's end-to-end leg runs it
    w = W.ramp()
    ref = run_gpu(w, topk_length=None)
    out, lse, mx = smla.sparse_mla_fwd_host(_host(w["q"]), _host(w["kv"]), _host(w["indices"]),
                                            sm_scale=w["sm_scale"], n_chunks=8)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref[0].cpu().view(torch.int16))
    assert torch.equal(lse, ref[1].cpu()) and torch.equal(mx, ref[2].cpu())


@pytest.mark.parametrize("world", [2, 3])
def test_row_sharded_forward_equals_one_call(world):
    # each rank's contiguous rows of one batch, computed alone, are exactly those rows of the
    # whole batch's result (rows are independent)
    w = W.random_case(78, 41, 1500, 128, 576, 260, with_len=True, with_sink=True, poison_suffix=True)
    from gpu_helpers import dev_tensor
    ref = run_gpu(w)
    q, kv, idx = dev_tensor(w["q"]), dev_tensor(w["kv"]), dev_tensor(w["indices"])
    tl, sink = dev_tensor(w["topk_length"]), dev_tensor(w["attn_sink"])
    seen = 0
    for rank in range(world):
        (r0, r1), (out, lse, mx) = smla.sparse_mla_fwd_sharded(q, kv, idx, rank, world, topk_length=tl,
                                                               attn_sink=sink, sm_scale=w["sm_scale"])
        torch.cuda.synchronize()
        assert r0 == seen
        seen = r1
        assert torch.equal(out.view(torch.int16), ref[0][r0:r1].view(torch.int16))
        assert torch.equal(lse, ref[1][r0:r1]) and torch.equal(mx, ref[2][r0:r1])
    assert seen == 41
