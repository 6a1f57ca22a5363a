"""The allocation-free split-KV entry point (sparse_mla_fwd_paged_splitkv_static): its partial
results live in the library's own 32 MiB __device__ scratch array.  This file is collected
last (its name sorts after every other test file), so it runs both alone and after the rest
of the suite.  The GPU test compares it with sparse_mla_fwd_paged_splitkv, which takes a
caller workspace, on two calls in a row: the same kernels over the same inputs must give the
same bits, and the second call must not see anything left from the first."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_mla_attention_fwd_gb300 as smla
import workloads as W
from sparse_mla_attention_fwd_gb300 import _native
from sparse_mla_attention_fwd_gb300.native_build import build

SCRATCH_BYTES = 32 << 20


def _decode_case(seed, n_req=2, s_q_per_req=2, topk=2048):
    w = W.decode_fixed(n_req=n_req, s_q_per_req=s_q_per_req, s_kv=4096, topk=topk)
    rng = np.random.default_rng(seed)
    s_q = n_req * s_q_per_req
    w["topk_length"] = rng.integers(0, topk + 1, size=s_q).astype(np.int32)
    w["topk_length"][0] = topk
    w["attn_sink"] = rng.standard_normal(128).astype(np.float32)
    return w


def _dev(a):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.int16 or a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def _args(w):
    return dict(q=_dev(w["q"]), kv_pool=_dev(w["kv"]), block_table=_dev(w["block_table"]),
                indices=_dev(w["indices"]), page_block=w["page_block"], s_kv_per_req=w["s_kv_per_req"],
                s_q_per_req=w["s_q_per_req"], topk_length=_dev(w["topk_length"]),
                attn_sink=_dev(w["attn_sink"]), sm_scale=w["sm_scale"])


def test_oversized_problems_are_rejected_before_launch():
    build()
    lib = _native.load_library()
    size = lib.sparse_mla_splitkv_workspace_size
    # 2 rows x 2 head groups x 64 ranges = 256 units of 128.75 KiB: too big for 32 MiB
    assert size(2, 128, 64) > SCRATCH_BYTES
    fake = 1 << 20
    rc = lib.sparse_mla_fwd_paged_splitkv_static(
        fake, fake, 4096, fake, 64, 64, None, 4096, 1, fake, None, None, ctypes.c_float(0.04), 512,
        fake, fake, fake, 2, 128, 576, 2048, 64, None)
    assert rc == 7   # SMLA_ERR_WORKSPACE
    # no rows: a no-op that returns SMLA_OK whatever n_split is (no scratch lookup, no launch)
    for n_split in (1, 2, 64):
        rc = lib.sparse_mla_fwd_paged_splitkv_static(
            fake, fake, 4096, fake, 64, 64, None, 4096, 1, fake, None, None, ctypes.c_float(0.04), 512,
            fake, fake, fake, 0, 128, 576, 2048, n_split, None)
        assert rc == 0, (n_split, rc)


@pytest.mark.gpu
def test_static_scratch_matches_workspace_call_twice():
    n_split = 8
    for seed in (1, 2):   # two calls in a row through the same scratch
        w = _decode_case(seed)
        a = _args(w)
        ref = smla.sparse_mla_fwd_paged(**a, n_split=n_split)
        got = smla.sparse_mla_fwd_paged_splitkv_static(**a, n_split=n_split)
        torch.cuda.synchronize()
        assert torch.equal(got[0].view(torch.int16), ref[0].view(torch.int16)), f"out differs (call {seed})"
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), f"lse/max differ (call {seed})"
    assert smla.sparse_mla_device_status() == 0
