"""Shared helpers for the GPU parity tests: move seeded inputs to the device, call the CUDA
path through its C ABI, and compare with the oracle under the acceptance bar:
  * validity / empty rows bit-exact: O exactly +0, lse exactly +inf, max_logits exactly -inf
    on exactly the oracle's empty rows, finite everywhere else;
  * O: max-abs error <= 2e-2 and relative L2 error <= 5e-3;
  * lse and max_logits: <= 1e-3 absolute.
"""
import numpy as np
import torch

import oracle
import sparse_mla_attention_fwd_gb300 as smla

O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
LSE_ABS = 1e-3


def dev_tensor(a, device="cuda:0"):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


def run_gpu(w, topk_length="auto", indices=None, n_split=1):
    """Run the workload dict `w` through the CUDA path.  topk_length="auto" uses w's; n_split > 1
    runs the split-KV variant."""
    tl = w["topk_length"] if isinstance(topk_length, str) else topk_length
    idx = w["indices"] if indices is None else indices
    if w.get("paged"):
        out = smla.sparse_mla_fwd_paged(
            dev_tensor(w["q"]), dev_tensor(w["kv"]), dev_tensor(w["block_table"]), dev_tensor(idx),
            page_block=w["page_block"], seqlens_k=dev_tensor(w.get("seqlens_k")),
            s_kv_per_req=w["s_kv_per_req"], s_q_per_req=w["s_q_per_req"], topk_length=dev_tensor(tl),
            attn_sink=dev_tensor(w["attn_sink"]), sm_scale=w["sm_scale"], d_v=w["d_v"], n_split=n_split)
    else:
        out = smla.sparse_mla_fwd(dev_tensor(w["q"]), dev_tensor(w["kv"]), dev_tensor(idx),
                                  dev_tensor(tl), dev_tensor(w["attn_sink"]), sm_scale=w["sm_scale"],
                                  d_v=w["d_v"], n_split=n_split)
    torch.cuda.synchronize()
    return out


def run_oracle(w, rows=None, topk_length="auto", indices=None):
    tl = w["topk_length"] if isinstance(topk_length, str) else topk_length
    idx = w["indices"] if indices is None else indices
    if w.get("paged"):
        return oracle.sparse_mla_fwd_paged(w["q"], w["kv"], w["block_table"], idx, w["page_block"],
                                           w.get("seqlens_k"), w["s_kv_per_req"], w["s_q_per_req"],
                                           tl, w["attn_sink"], w["sm_scale"], w["d_v"], rows=rows)
    return oracle.sparse_mla_fwd(w["q"], w["kv"], idx, tl, w["attn_sink"], w["sm_scale"], w["d_v"],
                                 rows=rows)


def to_np(gpu_out, rows=None):
    out, lse, mx = gpu_out
    if rows is not None:
        r = torch.as_tensor(np.asarray(rows), device=out.device)
        out, lse, mx = out[r], lse[r], mx[r]
    return (out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            mx.cpu().numpy().astype(np.float64))


def assert_parity(gpu, ref, what=""):
    og, lg, mg = gpu
    orf, lr, mr = ref
    empty = np.isinf(lr) & (lr > 0)
    # validity / empty rows: bit-exact
    assert np.array_equal(lg == np.inf, empty), f"{what}: +inf lse pattern differs"
    assert np.all(mg[empty] == -np.inf), f"{what}: max_logits of empty rows must be -inf"
    assert np.all(og[empty] == 0.0) and not np.any(np.signbit(og[empty])), f"{what}: O of empty rows must be +0"
    fin = ~empty
    assert np.all(np.isfinite(lg[fin])) and np.all(np.isfinite(mg[fin])), f"{what}: non-finite lse/max"
    assert np.all(np.isfinite(og)), f"{what}: non-finite O"
    err = np.abs(og - orf)
    assert err.max() <= O_MAX_ABS, f"{what}: O max-abs {err.max():.3e}"
    den = np.linalg.norm(orf)
    if den > 0:
        rel = np.linalg.norm(og - orf) / den
        assert rel <= O_REL_L2, f"{what}: O rel-L2 {rel:.3e}"
    if fin.any():
        el = np.abs(lg[fin] - lr[fin]).max()
        em = np.abs(mg[fin] - mr[fin]).max()
        assert el <= LSE_ABS, f"{what}: lse abs {el:.3e}"
        assert em <= LSE_ABS, f"{what}: max_logits abs {em:.3e}"
    return dict(o_max_abs=float(err.max()), o_rel_l2=float(np.linalg.norm(og - orf) / max(den, 1e-300)))
