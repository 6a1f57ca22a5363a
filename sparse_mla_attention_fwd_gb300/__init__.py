"""GB300-native sparse MLA attention forward and backward (DeepSeek-style DSA top-k), sm_103a.

Python names mirror the C ABI of include/sparse_mla.h.  Tensors are torch CUDA tensors (torch
supplies device memory and streams only); outputs are allocated here when not given.

    out, lse, max_logits = sparse_mla_fwd(q, kv, indices, topk_length=None, attn_sink=None,
                                          sm_scale=None, d_v=512)

Semantics (FlashMLA PR #196 "Problem"/"Fix", PR #216 "Summary", PR #198 "Summary" item 2): each
query row attends to the slots j < L_t of its index list whose index lies in [0, s_kv); L_t is
topk_length[t] clamped to [0, topk] when given, else topk.  O is bf16; lse (natural log, sink
excluded) and max_logits (max of sm_scale * q.k) are fp32; a row without a counted slot gives
O = 0, lse = +inf, max_logits = -inf.

    dq, dkv, dsink = sparse_mla_bwd(q, kv, out, dout, indices, lse, topk_length, attn_sink)

returns the gradients of sum(dout * out) (FlashMLA PR #198, "Summary" item 1) in fp32.
"""
from __future__ import annotations

import math

import torch

from ._native import EXPORTED, SmlaError, load_library, status_string
from .native_build import LIB_PATH, build as build_library

__all__ = ["sparse_mla_fwd", "sparse_mla_fwd_paged", "sparse_mla_fwd_paged_splitkv_static", "sparse_mla_fwd_host",
           "row_shard", "sparse_mla_fwd_sharded", "auto_splits",
           "sparse_mla_bwd", "sparse_mla_device_status",
           "sparse_mla_status_string", "SmlaError", "load_library", "build_library", "LIB_PATH"]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _check(t, name, dtype, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _outputs(q, h_q, d_v, out, lse, max_logits):
    s_q = q.shape[0]
    if out is None:
        out = torch.empty((s_q, h_q, d_v), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    if max_logits is None:
        max_logits = torch.empty((s_q, h_q), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, q.device)
    _check(lse, "lse", torch.float32, q.device)
    _check(max_logits, "max_logits", torch.float32, q.device)
    if tuple(out.shape) != (s_q, h_q, d_v) or tuple(lse.shape) != (s_q, h_q) \
            or tuple(max_logits.shape) != (s_q, h_q):
        raise ValueError("output tensors have the wrong shape")
    return out, lse, max_logits


def _host(t, name, dtype):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} host tensor")


def sparse_mla_fwd_host(q, kv, indices, topk_length=None, attn_sink=None, sm_scale=None, d_v=512,
                        out=None, lse=None, max_logits=None, device=None, dev_buffers=None, n_chunks=8,
                        stream=None, copy_streams=None):
    """The forward for host tensors (pinned for the copies to overlap), end to end: the C entry
    copies each row chunk's inputs to the device, runs the forward on it and copies its outputs
    back, with the copies of one chunk overlapping the compute of another.  Outputs are host
    tensors (pinned, allocated here when not given).  `dev_buffers` (a dict with the keys q, kv,
    indices, topk_length, attn_sink, out, lse, max_logits) and `copy_streams` (two streams: in,
    out) are allocated here when not given.  The call is asynchronous on `stream`: synchronise
    it before reading the outputs."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    _host(q, "q", torch.bfloat16)
    _host(kv, "kv", torch.bfloat16)
    _host(indices, "indices", torch.int32)
    _host(topk_length, "topk_length", torch.int32)
    _host(attn_sink, "attn_sink", torch.float32)
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    topk = indices.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    if out is None:
        out = torch.empty((s_q, h_q, d_v), dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((s_q, h_q), dtype=torch.float32).pin_memory()
    if max_logits is None:
        max_logits = torch.empty((s_q, h_q), dtype=torch.float32).pin_memory()
    _host(out, "out", torch.bfloat16)
    _host(lse, "lse", torch.float32)
    _host(max_logits, "max_logits", torch.float32)
    if dev_buffers is None:
        def like(t, shape=None):
            return None if t is None else torch.empty(t.shape if shape is None else shape, dtype=t.dtype, device=dev)
        dev_buffers = dict(q=like(q), kv=like(kv), indices=like(indices), topk_length=like(topk_length),
                           attn_sink=like(attn_sink), out=like(out), lse=like(lse), max_logits=like(max_logits))
    d = dev_buffers
    for k, dt in (("q", torch.bfloat16), ("kv", torch.bfloat16), ("indices", torch.int32),
                  ("topk_length", torch.int32), ("attn_sink", torch.float32), ("out", torch.bfloat16),
                  ("lse", torch.float32), ("max_logits", torch.float32)):
        _check(d.get(k), "dev_buffers[" + k + "]", dt, dev)
    if copy_streams is None:
        copy_streams = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    with torch.cuda.device(dev):
        rc = lib.sparse_mla_fwd_host(
            _ptr(q), _ptr(kv), _ptr(indices), _ptr(topk_length), _ptr(attn_sink), float(sm_scale), int(d_v),
            _ptr(out), _ptr(lse), _ptr(max_logits), int(s_q), int(s_kv), int(h_q), int(d_qk), int(topk),
            _ptr(d["q"]), _ptr(d["kv"]), _ptr(d["indices"]), _ptr(d.get("topk_length")), _ptr(d.get("attn_sink")),
            _ptr(d["out"]), _ptr(d["lse"]), _ptr(d["max_logits"]), int(n_chunks), _stream_handle(stream, dev),
            copy_streams[0].cuda_stream, copy_streams[1].cuda_stream)
    if rc != 0:
        raise SmlaError(rc, "sparse_mla_fwd_host")
    return out, lse, max_logits


def row_shard(s_q, rank, world):
    """The contiguous query rows [r0, r1) that rank `rank` of `world` owns in a batch of s_q rows.
    Rows are independent, so a batch splits across GPUs with no exchange; the first s_q % world
    ranks take one row more."""
    if world < 1 or not 0 <= rank < world or s_q < 0:
        raise ValueError("need 0 <= rank < world and s_q >= 0")
    base, extra = divmod(int(s_q), int(world))
    r0 = rank * base + min(rank, extra)
    return r0, r0 + base + (1 if rank < extra else 0)


def sparse_mla_fwd_sharded(q, kv, indices, rank, world, topk_length=None, attn_sink=None, sm_scale=None,
                           d_v=512, stream=None, n_split=1):
    """The forward on this rank's rows of the batch (see row_shard): every GPU holds the whole
    shared KV and the batch's tensors, computes its own contiguous rows, and keeps its outputs
    (an all-gather is needed only if a caller wants them replicated).  Returns (r0, r1) and the
    outputs of those rows."""
    r0, r1 = row_shard(q.shape[0], rank, world)
    tl = None if topk_length is None else topk_length[r0:r1]
    out = sparse_mla_fwd(q[r0:r1], kv, indices[r0:r1], tl, attn_sink, sm_scale=sm_scale, d_v=d_v,
                         stream=stream, n_split=n_split)
    return (r0, r1), out


def auto_splits(s_q, h_q, topk, device=None):
    """Split-KV factor for a call: 1 when the (row, 64-head group) items already fill more than
    half the SMs, else as many ranges per row as keep every (item, range) unit in one wave (at
    least one 64-slot block per range, at most 64 ranges)."""
    items = s_q * (h_q // 64)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    if items == 0 or 2 * items > sms:
        return 1
    # one wave of (item, range) units, each range at least one 64-slot block
    return int(max(1, min(64, sms // items, -(-topk // 64))))


def _workspace(lib, s_q, h_q, n_split, device):
    n = int(lib.sparse_mla_splitkv_workspace_size(int(s_q), int(h_q), int(n_split)))
    if n == 0:
        return None, 0
    return torch.empty(n, dtype=torch.uint8, device=device), n


def sparse_mla_fwd(q, kv, indices, topk_length=None, attn_sink=None, sm_scale=None, d_v=512,
                   out=None, lse=None, max_logits=None, stream=None, n_split=1):
    """q [s_q, h_q, d_qk] bf16; kv [s_kv, 1, d_qk] (or [s_kv, d_qk]) bf16; indices [s_q, 1, topk]
    (or [s_q, topk]) int32; topk_length [s_q] int32 or None; attn_sink [h_q] fp32 or None.
    Returns (out [s_q, h_q, d_v] bf16, lse [s_q, h_q] fp32, max_logits [s_q, h_q] fp32).
    n_split > 1 (or "auto": see auto_splits) runs the split-KV variant with a workspace
    allocated here."""
    lib = load_library()
    _check(q, "q", torch.bfloat16)
    dev = q.device
    _check(kv, "kv", torch.bfloat16, dev)
    _check(indices, "indices", torch.int32, dev)
    _check(topk_length, "topk_length", torch.int32, dev)
    _check(attn_sink, "attn_sink", torch.float32, dev)
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    if kv.numel() != s_kv * d_qk:
        raise ValueError("kv must be [s_kv, 1, d_qk] with the d_qk of q")
    topk = indices.shape[-1] if indices.dim() else 0
    if indices.numel() != s_q * topk:
        raise ValueError("indices must be [s_q, 1, topk]")
    if topk_length is not None and topk_length.numel() != s_q:
        raise ValueError("topk_length must have s_q entries")
    if attn_sink is not None and attn_sink.numel() != h_q:
        raise ValueError("attn_sink must have h_q entries")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    out, lse, max_logits = _outputs(q, h_q, d_v, out, lse, max_logits)
    if n_split == "auto":
        n_split = auto_splits(s_q, h_q, topk, dev)
    with torch.cuda.device(dev):
        if n_split == 1:
            rc = lib.sparse_mla_fwd(_ptr(q), _ptr(kv), _ptr(indices), _ptr(topk_length), _ptr(attn_sink),
                                    float(sm_scale), int(d_v), _ptr(out), _ptr(lse), _ptr(max_logits),
                                    int(s_q), int(s_kv), int(h_q), int(d_qk), int(topk),
                                    _stream_handle(stream, dev))
        else:
            ws, nbytes = _workspace(lib, s_q, h_q, n_split, dev)
            rc = lib.sparse_mla_fwd_splitkv(_ptr(q), _ptr(kv), _ptr(indices), _ptr(topk_length),
                                            _ptr(attn_sink), float(sm_scale), int(d_v), _ptr(out), _ptr(lse),
                                            _ptr(max_logits), int(s_q), int(s_kv), int(h_q), int(d_qk),
                                            int(topk), int(n_split), _ptr(ws), int(nbytes),
                                            _stream_handle(stream, dev))
    if rc != 0:
        raise SmlaError(rc, "sparse_mla_fwd")
    return out, lse, max_logits


def sparse_mla_fwd_paged(q, kv_pool, block_table, indices, page_block=64, seqlens_k=None,
                         s_kv_per_req=None, s_q_per_req=1, topk_length=None, attn_sink=None,
                         sm_scale=None, d_v=512, out=None, lse=None, max_logits=None, stream=None,
                         n_split=1):
    """Paged-KV variant: kv_pool [n_pages*page_block, 1, d_qk] bf16, block_table [n_req,
    max_blocks] int32, seqlens_k [n_req] int32 or None (then every request has s_kv_per_req
    tokens); indices hold token positions within the row's request."""
    lib = load_library()
    _check(q, "q", torch.bfloat16)
    dev = q.device
    _check(kv_pool, "kv_pool", torch.bfloat16, dev)
    _check(block_table, "block_table", torch.int32, dev)
    _check(indices, "indices", torch.int32, dev)
    _check(seqlens_k, "seqlens_k", torch.int32, dev)
    _check(topk_length, "topk_length", torch.int32, dev)
    _check(attn_sink, "attn_sink", torch.float32, dev)
    s_q, h_q, d_qk = q.shape
    pool_rows = kv_pool.shape[0]
    if kv_pool.numel() != pool_rows * d_qk:
        raise ValueError("kv_pool must be [rows, 1, d_qk] with the d_qk of q")
    if block_table.dim() != 2:
        raise ValueError("block_table must be [n_req, max_blocks]")
    max_blocks = block_table.shape[1]
    if s_kv_per_req is None:
        s_kv_per_req = max_blocks * page_block
    topk = indices.shape[-1] if indices.dim() else 0
    if indices.numel() != s_q * topk:
        raise ValueError("indices must be [s_q, 1, topk]")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    out, lse, max_logits = _outputs(q, h_q, d_v, out, lse, max_logits)
    if n_split == "auto":
        n_split = auto_splits(s_q, h_q, topk, dev)
    with torch.cuda.device(dev):
        if n_split == 1:
            rc = lib.sparse_mla_fwd_paged(_ptr(q), _ptr(kv_pool), int(pool_rows), _ptr(block_table),
                                          int(max_blocks), int(page_block), _ptr(seqlens_k),
                                          int(s_kv_per_req), int(s_q_per_req), _ptr(indices),
                                          _ptr(topk_length), _ptr(attn_sink), float(sm_scale), int(d_v),
                                          _ptr(out), _ptr(lse), _ptr(max_logits), int(s_q), int(h_q),
                                          int(d_qk), int(topk), _stream_handle(stream, dev))
        else:
            ws, nbytes = _workspace(lib, s_q, h_q, n_split, dev)
            rc = lib.sparse_mla_fwd_paged_splitkv(
                _ptr(q), _ptr(kv_pool), int(pool_rows), _ptr(block_table), int(max_blocks), int(page_block),
                _ptr(seqlens_k), int(s_kv_per_req), int(s_q_per_req), _ptr(indices), _ptr(topk_length),
                _ptr(attn_sink), float(sm_scale), int(d_v), _ptr(out), _ptr(lse), _ptr(max_logits), int(s_q),
                int(h_q), int(d_qk), int(topk), int(n_split), _ptr(ws), int(nbytes), _stream_handle(stream, dev))
    if rc != 0:
        raise SmlaError(rc, "sparse_mla_fwd_paged")
    return out, lse, max_logits


def sparse_mla_fwd_paged_splitkv_static(q, kv_pool, block_table, indices, n_split, page_block=64,
                                        seqlens_k=None, s_kv_per_req=None, s_q_per_req=1, topk_length=None,
                                        attn_sink=None, sm_scale=None, d_v=512, out=None, lse=None,
                                        max_logits=None, stream=None):
    """Split-KV paged forward whose partial results use the library's own 32 MiB scratch array
    (no workspace is allocated anywhere).  Calls on one device must not overlap; see the C
    header."""
    lib = load_library()
    _check(q, "q", torch.bfloat16)
    dev = q.device
    _check(kv_pool, "kv_pool", torch.bfloat16, dev)
    _check(block_table, "block_table", torch.int32, dev)
    _check(indices, "indices", torch.int32, dev)
    _check(seqlens_k, "seqlens_k", torch.int32, dev)
    _check(topk_length, "topk_length", torch.int32, dev)
    _check(attn_sink, "attn_sink", torch.float32, dev)
    s_q, h_q, d_qk = q.shape
    pool_rows = kv_pool.shape[0]
    max_blocks = block_table.shape[1]
    if s_kv_per_req is None:
        s_kv_per_req = max_blocks * page_block
    topk = indices.shape[-1] if indices.dim() else 0
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    out, lse, max_logits = _outputs(q, h_q, d_v, out, lse, max_logits)
    with torch.cuda.device(dev):
        rc = lib.sparse_mla_fwd_paged_splitkv_static(
            _ptr(q), _ptr(kv_pool), int(pool_rows), _ptr(block_table), int(max_blocks), int(page_block),
            _ptr(seqlens_k), int(s_kv_per_req), int(s_q_per_req), _ptr(indices), _ptr(topk_length),
            _ptr(attn_sink), float(sm_scale), int(d_v), _ptr(out), _ptr(lse), _ptr(max_logits), int(s_q),
            int(h_q), int(d_qk), int(topk), int(n_split), _stream_handle(stream, dev))
    if rc != 0:
        raise SmlaError(rc, "sparse_mla_fwd_paged_splitkv_static")
    return out, lse, max_logits


def sparse_mla_bwd(q, kv, out, dout, indices, lse, topk_length=None, attn_sink=None, sm_scale=None,
                   d_v=512, dq=None, dkv=None, dsink=None, stream=None):
    """Gradients of sum(dout * out) through the forward: q, kv, indices, topk_length, attn_sink and
    sm_scale as passed to :func:`sparse_mla_fwd`; out [s_q, h_q, d_v] bf16 and lse [s_q, h_q]
    fp32 as it returned them; dout [s_q, h_q, d_v] bf16.  Returns (dq [s_q, h_q, d_qk] fp32,
    dkv [s_kv, d_qk] fp32, dsink [h_q] fp32 or None)."""
    lib = load_library()
    _check(q, "q", torch.bfloat16)
    dev = q.device
    _check(kv, "kv", torch.bfloat16, dev)
    _check(out, "out", torch.bfloat16, dev)
    _check(dout, "dout", torch.bfloat16, dev)
    _check(indices, "indices", torch.int32, dev)
    _check(lse, "lse", torch.float32, dev)
    _check(topk_length, "topk_length", torch.int32, dev)
    _check(attn_sink, "attn_sink", torch.float32, dev)
    s_q, h_q, d_qk = q.shape
    s_kv = kv.shape[0]
    if kv.numel() != s_kv * d_qk:
        raise ValueError("kv must be [s_kv, 1, d_qk] with the d_qk of q")
    topk = indices.shape[-1] if indices.dim() else 0
    if indices.numel() != s_q * topk:
        raise ValueError("indices must be [s_q, 1, topk]")
    if out.numel() != s_q * h_q * d_v or dout.numel() != s_q * h_q * d_v or lse.numel() != s_q * h_q:
        raise ValueError("out / dout must be [s_q, h_q, d_v] and lse [s_q, h_q]")
    if topk_length is not None and topk_length.numel() != s_q:
        raise ValueError("topk_length must have s_q entries")
    if attn_sink is not None and attn_sink.numel() != h_q:
        raise ValueError("attn_sink must have h_q entries")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d_qk)
    if dq is None:
        dq = torch.empty((s_q, h_q, d_qk), dtype=torch.float32, device=dev)
    if dkv is None:
        dkv = torch.empty((s_kv, d_qk), dtype=torch.float32, device=dev)
    if dsink is None and attn_sink is not None:
        dsink = torch.empty((h_q,), dtype=torch.float32, device=dev)
    _check(dq, "dq", torch.float32, dev)
    _check(dkv, "dkv", torch.float32, dev)
    _check(dsink, "dsink", torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib.sparse_mla_bwd(_ptr(q), _ptr(kv), _ptr(out), _ptr(dout), _ptr(indices), _ptr(topk_length),
                                _ptr(attn_sink), _ptr(lse), float(sm_scale), int(d_v), _ptr(dq), _ptr(dkv),
                                _ptr(dsink), int(s_q), int(s_kv), int(h_q), int(d_qk), int(topk),
                                _stream_handle(stream, dev))
    if rc != 0:
        raise SmlaError(rc, "sparse_mla_bwd")
    return dq, dkv, dsink


def sparse_mla_device_status(reset=False) -> int:
    """Device-side status word (0, or 5 = a bounded wait gave up); synchronises."""
    return int(load_library().sparse_mla_device_status(1 if reset else 0))


def sparse_mla_status_string(code: int) -> str:
    return status_string(code)
