"""Seeded synthetic inputs for the sparse MLA forward.

This module is shared by the tests, the benchmark and the smoke check.  It draws random
numbers and lays out index lists; it contains none of the attention arithmetic.  Every array
is produced on the host with ``numpy.random.Generator(PCG64(seed))`` and handed bit-for-bit to
both the CUDA path and the CPU oracle.

Workloads follow the five configurations the pages benchmark or the build targets:
  * ``tiny``      -- s_q=128, s_kv=1024, h_q=64, d_qk=576, topk=128 correctness case with
                     empty rows, interior invalid slots, optional sink and topk_length.
  * ``ramp``      -- causal ramp-padded prefill: row i holds min(i+1, 1027) distinct indices
                     from [0, i], front-packed, padded with -1 to 1152 (FlashMLA PR #196,
                     "Numbers").
  * ``full``      -- every slot valid, distinct uniform indices (peak-throughput prefill).
  * ``scattered`` -- each slot invalid with probability 0.3 (-1 or >= s_kv), 1 % empty rows,
                     per-head sink.
  * ``decode``    -- paged decode: 256 requests, 64-token pages, random block table, first
                     1024 positions valid, suffix either INT_MAX (with topk_length) or -1
                     (FlashMLA PR #216, "Dynamic top-k").
bf16 values are drawn as N(0, 1) float32 and rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
INT_MAX = np.iinfo(np.int32).max


def rng_for(config_no: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + config_no + 1000003 * salt))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns.
    Inputs here are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) bf16 bit patterns, generated in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def distinct_rows(rng: np.random.Generator, n_rows: int, k: int, pop: int) -> np.ndarray:
    """[n_rows, k] int32: each row k distinct values drawn uniformly from [0, pop), in random
    order.  Vectorised: oversample with replacement, keep first occurrences."""
    assert k <= pop
    out = np.empty((n_rows, k), np.int32)
    extra = max(64, int(4 * k * k / pop) + 64)
    step = max(1, (1 << 22) // (k + extra))
    r0 = 0
    while r0 < n_rows:
        r1 = min(n_rows, r0 + step)
        m = r1 - r0
        draw = rng.integers(0, pop, size=(m, k + extra), dtype=np.int64)
        order = np.argsort(draw, axis=1, kind="stable")
        srt = np.take_along_axis(draw, order, axis=1)
        first = np.ones_like(srt, dtype=bool)
        first[:, 1:] = srt[:, 1:] != srt[:, :-1]
        keep = np.zeros_like(first)
        np.put_along_axis(keep, order, first, axis=1)
        cnt = keep.sum(axis=1)
        if np.any(cnt < k):  # rare: redo the short rows one by one
            for i in np.nonzero(cnt < k)[0]:
                draw[i, :k] = rng.choice(pop, size=k, replace=False)
                keep[i] = False
                keep[i, :k] = True
        pos = np.cumsum(keep, axis=1) - 1
        sel = keep & (pos < k)
        rr, cc = np.nonzero(sel)
        out[r0 + rr, pos[rr, cc]] = draw[rr, cc]
        r0 = r1
    return out


def _base(config, q, kv, indices, topk_length=None, attn_sink=None, sm_scale=None, d_v=512, **kw):
    d_qk = q.shape[-1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    w = dict(config=config, q=q, kv=kv, indices=indices, topk_length=topk_length,
             attn_sink=attn_sink, sm_scale=float(np.float32(sm_scale)), d_v=d_v, paged=False)
    w.update(kw)
    return w


def tiny(with_len: bool = False, with_sink: bool = False):
    """s_q=128, s_kv=1024, h_q=64, d_qk=576, d_v=512, topk=128.  Row i draws n_i ~ U[0,128]
    distinct indices from [0, i+896], front-packed and padded with -1; 8 rows are empty and 8
    rows carry interior -1 / s_kv+r / INT_MAX entries.  ``with_len`` passes topk_length = one
    past the last valid slot; ``with_sink`` adds a N(0,1) per-head sink."""
    rng = rng_for(1)
    s_q, s_kv, h_q, d_qk, topk = 128, 1024, 64, 576, 128
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = np.full((s_q, topk), -1, np.int32)
    n_valid = rng.integers(0, topk + 1, size=s_q)
    empty_rows = rng.choice(s_q, size=8, replace=False)
    rest = np.setdiff1d(np.arange(s_q), empty_rows)
    scattered_rows = rng.choice(rest, size=8, replace=False)
    n_valid[empty_rows] = 0
    for i in range(s_q):
        n = int(n_valid[i])
        vals = rng.choice(i + 897, size=n, replace=False).astype(np.int32)
        if i in scattered_rows:
            n = max(min(n, topk - 12), 16)
            vals = rng.choice(i + 897, size=n, replace=False).astype(np.int32)
            bad = np.array([-1, s_kv + int(rng.integers(0, 64)), INT_MAX, -1, s_kv, INT_MAX - 1,
                            -2, s_kv + 1000], np.int32)
            row = list(vals)
            for b in bad:
                row.insert(int(rng.integers(1, len(row))), int(b))  # interior positions
            idx[i, :len(row)] = row
        else:
            idx[i, :n] = vals
    tl = None
    if with_len:
        valid = (idx >= 0) & (idx < s_kv)
        tl = np.where(valid.any(1), topk - np.argmax(valid[:, ::-1], axis=1), 0).astype(np.int32)
    sink = rng_for(1, salt=1).standard_normal(h_q, dtype=np.float32) if with_sink else None
    return _base("tiny", q, kv.reshape(s_kv, 1, d_qk), idx.reshape(s_q, 1, topk), tl, sink,
                 float(np.float32(1.0 / np.sqrt(576.0))), s_kv=s_kv)


def ramp(s_q=8192, s_kv=8192, h_q=64, d_qk=512, topk=1152, max_valid=1027, with_len=False,
         config_no=2):
    """Causal ramp-padded prefill (FlashMLA PR #196, "Numbers"): row i holds min(i+1,
    max_valid) distinct indices from [0, i], front-packed, padded with -1 to topk."""
    rng = rng_for(config_no)
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = np.full((s_q, topk), -1, np.int32)
    for i in range(s_q):
        n = min(i + 1, max_valid, topk)
        pop = min(i + 1, s_kv)
        n = min(n, pop)
        idx[i, :n] = rng.choice(pop, size=n, replace=False)
    counts = np.minimum(np.minimum(np.arange(s_q) + 1, max_valid), np.minimum(np.arange(s_q) + 1, s_kv))
    counts = np.minimum(counts, topk).astype(np.int32)
    return _base("ramp", q, kv, idx.reshape(s_q, 1, topk), counts if with_len else None, None,
                 s_kv=s_kv, valid_counts=counts)


def full(s_q=8192, s_kv=65536, h_q=128, d_qk=576, topk=2048, config_no=3):
    """Every slot valid: topk distinct uniform indices in [0, s_kv) per row."""
    rng = rng_for(config_no)
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = distinct_rows(rng, s_q, topk, s_kv)
    return _base("full", q, kv, idx.reshape(s_q, 1, topk), None, None, s_kv=s_kv)


def scattered(s_q=4096, s_kv=32768, h_q=128, d_qk=576, topk=2048, p_invalid=0.3,
              empty_frac=0.01, config_no=4):
    """Each slot independently invalid with probability p_invalid (-1 or a value in
    [s_kv, INT_MAX] with equal odds); empty_frac of the rows fully invalid; per-head sink."""
    rng = rng_for(config_no)
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = distinct_rows(rng, s_q, topk, s_kv)
    bad = rng.random((s_q, topk)) < p_invalid
    neg = rng.random((s_q, topk)) < 0.5
    big = rng.integers(s_kv, INT_MAX, size=(s_q, topk), endpoint=True, dtype=np.int64).astype(np.int32)
    idx = np.where(bad, np.where(neg, np.int32(-1), big), idx).astype(np.int32)
    n_empty = max(1, int(round(empty_frac * s_q)))
    empty_rows = rng.choice(s_q, size=n_empty, replace=False)
    emp_neg = rng.random((n_empty, topk)) < 0.5
    emp_big = rng.integers(s_kv, INT_MAX, size=(n_empty, topk), endpoint=True, dtype=np.int64).astype(np.int32)
    idx[empty_rows] = np.where(emp_neg, np.int32(-1), emp_big)
    sink = rng.standard_normal(h_q, dtype=np.float32)
    return _base("scattered", q, kv, idx.reshape(s_q, 1, topk), None, sink, s_kv=s_kv,
                 empty_rows=np.sort(empty_rows))


def decode(n_req=256, s_kv=4096, h_q=128, d_qk=576, topk=2048, n_valid=1024, page_block=64,
           dynamic=True, config_no=5):
    """Paged decode (FlashMLA PR #216, "Dynamic top-k"): one query per request, each request's
    s_kv tokens live in page_block-token pages of a shared pool addressed by a random block
    table; the first n_valid slots are distinct positions in [0, s_kv); the rest is INT_MAX
    with topk_length = n_valid (dynamic) or -1 without topk_length (fixed)."""
    rng = rng_for(config_no)
    max_blocks = (s_kv + page_block - 1) // page_block
    n_pages = n_req * max_blocks
    q = normal_bf16(rng, (n_req, h_q, d_qk))
    pool = normal_bf16(rng, (n_pages * page_block, 1, d_qk))
    block_table = rng.permutation(n_pages).astype(np.int32).reshape(n_req, max_blocks)
    idx = np.empty((n_req, topk), np.int32)
    idx[:, :n_valid] = distinct_rows(rng, n_req, n_valid, s_kv)
    idx[:, n_valid:] = INT_MAX if dynamic else -1
    tl = np.full(n_req, n_valid, np.int32) if dynamic else None
    w = _base("decode", q, pool, idx.reshape(n_req, 1, topk), tl, None, s_kv=s_kv)
    w.update(paged=True, block_table=block_table, page_block=page_block, s_kv_per_req=s_kv,
             s_q_per_req=1, seqlens_k=None)
    return w


def decode_fixed(n_req=2, s_q_per_req=2, s_kv=32768, h_q=128, d_qk=576, topk=2048, page_block=64,
                 config_no=6):
    """Small-batch paged decode (the FlashMLA PR #216 "Reproduction" fixed-width sweep shape:
    S_q=2 queries per request, H=128, s_kv=32768, 64-token pages, top-k 2048): every slot holds
    a distinct valid position of its request, no topk_length."""
    rng = rng_for(config_no)
    max_blocks = (s_kv + page_block - 1) // page_block
    n_pages = n_req * max_blocks
    s_q = n_req * s_q_per_req
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    pool = normal_bf16(rng, (n_pages * page_block, 1, d_qk))
    block_table = rng.permutation(n_pages).astype(np.int32).reshape(n_req, max_blocks)
    idx = distinct_rows(rng, s_q, topk, s_kv)
    w = _base("decode_fixed", q, pool, idx.reshape(s_q, 1, topk), None, None, s_kv=s_kv)
    w.update(paged=True, block_table=block_table, page_block=page_block, s_kv_per_req=s_kv,
             s_q_per_req=s_q_per_req, seqlens_k=None)
    return w


def random_case(seed, s_q, s_kv, h_q, d_qk, topk, with_len=False, with_sink=False,
                poison_suffix=False, dup=False):
    """Small mixed-pattern case for parity tests: per row one of front-packed / scattered
    invalid / fully valid / empty, optional duplicated indices, optional INT_MAX suffix after
    topk_length."""
    rng = np.random.Generator(np.random.PCG64(SEED_BASE + 7919 * seed))
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = np.full((s_q, topk), -1, np.int32)
    lens = np.zeros(s_q, np.int32)
    for i in range(s_q):
        kind = i % 4
        n = int(rng.integers(0, min(topk, s_kv) + 1))
        if kind == 3 and i % 8 == 3:
            n = 0
        if kind == 2:
            n = min(topk, s_kv)
        vals = rng.choice(s_kv, size=n, replace=False).astype(np.int32)
        if dup and n > 2:
            vals[-1] = vals[0]
        if kind == 1 and n > 0:
            row = list(vals)
            for _ in range(min(6, topk - n)):
                row.insert(int(rng.integers(0, len(row) + 1)),
                           int(rng.choice([-1, s_kv, s_kv + 3, INT_MAX, -7])))
            row = row[:topk]
            idx[i, :len(row)] = row
            lens[i] = len(row)
        else:
            idx[i, :n] = vals
            lens[i] = n
        if with_len and poison_suffix:
            idx[i, lens[i]:] = INT_MAX
    tl = lens.copy() if with_len else None
    sink = rng.standard_normal(h_q, dtype=np.float32) if with_sink else None
    return _base("random", q, kv, idx.reshape(s_q, 1, topk), tl, sink, s_kv=s_kv)


def valid_slot_count(indices, s_kv, topk_length=None):
    """Number of counted (token, slot) pairs: slots below the row length with an index in
    [0, s_kv).  Used for the valid-token FLOP count 2*h_q*valid*(d_qk+d_v)."""
    idx = np.asarray(indices).reshape(np.asarray(indices).shape[0], -1)
    ok = (idx >= 0) & (idx < s_kv)
    if topk_length is not None:
        L = np.clip(np.asarray(topk_length), 0, idx.shape[1])
        ok &= np.arange(idx.shape[1])[None, :] < L[:, None]
    return ok.sum(axis=1)


def dout_for(w, salt: int = 17):
    """Seeded N(0,1) bf16 gradient of the loss w.r.t. O ([s_q, h_q, d_v] bit patterns) for the
    backward: the upstream gradient a training step would feed in."""
    s_q, h_q = w["q"].shape[0], w["q"].shape[1]
    rng = np.random.Generator(np.random.PCG64(SEED_BASE + 104729 * salt + s_q))
    return normal_bf16(rng, (s_q, h_q, w["d_v"]))


def bwd_prefill(s_q=4096, s_kv=32768, h_q=64, d_qk=576, topk=2048, config_no=8):
    """Backward benchmark shape of FlashMLA PR #198 ("Numerics": T = 4096, topk = 2048; "Notes":
    h_q = 64, d_qk = 576): every row holds topk distinct uniform indices in [0, s_kv), no
    invalid entry, no topk_length, no sink."""
    rng = rng_for(config_no)
    q = normal_bf16(rng, (s_q, h_q, d_qk))
    kv = normal_bf16(rng, (s_kv, 1, d_qk))
    idx = distinct_rows(rng, s_q, topk, s_kv)
    return _base("bwd_prefill", q, kv, idx.reshape(s_q, 1, topk), None, None, s_kv=s_kv)
