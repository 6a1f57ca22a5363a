"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test below checks the oracle against something the pages or plain mathematics fix:
  * a textbook special case (dense causal softmax attention in matrix form, with the
    library log-sum-exp) that the sparse definition must reduce to;
  * invariances the pages state (slot permutation, invalid entries anywhere in the row,
    topk_length versus masking a suffix poisoned with INT_MAX: FlashMLA PR #196 "Correctness
    notes", FlashMLA PR #216 "Correctness");
  * exact special values (empty rows: FlashMLA PR #196 "Correctness notes");
  * closed forms (uniform logits, one slot, two slots, duplicated slot, value-less sink key:
    FlashMLA PR #198 "Summary" item 2) including the hand-derived fixtures in
    tests/golden/closed_forms.json;
  * the paged address translation against an explicit per-request gather, and the paged
    validity rule (positions past the table row, unmapped pages, rows past the pool) against
    an independent numpy resolution into flat pool rows.
A plausible mistake in the oracle (dropped scale, wrong index, transposed operand, wrong V
columns, lse in the wrong base or including the sink, wrong validity bound, wrong clamp)
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
import workloads as W

INT_MAX = np.iinfo(np.int32).max
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


@pytest.fixture
def orc():
    """The oracle under test (a planted-mistake build is passed instead by the mutation
    tests)."""
    return oracle


def bits(x):
    return W.f32_to_bf16_bits(np.asarray(x, np.float32))


def vals(b):
    return W.bf16_bits_to_f32(b).astype(np.float64)


def small_inputs(rng, s_q, s_kv, h_q, d_qk, scale=1.0):
    q = bits(rng.standard_normal((s_q, h_q, d_qk)) * scale)
    kv = bits(rng.standard_normal((s_kv, 1, d_qk)))
    return q, kv


def dense_causal(q_bits, kv_bits, sm_scale, d_v, sink=None):
    """Matrix-form softmax(scale * Q K^T + causal mask) V with scipy's logsumexp, fp64."""
    Q = vals(q_bits)            # [s, h, d]
    K = vals(kv_bits)[:, 0, :]  # [s, d]
    V = K[:, :d_v]
    s = Q.shape[0]
    scores = sm_scale * np.einsum("shd,kd->shk", Q, K)
    mask = np.tril(np.ones((s, s), bool))[:, None, :]
    scores = np.where(mask, scores, -np.inf)
    lse = logsumexp(scores, axis=-1)
    mx = scores.max(axis=-1)
    if sink is None:
        P = np.exp(scores - lse[..., None])
        return P @ V, lse, mx
    # value-less virtual key with logit sink[h]: extra column with a zero value row
    sk = np.broadcast_to(np.asarray(sink, np.float64)[None, :, None], (s, Q.shape[1], 1))
    ext = np.concatenate([scores, sk], axis=-1)
    P = np.exp(ext - logsumexp(ext, axis=-1)[..., None])
    Vext = np.concatenate([V, np.zeros((1, d_v))], axis=0)
    return P @ Vext, lse, mx


def causal_indices(rng, s, topk, permute=True):
    idx = np.full((s, 1, topk), -1, np.int32)
    for i in range(s):
        row = rng.permutation(i + 1) if permute else np.arange(i + 1)
        idx[i, 0, : i + 1] = row
    return idx


@pytest.mark.parametrize("d_qk,d_v,h_q", [(8, 6, 2), (16, 16, 3), (12, 5, 1)])
def test_reduces_to_dense_causal_attention(orc, d_qk, d_v, h_q):
    rng = np.random.default_rng(11 + d_qk)
    s = 24
    q, kv = small_inputs(rng, s, s, h_q, d_qk)
    idx = causal_indices(rng, s, topk=s + 5)
    scale = float(np.float32(0.37))
    O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, sm_scale=scale, d_v=d_v)
    Od, lsed, mxd = dense_causal(q, kv, scale, d_v)
    np.testing.assert_allclose(O, Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lsed, rtol=0, atol=1e-12)
    np.testing.assert_allclose(mx, mxd, rtol=0, atol=1e-12)


def test_sink_is_a_valueless_extra_key(orc):
    rng = np.random.default_rng(5)
    s, h, d, dv = 20, 3, 8, 7
    q, kv = small_inputs(rng, s, s, h, d)
    idx = causal_indices(rng, s, topk=s)
    sink = rng.standard_normal(h).astype(np.float32)
    scale = float(np.float32(0.5))
    O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, attn_sink=sink, sm_scale=scale, d_v=dv)
    Od, lsed, mxd = dense_causal(q, kv, scale, dv, sink=sink)
    np.testing.assert_allclose(O, Od, rtol=0, atol=1e-12)
    # reading: lse and max_logits exclude the sink
    np.testing.assert_allclose(lse, lsed, rtol=0, atol=1e-12)
    np.testing.assert_allclose(mx, mxd, rtol=0, atol=1e-12)
    O0, lse0, mx0 = orc.sparse_mla_fwd(q, kv, idx, sm_scale=scale, d_v=dv)
    np.testing.assert_array_equal(lse, lse0)
    np.testing.assert_array_equal(mx, mx0)
    assert np.abs(O - O0).max() > 1e-3  # the sink does change O


def _random_rows(rng, s_q, s_kv, topk, fill=0.7):
    idx = np.full((s_q, 1, topk), -1, np.int32)
    for i in range(s_q):
        n = int(rng.integers(1, int(topk * fill) + 1))
        idx[i, 0, :n] = rng.choice(s_kv, size=n, replace=False)
    return idx


def test_permutation_invariance(orc):
    rng = np.random.default_rng(7)
    s_q, s_kv, h, d = 16, 50, 2, 16
    q, kv = small_inputs(rng, s_q, s_kv, h, d)
    idx = _random_rows(rng, s_q, s_kv, 40, fill=1.0)
    perm = np.stack([rng.permutation(40) for _ in range(s_q)])[:, None, :]
    idx_p = np.take_along_axis(idx, perm, axis=2)
    a = orc.sparse_mla_fwd(q, kv, idx, d_v=12)
    b = orc.sparse_mla_fwd(q, kv, idx_p, d_v=12)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_inserting_invalid_entries_anywhere(orc):
    rng = np.random.default_rng(8)
    s_q, s_kv, h, d = 12, 40, 2, 8
    q, kv = small_inputs(rng, s_q, s_kv, h, d)
    idx = _random_rows(rng, s_q, s_kv, 24, fill=0.8)
    bad = [-1, s_kv, s_kv + 1, INT_MAX, -5, np.iinfo(np.int32).min]
    ext = np.full((s_q, 1, 40), -1, np.int32)
    for i in range(s_q):
        row = list(idx[i, 0])
        for _ in range(16):
            row.insert(int(rng.integers(0, len(row) + 1)), int(rng.choice(bad)))
        ext[i, 0] = row[:40]
    a = orc.sparse_mla_fwd(q, kv, idx, d_v=8)
    b = orc.sparse_mla_fwd(q, kv, ext, d_v=8)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_index_equal_to_s_kv_is_invalid(orc):
    rng = np.random.default_rng(9)
    q, kv = small_inputs(rng, 1, 6, 1, 4)
    a = orc.sparse_mla_fwd(q, kv, np.array([[[2, 5]]], np.int32), d_v=4)
    b = orc.sparse_mla_fwd(q, kv[:5], np.array([[[2, 5]]], np.int32), d_v=4)  # 5 == s_kv now
    c = orc.sparse_mla_fwd(q, kv[:5], np.array([[[2, -1]]], np.int32), d_v=4)
    for x, y in zip(b, c):
        np.testing.assert_array_equal(x, y)
    assert not np.allclose(a[0], b[0])


def test_topk_length_equals_masking_a_poisoned_suffix(orc):
    rng = np.random.default_rng(10)
    s_q, s_kv, h, d, topk = 14, 64, 2, 8, 32
    q, kv = small_inputs(rng, s_q, s_kv, h, d)
    idx = np.empty((s_q, 1, topk), np.int32)
    for i in range(s_q):
        idx[i, 0] = rng.choice(s_kv, size=topk, replace=False)
    L = rng.integers(0, topk + 1, size=s_q).astype(np.int32)
    L[0], L[1] = 0, topk
    poisoned = idx.copy()
    masked = idx.copy()
    for i in range(s_q):
        poisoned[i, 0, L[i]:] = INT_MAX
        masked[i, 0, L[i]:] = -1
    a = orc.sparse_mla_fwd(q, kv, poisoned, topk_length=L, d_v=8)
    b = orc.sparse_mla_fwd(q, kv, masked, d_v=8)
    # valid indices beyond topk_length are ignored too
    c = orc.sparse_mla_fwd(q, kv, idx, topk_length=L, d_v=8)
    for x, y, z in zip(a, b, c):
        np.testing.assert_array_equal(x, y)
        np.testing.assert_array_equal(x, z)


def test_topk_length_is_clamped(orc):
    rng = np.random.default_rng(12)
    q, kv = small_inputs(rng, 3, 20, 1, 8)
    idx = np.stack([rng.choice(20, size=10, replace=False) for _ in range(3)])[:, None, :].astype(np.int32)
    full = orc.sparse_mla_fwd(q, kv, idx, d_v=8)
    big = orc.sparse_mla_fwd(q, kv, idx, topk_length=np.array([11, 10**6, INT_MAX], np.int32), d_v=8)
    for x, y in zip(full, big):
        np.testing.assert_array_equal(x, y)
    neg = orc.sparse_mla_fwd(q, kv, idx, topk_length=np.array([-1, -100, 0], np.int32), d_v=8)
    assert np.all(neg[0] == 0) and np.all(neg[1] == np.inf) and np.all(neg[2] == -np.inf)


@pytest.mark.parametrize("with_sink", [False, True])
def test_empty_rows_exact(orc, with_sink):
    rng = np.random.default_rng(13)
    q, kv = small_inputs(rng, 4, 10, 3, 8)
    idx = np.array([[[-1, -1, -1]], [[10, INT_MAX, -3]], [[1, 2, 3]], [[-1, 10, 11]]], np.int32)
    sink = rng.standard_normal(3).astype(np.float32) if with_sink else None
    O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, attn_sink=sink, d_v=8)
    for r in (0, 1, 3):
        assert np.all(O[r] == 0.0) and not np.any(np.signbit(O[r]))
        assert np.all(lse[r] == np.inf)
        assert np.all(mx[r] == -np.inf)
    assert np.all(np.isfinite(O[2])) and np.all(np.isfinite(lse[2]))


def test_zero_query_gives_mean_and_log_n(orc):
    rng = np.random.default_rng(14)
    s_kv, d, dv = 30, 8, 6
    q = np.zeros((1, 2, d), np.uint16)
    kv = bits(rng.standard_normal((s_kv, 1, d)))
    sel = rng.choice(s_kv, size=9, replace=False).astype(np.int32)
    idx = np.concatenate([sel, [-1, 40]]).astype(np.int32)[None, None, :]
    O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, d_v=dv)
    V = vals(kv)[sel, 0, :dv]
    np.testing.assert_allclose(O[0, 0], V.mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(9), rtol=0, atol=1e-14)
    assert np.all(mx == 0.0)
    s = np.float32(0.75)
    O2, lse2, _ = orc.sparse_mla_fwd(q, kv, idx, attn_sink=np.array([s, s], np.float32), d_v=dv)
    np.testing.assert_allclose(O2[0, 1], V.sum(axis=0) / (9 + math.exp(float(s))), rtol=0, atol=1e-14)
    np.testing.assert_array_equal(lse2, lse)


def test_single_slot_returns_its_value_row(orc):
    rng = np.random.default_rng(15)
    q, kv = small_inputs(rng, 1, 12, 2, 8)
    idx = np.array([[[-1, 7, 12, -1]]], np.int32)
    O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, d_v=5)
    np.testing.assert_array_equal(O[0, 0], vals(kv)[7, 0, :5])
    np.testing.assert_array_equal(O[0, 1], vals(kv)[7, 0, :5])
    np.testing.assert_array_equal(lse, mx)


def test_duplicated_slot_counts_twice(orc):
    rng = np.random.default_rng(16)
    q, kv = small_inputs(rng, 1, 12, 2, 8)
    one = orc.sparse_mla_fwd(q, kv, np.array([[[4, -1]]], np.int32), d_v=8)
    two = orc.sparse_mla_fwd(q, kv, np.array([[[4, 4]]], np.int32), d_v=8)
    np.testing.assert_allclose(two[0], one[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(two[1], one[1] + math.log(2), rtol=0, atol=1e-14)
    np.testing.assert_array_equal(two[2], one[2])


def _golden_case(name, base):
    case = dict(base)
    case.update({k: v for k, v in name.items()})
    return case


def test_hand_derived_golden_fixtures(orc):
    with open(GOLDEN) as f:
        g = json.load(f)
    base = g["two_slot"]
    for key in ("two_slot", "two_slot_sink", "length_bound", "empty_with_sink"):
        c = dict(base)
        c.update(g[key])
        q = bits(c["q"])
        kv = bits(c["kv"])
        idx = np.array(c["indices"], np.int32)
        tl = np.array(c["topk_length"], np.int32) if "topk_length" in c else None
        sink = np.array(c["attn_sink"], np.float32) if "attn_sink" in c else None
        O, lse, mx = orc.sparse_mla_fwd(q, kv, idx, topk_length=tl, attn_sink=sink,
                                           sm_scale=c["sm_scale"], d_v=c["d_v"])
        exp_lse = np.array([[float(v) for v in r] for r in c["lse"]])
        exp_mx = np.array([[float(v) for v in r] for r in c["max_logits"]])
        np.testing.assert_allclose(O, np.array(c["out"]), rtol=0, atol=1e-14, err_msg=key)
        np.testing.assert_allclose(lse, exp_lse, rtol=0, atol=1e-14, err_msg=key)
        np.testing.assert_allclose(mx, exp_mx, rtol=0, atol=1e-14, err_msg=key)


def test_paged_equals_explicit_per_request_gather(orc):
    rng = np.random.default_rng(17)
    n_req, s_kv, page, h, d, topk = 5, 40, 8, 2, 16, 24
    max_blocks = s_kv // page
    n_pages = n_req * max_blocks + 3
    pool = bits(rng.standard_normal((n_pages * page, 1, d)))
    q = bits(rng.standard_normal((n_req, h, d)))
    bt = rng.permutation(n_pages)[: n_req * max_blocks].astype(np.int32).reshape(n_req, max_blocks)
    seqlens = rng.integers(1, s_kv + 1, size=n_req).astype(np.int32)
    idx = np.empty((n_req, 1, topk), np.int32)
    for b in range(n_req):
        idx[b, 0] = rng.integers(-3, s_kv + 3, size=topk)
    O, lse, mx = orc.sparse_mla_fwd_paged(q, pool, bt, idx, page_block=page, seqlens_k=seqlens,
                                             s_q_per_req=1, d_v=12)
    for b in range(n_req):
        # explicit gather of request b's first seqlens[b] tokens into a flat kv
        pos = np.arange(seqlens[b])
        rows = bt[b, pos // page] * page + pos % page
        flat = pool[rows]
        Ob, lseb, mxb = orc.sparse_mla_fwd(q[b:b + 1], flat, idx[b:b + 1], d_v=12)
        np.testing.assert_array_equal(O[b], Ob[0])
        np.testing.assert_array_equal(lse[b], lseb[0])
        np.testing.assert_array_equal(mx[b], mxb[0])


def _paged_to_flat_rows(bt, idx, page, lengths, pool_rows, s_q_per_req=1):
    """Paged reading restated in numpy: each slot's token position becomes its pool row, or -1
    when the position is outside the request, past the request's block-table row, on a
    negative (unmapped) table entry, or on a row past the end of the pool."""
    s_q, topk = idx.shape[0], idx.shape[-1]
    max_blocks = bt.shape[1]
    flat = np.full((s_q, 1, topk), -1, np.int32)
    for t in range(s_q):
        b = t // s_q_per_req
        for j in range(topk):
            p = int(idx[t, 0, j])
            if p < 0 or p >= lengths[b] or p // page >= max_blocks:
                continue
            pg = int(bt[b, p // page])
            row = pg * page + p % page
            if pg < 0 or row >= pool_rows:
                continue
            flat[t, 0, j] = row
    return flat


def test_paged_positions_off_the_table_or_pool_are_invalid(orc):
    # Positions whose page lies past the request's block-table row, table entries that are
    # negative, and pages that run off the end of the pool are invalid slots (FlashMLA PR #216,
    # "Summary": a position that is not valid is never used as an address).  The paged oracle
    # must equal the flat oracle over the whole pool, with each slot resolved independently.
    rng = np.random.default_rng(23)
    n_req, s_q_per_req, page, max_blocks, h, d, topk = 4, 2, 8, 3, 2, 16, 30
    s_kv_per_req = 40                       # longer than the 24 positions the table covers
    n_pages = 16
    pool_rows = n_pages * page - 5          # the last page is partly off the pool
    pool = bits(rng.standard_normal((pool_rows, 1, d)))
    bt = rng.choice(n_pages - 1, size=(n_req, max_blocks), replace=False).astype(np.int32)
    bt[0, 1] = -1                           # unmapped page
    bt[1, 2] = n_pages - 1                  # page partly past the pool
    bt[2, 0] = n_pages + 3                  # page wholly past the pool
    bt[3, 2] = -7
    s_q = n_req * s_q_per_req
    q = bits(rng.standard_normal((s_q, h, d)))
    idx = rng.integers(-2, s_kv_per_req + 4, size=(s_q, 1, topk)).astype(np.int32)
    idx[0, 0, :4] = [8, 9, 15, 30]          # on the unmapped page, and past the table
    idx[2, 0, :3] = [16 + 2, 16 + 7, 21]    # on the partly-off page: row 122 valid, 127 and 125 not
    idx[4, 0, :3] = [0, 5, 7]               # on the page wholly past the pool
    sink = rng.standard_normal(h).astype(np.float32)
    lengths = np.full(n_req, s_kv_per_req)
    flat_idx = _paged_to_flat_rows(bt, idx, page, lengths, pool_rows, s_q_per_req)
    assert (flat_idx >= 0).sum() > 20 and (flat_idx < 0).sum() > 20
    got = orc.sparse_mla_fwd_paged(q, pool, bt, idx, page_block=page, s_kv_per_req=s_kv_per_req,
                                   s_q_per_req=s_q_per_req, attn_sink=sink, d_v=12)
    ref = orc.sparse_mla_fwd(q, pool, flat_idx, attn_sink=sink, d_v=12)
    for x, y in zip(got, ref):
        np.testing.assert_array_equal(x, y)
    # a row whose every position is invalid in these ways is an exactly empty row
    idx2 = idx.copy()
    idx2[1, 0, :] = 8                       # request 0, unmapped page only
    got2 = orc.sparse_mla_fwd_paged(q, pool, bt, idx2, page_block=page, s_kv_per_req=s_kv_per_req,
                                    s_q_per_req=s_q_per_req, attn_sink=sink, d_v=12)
    assert np.all(got2[0][1] == 0) and np.all(got2[1][1] == np.inf) and np.all(got2[2][1] == -np.inf)


def test_last_valid_length_matches_definition_and_is_neutral(orc):
    rng = np.random.default_rng(18)
    s_q, s_kv, topk = 30, 50, 20
    idx = rng.integers(-2, s_kv + 3, size=(s_q, 1, topk)).astype(np.int32)
    idx[0] = -1
    idx[1, 0, -1] = 3
    L = orc.last_valid_length(idx, s_kv)
    for i in range(s_q):
        ok = [j for j in range(topk) if 0 <= idx[i, 0, j] < s_kv]
        assert L[i] == (ok[-1] + 1 if ok else 0)
    q, kv = small_inputs(rng, s_q, s_kv, 2, 8)
    a = orc.sparse_mla_fwd(q, kv, idx, d_v=8)
    b = orc.sparse_mla_fwd(q, kv, idx, topk_length=L, d_v=8)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_row_subset_matches_full_run(orc):
    w = W.random_case(3, s_q=9, s_kv=70, h_q=64, d_qk=512, topk=40, with_sink=True)
    full = orc.sparse_mla_fwd(w["q"], w["kv"], w["indices"], attn_sink=w["attn_sink"])
    rows = np.array([8, 0, 5], np.int64)
    sub = orc.sparse_mla_fwd(w["q"], w["kv"], w["indices"], attn_sink=w["attn_sink"], rows=rows)
    for x, y in zip(full, sub):
        np.testing.assert_array_equal(x[rows], y)


def brute_force(q_bits, kv_bits, idx, topk_length, sink, sm_scale, d_v):
    """Pure-Python loops over tiny shapes: the definition evaluated slot by slot with math.exp,
    sharing nothing with the C oracle."""
    qv, kvv = vals(q_bits), vals(kv_bits)[:, 0, :]
    s_q, h_q, d_qk = qv.shape
    s_kv, topk = kvv.shape[0], idx.shape[-1]
    O = [[[0.0] * d_v for _ in range(h_q)] for _ in range(s_q)]
    lse = [[math.inf] * h_q for _ in range(s_q)]
    mx = [[-math.inf] * h_q for _ in range(s_q)]
    for t in range(s_q):
        L = topk if topk_length is None else min(max(int(topk_length[t]), 0), topk)
        slots = [int(idx[t, 0, j]) for j in range(L) if 0 <= int(idx[t, 0, j]) < s_kv]
        if not slots:
            continue
        for h in range(h_q):
            logits = []
            for r in slots:
                acc = 0.0
                for d in range(d_qk):
                    acc += float(qv[t, h, d]) * float(kvv[r, d])
                logits.append(sm_scale * acc)
            m = max(logits)
            ws = [math.exp(x - m) for x in logits]
            se = sum(ws)
            den = se + (math.exp(float(sink[h]) - m) if sink is not None else 0.0)
            for d in range(d_v):
                O[t][h][d] = sum(wj * float(kvv[r, d]) for wj, r in zip(ws, slots)) / den
            lse[t][h] = m + math.log(se)
            mx[t][h] = m
    return np.array(O), np.array(lse), np.array(mx)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_on_tiny_shapes(orc, seed):
    rng = np.random.default_rng(100 + seed)
    s_q, s_kv = 5, int(rng.integers(1, 9))
    h_q, d_qk = int(rng.integers(1, 3)), int(rng.integers(4, 9))
    d_v = int(rng.integers(1, d_qk + 1))
    topk = int(rng.integers(1, 5))
    q, kv = small_inputs(rng, s_q, s_kv, h_q, d_qk)
    idx = rng.integers(-2, s_kv + 2, size=(s_q, 1, topk)).astype(np.int32)
    idx[0, 0, 0] = INT_MAX
    tl = rng.integers(-1, topk + 2, size=s_q).astype(np.int32) if seed % 2 else None
    sink = rng.standard_normal(h_q).astype(np.float32) if seed % 3 == 0 else None
    scale = float(np.float32(rng.uniform(0.2, 1.5)))
    got = orc.sparse_mla_fwd(q, kv, idx, topk_length=tl, attn_sink=sink, sm_scale=scale, d_v=d_v)
    ref = brute_force(q, kv, idx, tl, sink, scale, d_v)
    for x, y in zip(got, ref):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)
