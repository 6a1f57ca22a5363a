"""Pins of the backward oracle (oracle/sparse_mla_bwd_oracle.c) to things other than itself.

The backward is the gradient of L = sum(dO * O) through the sparse MLA forward (FlashMLA PR #198,
"Summary" item 1, for the operation; PR #196 / #216 / #198 item 2 for the forward it
differentiates).  It is pinned by:
  * reverse-mode autograd (a library routine) through a plain PyTorch fp64 forward, which is
    itself checked against the pinned C forward oracle;
  * central finite differences of that forward;
  * closed forms: one counted slot without a sink gives dq = 0, dkv = sum_h dO_h on the value
    columns and 0 on the rest; one slot with a sink gives the sink gradient -p_sink * <dO, O>;
  * invariances the pages fix: permuting a row's slots, inserting invalid entries, and passing
    topk_length instead of a suffix poisoned with INT_MAX leave every gradient unchanged; a row
    with no counted slot contributes nothing.
"""
import numpy as np
import pytest
import torch

import oracle

INT_MAX = 2**31 - 1


def torch_forward(q, kv, indices, topk_length=None, attn_sink=None, sm_scale=None, d_v=None):
    """Plain fp64 sparse MLA forward in PyTorch: a list of valid slots per row, softmax over
    their logits with the sink as an extra value-less term, O = sum p v.  Empty rows give 0."""
    s_q, h_q, d_qk = q.shape
    topk = indices.shape[1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    outs = []
    for t in range(s_q):
        L = topk if topk_length is None else int(min(max(int(topk_length[t]), 0), topk))
        rows = [int(v) for v in indices[t, :L] if 0 <= int(v) < kv.shape[0]]
        if not rows:
            outs.append(torch.zeros(h_q, d_v, dtype=torch.float64) + 0.0 * q[t, :, :1].sum())
            continue
        K = kv[rows, :]                                   # [n, d_qk]
        V = kv[rows, :d_v]                                # [n, d_v]
        logits = sm_scale * (q[t] @ K.T)                  # [h, n]
        if attn_sink is not None:
            logits = torch.cat([logits, attn_sink.reshape(h_q, 1)], dim=1)
        p = torch.softmax(logits, dim=1)
        outs.append(p[:, : len(rows)] @ V)
    return torch.stack(outs)


def autograd_grads(q, kv, dout, indices, topk_length=None, attn_sink=None, sm_scale=None):
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    kvt = torch.tensor(kv, dtype=torch.float64, requires_grad=True)
    st = None if attn_sink is None else torch.tensor(np.asarray(attn_sink, np.float64), requires_grad=True)
    O = torch_forward(qt, kvt, np.asarray(indices), topk_length, st, sm_scale, d_v=dout.shape[2])
    (O * torch.tensor(dout)).sum().backward()
    return qt.grad.numpy(), kvt.grad.numpy(), None if st is None else st.grad.numpy()


def random_case(seed, s_q=5, s_kv=37, h_q=3, d_qk=24, d_v=16, topk=12, sink=False, lengths=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((s_q, h_q, d_qk))
    kv = rng.standard_normal((s_kv, d_qk))
    dout = rng.standard_normal((s_q, h_q, d_v))
    idx = rng.integers(0, s_kv, size=(s_q, topk)).astype(np.int32)   # duplicates allowed
    idx[rng.random((s_q, topk)) < 0.25] = -1
    idx[rng.random((s_q, topk)) < 0.1] = s_kv + 3                  # invalid: beyond s_kv
    idx[1, :] = -1                                                  # one empty row
    tl = rng.integers(0, topk + 3, size=s_q).astype(np.int32) if lengths else None
    sk = rng.standard_normal(h_q).astype(np.float32) if sink else None
    return q, kv, dout, idx, tl, sk


@pytest.mark.parametrize("seed,sink,lengths", [(1, False, False), (2, True, False), (3, True, True), (4, False, True)])
def test_matches_autograd(seed, sink, lengths):
    q, kv, dout, idx, tl, sk = random_case(seed, sink=sink, lengths=lengths)
    dq, dkv, ds = oracle.sparse_mla_bwd_f64(q, kv, dout, idx, tl, sk)
    gq, gkv, gs = autograd_grads(q, kv, dout, idx, tl, sk)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dkv, gkv, rtol=0, atol=1e-12)
    if sink:
        np.testing.assert_allclose(ds, gs, rtol=0, atol=1e-12)
    else:
        assert ds is None


def test_torch_forward_matches_c_forward_oracle():
    rng = np.random.default_rng(7)
    s_q, s_kv, h_q, d_qk, d_v, topk = 4, 29, 2, 32, 16, 10
    q_bits = (rng.standard_normal((s_q, h_q, d_qk)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kv_bits = (rng.standard_normal((s_kv, d_qk)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    idx = rng.integers(-3, s_kv + 3, size=(s_q, topk)).astype(np.int32)
    sink = rng.standard_normal(h_q).astype(np.float32)
    O_c, _, _ = oracle.sparse_mla_fwd(q_bits, kv_bits.reshape(s_kv, 1, d_qk), idx, None, sink, d_v=d_v)
    O_t = torch_forward(torch.tensor(oracle.bf16_bits_to_f64(q_bits)), torch.tensor(oracle.bf16_bits_to_f64(kv_bits)),
                        idx, None, torch.tensor(sink.astype(np.float64)), d_v=d_v)
    np.testing.assert_allclose(O_t.numpy(), O_c, rtol=0, atol=1e-12)


def test_central_finite_differences():
    q, kv, dout, idx, tl, sk = random_case(11, s_q=3, s_kv=13, h_q=2, d_qk=8, d_v=6, topk=6, sink=True)
    dq, dkv, ds = oracle.sparse_mla_bwd_f64(q, kv, dout, idx, tl, sk)

    def loss(qq, kk, ss):
        O = torch_forward(torch.tensor(qq), torch.tensor(kk), idx, tl, torch.tensor(ss), d_v=dout.shape[2])
        return float((O.numpy() * dout).sum())

    eps = 1e-6
    sk64 = sk.astype(np.float64)
    rng = np.random.default_rng(0)
    for _ in range(12):
        t, h, d = rng.integers(3), rng.integers(2), rng.integers(8)
        qp, qm = q.copy(), q.copy()
        qp[t, h, d] += eps
        qm[t, h, d] -= eps
        assert abs((loss(qp, kv, sk64) - loss(qm, kv, sk64)) / (2 * eps) - dq[t, h, d]) < 1e-7
    for r in {int(v) for v in idx.ravel() if 0 <= v < 13} | {0}:
        for d in (0, 5, 7):
            kp, km = kv.copy(), kv.copy()
            kp[r, d] += eps
            km[r, d] -= eps
            assert abs((loss(q, kp, sk64) - loss(q, km, sk64)) / (2 * eps) - dkv[r, d]) < 1e-7
    for h in range(2):
        sp, sm = sk64.copy(), sk64.copy()
        sp[h] += eps
        sm[h] -= eps
        assert abs((loss(q, kv, sp) - loss(q, kv, sm)) / (2 * eps) - ds[h]) < 1e-7


def test_single_slot_closed_form():
    rng = np.random.default_rng(5)
    h_q, d_qk, d_v = 3, 20, 12
    q = rng.standard_normal((1, h_q, d_qk))
    kv = rng.standard_normal((9, d_qk))
    dout = rng.standard_normal((1, h_q, d_v))
    idx = np.array([[-1, 4, 12, -7]], np.int32)                   # only slot 1 counts (row 4)
    dq, dkv, _ = oracle.sparse_mla_bwd_f64(q, kv, dout, idx)
    assert np.all(dq == 0.0)                                        # p = 1: dS = dP - D = 0
    expect = np.zeros_like(kv)
    expect[4, :d_v] = dout[0].sum(axis=0)
    np.testing.assert_allclose(dkv, expect, rtol=0, atol=1e-14)
    # with a sink: d sink_h = -p_sink * <dO_h, O_h>, O_h = p_key v
    sink = np.array([0.4, -1.1, 2.0], np.float32)
    dq, dkv, ds = oracle.sparse_mla_bwd_f64(q, kv, dout, idx, attn_sink=sink)
    sm_scale = float(np.float32(1.0 / np.sqrt(d_qk)))
    for h in range(h_q):
        l = sm_scale * q[0, h] @ kv[4]
        p_key = 1.0 / (1.0 + np.exp(float(sink[h]) - l))
        p_sink = 1.0 - p_key
        D = p_key * (dout[0, h] @ kv[4, :d_v])
        assert abs(ds[h] - (-p_sink * D)) < 1e-12


def test_empty_row_contributes_nothing():
    q, kv, dout, idx, _, sk = random_case(21, sink=True)
    base = oracle.sparse_mla_bwd_f64(q, kv, dout, idx, attn_sink=sk)
    assert np.all(base[0][1] == 0.0)                               # row 1 is all invalid
    idx2 = idx.copy()
    idx2[1, :] = [-1, 2**31 - 1, -5, 37, 40, -1, -1, 99, -2, 38, -1, -1]
    other = oracle.sparse_mla_bwd_f64(q, kv, dout, idx2, attn_sink=sk)
    for a, b in zip(base, other):
        np.testing.assert_array_equal(a, b)


def test_permutation_and_invalid_insertion_invariance():
    q, kv, dout, idx, _, sk = random_case(31, sink=True)
    base = oracle.sparse_mla_bwd_f64(q, kv, dout, idx, attn_sink=sk)
    rng = np.random.default_rng(9)
    perm = np.stack([rng.permutation(row) for row in idx])
    wide = np.full((idx.shape[0], idx.shape[1] * 2), -1, np.int32)
    for t in range(idx.shape[0]):
        pos = np.sort(rng.choice(wide.shape[1], idx.shape[1], replace=False))
        wide[t, pos] = perm[t]
        wide[t, np.setdiff1d(np.arange(wide.shape[1]), pos)[::3]] = INT_MAX
    for variant in (perm, wide):
        got = oracle.sparse_mla_bwd_f64(q, kv, dout, variant, attn_sink=sk)
        for a, b in zip(base, got):
            np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_topk_length_equals_masking_a_poisoned_suffix():
    q, kv, dout, idx, _, sk = random_case(41, sink=True)
    L = np.array([0, 3, 12, 7, 5], np.int32)
    masked = idx.copy()
    poisoned = idx.copy()
    for t in range(idx.shape[0]):
        masked[t, L[t]:] = -1
        poisoned[t, L[t]:] = INT_MAX
    a = oracle.sparse_mla_bwd_f64(q, kv, dout, masked, attn_sink=sk)
    b = oracle.sparse_mla_bwd_f64(q, kv, dout, poisoned, topk_length=L, attn_sink=sk)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_bf16_entry_converts_exactly():
    rng = np.random.default_rng(3)
    bits = lambda shape: (rng.standard_normal(shape).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qb, kb, db = bits((2, 2, 16)), bits((11, 16)), bits((2, 2, 8))
    idx = rng.integers(-2, 13, size=(2, 5)).astype(np.int32)
    a = oracle.sparse_mla_bwd(qb, kb, db, idx)
    b = oracle.sparse_mla_bwd_f64(oracle.bf16_bits_to_f64(qb), oracle.bf16_bits_to_f64(kb),
                                  oracle.bf16_bits_to_f64(db), idx)
    for x, y in zip(a[:2], b[:2]):
        np.testing.assert_array_equal(x, y)
