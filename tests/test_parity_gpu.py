"""GPU parity: the CUDA path (through its C ABI) against the fp64 CPU oracle on the same seeded
inputs, element by element at small sizes that span several 64-key blocks and ragged tails, and
on sampled rows at the full configuration sizes.  Also the bit-level self-consistency the pages
rely on: a run without topk_length equals a run with topk_length set to the derived length
(FlashMLA PR #196, "Numbers": bitwise A/B of out / lse / max_logits)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_parity, dev_tensor, run_gpu, run_oracle, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("with_len", [False, True])
@pytest.mark.parametrize("with_sink", [False, True])
def test_tiny_config_all_rows(with_len, with_sink):
    w = W.tiny(with_len=with_len, with_sink=with_sink)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"tiny len={with_len} sink={with_sink}")


CASES = [
    # seed, s_q, s_kv, h_q, d_qk, topk
    (1, 37, 300, 64, 512, 200),
    (2, 21, 1000, 128, 576, 333),
    (3, 16, 70, 64, 576, 64),
    (4, 9, 5000, 128, 512, 1),
    (5, 13, 129, 64, 512, 130),
]


@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}" for c in CASES])
@pytest.mark.parametrize("mode", ["plain", "len_poison", "sink_dup"])
def test_random_shapes(case, mode):
    seed, s_q, s_kv, h_q, d_qk, topk = case
    w = W.random_case(seed, s_q, s_kv, h_q, d_qk, topk, with_len=(mode == "len_poison"),
                      with_sink=(mode == "sink_dup"), poison_suffix=(mode == "len_poison"),
                      dup=(mode == "sink_dup"))
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"{case} {mode}")


@pytest.mark.parametrize("case", CASES[:3], ids=[f"s{c[0]}" for c in CASES[:3]])
def test_derived_length_is_bit_identical_to_passed_length(case):
    seed, s_q, s_kv, h_q, d_qk, topk = case
    w = W.random_case(seed, s_q, s_kv, h_q, d_qk, topk, with_sink=True)
    L = oracle.last_valid_length(w["indices"], s_kv)
    a = run_gpu(w, topk_length=None)
    b = run_gpu(w, topk_length=L)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))


@pytest.mark.parametrize("tail", [0, 1, 17, 63, 64, 65, 127, 128])
def test_tail_lengths(tail):
    # FlashMLA PR #216, "Correctness": tail lengths 0,1,17,63,64,65,127,128 with the suffix
    # after topk_length poisoned with INT_MAX.
    rng = np.random.default_rng(100 + tail)
    s_q, s_kv, h_q, d_qk, topk = 6, 600, 64, 576, 192
    q = W.normal_bf16(rng, (s_q, h_q, d_qk))
    kv = W.normal_bf16(rng, (s_kv, 1, d_qk))
    idx = np.stack([rng.choice(s_kv, topk, replace=False) for _ in range(s_q)]).astype(np.int32)
    L = np.full(s_q, tail, np.int32)
    L[1] = min(tail + 1, topk)
    idx_p = idx.copy()
    for i in range(s_q):
        idx_p[i, L[i]:] = W.INT_MAX
    w = dict(q=q, kv=kv, indices=idx_p.reshape(s_q, 1, topk), topk_length=L, attn_sink=None,
             sm_scale=float(np.float32(1 / np.sqrt(576))), d_v=512, paged=False)
    gpu = run_gpu(w)
    assert_parity(to_np(gpu), run_oracle(w), f"tail {tail}")
    # same result as the -1 suffix without topk_length (bit-identical: same blocks, same order)
    idx_m = idx.copy()
    for i in range(s_q):
        idx_m[i, L[i]:] = -1
    w2 = dict(w, indices=idx_m.reshape(s_q, 1, topk), topk_length=None)
    gpu2 = run_gpu(w2)
    for i in range(s_q):
        # the derived length equals L[i] only when slot L[i]-1 is valid (always, here)
        assert torch.equal(gpu[0][i].view(torch.int16), gpu2[0][i].view(torch.int16))
        assert torch.equal(gpu[1][i], gpu2[1][i]) and torch.equal(gpu[2][i], gpu2[2][i])


def test_zero_rows_is_a_noop():
    import sparse_mla_attention_fwd_gb300 as smla
    q = torch.empty((0, 64, 512), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((10, 1, 512), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((0, 1, 8), dtype=torch.int32, device="cuda")
    out, lse, mx = smla.sparse_mla_fwd(q, kv, idx)
    assert out.shape == (0, 64, 512) and lse.shape == (0, 64)


def test_empty_kv_gives_empty_rows():
    w = W.random_case(9, 5, 40, 64, 512, 16)
    w = dict(w, kv=w["kv"][:0], indices=w["indices"])
    gpu = to_np(run_gpu(w))
    assert np.all(gpu[0] == 0) and np.all(gpu[1] == np.inf) and np.all(gpu[2] == -np.inf)


def test_single_valid_slot_is_bit_exact():
    # one valid slot and no sink: O must be exactly that row's first d_v values
    rng = np.random.default_rng(3)
    s_q, s_kv = 8, 100
    w = W.random_case(11, s_q, s_kv, 64, 576, 70)
    idx = np.full((s_q, 1, 70), -1, np.int32)
    pick = rng.integers(0, s_kv, size=s_q)
    for i in range(s_q):
        idx[i, 0, (7 * i) % 70] = pick[i]
    w = dict(w, indices=idx, attn_sink=None, topk_length=None)
    out = run_gpu(w)[0].view(torch.int16).cpu().numpy().view(np.uint16)
    for i in range(s_q):
        expect = w["kv"][pick[i], 0, :512]
        assert np.array_equal(out[i], np.broadcast_to(expect, (64, 512)))


# ---------------------------------------------------------------- full-size configurations
# At the benchmark sizes every row is compared with the oracle (C3: 1024 rows plus fixed ones),
# in chunks of rows so that the fp64 reference stays small; each chunk must meet the bar.
CHUNK = 1024
_ORACLE_CACHE = {}


def _oracle_rows(w, key, rows):
    """Oracle outputs for `rows` of workload `key`, cached across tests that share the inputs
    (the ramp runs with and without topk_length have the same expected output)."""
    ck = (key, rows.tobytes())
    if ck not in _ORACLE_CACHE:
        _ORACLE_CACHE[ck] = run_oracle(w, rows=rows)
    return _ORACLE_CACHE[ck]


def _check_full(w, what, key, rows=None):
    s_q = w["q"].shape[0]
    gpu = run_gpu(w)
    rows = np.arange(s_q, dtype=np.int64) if rows is None else rows
    for c0 in range(0, len(rows), CHUNK):
        r = rows[c0:c0 + CHUNK]
        assert_parity(to_np(gpu, r), _oracle_rows(w, key, r), f"{what} rows {r[0]}..{r[-1]}")
    # properties at every row: finite where the row has a counted slot, exact empties elsewhere
    counts = W.valid_slot_count(w["indices"], w["s_kv"], w["topk_length"])
    lse = gpu[1].cpu().numpy()
    mx = gpu[2].cpu().numpy()
    has = counts > 0
    assert np.all(np.isfinite(lse[has])) and np.all(lse[~has] == np.inf)
    assert np.all(mx[~has] == -np.inf)
    assert bool(torch.isfinite(gpu[0].float()).all())
    return gpu


@pytest.mark.parametrize("with_len", [False, True])
def test_ramp_config_all_rows(with_len):
    w = W.ramp(with_len=with_len)
    _check_full(w, f"ramp len={with_len}", "ramp")


def test_ramp_len_vs_no_len_bit_identical():
    w = W.ramp()
    a = run_gpu(w, topk_length=None)
    b = run_gpu(w, topk_length=w["valid_counts"])
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_full_config_sampled_rows():
    w = W.full()
    rng = np.random.default_rng(1234)
    rows = set(rng.choice(w["q"].shape[0], size=1024, replace=False).tolist()) | {0, 1, w["q"].shape[0] - 1}
    _check_full(w, "full", "full", rows=np.array(sorted(rows), np.int64))


def test_scattered_config_all_rows():
    w = W.scattered()
    _check_full(w, "scattered", "scattered")


@pytest.mark.parametrize("dynamic", [True, False])
def test_decode_config(dynamic):
    w = W.decode(dynamic=dynamic)
    gpu = run_gpu(w)
    assert_parity(to_np(gpu), run_oracle(w), f"decode dynamic={dynamic}")


def test_decode_fixed_equals_dynamic():
    # FlashMLA PR #216 harness: fixed (-1 suffix, no topk_length) and dynamic (INT_MAX suffix,
    # topk_length=1024) produce the same output
    a = run_gpu(W.decode(dynamic=True))
    b = run_gpu(W.decode(dynamic=False))
    torch.testing.assert_close(a[0], b[0], atol=1e-3, rtol=2.01 / 128)
    torch.testing.assert_close(a[1], b[1], atol=1e-6, rtol=8.01 / 65536)


def test_bounded_wait_times_out_and_reports_it():
    # failure detection without a fault: a wait on a barrier nothing completes gives up after
    # 20 ms, the status word says so, and the context still runs the forward correctly
    import sparse_mla_attention_fwd_gb300 as smla
    from sparse_mla_attention_fwd_gb300 import _native
    lib = _native.load_library()
    assert smla.sparse_mla_device_status(reset=True) == 0
    assert lib.sparse_mla_selftest_wait_timeout(20_000_000, None) == 0
    torch.cuda.synchronize()
    assert smla.sparse_mla_device_status(reset=True) == 5      # SMLA_ERR_DEVICE_TIMEOUT
    assert smla.sparse_mla_device_status() == 0
    w = W.tiny(with_len=True, with_sink=True)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), "tiny after a timeout")
    assert lib.sparse_mla_selftest_wait_timeout(0, None) == 2


def test_no_device_timeouts_recorded():
    import sparse_mla_attention_fwd_gb300 as smla
    assert smla.sparse_mla_device_status() == 0


# ---------------------------------------------------------------- block packing
def _scattered_row_case(seed, s_q=12, s_kv=900, h_q=64, d_qk=576, topk=640):
    """Rows whose counted slots are spread among invalid entries (-1, >= s_kv, INT_MAX, other
    negatives), with counts on and around block boundaries, and the same rows front-packed."""
    rng = np.random.default_rng(seed)
    q = W.normal_bf16(rng, (s_q, h_q, d_qk))
    kv = W.normal_bf16(rng, (s_kv, 1, d_qk))
    counts = [0, 1, 63, 64, 65, 127, 128, 129, 200, 333, 511, 640][:s_q]
    spread = np.full((s_q, topk), -1, np.int32)
    packed = np.full((s_q, topk), -1, np.int32)
    bad = np.array([-1, s_kv, s_kv + 7, W.INT_MAX, -9], np.int32)
    for i, n in enumerate(counts):
        vals = rng.choice(s_kv, size=n, replace=False).astype(np.int32)
        pos = np.sort(rng.choice(topk, size=n, replace=False))
        if i == 4:
            pos = np.arange(topk - n, topk)          # counted slots only at the far end
        row = rng.choice(bad, size=topk)
        row[pos] = vals
        spread[i] = row
        packed[i, :n] = vals
    base = dict(q=q, kv=kv, topk_length=None, attn_sink=rng.standard_normal(h_q).astype(np.float32),
                sm_scale=float(np.float32(1 / np.sqrt(d_qk))), d_v=512, paged=False)
    return (dict(base, indices=spread.reshape(s_q, 1, topk)), dict(base, indices=packed.reshape(s_q, 1, topk)))


@pytest.mark.parametrize("seed", [1, 2])
def test_packed_blocks_match_oracle(seed):
    spread, _ = _scattered_row_case(seed)
    assert_parity(to_np(run_gpu(spread)), run_oracle(spread), f"scattered rows seed {seed}")


@pytest.mark.parametrize("seed", [1, 2])
def test_invalid_entries_do_not_change_a_bit(seed):
    # Counted slots are packed in slot order into dense blocks, so a row with invalid entries
    # anywhere computes exactly the same blocks, in the same order, as the row with them
    # removed: outputs must agree bit for bit (FlashMLA PR #196, "Correctness notes": invalid
    # entries are masked wherever they sit).
    spread, packed = _scattered_row_case(seed)
    a, b = run_gpu(spread), run_gpu(packed)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


# ---------------------------------------------------------------- wider shapes and paged variants
@pytest.mark.parametrize("h_q,d_qk,topk", [(256, 512, 3000), (192, 576, 700), (1024, 512, 96)])
def test_many_head_groups_and_long_lists(h_q, d_qk, topk):
    # several 64-head groups per token (items of one token on different CTAs), lists far
    # longer than one block, and the largest supported head count
    w = W.random_case(21 + h_q, 5, 4096, h_q, d_qk, topk, with_sink=True, dup=True)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"h_q={h_q} d_qk={d_qk} topk={topk}")


def _paged_case(seed, n_req=6, s_q_per_req=3, page=32, max_blocks=12, h_q=128, d_qk=576, topk=300,
                with_len=True):
    rng = np.random.default_rng(seed)
    n_pages = n_req * max_blocks + 5
    pool = W.normal_bf16(rng, (n_pages * page, 1, d_qk))
    q = W.normal_bf16(rng, (n_req * s_q_per_req, h_q, d_qk))
    bt = rng.permutation(n_pages)[: n_req * max_blocks].astype(np.int32).reshape(n_req, max_blocks)
    seqlens = rng.integers(0, max_blocks * page + 1, size=n_req).astype(np.int32)
    seqlens[0] = 0                                   # a request with an empty cache
    s_q = n_req * s_q_per_req
    idx = rng.integers(-3, max_blocks * page + 40, size=(s_q, 1, topk)).astype(np.int32)
    tl = rng.integers(0, topk + 1, size=s_q).astype(np.int32) if with_len else None
    return dict(q=q, kv=pool, indices=idx, topk_length=tl, attn_sink=rng.standard_normal(h_q).astype(np.float32),
                sm_scale=float(np.float32(1 / np.sqrt(d_qk))), d_v=512, paged=True, block_table=bt,
                page_block=page, s_kv_per_req=max_blocks * page, s_q_per_req=s_q_per_req, seqlens_k=seqlens)


@pytest.mark.parametrize("with_len", [True, False])
def test_paged_per_request_lengths(with_len):
    # per-request cache lengths (seqlens_k), several queries per request, positions beyond a
    # request's length or its block table, and a request with an empty cache
    w = _paged_case(31, with_len=with_len)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"paged seqlens len={with_len}")


@pytest.mark.parametrize("with_len", [False, True])
def test_very_long_lists(with_len):
    # 40000-slot lists (up to 625 blocks in one row, slot numbers past 2^15), mixed row kinds
    w = W.random_case(91, 4, 70000, 64, 512, 40000, with_len=with_len, poison_suffix=with_len)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"very long lists len={with_len}")


def test_kv_rows_past_2_gib():
    # a 2.5 M-row KV (2.9 GB): half of every row's slots point past byte offset 2^31 of the KV,
    # one of them at its very last row; only the referenced rows carry data
    rng = np.random.default_rng(77)
    s_kv, s_q, h_q, d_qk, topk = 2_500_000, 6, 64, 576, 256
    high = np.arange(s_kv - 2000, s_kv)
    assert int(high[0]) * d_qk * 2 > 2 ** 31
    idx = np.empty((s_q, 1, topk), np.int32)
    for i in range(s_q):
        row = np.concatenate([rng.choice(high, size=topk // 2, replace=False),
                              rng.choice(s_kv - 2000, size=topk // 2, replace=False)])
        idx[i, 0] = rng.permutation(row)
    idx[0, 0, 0] = s_kv - 1
    kv = np.zeros((s_kv, 1, d_qk), np.uint16)
    used = np.unique(idx)
    kv[used] = W.normal_bf16(rng, (len(used), 1, d_qk))
    w = W._base("kv_past_2gib", W.normal_bf16(rng, (s_q, h_q, d_qk)), kv, idx, s_kv=s_kv)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), "kv rows past 2 GiB")


@pytest.mark.parametrize("page, max_blocks, h_q, d_qk", [(1, 400, 64, 512), (48, 9, 128, 576), (100, 5, 192, 512)])
def test_paged_page_sizes(page, max_blocks, h_q, d_qk):
    # one-token pages, and page sizes that are not powers of two: the position -> (page, row)
    # split is plain integer division on both sides
    w = _paged_case(50 + page, page=page, max_blocks=max_blocks, h_q=h_q, d_qk=d_qk)
    assert_parity(to_np(run_gpu(w)), run_oracle(w), f"paged page={page} h_q={h_q} d_qk={d_qk}")


def _paged_edge_case(seed, n_req=5, s_q_per_req=2, page=64, max_blocks=6, h_q=64, d_qk=576, topk=520):
    """Paged cache whose requests are longer than their block-table rows (positions past the
    table), with unmapped (negative) table entries and pages that run off the end of the pool."""
    rng = np.random.default_rng(seed)
    n_pages = n_req * max_blocks + 4
    pool_rows = n_pages * page - 21              # the last page is partly off the pool
    pool = W.normal_bf16(rng, (pool_rows, 1, d_qk))
    bt = rng.permutation(n_pages - 1)[: n_req * max_blocks].astype(np.int32).reshape(n_req, max_blocks)
    bt[0, 1] = -1
    bt[1, 3] = n_pages - 1                       # partly past the pool
    bt[2, 0] = n_pages + 5                       # wholly past the pool
    bt[3, 5] = -100
    s_kv_per_req = max_blocks * page + 150       # positions up to 150 past each table row
    s_q = n_req * s_q_per_req
    q = W.normal_bf16(rng, (s_q, h_q, d_qk))
    idx = rng.integers(-2, s_kv_per_req + 8, size=(s_q, 1, topk)).astype(np.int32)
    idx[2, 0, :64] = 3 * page + np.arange(64)    # request 1, the partly-off page
    idx[0, 0, :] = page + rng.integers(0, page, size=topk)   # request 0, unmapped page only
    return dict(q=q, kv=pool, indices=idx, topk_length=None,
                attn_sink=rng.standard_normal(h_q).astype(np.float32),
                sm_scale=float(np.float32(1 / np.sqrt(d_qk))), d_v=512, paged=True, block_table=bt,
                page_block=page, s_kv_per_req=s_kv_per_req, s_q_per_req=s_q_per_req, seqlens_k=None)


@pytest.mark.parametrize("n_split", [1, 3])
def test_paged_positions_off_the_table_or_pool(n_split):
    # positions whose page lies past the request's table row, negative table entries and rows
    # past the pool are invalid slots on both sides; row 0 has only such slots and is empty
    w = _paged_edge_case(41)
    gpu = to_np(run_gpu(w, n_split=n_split))
    ref = run_oracle(w)
    assert np.all(ref[1][0] == np.inf)
    assert_parity(gpu, ref, f"paged edge positions n_split={n_split}")


# ---------------------------------------------------------------- split-KV
@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}" for c in CASES])
@pytest.mark.parametrize("n_split", [2, 5, 64])
def test_splitkv_matches_oracle(case, n_split):
    # rows cut into n_split ranges (many of them empty when n_split * 64 > L_t), merged with
    # log-sum-exp weights; empty rows, sinks, duplicates and poisoned suffixes as in the base case
    seed, s_q, s_kv, h_q, d_qk, topk = case
    w = W.random_case(seed, s_q, s_kv, h_q, d_qk, topk, with_len=(n_split != 5), with_sink=True,
                      poison_suffix=(n_split != 5), dup=(n_split == 5))
    assert_parity(to_np(run_gpu(w, n_split=n_split)), run_oracle(w), f"{case} n_split={n_split}")


@pytest.mark.parametrize("with_len", [True, False])
def test_splitkv_paged(with_len):
    w = _paged_case(32, with_len=with_len)
    assert_parity(to_np(run_gpu(w, n_split=3)), run_oracle(w), f"paged split len={with_len}")


def test_splitkv_small_batch_decode_shape():
    # two requests of two queries each over 2048-slot lists: 8 (row, head group) items, cut
    # into enough ranges to cover the SMs
    import sparse_mla_attention_fwd_gb300 as smla
    w = _paged_case(33, n_req=2, s_q_per_req=2, page=64, max_blocks=64, h_q=128, d_qk=576, topk=2048,
                    with_len=False)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(64 * 64, size=2048, replace=False) for _ in range(4)]).astype(np.int32)
    w = dict(w, indices=idx.reshape(4, 1, 2048), seqlens_k=None)
    n = smla.auto_splits(4, 128, 2048)
    assert n > 1
    assert_parity(to_np(run_gpu(w, n_split=n)), run_oracle(w), f"small-batch decode n_split={n}")


# ---------------------------------------------------------------- randomized sweep
def _sweep_case(k):
    rng = np.random.default_rng(9000 + k)
    h_q = int(rng.choice([64, 128, 192, 256]))
    d_qk = int(rng.choice([512, 576]))
    s_q = int(rng.integers(1, 12))
    topk = int(rng.integers(1, 1400))
    s_kv = int(rng.integers(1, 3000))
    w = W.random_case(9100 + k, s_q, s_kv, h_q, d_qk, topk, with_len=bool(k % 2), with_sink=bool(k % 3 == 0),
                      poison_suffix=bool(k % 2), dup=bool(k % 5 == 0))
    n_split = int(rng.choice([1, 1, 2, 3, 7]))
    return w, n_split


@pytest.mark.parametrize("k", range(24))
def test_randomized_sweep(k):
    w, n_split = _sweep_case(k)
    assert_parity(to_np(run_gpu(w, n_split=n_split)), run_oracle(w), f"sweep {k} n_split={n_split}")
