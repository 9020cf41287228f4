"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Each test checks the oracle against something it does not contain: library
conversions, hand-worked fixtures under tests/golden/, closed forms, brute
force on tiny inputs, a library attention routine, or invariances that a
dropped term, wrong index or transposed operand would break.
"""
import dataclasses
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_decode_paged_gb300 import workloads as W


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _bf16_bits(x):
    """float -> bf16 bits via torch (exact for the values used here)."""
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _tiny_wl(**kw):
    base = W.workload(0)
    return dataclasses.replace(base, **kw)


# ----------------------------------------------------------------------------
# decoders: all codes against torch's own conversions
# ----------------------------------------------------------------------------
def test_bf16_decoder_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = O.bf16_bits_to_f64(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(ref[~both_nan], got[~both_nan])
    assert np.array_equal(np.isnan(ref), np.isnan(got))


def test_e4m3_decoder_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = O.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9  # smallest subnormal


# ----------------------------------------------------------------------------
# row builder
# ----------------------------------------------------------------------------
def test_build_rows_worked_example(golden_dir):
    g = _golden(golden_dir, "build_rows_worked_example.json")
    rows = O.build_rows(g["cache_len"], g["new_tokens"], g["max_rows"], g["block_rows"])
    for key in ("row_req", "row_len", "row_pos", "block_first", "block_nrows"):
        assert rows[key].tolist() == g[key], key
    assert rows["num_rows"] == g["num_rows"]
    assert rows["num_blocks"] == g["num_blocks"]


@pytest.mark.parametrize("i", range(5))
def test_build_rows_invariants(i):
    wl = W.workload(i)
    cache_len, new = W.request_mix(wl)
    rows = O.build_rows(cache_len, new, wl.max_rows, wl.block_rows)
    n = rows["num_rows"]
    assert n == int(new.sum())
    assert np.array_equal(rows["row_len"][:n], rows["row_pos"][:n] + 1)
    assert (rows["row_len"][n:] == 0).all() and (rows["row_req"][n:] == 0).all()
    # every row's length is at most its request's cache length, and the last
    # row of each request sees the whole cache
    for b in range(len(cache_len)):
        rr = np.nonzero((rows["row_req"][:n] == b))[0]
        assert rr.size == new[b]
        if rr.size:
            assert np.all(np.diff(rr) == 1)
            assert rows["row_len"][rr[-1]] == cache_len[b]
    # blocks tile the rows exactly once, each inside one request
    covered = np.zeros(n, int)
    for k in range(rows["num_blocks"]):
        f, c = rows["block_first"][k], rows["block_nrows"][k]
        assert 1 <= c <= wl.block_rows
        assert len(set(rows["row_req"][f:f + c])) == 1
        covered[f:f + c] += 1
    assert (covered == 1).all()
    assert (rows["block_nrows"][rows["num_blocks"]:] == 0).all()


def test_build_rows_rejects_overflow():
    with pytest.raises(ValueError):
        O.build_rows([4, 4], [3, 3], 5, 1)
    with pytest.raises(ValueError):
        O.build_rows([2], [3], 8, 1)


# ----------------------------------------------------------------------------
# indexer
# ----------------------------------------------------------------------------
def _fixture_inputs(g, fp8: bool):
    wl = _tiny_wl(idx_heads=2, idx_dim=2, page_size=g["page_size"], max_rows=1,
                  max_reqs=1, max_pages_per_req=2, score_width=4,
                  idx_key_dtype=W.KEY_FP8_E4M3 if fp8 else W.KEY_BF16)
    inp = dict(workload=wl, page_table=np.array(g["page_table"], np.int32),
               q_idx=_bf16_bits(g["q_idx"])[None], w=np.array([g["w"]], np.float32))
    if fp8:
        inp["idx_cache"] = np.array(g["physical_keys_e4m3"], np.uint8)
        inp["idx_scale"] = np.array(g["physical_scales"], np.float32)
    else:
        inp["idx_cache"] = _bf16_bits(g["physical_keys"])
        inp["idx_scale"] = None
    rows = dict(num_rows=1, row_req=np.array([0]), row_len=np.array([g["length"]]))
    return inp, rows


@pytest.mark.parametrize("fp8", [False, True])
def test_indexer_worked_example(golden_dir, fp8):
    g = _golden(golden_dir, "indexer_worked_example.json")
    inp, rows = _fixture_inputs(g, fp8)
    s = O.indexer_scores(inp, rows)
    want = g["scores_fp8"] if fp8 else g["scores_bf16"]
    assert s[0, :3].tolist() == want
    assert np.isnan(s[0, 3])  # past the length: never written
    for k, idx in g["topk_fp8" if fp8 else "topk_bf16"].items():
        assert O.topk_row(s[0], 3, int(k)).tolist() == idx


def test_indexer_closed_form_nonnegative():
    # with q, k >= 0 every ReLU is the identity and the score collapses to
    # (sum_h w_h q_h) . k_t * s_t, a single matrix-vector product
    rng = np.random.default_rng(7)
    q = rng.random((8, 16))
    k = rng.random((40, 16))
    w = rng.standard_normal(8)
    s = rng.random(40) + 0.5
    got = O.indexer_scores_row(q, w, k, s)
    want = (k @ (w @ q)) * s
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_indexer_all_negative_dots_give_zero():
    rng = np.random.default_rng(8)
    q = rng.random((4, 8)) + 0.1
    k = -(rng.random((10, 8)) + 0.1)
    w = rng.standard_normal(4)
    assert np.array_equal(O.indexer_scores_row(q, w, k, np.ones(10)), np.zeros(10))


def test_indexer_single_head_is_relu_dot():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 8))
    k = rng.standard_normal((30, 8))
    got = O.indexer_scores_row(q, np.array([3.0]), k, np.ones(30))
    want = 3.0 * np.maximum(k @ q[0], 0.0)
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)


def _relabel_pages(inp, perm):
    """Move physical page p to perm[p] and rewrite the page table to match."""
    out = dict(inp)
    inv_target = np.empty_like(perm)
    inv_target[perm] = np.arange(perm.size)
    for key in ("idx_cache", "idx_scale", "k_cache", "v_cache"):
        if out.get(key) is not None:
            out[key] = inp[key][inv_target]
    pt = inp["page_table"].copy()
    m = pt >= 0
    pt[m] = perm[pt[m]]
    out["page_table"] = pt
    return out


@pytest.mark.parametrize("i", [0, 1])
def test_page_permutation_invariance(i):
    inp = W.generate(i)
    ref = O.step(inp)
    rng = np.random.default_rng(100 + i)
    perm = rng.permutation(inp["num_pages"]).astype(np.int32)
    got = O.step(_relabel_pages(inp, perm))
    assert np.array_equal(np.nan_to_num(ref["scores"], nan=-7.0), np.nan_to_num(got["scores"], nan=-7.0))
    assert np.array_equal(ref["topk_idx"], got["topk_idx"])
    assert np.array_equal(ref["out"], got["out"])


def test_poison_past_length_changes_nothing():
    inp = W.generate(0)
    ref = O.step(inp)
    wl = inp["workload"]
    bad = dict(inp)
    for key in ("idx_cache", "k_cache", "v_cache"):
        bad[key] = inp[key].copy()
    for b, L in enumerate(inp["cache_len"]):
        last_page = inp["page_table"][b, (L - 1) // wl.page_size]
        slot0 = L % wl.page_size
        if slot0:
            bad["idx_cache"][last_page, slot0:] = 0x7FC0  # bf16 NaN
            bad["k_cache"][last_page, slot0:] = 0x7F80    # +inf
            bad["v_cache"][last_page, slot0:] = 0x7FC0
    got = O.step(bad)
    assert np.array_equal(ref["topk_idx"], got["topk_idx"])
    assert np.array_equal(ref["out"], got["out"])


# ----------------------------------------------------------------------------
# top-k
# ----------------------------------------------------------------------------
def _beats(s, i, j):
    """Ranking of the selection: numbers beat NaN, higher beats lower, ties to lower index."""
    ni, nj = math.isnan(s[i]), math.isnan(s[j])
    if ni != nj:
        return nj
    if not ni and s[i] != s[j]:
        return s[i] > s[j]
    return i < j


def test_topk_bruteforce_subsets():
    rng = np.random.default_rng(11)
    values = np.array([-np.inf, -1.0, 0.0, 0.5, 2.0, np.inf, np.nan])
    for trial in range(300):
        L = int(rng.integers(1, 9))
        k = int(rng.integers(1, 11))
        s = values[rng.integers(0, values.size, L)]
        n = min(k, L)
        # brute force: the unique subset every member of which beats every non-member
        winners = [c for c in itertools.combinations(range(L), n)
                   if all(_beats(s, i, j) for i in c for j in range(L) if j not in c)]
        assert len(winners) == 1
        want = list(winners[0]) + [-1] * (k - n)
        assert O.topk_row(s, L, k).tolist() == want, (s, k)


def test_topk_matches_torch_on_distinct_values():
    rng = np.random.default_rng(12)
    for _ in range(20):
        L = int(rng.integers(50, 3000))
        k = int(rng.integers(1, 600))
        s = rng.permutation(L * 3)[:L].astype(np.float64) / 7.0  # distinct
        got = O.topk_row(s, L, k)
        ref = torch.topk(torch.from_numpy(s), min(k, L)).indices.sort().values.numpy()
        assert np.array_equal(got[:min(k, L)], ref)
        assert (got[min(k, L):] == -1).all()


def test_topk_reads_only_up_to_length():
    s = np.array([1.0, 5.0, 2.0, 9.0, 100.0, 200.0])
    assert O.topk_row(s, 4, 2).tolist() == [1, 3]
    assert O.topk_row(s, 4, 6).tolist() == [0, 1, 2, 3, -1, -1]


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------
def test_attention_worked_example(golden_dir):
    g = _golden(golden_dir, "attention_worked_example.json")
    k = np.array(g["k"])[:, None, :]
    v = np.array(g["v"])[:, None, :]
    out, lse = O.attention_row(np.array(g["q"]), k, v, g["sm_scale"], 1)
    np.testing.assert_allclose(out, g["out"], rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(lse, g["lse"], rtol=1e-15, atol=1e-15)


def _paged_golden_input(g):
    wl = _tiny_wl(page_size=g["page_size"], num_q_heads=g["num_q_heads"], num_kv_heads=g["num_kv_heads"],
                  head_dim=g["head_dim"], max_rows=len(g["cache_len"]), max_reqs=len(g["cache_len"]),
                  max_pages_per_req=len(g["page_table"][0]), topk=len(g["topk_idx"][0]), block_rows=1)
    assert wl.sm_scale == 0.5  # the fixture's scale, 1/sqrt(4)
    inp = dict(workload=wl, cache_len=np.array(g["cache_len"]), new_tokens=np.array(g["new_tokens"]),
               page_table=np.array(g["page_table"], np.int32), q=_bf16_bits(g["q"]),
               k_cache=_bf16_bits(g["k_cache"]), v_cache=_bf16_bits(g["v_cache"]))
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    return inp, rows


def test_paged_kv_rows_worked_example(golden_dir):
    # the paged fetch alone: K and V of the selected logical positions, through
    # the page table, each from its own cache
    g = _golden(golden_dir, "paged_attention_worked_example.json")
    inp, rows = _paged_golden_input(g)
    for r in range(2):
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), g["topk_idx"][r])
        assert np.array_equal(k, np.array(g["selected_k"][r], np.float64)), r
        assert np.array_equal(v, np.array(g["selected_v"][r], np.float64)), r


def test_paged_attention_worked_example(golden_dir):
    # the whole paged driver (rows -> request -> page table -> K, V ->
    # softmax) against the hand-worked closed form: a K/V swap, a page/slot
    # mix-up or a wrong request's table changes every output
    g = _golden(golden_dir, "paged_attention_worked_example.json")
    inp, rows = _paged_golden_input(g)
    assert rows["row_len"].tolist() == [4, 2]
    out, lse = O.attention(inp, rows, np.array(g["topk_idx"], np.int32))
    np.testing.assert_allclose(out, g["out"], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse, g["lse"], rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 2), (8, 4)])
def test_attention_full_prefix_matches_sdpa(hq, hkv):
    # with top-k >= length the selection is the whole causal prefix and the
    # method reduces to dense softmax attention: compare with torch's SDPA
    rng = np.random.default_rng(13 + hq + hkv)
    D, L = 16, 23
    q = rng.standard_normal((hq, D))
    k = rng.standard_normal((L, hkv, D))
    v = rng.standard_normal((L, hkv, D))
    scale = 1.0 / math.sqrt(D)
    out, lse = O.attention_row(q, k, v, scale, hkv)
    tq = torch.from_numpy(q)[None, :, None, :]            # [1, Hq, 1, D]
    tk = torch.from_numpy(k).permute(1, 0, 2)[None]       # [1, Hkv, L, D]
    tv = torch.from_numpy(v).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale, enable_gqa=True)
    np.testing.assert_allclose(out, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-12)
    # lse against the library log-sum-exp
    import scipy.special
    for h in range(hq):
        x = scale * (k[:, h // (hq // hkv)] @ q[h])
        assert abs(lse[h] - scipy.special.logsumexp(x)) < 1e-12


def test_attention_single_key_reproduces_v():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((8, 32))
    k = rng.standard_normal((1, 2, 32))
    v = rng.standard_normal((1, 2, 32))
    out, lse = O.attention_row(q, k, v, 0.3, 2)
    for h in range(8):
        assert np.array_equal(out[h], v[0, h // 4])
        assert lse[h] == 0.3 * (k[0, h // 4] @ q[h])


def test_attention_empty_selection():
    out, lse = O.attention_row(np.ones((4, 8)), np.zeros((0, 1, 8)), np.zeros((0, 1, 8)), 1.0, 1)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_row_and_request_order_invariance():
    inp = W.generate(1)
    wl = inp["workload"]
    ref = O.step(inp)
    perm = np.random.default_rng(15).permutation(len(inp["cache_len"]))
    swapped = dict(inp)
    swapped["cache_len"] = inp["cache_len"][perm]
    swapped["new_tokens"] = inp["new_tokens"][perm]
    swapped["page_table"] = inp["page_table"][perm]
    # decode: request b has exactly row b, so rows move with the requests
    for key in ("q_idx", "w", "q"):
        swapped[key] = inp[key][perm]
    got = O.step(swapped)
    assert np.array_equal(got["topk_idx"], ref["topk_idx"][perm])
    assert np.array_equal(got["out"], ref["out"][perm])
    assert wl.block_rows == 1


# ----------------------------------------------------------------------------
# split partials + merge
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("S", [1, 2, 3, 8, 40])
def test_merge_of_splits_equals_unsplit(S):
    rng = np.random.default_rng(16 + S)
    q = rng.standard_normal((8, 32))
    n = 29
    k = rng.standard_normal((n, 2, 32)) * 2.0
    v = rng.standard_normal((n, 2, 32))
    m, l, acc = O.split_partials_row(q, k, v, 0.4, 2, S)
    out, lse = O.merge(m, l, acc)
    ref_out, ref_lse = O.attention_row(q, k, v, 0.4, 2)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    if S > n:
        # S - n splits are empty: (m=-inf, l=0, acc=0), and the merge above
        # already showed that they are neutral
        empty = (l == 0)
        assert (empty.sum(axis=1) == S - n).all()
        assert np.isneginf(m[empty]).all() and (acc[empty] == 0).all()


def test_merge_all_empty():
    out, lse = O.merge(np.full((3, 4), -np.inf), np.zeros((3, 4)), np.zeros((3, 4, 5)))
    assert (out == 0).all() and np.isneginf(lse).all()


def test_split_bounds_cover_once():
    for n in range(0, 50):
        for S in (1, 2, 3, 7, 8):
            b = O.split_bounds(n, S)
            assert b[0][0] == 0 and b[-1][1] == n
            assert all(b[i][1] == b[i + 1][0] for i in range(S - 1))


def test_step_tiny_end_to_end():
    inp = W.generate(0)
    res = O.step(inp)
    wl = inp["workload"]
    rows = res["rows"]
    assert rows["num_rows"] == 2
    for r in range(2):
        L = rows["row_len"][r]
        idx = res["topk_idx"][r]
        n = min(wl.topk, L)
        assert (idx[:n] >= 0).all() and (idx[:n] < L).all() and (idx[n:] == -1).all()
        assert np.all(np.diff(idx[:n]) > 0)
        assert np.isfinite(res["out"][r]).all()
