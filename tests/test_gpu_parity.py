"""CUDA path (through the C-ABI) against the fp64 CPU oracle.

Every workload runs in both K/V cache layouts: the separate K and V caches
and the interleaved one (a token's K row then its V row in one cache) that
the benchmark times.

Tolerances (written here, applied element by element):
  indexer scores : |g - o| <= rtol*|o| + rtol*rms(o over the row),
                   rtol 2e-2 for bf16 keys, 6e-2 for fp8 keys;
  top-k indices  : bit-exact, given the GPU's own scores as input to both;
  attention      : |g - o| <= 1e-2 + 2e-2*|o| on the GPU's selected set
                   (output and lse);
  split partials : m within the attention bound; l relative 2e-2 (l >= 1
                   for a non-empty split, it is a sum whose largest term is
                   1); acc / l — the split's own normalised attention output —
                   within the attention bound (acc itself scales with l).
"""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_decode_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu

RTOL_SCORE = {W.KEY_BF16: 2e-2, W.KEY_FP8_E4M3: 6e-2}
ATOL_OUT, RTOL_OUT = 1e-2, 2e-2
RTOL_L = 2e-2

# rows the oracle recomputes one by one for the attention checks (None: all
# rows).  Mixed workload: its 48 decode rows, 128 of its 512 prefill rows
# (every fourth, stepping through the four rows of a score block, and both
# ends of the prefill request) and pad rows.
_MIXED = sorted(set(range(48)) | {48 + 4 * k + (k % 4) for k in range(128)} | {49, 50, 51, 558, 559}
                | {560, 561, 1023})
SAMPLE_ROWS = {0: None, 1: None, 2: None, 3: _MIXED, 4: None}

# (workload, K/V layout); a workload's two layouts are adjacent so its
# generated inputs are drawn once
CASES = [(i, lay) for i in range(5) for lay in ("separate", "interleaved")]
_inputs = {}


def _generated(i):
    if i not in _inputs:
        _inputs.clear()
        _inputs[i] = W.generate(i)
    return _inputs[i]


@pytest.fixture(scope="module", params=CASES, ids=lambda c: f"workload{c[0]}-{c[1]}")
def problem(request, dsa_lib, cuda_ok):
    """Generated inputs + device buffers of one workload in one K/V layout,
    after one step.

    Module-scoped and parametrized, so pytest runs every test of a case
    before building the next one."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    i, layout = request.param
    inp = _generated(i)
    flags = dsa_lib.DSA_FLAG_KV_INTERLEAVED if layout == "interleaved" else 0
    dev = DeviceStep(inp, flags=flags)
    assert (dev.cfg.flags & dsa_lib.DSA_FLAG_KV_INTERLEAVED) == flags
    dev.step()
    torch.cuda.synchronize()
    yield i, inp, dev
    del dev
    torch.cuda.empty_cache()


def _rows(inp):
    wl = inp["workload"]
    return O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)


def _sample(i, rows):
    s = SAMPLE_ROWS[i]
    if s is None:
        return list(range(rows["num_rows"]))
    return [r for r in s if r < len(rows["row_len"])]


def _score_ok(g, o, rtol):
    o = np.asarray(o, np.float64)
    rms = np.sqrt(np.mean(o * o)) if o.size else 0.0
    err = np.abs(np.asarray(g, np.float64) - o)
    bound = rtol * np.abs(o) + rtol * rms
    return bool(np.all(err <= bound)), float(np.max(err / np.maximum(bound, 1e-30))) if o.size else 0.0


def _bf16_to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


# ----------------------------------------------------------------------------
def test_step_status_clean(problem):
    i, inp, dev = problem
    assert dev.status() == 0
    assert dev.rows["num_rows"] == _rows(inp)["num_rows"]


def test_indexer_scores_vs_oracle(problem):
    i, inp, dev = problem
    wl = inp["workload"]
    rows = _rows(inp)
    scores = dev.views["scores"].cpu().numpy()
    qi = O.bf16_bits_to_f64(inp["q_idx"])
    worst = 0.0
    for r in range(rows["num_rows"]):
        L = int(rows["row_len"][r])
        if L == 0:
            continue
        keys, sc = O.index_keys(inp, int(rows["row_req"][r]), L)
        want = O.indexer_scores_row(qi[r], inp["w"][r], keys, sc)
        ok, ratio = _score_ok(scores[r, :L], want, RTOL_SCORE[wl.idx_key_dtype])
        worst = max(worst, ratio)
        assert ok, (r, ratio)
    print(f"workload {i}: worst score error / tolerance = {worst:.3e}")


def test_indexer_writes_nothing_past_length(problem, dsa_lib):
    i, inp, dev = problem
    cfg = dev.cfg
    sentinel = torch.full((cfg.max_rows, cfg.score_width), 12345.0, device="cuda")
    t = dev.t
    dsa_lib.dsa_indexer_scores(cfg, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"],
                               t["row_req"], t["row_len"], t["block_first"], t["block_nrows"],
                               sentinel, dev.workspace)
    s = sentinel.cpu().numpy()
    L = dev.rows["row_len"]
    for r in range(cfg.max_rows):
        assert (s[r, L[r]:] == 12345.0).all(), r
        if L[r]:
            assert np.array_equal(s[r, :L[r]], dev.views["scores"][r, :L[r]].cpu().numpy())
    assert dev.status() == 0


def test_topk_bit_exact_on_gpu_scores(problem):
    i, inp, dev = problem
    wl = inp["workload"]
    rows = _rows(inp)
    scores = dev.views["scores"].cpu().numpy()
    got = dev.views["topk_idx"].cpu().numpy()
    for r in range(wl.max_rows):
        L = int(rows["row_len"][r])
        want = O.topk_row(scores[r], L, wl.topk) if L else np.full(wl.topk, -1, np.int32)
        assert np.array_equal(got[r], want), r


def test_attention_vs_oracle_on_gpu_selection(problem):
    i, inp, dev = problem
    wl = inp["workload"]
    rows = _rows(inp)
    idx = dev.views["topk_idx"].cpu().numpy()
    out = _bf16_to_f64(dev.t["out"])
    lse = dev.t["lse"].cpu().numpy().astype(np.float64)
    q = O.bf16_bits_to_f64(inp["q"])
    for r in _sample(i, rows):
        L = int(rows["row_len"][r])
        if L == 0:
            continue
        sel = idx[r][idx[r] >= 0]
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel)
        o, ls = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[r], o, atol=ATOL_OUT, rtol=RTOL_OUT, err_msg=f"row {r}")
        np.testing.assert_allclose(lse[r], ls, atol=ATOL_OUT, rtol=RTOL_OUT, err_msg=f"row {r}")


def _grouped_rows(dev, dsa_lib):
    """Rows the library put into prefill row groups (its `group` region)."""
    R = dev.cfg.max_rows
    lay = dsa_lib.dsa_workspace_layout(dev.cfg)
    if lay["group"] == lay["key_hist"]:  # the config has no prefill groups
        return np.zeros(R, bool)
    return dev.workspace[lay["group"]:lay["group"] + 4 * R].view(torch.int32).cpu().numpy() != 0


def _group_row_partials(inp, rows, idx, grouped, q, r):
    """Oracle partial state of group row r: split s covers the tiles
    [s*T/S, (s+1)*T/S) of the T 128-position tiles holding a position some
    row of its group (the grouped rows of its 16-row slot) selected, and the
    row's state there is over its own selected positions in those tiles."""
    wl = inp["workload"]
    S = wl.num_splits
    slot = r // 16
    members = [j for j in range(16 * slot, 16 * slot + 16) if grouped[j]]
    union = np.unique(np.concatenate([idx[j][idx[j] >= 0] for j in members]))
    tiles = np.unique(union // 128)
    T = tiles.size
    sel = idx[r][idx[r] >= 0]
    Hq, D = wl.num_q_heads, wl.head_dim
    m, l, acc = np.full((Hq, S), -np.inf), np.zeros((Hq, S)), np.zeros((Hq, S, D))
    for s in range(S):
        part = sel[np.isin(sel // 128, tiles[s * T // S:(s + 1) * T // S])]
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), part)
        ms, ls, accs = O.split_partials_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads, 1)
        m[:, s], l[:, s], acc[:, s] = ms[:, 0], ls[:, 0], accs[:, 0]
    return m, l, acc


def test_split_partials_vs_oracle(problem, dsa_lib):
    i, inp, dev = problem
    wl = inp["workload"]
    rows = _rows(inp)
    idx = dev.views["topk_idx"].cpu().numpy()
    pm = dev.views["part_m"].cpu().numpy().astype(np.float64)
    pl = dev.views["part_l"].cpu().numpy().astype(np.float64)
    pa = dev.views["part_acc"].cpu().numpy().astype(np.float64)
    q = O.bf16_bits_to_f64(inp["q"])
    sample = _sample(i, rows)
    if len(sample) > 48:  # spread the split checks over the sample
        sample = sample[::max(1, len(sample) // 48)]
    grouped = _grouped_rows(dev, dsa_lib)
    for r in sample:
        L = int(rows["row_len"][r])
        if L == 0:  # dsa_step writes no partials for pad rows (the separate call does: see below)
            continue
        sel = idx[r][idx[r] >= 0]
        if grouped[r]:
            m, l, acc = _group_row_partials(inp, rows, idx, grouped, q, r)
        else:
            k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel) if L else (np.zeros((0, wl.num_kv_heads, wl.head_dim)),) * 2
            m, l, acc = O.split_partials_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads, wl.num_splits)
        fin = np.isfinite(m)
        assert np.array_equal(fin, np.isfinite(pm[r])), r
        # empty splits: l = 0 and acc = 0 exactly
        assert (pl[r][~fin] == 0).all() and (pa[r][~fin] == 0).all(), r
        np.testing.assert_allclose(pm[r][fin], m[fin], atol=ATOL_OUT, rtol=RTOL_OUT, err_msg=f"m, row {r}")
        np.testing.assert_allclose(pl[r][fin], l[fin], rtol=RTOL_L, atol=0, err_msg=f"l, row {r}")
        np.testing.assert_allclose(pa[r][fin] / pl[r][fin][:, None], acc[fin] / l[fin][:, None],
                                   atol=ATOL_OUT, rtol=RTOL_OUT, err_msg=f"acc / l, row {r}")


def test_pad_rows_are_empty(problem):
    i, inp, dev = problem
    if i != 3:
        pytest.skip("only workload 3 has pad rows")
    n = dev.rows["num_rows"]
    assert n == 560
    assert (dev.views["topk_idx"][n:] == -1).all()
    assert (dev.t["out"][n:].float() == 0).all()
    assert torch.isneginf(dev.t["lse"][n:]).all()


def test_step_equals_separate_calls_bitwise(problem, dsa_lib):
    i, inp, dev = problem
    cfg, t = dev.cfg, dev.t
    ws = dsa_lib.alloc_workspace(cfg)
    v = dsa_lib.workspace_views(cfg, ws)
    out = torch.empty_like(t["out"])
    lse = torch.empty_like(t["lse"])
    dsa_lib.dsa_indexer_scores(cfg, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"],
                               t["row_req"], t["row_len"], t["block_first"], t["block_nrows"], v["scores"], ws)
    dsa_lib.dsa_topk(cfg, v["scores"], t["row_len"], v["topk_idx"], ws)
    dsa_lib.dsa_sparse_attn(cfg, t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["row_req"], t["row_len"],
                            v["topk_idx"], v["part_m"], v["part_l"], v["part_acc"], ws)
    dsa_lib.dsa_merge(cfg, v["part_m"], v["part_l"], v["part_acc"], out, lse)
    torch.cuda.synchronize()
    assert torch.equal(v["topk_idx"], dev.views["topk_idx"])
    assert torch.equal(out.view(torch.int16), t["out"].view(torch.int16))
    assert torch.equal(lse, t["lse"])
    # dsa_sparse_attn on its own writes empty partials for the pad rows
    # (m = -inf, l = 0, acc = 0): its merge reads every row
    n = dev.rows["num_rows"]
    assert torch.isneginf(v["part_m"][n:]).all()
    assert (v["part_l"][n:] == 0).all() and (v["part_acc"][n:] == 0).all()
