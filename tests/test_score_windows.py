"""Score windows under a byte budget (Megatron-LM PR #7211, commit message 3):
the indexer and the top-k run over row windows that share one score buffer
of window_rows rows, and the step's results equal those of one window.

Host tests check the window arithmetic and the argument checks; the GPU
tests check that windowed steps and window calls give bit-identical scores,
selections and outputs, including windows whose edges cut a prefill score
block in two."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_decode_paged_gb300 import workloads as W


def _cfg(dsa_lib, **kw):
    base = dict(num_q_heads=64, num_kv_heads=8, head_dim=128, idx_heads=64, idx_dim=128, page_size=64,
                topk=2048, num_splits=4, max_rows=1024, max_reqs=49, max_pages_per_req=512,
                score_width=32768, num_pages=4096, block_rows=4)
    base.update(kw)
    return dsa_lib.make_config(**base)


# ----------------------------------------------------------------------------
# host: window sizes, workspace, argument checks
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("budget_rows,extra,want", [
    (None, 0, (1024, 1)),       # no budget: one window of every row
    (256, 0, (256, 4)),
    (250, 0, (250, 5)),         # last window 24 rows
    (250, 4 * 32768 - 4, (250, 5)),  # a partial row of budget does not count
    (1, 0, (1, 1024)),
    (5000, 0, (1024, 1)),       # more than max_rows: one window
])
def test_window_sizes(budget_rows, extra, want, dsa_lib):
    budget = 0 if budget_rows is None else budget_rows * 32768 * 4 + extra
    cfg = _cfg(dsa_lib, score_buffer_bytes=budget)
    wr, nw = dsa_lib.dsa_score_windows(cfg)
    assert (wr, nw) == want
    # the windows cover [0, max_rows) once, in order, each within the budget
    edges = [(i * wr, min((i + 1) * wr, cfg.max_rows)) for i in range(nw)]
    assert edges[0][0] == 0 and edges[-1][1] == cfg.max_rows
    assert all(a < b for a, b in edges) and all(e[1] == f[0] for e, f in zip(edges, edges[1:]))
    if budget:
        assert wr * cfg.score_width * 4 <= budget
    lay = dsa_lib.dsa_workspace_layout(cfg)
    span = lay["topk_idx"] - lay["scores"]
    assert wr * cfg.score_width * 4 <= span < wr * cfg.score_width * 4 + 256


def test_window_budget_shrinks_workspace(dsa_lib):
    full = dsa_lib.dsa_workspace_size(_cfg(dsa_lib))
    win = dsa_lib.dsa_workspace_size(_cfg(dsa_lib, score_buffer_bytes=128 * 32768 * 4))
    assert full - win == (1024 - 128) * 32768 * 4


@pytest.mark.parametrize("budget", [-1, 4, 32768 * 4 - 1])
def test_window_budget_below_one_row_rejected(budget, dsa_lib):
    with pytest.raises(dsa_lib.DsaError) as e:
        dsa_lib.dsa_validate_config(_cfg(dsa_lib, score_buffer_bytes=budget))
    assert e.value.status == dsa_lib.DSA_ERR_INVALID_ARG
    assert "score_buffer_bytes" in str(e.value)


@pytest.mark.parametrize("lo,hi", [(-1, 4), (0, 0), (5, 5), (6, 2), (0, 1025), (1024, 1025)])
def test_window_bounds_rejected_before_launch(lo, hi, dsa_lib):
    """A window outside [0, max_rows) is refused before any pointer is looked
    at (NULL pointers here; nothing reaches a GPU)."""
    lib = dsa_lib._lib
    cfg = _cfg(dsa_lib)
    st = lib.dsa_indexer_scores_window(ctypes.byref(cfg), lo, hi, *([None] * 12))
    assert st == dsa_lib.DSA_ERR_INVALID_ARG
    assert "row window" in lib.dsa_last_error().decode()
    st = lib.dsa_topk_window(ctypes.byref(cfg), lo, hi, *([None] * 5))
    assert st == dsa_lib.DSA_ERR_INVALID_ARG
    assert "row window" in lib.dsa_last_error().decode()


# ----------------------------------------------------------------------------
# GPU: windowed results are the whole-batch results
# ----------------------------------------------------------------------------
# rows per window for each workload: edges that fall inside prefill score
# blocks (mixed workload: blocks of 4 rows from row 48, edges at 250, 500...)
_WINDOW_ROWS = {0: 1, 1: 3, 3: 250, 4: 5, 5: 16}


@pytest.mark.gpu
@pytest.mark.parametrize("i", [0, 1, 3, 4, 5])
def test_windowed_step_identical(i, dsa_lib, cuda_ok):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    wl = inp["workload"]
    budget = _WINDOW_ROWS[i] * wl.score_width * 4
    whole = DeviceStep(inp)
    win = DeviceStep(inp, score_buffer_bytes=budget)
    wr, nw = dsa_lib.dsa_score_windows(win.cfg)
    assert wr == _WINDOW_ROWS[i] and nw > 1
    assert win.views["scores"].shape == (wr, wl.score_width)
    for dev in (whole, win):
        dev.step()
    torch.cuda.synchronize()
    assert whole.status() == 0 and win.status() == 0
    assert torch.equal(whole.views["topk_idx"], win.views["topk_idx"])
    assert torch.equal(whole.t["out"], win.t["out"])
    assert torch.equal(whole.t["lse"], win.t["lse"])
    # the histogram each window's indexer hands over is used up and zeroed
    lay = dsa_lib.dsa_workspace_layout(win.cfg)
    assert int(win.workspace[lay["key_hist"]:lay["total"]].count_nonzero()) == 0
    # the windowed step replays from a CUDA graph with the same results
    win.t["out"].zero_()
    win.views["topk_idx"].fill_(-5)
    g = win.capture()
    g.replay()
    torch.cuda.synchronize()
    assert win.status() == 0
    assert torch.equal(whole.views["topk_idx"], win.views["topk_idx"])
    assert torch.equal(whole.t["out"], win.t["out"])


@pytest.mark.gpu
@pytest.mark.parametrize("i,windows", [(3, [(0, 50), (50, 250), (250, 251), (251, 1024)]),
                                       (1, [(2, 5), (0, 2), (5, 8)])])
def test_window_calls_match_whole(i, windows, dsa_lib, cuda_ok):
    """dsa_indexer_scores_window writes exactly the window's rows (each row's
    first row_len scores, bit-identical to the whole-batch call, nothing past
    them) at row - row_begin; dsa_topk_window writes exactly the window's
    rows of topk_idx, bit-identical to dsa_topk."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    dev = DeviceStep(inp)
    cfg, t, v = dev.cfg, dev.t, dev.views
    R, Wd, K = cfg.max_rows, cfg.score_width, cfg.topk
    lens = dev.rows["row_len"]
    idx_args = (t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"], t["row_req"],
                t["row_len"], t["block_first"], t["block_nrows"])
    dsa_lib.dsa_indexer_scores(cfg, *idx_args, v["scores"], dev.workspace)
    dsa_lib.dsa_topk(cfg, v["scores"], t["row_len"], v["topk_idx"], dev.workspace)
    torch.cuda.synchronize()
    full_scores = v["scores"].clone()
    full_sel = v["topk_idx"].clone()

    sel = torch.full((R, K), -7, dtype=torch.int32, device="cuda")
    covered = np.zeros(R, bool)
    for lo, hi in windows:
        buf = torch.full((hi - lo, Wd), float("nan"), dtype=torch.float32, device="cuda")
        dsa_lib.dsa_indexer_scores(cfg, *idx_args, buf, dev.workspace, window=(lo, hi))
        before = sel.clone()
        dsa_lib.dsa_topk(cfg, buf, t["row_len"], sel, dev.workspace, window=(lo, hi))
        torch.cuda.synchronize()
        assert dev.status() == 0
        got = buf.cpu().numpy()
        ref = full_scores[lo:hi].cpu().numpy()
        for j, r in enumerate(range(lo, hi)):
            L = int(lens[r])
            assert np.array_equal(got[j, :L].view(np.uint32), ref[j, :L].view(np.uint32)), f"row {r}"
            assert np.isnan(got[j, L:]).all(), f"row {r}: written past its length"
        assert torch.equal(sel[lo:hi], full_sel[lo:hi])
        outside = torch.ones(R, dtype=torch.bool, device="cuda")
        outside[lo:hi] = False
        assert torch.equal(sel[outside], before[outside])
        covered[lo:hi] = True
    assert covered.all()
    assert torch.equal(sel, full_sel)


# ----------------------------------------------------------------------------
# GPU: a windowed step against the oracle
# ----------------------------------------------------------------------------
# sampled rows: on the mixed workload both sides of the window edge at row
# 250, which cuts the prefill score block of rows 248..251, the edge at 500
# (a block boundary), decode rows and pad rows; on the long fp8 workload
# (5-row windows) every row; on the 1M-key prefill (16-row windows, 80 MB
# of scores per window instead of 320 MB) the decode row near 1M keys, both
# sides of the edges at rows 16 and 64 (inside the prefill blocks 13..16 and
# 61..64), the short decode row and a pad row
_ORACLE_ROWS = {3: [0, 23, 47, 48, 49, 246, 247, 248, 249, 250, 251, 252, 253, 498, 499, 500, 501, 558, 559, 560,
                    1023],
                4: list(range(16)),
                5: [0, 1, 15, 16, 17, 63, 64, 65, 66]}


@pytest.mark.gpu
@pytest.mark.parametrize("i", [3, 4, 5])
def test_windowed_step_vs_oracle(i, dsa_lib, cuda_ok):
    """A step with a score budget (several row windows) compared with the
    oracle: each window's scores within the score tolerance, its top-k
    bit-exact given those scores, and the windowed dsa_step's output and lse
    on its own selection within the attention tolerance.  The selection is
    also checked as a valid top-k under the oracle's own scores: every
    selected position ranks within the score tolerance of the k-th best."""
    from oracle import dsa_oracle as O
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    wl = inp["workload"]
    rtol = 6e-2 if wl.idx_key_dtype == W.KEY_FP8_E4M3 else 2e-2
    dev = DeviceStep(inp, score_buffer_bytes=_WINDOW_ROWS[i] * wl.score_width * 4,
                     flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    cfg, t, v = dev.cfg, dev.t, dev.views
    wr, nw = dsa_lib.dsa_score_windows(cfg)
    assert nw > 1
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    sel_step = v["topk_idx"].cpu().numpy()
    out = dev.t["out"].float().cpu().numpy().astype(np.float64)
    lse = dev.t["lse"].cpu().numpy().astype(np.float64)

    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    qi = O.bf16_bits_to_f64(inp["q_idx"])
    q = O.bf16_bits_to_f64(inp["q"])
    sample = [r for r in _ORACLE_ROWS[i] if r < wl.max_rows]
    # the window calls dsa_step makes, with each window's scores kept
    idx_args = (t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"], t["row_req"],
                t["row_len"], t["block_first"], t["block_nrows"])
    sel = torch.full_like(v["topk_idx"], -7)
    win_scores = {}
    for lo in range(0, cfg.max_rows, wr):
        hi = min(lo + wr, cfg.max_rows)
        if not any(lo <= r < hi for r in sample):
            continue
        dsa_lib.dsa_indexer_scores(cfg, *idx_args, v["scores"], dev.workspace, window=(lo, hi))
        dsa_lib.dsa_topk(cfg, v["scores"], t["row_len"], sel, dev.workspace, window=(lo, hi))
        torch.cuda.synchronize()
        got = v["scores"].cpu().numpy()
        for r in range(lo, hi):
            if r in sample:
                win_scores[r] = got[r - lo].copy()
    assert dev.status() == 0
    sel = sel.cpu().numpy()
    for r in sample:
        L = int(rows["row_len"][r])
        if L == 0:
            assert (sel_step[r] == -1).all() and (out[r] == 0).all() and np.isneginf(lse[r]).all()
            continue
        keys, sc = O.index_keys(inp, int(rows["row_req"][r]), L)
        want = O.indexer_scores_row(qi[r], inp["w"][r], keys, sc)
        g = win_scores[r][:L].astype(np.float64)
        rms = np.sqrt(np.mean(want * want))
        assert np.all(np.abs(g - want) <= rtol * np.abs(want) + rtol * rms), f"scores, row {r}"
        assert np.array_equal(sel[r], O.topk_row(win_scores[r], L, wl.topk)), f"top-k, row {r}"
        assert np.array_equal(sel_step[r], sel[r]), f"step selection, row {r}"
        chosen = sel_step[r][sel_step[r] >= 0]
        n = min(wl.topk, L)
        assert chosen.size == n and np.all(np.diff(chosen) > 0) and chosen[-1] < L
        if n < L:  # valid under the oracle's scores up to the score tolerance
            kth = np.sort(want)[::-1][n - 1]
            assert np.all(want[chosen] >= kth - 2 * (rtol * np.abs(kth) + rtol * rms)), f"selection, row {r}"
        k, vv = O.kv_rows(inp, int(rows["row_req"][r]), chosen)
        o, ls = O.attention_row(q[r], k, vv, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")
        np.testing.assert_allclose(lse[r], ls, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")
