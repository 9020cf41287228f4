"""Edge cases of the CUDA path: exact integer cases, top-k ties and
infinities, CUDA-graph replay with changed metadata, device-side bounds
flags, poisoned cache slots and page relabelling."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from sparse_attention_decode_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dev_step(inp, **kw):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    dev = DeviceStep(inp, **kw)
    dev.step()
    torch.cuda.synchronize()
    return dev


def _bf16_bits_of(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# indexer: integer-valued inputs make every fp32 sum exact
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("fp8,P,br", [(False, 64, 1), (False, 64, 4), (True, 64, 1), (True, 16, 1), (True, 32, 1),
                                      (True, 128, 1), (True, 64, 2), (True, 64, 4)])
def test_indexer_exact_on_integer_inputs(fp8, P, br, dsa_lib, cuda_ok):
    """Exact scores for bf16 and fp8 keys, at every page size (the producer
    issues one box per page, 1 to 8 per tile) and with score blocks of 1, 2
    and 4 rows.  With br > 1 the last request appends 9 tokens, so its rows
    form 2- or 4-row blocks and a shorter last block."""
    wl = dataclasses.replace(W.workload(1), page_size=P, max_pages_per_req=4096 // P, block_rows=br,
                             max_rows=16 if br > 1 else 8)
    if fp8:
        wl = dataclasses.replace(wl, idx_key_dtype=W.KEY_FP8_E4M3)
    inp = W.generate(wl)
    if br > 1:
        inp["new_tokens"] = inp["new_tokens"].copy()
        inp["new_tokens"][-1] = 9
    rng = np.random.default_rng(21)
    R, HI, DI = wl.max_rows, wl.idx_heads, wl.idx_dim
    q = rng.integers(-3, 4, (R, HI, DI)).astype(np.float32)
    if fp8:
        # fp8 keys: the kernel quantises each query head to e4m3 with scale
        # amax/448; a head whose largest entry is 448 has scale 1 and small
        # integers are e4m3 values, so that quantisation is lossless here
        q[..., 0] = 448.0
    inp["q_idx"] = _bf16_bits_of(q)
    inp["w"] = (2.0 ** rng.integers(-2, 2, (R, HI)) * rng.choice([-1.0, 1.0], (R, HI))).astype(np.float32)
    keys = rng.integers(-4, 5, inp["idx_cache"].shape).astype(np.float32)
    if fp8:
        inp["idx_cache"] = torch.from_numpy(keys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        inp["idx_scale"] = (2.0 ** rng.integers(-3, 3, inp["idx_scale"].shape)).astype(np.float32)
    else:
        inp["idx_cache"] = _bf16_bits_of(keys)
    dev = _dev_step(inp)
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    want = O.indexer_scores(inp, rows)
    got = dev.views["scores"].cpu().numpy().astype(np.float64)
    for r in range(rows["num_rows"]):
        L = rows["row_len"][r]
        assert np.array_equal(got[r, :L], want[r, :L]), r
    assert dev.status() == 0

    if fp8 and P == 32:
        # a page id outside the pool inside row 1: flagged, and every key on
        # the other pages (the same tiles included) still scores exactly
        r = 1
        req, j = int(rows["row_req"][r]), 3
        assert rows["row_len"][r] > (j + 1) * P
        dev.t["page_table"][req, j] = inp["num_pages"] + 3
        dev.step()
        torch.cuda.synchronize()
        assert dev.status() & dsa_lib.DSA_DEV_BAD_PAGE
        got = dev.views["scores"].cpu().numpy().astype(np.float64)
        keep = np.ones(rows["row_len"][r], bool)
        keep[j * P:(j + 1) * P] = False
        assert np.array_equal(got[r, :rows["row_len"][r]][keep], want[r, :rows["row_len"][r]][keep])
        for r2 in range(rows["num_rows"]):
            if rows["row_req"][r2] != req:
                L = rows["row_len"][r2]
                assert np.array_equal(got[r2, :L], want[r2, :L]), r2


# ----------------------------------------------------------------------------
# top-k: crafted rows
# ----------------------------------------------------------------------------
def _topk_cfg(dsa_lib, R, W_, K):
    return dsa_lib.make_config(num_q_heads=8, num_kv_heads=1, head_dim=64, idx_heads=8, idx_dim=32,
                               page_size=64, topk=K, num_splits=1, max_rows=R, max_reqs=R,
                               max_pages_per_req=(W_ + 63) // 64, score_width=W_, num_pages=1)


# widths reach each cluster size of the in-shared-memory top-k: 1 CTA (300,
# 4096), 2 (32768), 4 (65536, 131072) and 8 (262144, the longest row it
# holds); past that the streaming top-k reads the score buffer: 262148 and
# 1M / 4M keys (float4 loads), 262147 (a row stride that is not a multiple
# of 4: scalar loads).  It reads a row once when k <= 4096 and the
# threshold bin holds at most 4096 keys (the all-ties rows do not), else in
# several passes (also k = 5000)
@pytest.mark.parametrize("W_,K", [(4096, 512), (32768, 2048), (65536, 1024), (131072, 2048), (262144, 2048),
                                  (300, 16), (262147, 300), (262148, 512), (262148, 5000), (1 << 20, 2048),
                                  (1 << 22, 2048)])
def test_topk_crafted_rows(W_, K, dsa_lib, cuda_ok):
    rng = np.random.default_rng(W_ + K)
    R = 12
    cfg = _topk_cfg(dsa_lib, R, W_, K)
    lens = [0, 1, K - 1, K, K + 1, W_, W_, W_, W_, int(rng.integers(K, W_ + 1)), W_ - 1, W_]
    s = rng.standard_normal((R, W_)).astype(np.float32)
    s[5] = 1.0                                                   # all equal: lowest positions win
    s[6] = rng.choice(np.array([-np.inf, -1.0, 0.0, 2.0, np.nan], np.float32), W_)  # heavy ties + inf + nan
    s[7] = -np.inf
    s[7, rng.integers(0, W_, K // 3)] = 3.0                      # few finite, rest -inf
    s[8] = np.nan
    s[8, rng.integers(0, W_, K // 2)] = -np.inf                  # -inf beats NaN
    s[10] = np.round(rng.standard_normal(W_) * 4) / 4            # quantised ties
    s[10][::7] = -0.0                                            # -0 ties with +0
    s[11] = np.float32(0.0)
    s[11, ::3] = -0.0
    scores = torch.from_numpy(s).cuda()
    row_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = torch.full((R, K), -7, dtype=torch.int32, device="cuda")
    ws = dsa_lib.alloc_workspace(cfg)
    dsa_lib.dsa_topk(cfg, scores, row_len, out, ws)
    got = out.cpu().numpy()
    for r in range(R):
        want = O.topk_row(s[r], lens[r], K) if lens[r] else np.full(K, -1, np.int32)
        assert np.array_equal(got[r], want), (r, lens[r])
    assert dsa_lib.dsa_read_device_status(ws) == 0


def test_topk_random_ragged(dsa_lib, cuda_ok):
    rng = np.random.default_rng(99)
    R, W_, K = 64, 8192, 700
    cfg = _topk_cfg(dsa_lib, R, W_, K)
    for trial in range(3):
        lens = rng.integers(0, W_ + 1, R)
        pool = rng.standard_normal(int(rng.integers(2, 5000))).astype(np.float32)
        s = pool[rng.integers(0, pool.size, (R, W_))]
        scores = torch.from_numpy(s).cuda()
        out = torch.empty((R, K), dtype=torch.int32, device="cuda")
        ws = dsa_lib.alloc_workspace(cfg)
        dsa_lib.dsa_topk(cfg, scores, torch.from_numpy(lens.astype(np.int32)).cuda(), out, ws)
        got = out.cpu().numpy()
        for r in range(R):
            want = O.topk_row(s[r], int(lens[r]), K) if lens[r] else np.full(K, -1, np.int32)
            assert np.array_equal(got[r], want), (trial, r)


# ----------------------------------------------------------------------------
# CUDA graphs: capture once, replay with new device metadata
# ----------------------------------------------------------------------------
def test_graph_replay_follows_metadata(dsa_lib, cuda_ok):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(1)
    wl = inp["workload"]
    dev = DeviceStep(inp)
    graph = dev.capture()
    graph.replay()
    torch.cuda.synchronize()
    out_g1 = dev.t["out"].clone()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_g1.view(torch.int16), dev.t["out"].view(torch.int16))  # deterministic
    dev.step()
    torch.cuda.synchronize()
    assert torch.equal(out_g1.view(torch.int16), dev.t["out"].view(torch.int16))  # graph == eager

    # new lengths (within each request's pages), fewer live requests, and a
    # relabelled page table: same buffers, no re-capture
    rng = np.random.default_rng(3)
    cl = inp["cache_len"].copy()
    new_cl = np.array([int(rng.integers(1, c + 1)) for c in cl], np.int32)
    new_cl[0] = 1
    new_cl[1] = wl.topk + 1
    nt = np.ones_like(new_cl)
    nt[5:] = 0  # requests 5..7 idle this step
    perm = rng.permutation(inp["num_pages"]).astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    for key in ("idx_cache", "k_cache", "v_cache"):
        src = inp[key][inv]
        dst = dev.t[key]
        dst.view(torch.int16 if dst.dtype == torch.bfloat16 else dst.dtype).copy_(
            torch.from_numpy(src.view(np.int16) if src.dtype == np.uint16 else src))
    dev.set_rows(new_cl, nt, pt)
    graph.replay()
    torch.cuda.synchronize()
    out_g2 = dev.t["out"].clone()
    idx_g2 = dev.views["topk_idx"].clone()
    dev.step()
    torch.cuda.synchronize()
    assert torch.equal(out_g2.view(torch.int16), dev.t["out"].view(torch.int16))
    assert dev.status() == 0

    inp2 = dict(inp)
    inp2["cache_len"], inp2["new_tokens"] = new_cl, nt
    inp2["page_table"] = pt
    for key in ("idx_cache", "k_cache", "v_cache"):
        inp2[key] = inp[key][inv]
    rows = O.build_rows(new_cl, nt, wl.max_rows, wl.block_rows)
    assert rows["num_rows"] == 5
    q = O.bf16_bits_to_f64(inp2["q"])
    got_out = out_g2.float().cpu().numpy()
    idx = idx_g2.cpu().numpy()
    scores = dev.views["scores"].cpu().numpy()
    for r in range(wl.max_rows):
        L = int(rows["row_len"][r])
        if L == 0:
            assert (idx[r] == -1).all() and (got_out[r] == 0).all()
            continue
        assert np.array_equal(idx[r], O.topk_row(scores[r], L, wl.topk))
        sel = idx[r][idx[r] >= 0]
        k, v = O.kv_rows(inp2, int(rows["row_req"][r]), sel)
        o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(got_out[r], o, atol=1e-2, rtol=2e-2)


# ----------------------------------------------------------------------------
# invariances on the GPU
# ----------------------------------------------------------------------------
def test_poisoned_slots_past_length_change_nothing(dsa_lib, cuda_ok):
    inp = W.generate(0)
    wl = inp["workload"]
    ref = _dev_step(inp)
    bad = dict(inp)
    for key in ("idx_cache", "k_cache", "v_cache"):
        bad[key] = inp[key].copy()
    for b, L in enumerate(inp["cache_len"]):
        page = inp["page_table"][b, (L - 1) // wl.page_size]
        if L % wl.page_size:
            bad["idx_cache"][page, L % wl.page_size:] = 0x7FC0
            bad["k_cache"][page, L % wl.page_size:] = 0x7F80
            bad["v_cache"][page, L % wl.page_size:] = 0x7FC0
    got = _dev_step(bad)
    assert torch.equal(ref.views["topk_idx"], got.views["topk_idx"])
    assert torch.equal(ref.t["out"].view(torch.int16), got.t["out"].view(torch.int16))


def test_page_relabelling_is_bit_identical(dsa_lib, cuda_ok):
    inp = W.generate(1)
    ref = _dev_step(inp)
    rng = np.random.default_rng(8)
    perm = rng.permutation(inp["num_pages"]).astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    moved = dict(inp)
    for key in ("idx_cache", "k_cache", "v_cache"):
        moved[key] = inp[key][inv]
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    moved["page_table"] = pt
    got = _dev_step(moved)
    assert torch.equal(ref.views["scores"], got.views["scores"])
    assert torch.equal(ref.t["out"].view(torch.int16), got.t["out"].view(torch.int16))


# ----------------------------------------------------------------------------
# device-side bounds checks: flagged, skipped, never a fault
# ----------------------------------------------------------------------------
def test_device_bounds_flags(dsa_lib, cuda_ok):
    inp = W.generate(0)
    dev = _dev_step(inp)
    assert dev.status() == 0
    t, cfg = dev.t, dev.cfg

    # a page id outside the pool, inside request 1's length
    saved = t["page_table"].clone()
    t["page_table"][1, 2] = cfg.num_pages + 3
    dev.step()
    st = dev.status()
    assert st & dsa_lib.DSA_DEV_BAD_PAGE
    t["page_table"].copy_(saved)
    dsa_lib.dsa_reset_device_status(dev.workspace)

    # a row longer than the score width
    saved_len = t["row_len"].clone()
    t["row_len"][0] = cfg.score_width + 1
    dev.step()
    st = dev.status()
    assert st & dsa_lib.DSA_DEV_BAD_BLOCK and st & dsa_lib.DSA_DEV_BAD_ROW
    assert (dev.views["topk_idx"][0] == -1).all()
    t["row_len"].copy_(saved_len)
    dsa_lib.dsa_reset_device_status(dev.workspace)

    # a selected position at or past the row's length
    idx = dev.views["topk_idx"].clone()
    dev.step()
    idx = dev.views["topk_idx"].clone()
    idx[0, 0] = int(dev.rows["row_len"][0]) + 5
    idx[1, 1] = -9
    v = dev.views
    dsa_lib.dsa_sparse_attn(cfg, t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["row_req"],
                            t["row_len"], idx, v["part_m"], v["part_l"], v["part_acc"], dev.workspace)
    assert dev.status() & dsa_lib.DSA_DEV_BAD_INDEX
    dsa_lib.dsa_reset_device_status(dev.workspace)
    dev.step()
    assert dev.status() == 0


# ----------------------------------------------------------------------------
# indexer -> top-k histogram hand-off (DSA_FLAG_TOPK_HISTOGRAM, always on in dsa_step)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("i", [1, 3, 4, 5])  # 5: 1M-key rows, the streaming top-k
def test_topk_histogram_handoff(i, dsa_lib, cuda_ok):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    plain = DeviceStep(inp)
    fused = DeviceStep(inp, flags=dsa_lib.DSA_FLAG_TOPK_HISTOGRAM)
    for dev in (plain, fused):
        cfg, t, v = dev.cfg, dev.t, dev.views
        for _ in range(2):  # the second pass needs the histogram re-zeroed by the first top-k
            dsa_lib.dsa_indexer_scores(cfg, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"],
                                       t["row_req"], t["row_len"], t["block_first"], t["block_nrows"],
                                       v["scores"], dev.workspace)
            dsa_lib.dsa_topk(cfg, v["scores"], t["row_len"], v["topk_idx"], dev.workspace)
        torch.cuda.synchronize()
        assert dev.status() == 0
    assert torch.equal(plain.views["scores"], fused.views["scores"])
    assert torch.equal(plain.views["topk_idx"], fused.views["topk_idx"])
    hist = dsa_lib.dsa_workspace_layout(fused.cfg)
    kh = fused.workspace[hist["key_hist"]:hist["total"]]
    assert int(kh.count_nonzero()) == 0  # left at zero for the next step
    fused.step()  # dsa_step hands the histogram over internally
    torch.cuda.synchronize()
    assert torch.equal(plain.views["topk_idx"], fused.views["topk_idx"])
    assert int(kh.count_nonzero()) == 0


def test_topk_histogram_mismatch(dsa_lib, cuda_ok):
    """A hand-over histogram that does not count the row's scores is recounted
    (same selection, clean status); one with the right total but the wrong
    bins sets DSA_DEV_BAD_HIST and stays inside the buffers."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(1)
    plain = DeviceStep(inp)
    plain.step()
    dev = DeviceStep(inp, flags=dsa_lib.DSA_FLAG_TOPK_HISTOGRAM)
    cfg, t, v = dev.cfg, dev.t, dev.views
    cfg_nohist = type(cfg).from_buffer_copy(cfg)
    cfg_nohist.flags = 0
    lay = dsa_lib.dsa_workspace_layout(cfg)
    kh = dev.workspace[lay["key_hist"]:lay["total"]]

    def indexer(c):
        dsa_lib.dsa_indexer_scores(c, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"],
                                   t["row_req"], t["row_len"], t["block_first"], t["block_nrows"],
                                   v["scores"], dev.workspace)

    def topk():
        dsa_lib.dsa_topk(cfg, v["scores"], t["row_len"], v["topk_idx"], dev.workspace)

    # the indexer ran without the bit: nothing counted, the top-k recounts
    indexer(cfg_nohist)
    v["topk_idx"].fill_(-7)
    topk()
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(v["topk_idx"], plain.views["topk_idx"])
    # the indexer ran twice with the bit: every bin counted twice, recounted
    indexer(cfg)
    indexer(cfg)
    v["topk_idx"].fill_(-7)
    topk()
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(v["topk_idx"], plain.views["topk_idx"])
    assert int(kh.count_nonzero()) == 0
    # right total, wrong bins: the scores of one long row change after counting
    lens = t["row_len"].cpu().numpy()
    K = cfg.topk
    r = int(next(i for i, L in enumerate(lens) if L > K))
    indexer(cfg)
    v["scores"][r, : int(lens[r])] = -1e30
    topk()
    torch.cuda.synchronize()
    st = dev.status()
    assert st & dsa_lib.DSA_DEV_BAD_HIST, hex(st)
    others = [i for i in range(cfg.max_rows) if i != r]
    assert torch.equal(v["topk_idx"][others], plain.views["topk_idx"][others])
    assert int(kh.count_nonzero()) == 0
    dsa_lib.dsa_reset_device_status(dev.workspace)
    dev.step()  # a clean step afterwards
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(v["topk_idx"], plain.views["topk_idx"])


@pytest.mark.parametrize("i", [0, 1, 3])
def test_kv_interleaved_layout_identical(i, dsa_lib, cuda_ok):
    """DSA_FLAG_KV_INTERLEAVED (a token's K and V rows adjacent, one copy per
    token) gives bit-identical outputs to the separate K and V caches."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    sep = DeviceStep(inp)
    itl = DeviceStep(inp, flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    assert itl.t["k_cache"].shape[2] == 2
    for dev in (sep, itl):
        dev.step()
    torch.cuda.synchronize()
    assert sep.status() == 0 and itl.status() == 0
    assert torch.equal(sep.t["out"], itl.t["out"])
    assert torch.equal(sep.t["lse"], itl.t["lse"])
    # the separate calls take the same layout
    cfg, t, v = itl.cfg, itl.t, itl.views
    v["part_acc"].zero_()
    dsa_lib.dsa_sparse_attn(cfg, t["q"], t["k_cache"], None, t["page_table"], t["row_req"], t["row_len"],
                            v["topk_idx"], v["part_m"], v["part_l"], v["part_acc"], itl.workspace)
    dsa_lib.dsa_merge(cfg, v["part_m"], v["part_l"], v["part_acc"], t["out"], t["lse"])
    torch.cuda.synchronize()
    assert torch.equal(sep.t["out"], itl.t["out"])


# ----------------------------------------------------------------------------
# the bounded-wait failure path, without a fault
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("i", [0, 4])
def test_wait_that_runs_out_flags_timeout_and_the_next_step_is_clean(i, dsa_lib, cuda_ok):
    """With the test-only flag the indexer's MMA thread waits on a barrier
    that nothing completes, with a ~1 ms budget: the wait runs out, the
    kernel sets DSA_DEV_TIMEOUT, every role leaves its loop (the producer
    still waits for its copies in flight) and the launch returns well within
    a second.  The context stays usable: after resetting the status word, a
    step without the flag gives the same result as before (bf16 keys and
    fp8 keys, whose epilogue path differs)."""
    import time
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i, with_kv=True)
    dev = DeviceStep(inp)
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    ref_out, ref_lse = dev.t["out"].clone(), dev.t["lse"].clone()
    ref_scores = dev.views["scores"].clone()

    t = dev.t
    cfg = dsa_lib.config_from_workload(inp["workload"], inp["num_pages"],
                                       flags=dev.cfg.flags | dsa_lib.DSA_FLAG_TEST_WAIT_TIMEOUT)
    dsa_lib.dsa_validate_config(cfg)
    scores = torch.full_like(dev.views["scores"], 7.0)
    t0 = time.perf_counter()
    dsa_lib.dsa_indexer_scores(cfg, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"],
                               t["row_req"], t["row_len"], t["block_first"], t["block_nrows"], scores,
                               dev.workspace)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = dev.status()
    assert status & dsa_lib.DSA_DEV_TIMEOUT, hex(status)
    assert status == dsa_lib.DSA_DEV_TIMEOUT, hex(status)  # nothing else went wrong
    assert elapsed < 0.5, elapsed  # the ~1 ms wait, not the ~1 s one
    assert (scores == 7.0).all()   # no MMA ran, so no score was written

    dsa_lib.dsa_reset_device_status(dev.workspace)
    dev.t["out"].zero_()
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    assert torch.equal(dev.views["scores"], ref_scores)
    assert torch.equal(dev.t["out"].view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(dev.t["lse"], ref_lse)


# ----------------------------------------------------------------------------
# prefill row groups (tensor-core attention over the union of a group's
# selections)
# ----------------------------------------------------------------------------
def _group_slots(row_req, row_len, idx, wl):
    """The grouping rule the library states: in each slot of 16 rows, the
    rows of the request with the most rows there (ties: the lowest row's),
    if there are at least 8, their longest row spans at most
    min(score_width, 64 * topk) rounded up to 128 positions, and their union
    of selected positions fills at least a quarter of it."""
    umax = -(-min(wl.score_width, 64 * wl.topk) // 128) * 128
    groups = {}
    for slot in range((wl.max_rows + 15) // 16):
        rows = [r for r in range(16 * slot, min(16 * slot + 16, wl.max_rows)) if row_len[r] > 0]
        if not rows:
            continue
        counts = {}
        for r in rows:
            counts.setdefault(int(row_req[r]), []).append(r)
        best = max(counts.values(), key=lambda rs: (len(rs), -rs[0]))
        lmax = max(int(row_len[r]) for r in best)
        if len(best) < 8 or lmax > umax:
            continue
        union = np.unique(np.concatenate([idx[r][idx[r] >= 0] for r in best]))
        if 4 * union.size >= lmax:
            groups[slot] = (best, union)
    return groups


@pytest.mark.parametrize("i,splits", [(3, 1), (3, 3), (6, 4)])
def test_prefill_groups_vs_oracle(i, splits, dsa_lib, cuda_ok):
    """The mixed step's prefill rows go through the group kernel: their
    outputs match the oracle on their own selections, and each split's
    partial state matches the oracle over the row's selected positions in
    that split's union tiles; the decode rows keep the slot splits.  Workload
    6 is the same step with correlated indexer queries."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(i)
    wl = inp["workload"]
    dev = DeviceStep(inp, num_splits=splits, flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    idx = dev.views["topk_idx"].cpu().numpy()
    groups = _group_slots(rows["row_req"], rows["row_len"], idx, wl)
    assert len(groups) == 32 and all(len(m) == 16 for m, _ in groups.values())  # rows 48..559
    lay = dsa_lib.dsa_workspace_layout(dev.cfg)
    grouped = dev.workspace[lay["group"]:lay["group"] + 4 * wl.max_rows].view(torch.int32).cpu().numpy()
    want_grouped = np.zeros(wl.max_rows, np.int32)
    for m, _ in groups.values():
        want_grouped[m] = 1
    assert np.array_equal(grouped, want_grouped)

    out = dev.t["out"].float().cpu().numpy().astype(np.float64)
    pm = dev.views["part_m"].cpu().numpy().astype(np.float64)
    pl = dev.views["part_l"].cpu().numpy().astype(np.float64)
    pa = dev.views["part_acc"].cpu().numpy().astype(np.float64)
    q = O.bf16_bits_to_f64(inp["q"])
    for slot in sorted(groups)[::5] + [max(groups)]:
        members, union = groups[slot]
        tiles = np.unique(union // 128)  # the 128-position tiles holding a selected position
        T = tiles.size
        for r in members[::5] + [members[-1]]:
            sel = idx[r][idx[r] >= 0]
            k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel)
            o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
            np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")
            for s in range(splits):
                mine = tiles[s * T // splits:(s + 1) * T // splits]
                part = sel[np.isin(sel // 128, mine)]
                k, v = O.kv_rows(inp, int(rows["row_req"][r]), part)
                m, l, acc = O.split_partials_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads, 1)
                fin = np.isfinite(m[:, 0])
                assert np.array_equal(fin, np.isfinite(pm[r, :, s])), (r, s)
                assert (pl[r, ~fin, s] == 0).all() and (pa[r, ~fin, s] == 0).all(), (r, s)
                np.testing.assert_allclose(pm[r, fin, s], m[fin, 0], atol=1e-2, rtol=2e-2, err_msg=f"m {r} {s}")
                np.testing.assert_allclose(pl[r, fin, s], l[fin, 0], rtol=2e-2, atol=0, err_msg=f"l {r} {s}")
                np.testing.assert_allclose(pa[r, fin, s] / pl[r, fin, s][:, None], acc[fin, 0] / l[fin, 0][:, None],
                                           atol=1e-2, rtol=2e-2, err_msg=f"acc/l {r} {s}")
    for r in (0, 23, 47):  # decode rows
        sel = idx[r][idx[r] >= 0]
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel)
        o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")


def test_no_prefill_groups_flag_takes_the_row_path(dsa_lib, cuda_ok):
    """With DSA_FLAG_NO_PREFILL_GROUPS the mixed step has no group region and
    every prefill row takes the per-row attention: outputs and top-k slot
    split partials match the oracle, and the selection is the grouped
    step's."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(3)
    wl = inp["workload"]
    flags = dsa_lib.DSA_FLAG_KV_INTERLEAVED
    dev = DeviceStep(inp, flags=flags | dsa_lib.DSA_FLAG_NO_PREFILL_GROUPS)
    lay = dsa_lib.dsa_workspace_layout(dev.cfg)
    assert lay["group"] == lay["key_hist"]
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    ref = DeviceStep(inp, flags=flags)
    ref.step()
    torch.cuda.synchronize()
    idx = dev.views["topk_idx"].cpu().numpy()
    assert np.array_equal(idx, ref.views["topk_idx"].cpu().numpy())
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    out = dev.t["out"].float().cpu().numpy().astype(np.float64)
    pm = dev.views["part_m"].cpu().numpy().astype(np.float64)
    pl = dev.views["part_l"].cpu().numpy().astype(np.float64)
    pa = dev.views["part_acc"].cpu().numpy().astype(np.float64)
    q = O.bf16_bits_to_f64(inp["q"])
    for r in list(range(48, 560, 37)) + [559]:  # prefill rows
        sel = idx[r][idx[r] >= 0]
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel)
        o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")
        m, l, acc = O.split_partials_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads, wl.num_splits)
        fin = np.isfinite(m)
        assert np.array_equal(fin, np.isfinite(pm[r])), r
        np.testing.assert_allclose(pm[r][fin], m[fin], atol=1e-2, rtol=2e-2, err_msg=f"m {r}")
        np.testing.assert_allclose(pl[r][fin], l[fin], rtol=2e-2, atol=0, err_msg=f"l {r}")
        np.testing.assert_allclose(pa[r][fin] / pl[r][fin][:, None], acc[fin] / l[fin][:, None],
                                   atol=1e-2, rtol=2e-2, err_msg=f"acc/l {r}")


@pytest.mark.parametrize("P", [16, 32, 128])
def test_prefill_groups_other_page_sizes(P, dsa_lib, cuda_ok):
    """The group kernel moves whole pages per 128-position tile (8, 4 or 1
    page boxes per tile, or one box per tile for 128-token pages): the mixed
    step with other page sizes forms the same groups and its group rows'
    outputs match the oracle."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    wl = dataclasses.replace(W.workload(3), page_size=P, max_pages_per_req=32768 // P)
    inp = W.generate(wl)
    dev = DeviceStep(inp, flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    idx = dev.views["topk_idx"].cpu().numpy()
    groups = _group_slots(rows["row_req"], rows["row_len"], idx, wl)
    assert len(groups) == 32
    out = dev.t["out"].float().cpu().numpy().astype(np.float64)
    q = O.bf16_bits_to_f64(inp["q"])
    for slot in sorted(groups)[::8]:
        members, _ = groups[slot]
        for r in (members[0], members[-1]):
            sel = idx[r][idx[r] >= 0]
            k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel)
            o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
            np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"P {P} row {r}")


# ----------------------------------------------------------------------------
# the largest row count
# ----------------------------------------------------------------------------
def test_maximum_rows_vs_oracle(dsa_lib, cuda_ok):
    """4096 rows, the most a config takes: a fresh 4095-token prompt (row j
    sees j + 1 keys, so rows up to 256 keys select every position) in 4-row
    score blocks plus one decode row.  The indexer's first CTAs span more
    short blocks than their block cache holds (the rest are read from global
    memory), the top-k runs 4096 one-CTA rows, and the prompt's 16-row slots
    form prefill groups.  Sampled rows' scores, selections and outputs match
    the oracle; the grouped rows are the ones the stated rule picks."""
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    inp = W.generate(7)
    wl = inp["workload"]
    dev = DeviceStep(inp, flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    assert rows["num_rows"] == 4096
    scores = dev.views["scores"].cpu().numpy()
    idx = dev.views["topk_idx"].cpu().numpy()
    out = dev.t["out"].float().cpu().numpy().astype(np.float64)
    qi = O.bf16_bits_to_f64(inp["q_idx"])
    q = O.bf16_bits_to_f64(inp["q"])
    for r in (0, 1, 2, 3, 4, 127, 255, 256, 257, 1023, 2048, 2049, 3001, 4093, 4094, 4095):
        L, req = int(rows["row_len"][r]), int(rows["row_req"][r])
        keys, sc = O.index_keys(inp, req, L)
        want = O.indexer_scores_row(qi[r], inp["w"][r], keys, sc)
        tol = 2e-2 * np.abs(want) + 2e-2 * np.sqrt(np.mean(want ** 2))
        assert (np.abs(scores[r, :L] - want) <= tol).all(), r
        assert np.array_equal(idx[r], O.topk_row(scores[r], L, wl.topk)), r
        sel = idx[r][idx[r] >= 0]
        assert sel.size == min(L, wl.topk), r
        k, v = O.kv_rows(inp, req, sel)
        o, _ = O.attention_row(q[r], k, v, wl.sm_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[r], o, atol=1e-2, rtol=2e-2, err_msg=f"row {r}")
    groups = _group_slots(rows["row_req"], rows["row_len"], idx, wl)
    assert len(groups) > 200
    lay = dsa_lib.dsa_workspace_layout(dev.cfg)
    grouped = dev.workspace[lay["group"]:lay["group"] + 4 * wl.max_rows].view(torch.int32).cpu().numpy()
    want_grouped = np.zeros(wl.max_rows, np.int32)
    for m, _ in groups.values():
        want_grouped[m] = 1
    assert np.array_equal(grouped, want_grouped)
