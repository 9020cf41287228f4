"""Host-side checks of the C-ABI (no GPU work is launched here)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from oracle import dsa_oracle as O
from sparse_attention_decode_paged_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_path():
    names = _declared()
    for n in ("dsa_build_rows", "dsa_indexer_scores", "dsa_topk", "dsa_sparse_attn",
              "dsa_merge", "dsa_step"):
        assert n in names


def test_library_exports_every_declared_symbol(dsa_lib):
    lib = ctypes.CDLL(dsa_lib.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", dsa_lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dsa_\w+)", out))
    assert set(_declared()) <= exported
    assert set(dsa_lib.EXPORTED) == set(_declared())


def _cfg(dsa, **kw):
    base = dict(num_q_heads=64, num_kv_heads=8, head_dim=128, idx_heads=64, idx_dim=128,
                page_size=64, topk=2048, num_splits=8, max_rows=64, max_reqs=64,
                max_pages_per_req=512, score_width=32768, num_pages=32768)
    base.update(kw)
    return dsa.make_config(**base)


def test_validate_config_accepts_all_workloads(dsa_lib):
    for i in range(5):
        inp_wl = W.workload(i)
        cfg = dsa_lib.config_from_workload(inp_wl, 1000)
        dsa_lib.dsa_validate_config(cfg)


@pytest.mark.parametrize("bad,status", [
    (dict(num_q_heads=60), 1), (dict(num_q_heads=128), 2), (dict(head_dim=96), 2),
    (dict(idx_dim=48), 2), (dict(idx_heads=0), 2), (dict(page_size=48), 2),
    (dict(topk=0), 1), (dict(topk=40000), 1), (dict(score_width=40000), 1),
    (dict(num_splits=0), 2), (dict(block_rows=5), 2), (dict(idx_key_dtype=7), 1),
    (dict(sm_scale=-1.0), 1), (dict(sm_scale=float("inf")), 1), (dict(max_rows=0), 1),
    (dict(flags=16), 1),
])
def test_validate_config_rejects(dsa_lib, bad, status):
    cfg = _cfg(dsa_lib, **bad)
    with pytest.raises(dsa_lib.DsaError) as e:
        dsa_lib.dsa_validate_config(cfg)
    assert e.value.status == status
    assert dsa_lib._lib.dsa_last_error()  # message text is set


@pytest.mark.parametrize("i", range(5))
def test_build_rows_matches_oracle(dsa_lib, i):
    wl = W.workload(i)
    cl, nt = W.request_mix(wl)
    cfg = dsa_lib.config_from_workload(wl, 1000)
    got = dsa_lib.dsa_build_rows(cfg, cl, nt)
    want = O.build_rows(cl, nt, wl.max_rows, wl.block_rows)
    for k in ("row_req", "row_len", "row_pos", "block_first", "block_nrows", "num_rows", "num_blocks"):
        assert np.array_equal(np.asarray(got[k]), np.asarray(want[k])), k


def test_build_rows_worked_example(dsa_lib, golden_dir):
    import json
    g = json.load(open(os.path.join(golden_dir, "build_rows_worked_example.json")))
    cfg = _cfg(dsa_lib, max_rows=g["max_rows"], max_reqs=4, block_rows=g["block_rows"])
    got = dsa_lib.dsa_build_rows(cfg, g["cache_len"], g["new_tokens"])
    for k in ("row_req", "row_len", "row_pos", "block_first", "block_nrows"):
        assert got[k].tolist() == g[k], k
    assert got["num_rows"] == g["num_rows"] and got["num_blocks"] == g["num_blocks"]


def test_build_rows_random_mixes_match_oracle(dsa_lib):
    rng = np.random.default_rng(5)
    for _ in range(50):
        B = int(rng.integers(0, 12))
        new = rng.integers(0, 9, B)
        cl = new + rng.integers(0, 300, B)
        G = int(rng.integers(1, 5))
        cfg = _cfg(dsa_lib, max_rows=96, max_reqs=12, block_rows=G, score_width=4096,
                   max_pages_per_req=64, topk=64)
        got = dsa_lib.dsa_build_rows(cfg, cl, new)
        want = O.build_rows(cl, new, 96, G)
        for k in ("row_req", "row_len", "row_pos", "block_first", "block_nrows"):
            assert np.array_equal(got[k], want[k]), k


@pytest.mark.parametrize("cl,nt,status", [
    ([10, 10], [3, 11], 1),          # more new tokens than cache
    ([10], [-1], 1),                 # negative count
    ([40000], [1], 3),               # longer than score_width
    ([100] * 65, [1] * 65, 3),       # more requests than max_reqs
    ([100, 100], [40, 40], 3),       # more rows than max_rows
])
def test_build_rows_errors(dsa_lib, cl, nt, status):
    cfg = _cfg(dsa_lib)
    with pytest.raises(dsa_lib.DsaError) as e:
        dsa_lib.dsa_build_rows(cfg, cl, nt)
    assert e.value.status == status


def test_workspace_layout(dsa_lib):
    cfg = _cfg(dsa_lib)
    lay = dsa_lib.dsa_workspace_layout(cfg)
    assert lay["status"] == 0
    order = ["status", "scores", "topk_idx", "part_m", "part_l", "part_acc", "group", "key_hist", "total"]
    offs = [lay[k] for k in order]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay["topk_idx"] - lay["scores"] >= 64 * 32768 * 4
    assert lay["key_hist"] - lay["part_acc"] >= 64 * 64 * 8 * 128 * 4
    assert lay["total"] - lay["key_hist"] >= 64 * 4096 * 4
    assert dsa_lib.dsa_workspace_size(cfg) == lay["total"]


def test_null_and_misaligned_pointers_are_rejected_before_launch(dsa_lib):
    lib = dsa_lib._lib
    cfg = _cfg(dsa_lib)
    c = ctypes.byref(cfg)
    vp = ctypes.c_void_p
    assert lib.dsa_topk(c, None, vp(16), vp(16), vp(16), None) == dsa_lib.DSA_ERR_INVALID_ARG
    assert b"scores" in lib.dsa_last_error()
    assert lib.dsa_topk(c, vp(16), vp(16), vp(24), vp(16), None) == dsa_lib.DSA_ERR_INVALID_ARG
    assert b"aligned" in lib.dsa_last_error()
    assert lib.dsa_merge(c, vp(16), vp(16), vp(16), None, None, None) == dsa_lib.DSA_ERR_INVALID_ARG
    assert lib.dsa_step(c, None, vp(16), None) == dsa_lib.DSA_ERR_INVALID_ARG
    bad = _cfg(dsa_lib, head_dim=80)
    assert lib.dsa_sparse_attn(ctypes.byref(bad), *([vp(16)] * 11), None) == dsa_lib.DSA_ERR_UNSUPPORTED
    # fp8 keys need a scale pointer
    f8 = _cfg(dsa_lib, idx_key_dtype=1)
    args = [vp(16)] * 3 + [None] + [vp(16)] * 7 + [None]
    assert lib.dsa_indexer_scores(ctypes.byref(f8), *args) == dsa_lib.DSA_ERR_INVALID_ARG
    assert b"idx_scale" in lib.dsa_last_error()


def test_read_probe_library_exports(dsa_lib):
    """The benchmark's read-only stream probe is built beside the library
    (its own .so, not part of the DSA path) and exports its one entry."""
    import ctypes
    from sparse_attention_decode_paged_gb300 import build as B

    assert os.path.exists(B.PROBE_LIB)
    lib = ctypes.CDLL(B.PROBE_LIB)
    assert hasattr(lib, "dsa_probe_read_pages")
    # host-side argument checks run before any device call
    lib.dsa_probe_read_pages.restype = ctypes.c_int
    assert lib.dsa_probe_read_pages(None, None, 1, 16, None, 1, 256, None) != 0


def test_kv_interleaved_requires_adjacent_v(dsa_lib):
    """With DSA_FLAG_KV_INTERLEAVED the V pointer must be the K pointer plus
    one K row; anything else is rejected before any launch."""
    cfg = dsa_lib.make_config(num_q_heads=64, num_kv_heads=8, head_dim=128, idx_heads=64, idx_dim=128,
                              page_size=64, topk=2048, num_splits=8, max_rows=64, max_reqs=64,
                              max_pages_per_req=512, score_width=32768, num_pages=32768, block_rows=1,
                              idx_key_dtype=0, flags=dsa_lib.DSA_FLAG_KV_INTERLEAVED)
    lib = ctypes.CDLL(dsa_lib.LIB_PATH)
    lib.dsa_sparse_attn.restype = ctypes.c_int
    base = 0x10000000
    p = [ctypes.c_void_p(base + 0x100000 * k) for k in range(12)]
    row = 8 * 128 * 2
    bad = lib.dsa_sparse_attn(ctypes.byref(cfg), p[0], p[1], ctypes.c_void_p(p[1].value + row + 16), p[3], p[4],
                              p[5], p[6], p[7], p[8], p[9], p[10], None)
    assert bad == dsa_lib.DSA_ERR_INVALID_ARG
    assert "KV_INTERLEAVED" in lib_last_error(lib)


def lib_last_error(lib):
    lib.dsa_last_error.restype = ctypes.c_char_p
    return lib.dsa_last_error().decode()


# ----------------------------------------------------------------------------
# dsa_suggest_num_splits: the documented rule, on the host
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("rows,topk,sms,want", [
    (64, 2048, 152, 19),    # 4 programs per resident CTA: round(4 * 304 / 64)
    (8, 512, 152, 16),      # capped at topk / 32, one wave instead
    (16, 2048, 152, 19),    # round(4 * 304 / 16) = 76 > cap 64: one wave, 304 // 16
    (1024, 2048, 152, 1),
    (2, 16, 152, 1),        # topk / 32 = 0: at least one split
    (64, 2048, 76, 10),     # half the SMs: round(4 * 152 / 64) = round(9.5)
    (4096, 2048, 152, 1),
    (1, 4096, 152, 64),     # cap at 64
])
def test_suggest_num_splits_rule(rows, topk, sms, want, dsa_lib):
    cfg = _cfg(dsa_lib, max_rows=rows, max_reqs=rows, topk=topk)
    assert dsa_lib.dsa_suggest_num_splits(cfg, sms) == want
    # what it suggests is itself a valid config
    dsa_lib.dsa_validate_config(_cfg(dsa_lib, max_rows=rows, max_reqs=rows, topk=topk, num_splits=want))


def test_suggest_num_splits_matches_the_workloads(dsa_lib):
    """The parity workloads use the suggestion for a 152-SM GB300 (the tiny
    case keeps 2 splits so the merge runs on it)."""
    for i in (1, 2, 3, 4, 6):
        wl = W.workload(i)
        assert dsa_lib.dsa_suggest_num_splits(dsa_lib.config_from_workload(wl, 1000), 152) == wl.num_splits


def test_suggest_num_splits_needs_a_device_or_a_count(dsa_lib):
    import torch
    cfg = _cfg(dsa_lib)
    if torch.cuda.is_available():
        assert 1 <= dsa_lib.dsa_suggest_num_splits(cfg) <= 64
    else:
        with pytest.raises(dsa_lib.DsaError) as e:
            dsa_lib.dsa_suggest_num_splits(cfg)
        assert e.value.status == dsa_lib.DSA_ERR_CUDA


# ----------------------------------------------------------------------------
# the harness's input / output arenas (host logic, CPU tensors)
# ----------------------------------------------------------------------------
def test_arena_views_are_aligned_disjoint_and_shaped():
    import torch
    from sparse_attention_decode_paged_gb300.harness import DEVICE_ROW_KEYS, _arena

    R = 3  # a row count whose int32 arrays are not a multiple of 16 bytes
    parts = [(k, torch.int32, (R,)) for k in DEVICE_ROW_KEYS] + [
        ("page_table", torch.int32, (3, 5)), ("q_idx", torch.bfloat16, (R, 4, 32)),
        ("w", torch.float32, (R, 4)), ("q", torch.bfloat16, (R, 4, 64))]
    buf, views = _arena(parts, "cpu")
    spans = []
    for name, dtype, shape in parts:
        v = views[name]
        assert v.dtype == dtype and tuple(v.shape) == shape and v.is_contiguous()
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0, name  # every view meets the library's 16-byte pointer rule
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))  # no overlap
    assert spans[-1][1] <= buf.numel()
    # writes through one view land in the buffer a single copy moves
    views["q"].fill_(1.5)
    views["row_len"].copy_(torch.tensor([7, 8, 9], dtype=torch.int32))
    again = {n: buf[v.data_ptr() - buf.data_ptr():][:v.numel() * v.element_size()] for n, v in views.items()}
    assert torch.equal(again["row_len"].view(torch.int32), torch.tensor([7, 8, 9], dtype=torch.int32))
    assert bool((again["q"].view(torch.bfloat16) == 1.5).all())


def test_no_prefill_groups_flag_drops_the_group_region(dsa_lib):
    """DSA_FLAG_NO_PREFILL_GROUPS: no group region in the workspace and no
    group term in the split suggestion."""
    wl = W.workload(3)
    cfg = dsa_lib.config_from_workload(wl, 1000)
    lay = dsa_lib.dsa_workspace_layout(cfg)
    assert lay["key_hist"] > lay["group"]
    cfg2 = dsa_lib.config_from_workload(wl, 1000, flags=dsa_lib.DSA_FLAG_NO_PREFILL_GROUPS)
    lay2 = dsa_lib.dsa_workspace_layout(cfg2)
    assert lay2["group"] == lay2["key_hist"] and lay2["total"] < lay["total"]
    assert dsa_lib.dsa_suggest_num_splits(cfg, 152) == 4
    assert dsa_lib.dsa_suggest_num_splits(cfg2, 152) == 1
