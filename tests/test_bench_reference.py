"""The reference arm's JSON line (the CPU oracle timed on the host), run on
the tiny workload so it takes seconds and needs no GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line_contract():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "0", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # one JSON line, nothing else on stdout that looks like one
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["unit"] == "us" and d["higher_is_better"] is False and d["value"] > 0
    assert abs(d["ms_per_step"] * 1e3 - d["value"]) < 1e-6 * d["value"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["sample"]
    # the host is stated: its CPUs, the ones used, and the model
    assert cb["cores"] == cb["threads"] == min(cb["usable_cpus"], 2)  # the tiny step has 2 rows
    assert cb["cpu_count"] >= cb["usable_cpus"] >= 1 and "cpu_model" in cb
    assert cb["one_thread"]["threads"] == 1 and cb["one_thread"]["value"] > 0
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "tiny_decode_b2" in d["config"]["workload"]


def _bench():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_cpu_sample_rows_spread_over_lengths():
    import numpy as np
    b = _bench()
    L = np.array([5, 1, 9, 0, 3, 7, 2, 8])  # row 3 is a pad row
    # sorted by length: rows 1, 6, 4, 0, 5, 7, 2 (lengths 1, 2, 3, 5, 7, 8, 9)
    assert b.sample_rows(L, 8, 2) == [6, 7]     # the middles of the lower and upper halves
    assert b.sample_rows(L, 8, 1) == [0]        # the median length
    assert b.sample_rows(L, 8, 7) == [0, 1, 2, 4, 5, 6, 7]
    assert b.sample_rows(L, 8, 20) == [0, 1, 2, 4, 5, 6, 7]   # never a pad row, never twice
    assert b.sample_rows(np.zeros(4, int), 4, 2) == []


def test_cpu_sample_is_the_rows_own_work():
    """The sampled rows' sub-problem gives the oracle the same results for
    those rows as the full step (same scores, selection and output)."""
    import numpy as np
    from oracle import dsa_oracle as O
    from sparse_attention_decode_paged_gb300 import workloads as W
    b = _bench()
    inp = W.generate(3, with_kv=True)
    wl = inp["workload"]
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    picks = [0, 60, 300]  # a decode row and two prefill rows of the mixed step
    sub_wl, arrays = b.cpu_sample(inp, rows, picks)
    sub = dict(arrays, workload=sub_wl, num_pages=int(arrays["idx_cache"].shape[0]))
    sub.setdefault("idx_scale", None)
    got = O.step(sub)
    for j, r in enumerate(picks):
        L = int(rows["row_len"][r])
        assert got["rows"]["row_len"][j] == L
        keys, sc = O.index_keys(inp, int(rows["row_req"][r]), L)
        want = O.indexer_scores_row(O.bf16_bits_to_f64(inp["q_idx"][r]), inp["w"][r], keys, sc)
        assert np.array_equal(got["scores"][j, :L], want)
        sel = O.topk_row(want, L, wl.topk)
        assert np.array_equal(got["topk_idx"][j], sel)
        k, v = O.kv_rows(inp, int(rows["row_req"][r]), sel[sel >= 0])
        o, _ = O.attention_row(O.bf16_bits_to_f64(inp["q"][r]), k, v, wl.sm_scale, wl.num_kv_heads)
        assert np.array_equal(got["out"][j], o)
