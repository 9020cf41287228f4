"""Plain, slow fp64 CPU oracle of the DSA decode/prefill step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the benchmark's
CPU-baseline / reference arm use it.  It shares no code with the CUDA path
(the library under sparse_attention_decode_paged_gb300/csrc); the only module
both sides import is the seeded input generator, which holds no arithmetic
of the method.

Source of truth: Megatron-LM PR #7211 (dynamic-inference DSA over GQA with
paged caches).  The PR page describes the method in its commit messages;
they are cited here as "commit message N" in the order the page lists them, and the closing summary as the "What does
this PR do?" section.  The indexer formula itself, score[t] =
sum_h w_h * ReLU(q_h . k_t) times a per-token key scale, is the standard
lightning-indexer score the PR's indexer kernels compute; the page names the
scores but does not print the formula.

Readings taken where the page is silent:
  * one index key per token, shared by all indexer heads;
  * a row's causal prefix includes its own token: length = position + 1;
  * equal scores are ranked by lower position; NaN ranks below -inf but is
    still a candidate; any position inside the length outranks padding;
  * if top-k >= length, every position is selected; unused slots are -1;
    selected positions are returned in ascending order;
  * the softmax scale is 1/sqrt(head_dim); an empty selection yields a zero
    output and lse = -inf.

Parity status per function (pins live in tests/test_oracle_pins.py):
  bf16_bits_to_f64, e4m3_to_f64   pinned (torch's own conversions, all codes)
  build_rows                      pinned (hand-worked fixture + invariants)
  indexer_scores                  pinned (hand-worked fixture, closed forms,
                                  page-permutation and poison invariance)
  topk                            pinned (subset brute force, torch.topk on
                                  distinct values, tie fixture)
  attention                       pinned (torch SDPA fp64 when k >= length,
                                  single key reproduces V, invariances)
  split_partials / merge          pinned (split+merge == unsplit, scipy
                                  logsumexp)
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------------------
# element decoders
# ----------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly.

    bf16 is the top half of an IEEE binary32, so the value is the binary32
    whose high 16 bits are the pattern and whose low 16 bits are zero.
    """
    b = np.asarray(bits).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 codes (uint8) -> float64, by the format's definition.

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent field 0
    encodes subnormals m/8 * 2^-6; exponent 15 with mantissa 7 encodes NaN
    (S.1111.111); there is no infinity, so 0x7E / 0xFE are +-448.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * np.exp2(-6.0)
    val = np.where(e == 0, sub, normal) * sign
    return np.where((e == 15) & (m == 7), np.nan, val)


# ----------------------------------------------------------------------------
# rows and score blocks (commit message 2: every query token is a row)
# ----------------------------------------------------------------------------
def build_rows(cache_len, new_tokens, max_rows: int, block_rows: int):
    """One row per query token of the step, padded to max_rows slots.

    Commit message 2 of the PR: every query token, decode or prefill, is a
    row (request, causal length) routed to the top-k of its causal prefix;
    score blocks are runs of consecutive rows of one request.  Request b has
    cache length C_b after this step's n_b tokens were appended, so its row
    j (0 <= j < n_b) sits at position C_b - n_b + j and sees the prefix of
    length C_b - n_b + j + 1.  Pad slots have request 0 and length 0.
    Blocks cut each request's rows into runs of at most block_rows.
    """
    cache_len = [int(x) for x in cache_len]
    new_tokens = [int(x) for x in new_tokens]
    if len(cache_len) != len(new_tokens):
        raise ValueError("cache_len and new_tokens differ in length")
    row_req = np.zeros(max_rows, np.int32)
    row_len = np.zeros(max_rows, np.int32)
    row_pos = np.zeros(max_rows, np.int32)
    block_first = np.zeros(max_rows, np.int32)
    block_nrows = np.zeros(max_rows, np.int32)
    r = 0
    nb = 0
    for b, (c, n) in enumerate(zip(cache_len, new_tokens)):
        if n < 0 or c < n:
            raise ValueError(f"request {b}: cache length {c} < new tokens {n}")
        if r + n > max_rows:
            raise ValueError("more rows than static slots")
        first = r
        for j in range(n):
            row_req[r] = b
            row_pos[r] = c - n + j
            row_len[r] = c - n + j + 1
            r += 1
        j = 0
        while j < n:
            cnt = min(block_rows, n - j)
            block_first[nb] = first + j
            block_nrows[nb] = cnt
            nb += 1
            j += cnt
    return dict(row_req=row_req, row_len=row_len, row_pos=row_pos,
                block_first=block_first, block_nrows=block_nrows,
                num_rows=r, num_blocks=nb)


# ----------------------------------------------------------------------------
# paged cache access
# ----------------------------------------------------------------------------
def token_slots(page_table, req: int, length: int, page_size: int):
    """(physical page, slot in page) of logical positions 0..length-1.

    Paged KV (the PR's summary section): logical position t of a request
    lives in its page page_table[req][t // P] at slot t % P.
    """
    t = np.arange(length, dtype=np.int64)
    pages = np.asarray(page_table)[req, t // page_size].astype(np.int64)
    if length and (pages < 0).any():
        raise ValueError("page table entry -1 inside a row's length")
    return pages, t % page_size


def index_keys(inp, req: int, length: int):
    """Decoded index keys [length, idx_dim] (fp64) and per-token scales."""
    wl = inp["workload"]
    pages, slots = token_slots(inp["page_table"], req, length, wl.page_size)
    raw = inp["idx_cache"][pages, slots]
    if inp.get("idx_scale") is None:
        return bf16_bits_to_f64(raw), np.ones(length)
    return e4m3_to_f64(raw), inp["idx_scale"][pages, slots].astype(np.float64)


# ----------------------------------------------------------------------------
# lightning indexer (commit message 1: indexer scores up to each length)
# ----------------------------------------------------------------------------
def indexer_scores_row(q_idx_r, w_r, keys, scales):
    """score[t] = s_t * sum_h w_h * max(0, q_h . k_t), for one row.

    q_idx_r [H_I, D_I] fp64, w_r [H_I], keys [L, D_I] fp64, scales [L].
    One key per token shared by all indexer heads; s_t = 1 for bf16 keys.
    """
    dots = np.asarray(q_idx_r, np.float64) @ np.asarray(keys, np.float64).T  # [H_I, L]
    relu = np.maximum(dots, 0.0)
    return (np.asarray(w_r, np.float64) @ relu) * np.asarray(scales, np.float64)


def indexer_scores(inp, rows):
    """Scores [max_rows, score_width] (fp64); NaN outside each row's length.

    Commit message 1: each row is scored only up to its own length; the
    positions past it are neither read nor written (left NaN here).
    """
    wl = inp["workload"]
    out = np.full((wl.max_rows, wl.score_width), np.nan)
    qi = bf16_bits_to_f64(inp["q_idx"])
    for r in range(rows["num_rows"]):
        L = int(rows["row_len"][r])
        if L == 0:
            continue
        keys, scales = index_keys(inp, int(rows["row_req"][r]), L)
        out[r, :L] = indexer_scores_row(qi[r], inp["w"][r], keys, scales)
    return out


# ----------------------------------------------------------------------------
# length-aware top-k (commit messages 1, 6 and 10)
# ----------------------------------------------------------------------------
def topk_row(scores_row, length: int, k: int):
    """Positions of the k best scores among 0..length-1, ascending, -1 padded.

    Commit message 1: selection reads a row only up to its length.  Commit
    message 10: a position inside the length whose score is -inf still beats
    every position past the length.  Order: higher
    score first, equal scores by lower position, NaN below every number.
    If k >= length every position is selected.
    """
    s = np.asarray(scores_row[:length], dtype=np.float64)
    t = np.arange(length)
    isnan = np.isnan(s)
    neg = np.where(isnan, 0.0, -s)
    order = np.lexsort((t, neg, isnan))  # primary: not NaN; then -score; then t
    chosen = np.sort(order[:min(k, length)])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.size] = chosen
    return out


def topk(scores, row_len, k: int):
    scores = np.asarray(scores)
    R = scores.shape[0]
    out = np.full((R, k), -1, dtype=np.int32)
    for r in range(R):
        L = int(row_len[r])
        if L:
            out[r] = topk_row(scores[r], L, k)
    return out


# ----------------------------------------------------------------------------
# sparse GQA attention over the selected set (commit messages 1 and 8)
# ----------------------------------------------------------------------------
def kv_rows(inp, req: int, positions):
    """K and V rows [n, Hkv, D] (fp64) of a request's logical positions."""
    wl = inp["workload"]
    pos = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(inp["page_table"])[req, pos // wl.page_size].astype(np.int64)
    if pos.size and (pages < 0).any():
        raise ValueError("selected position outside the request's pages")
    slots = pos % wl.page_size
    return (bf16_bits_to_f64(inp["k_cache"][pages, slots]),
            bf16_bits_to_f64(inp["v_cache"][pages, slots]))


def attention_row(q_r, k_sel, v_sel, sm_scale: float, num_kv_heads: int):
    """Softmax attention of one row over its selected keys, fp64.

    q_r [Hq, D]; k_sel, v_sel [n, Hkv, D].  Query head h reads KV head
    h // (Hq/Hkv) (all heads of a KV group share the group's selected keys,
    commit message 1).  x_t = sm_scale * q_h . k_t; out_h = sum_t p_t v_t
    with p the softmax of x over the selected set, probabilities kept in full
    precision before the value reduction (commit message 8).
    Returns (out [Hq, D], lse [Hq]); an empty set gives zeros and -inf.
    """
    q_r = np.asarray(q_r, np.float64)
    Hq, D = q_r.shape
    G = Hq // num_kv_heads
    out = np.zeros((Hq, D))
    lse = np.full(Hq, -np.inf)
    if k_sel.shape[0] == 0:
        return out, lse
    for h in range(Hq):
        g = h // G
        x = sm_scale * (k_sel[:, g, :] @ q_r[h])
        m = x.max()
        e = np.exp(x - m)
        l = e.sum()
        out[h] = (e @ v_sel[:, g, :]) / l
        lse[h] = m + np.log(l)
    return out, lse


def attention(inp, rows, topk_idx):
    """Output [max_rows, Hq, D] and lse [max_rows, Hq] over given selections."""
    wl = inp["workload"]
    q = bf16_bits_to_f64(inp["q"])
    out = np.zeros((wl.max_rows, wl.num_q_heads, wl.head_dim))
    lse = np.full((wl.max_rows, wl.num_q_heads), -np.inf)
    for r in range(rows["num_rows"]):
        L = int(rows["row_len"][r])
        if L == 0:
            continue
        sel = np.asarray(topk_idx[r])
        sel = sel[sel >= 0]
        k_sel, v_sel = kv_rows(inp, int(rows["row_req"][r]), sel)
        out[r], lse[r] = attention_row(q[r], k_sel, v_sel, wl.sm_scale, wl.num_kv_heads)
    return out, lse


# ----------------------------------------------------------------------------
# split partials and flash-decoding merge (commit messages 1 and 6)
# ----------------------------------------------------------------------------
def split_bounds(n_sel: int, num_splits: int):
    """Split s covers selected slots [s*n/S, (s+1)*n/S) (integer division)."""
    return [((s * n_sel) // num_splits, ((s + 1) * n_sel) // num_splits)
            for s in range(num_splits)]


def split_partials_row(q_r, k_sel, v_sel, sm_scale, num_kv_heads, num_splits):
    """Unnormalised per-split softmax state (m, l, acc) for one row.

    Commit message 1 splits the top-k slots across programs; each split keeps
    m = max x, l = sum e^(x-m), acc = sum e^(x-m) v over its slots.  An empty
    split is (m=-inf, l=0, acc=0).
    """
    q_r = np.asarray(q_r, np.float64)
    Hq, D = q_r.shape
    G = Hq // num_kv_heads
    m = np.full((Hq, num_splits), -np.inf)
    l = np.zeros((Hq, num_splits))
    acc = np.zeros((Hq, num_splits, D))
    for s, (a, b) in enumerate(split_bounds(k_sel.shape[0], num_splits)):
        if b <= a:
            continue
        for h in range(Hq):
            g = h // G
            x = sm_scale * (k_sel[a:b, g, :] @ q_r[h])
            m[h, s] = x.max()
            e = np.exp(x - m[h, s])
            l[h, s] = e.sum()
            acc[h, s] = e @ v_sel[a:b, g, :]
    return m, l, acc


def merge(m, l, acc):
    """Flash-decoding merge of split partials (commit messages 1 and 6).

    m, l [..., S]; acc [..., S, D].  m* = max_s m_s, l* = sum_s l_s e^(m_s-m*),
    out = sum_s acc_s e^(m_s-m*) / l*; splits with l = 0 contribute nothing and
    an all-empty input gives out = 0, lse = -inf.  lse = m* + ln l*.
    """
    m = np.asarray(m, np.float64)
    l = np.asarray(l, np.float64)
    acc = np.asarray(acc, np.float64)
    mstar = m.max(axis=-1)
    safe = np.where(np.isfinite(mstar), mstar, 0.0)
    f = np.where(l > 0, np.exp(np.where(l > 0, m, 0.0) - safe[..., None]), 0.0)
    lstar = (l * f).sum(axis=-1)
    num = (acc * f[..., None]).sum(axis=-2)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(lstar[..., None] > 0, num / np.where(lstar > 0, lstar, 1.0)[..., None], 0.0)
        lse = np.where(lstar > 0, safe + np.log(np.where(lstar > 0, lstar, 1.0)), -np.inf)
    return out, lse


# ----------------------------------------------------------------------------
# the whole step
# ----------------------------------------------------------------------------
def step(inp, rows=None):
    """rows -> indexer -> top-k -> attention, all in fp64 (unsplit)."""
    wl = inp["workload"]
    if rows is None:
        rows = build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    scores = indexer_scores(inp, rows)
    idx = topk(scores, rows["row_len"], wl.topk)
    out, lse = attention(inp, rows, idx)
    return dict(rows=rows, scores=scores, topk_idx=idx, out=out, lse=lse)
