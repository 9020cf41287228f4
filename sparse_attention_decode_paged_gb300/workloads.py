"""Seeded synthetic inputs for the DSA decode/prefill step.

This module only draws numbers.  It holds none of the method's arithmetic:
no row building, no scoring, no selection and no attention.  It is shared by
the CUDA path's tests and benchmark and by the CPU oracle's tests, so both
sides see identical inputs.

Seven workloads, numbered by their seed:

  0  tiny decode   B=2, lengths {37, 200}, page 16, indexer 4x32, top-k 16,
                   4 q heads / 1 KV head, head dim 64
  1  decode        B=8, lengths U{512..4096}, page 64, indexer 64x128 bf16,
                   top-k 512, 64 q / 8 KV heads, head dim 128
  2  decode B64    B=64, all lengths 32768, page 64, indexer 64x128 bf16,
                   top-k 2048, 64 q / 8 KV heads, head dim 128
  3  mixed         48 decode rows (lengths U{1024..32768}) + one chunked
                   prefill request of 512 tokens at prefix offset 8192,
                   score blocks of up to 4 rows, 1024 static row slots
  4  long fp8      B=16, lengths U{1024..131072}, indexer keys fp8 e4m3
                   with a per-token fp32 scale, top-k 2048
  5  1M prefill    a 64-token prefill chunk at 1M (1,048,576) keys of
                   context, one decode request just under 1M and one
                   short decode request; score blocks of up to 4 rows,
                   80 row slots, indexer 64x128 bf16, top-k 2048, 8 q /
                   1 KV head, head dim 128 (the score-window case of a
                   prefill chunk at 1M context, with one KV head so the
                   caches stay a few GB)
  6  correlated    workload 3's shape and request mix, with the
                   indexer queries of each 16-row slot [16i, 16i+16) drawn
                   around one shared base vector (q_idx = base_i + 0.25 e_r),
                   so consecutive prefill tokens select overlapping keys

The problem statement these follow is Megatron-LM PR #7211 (DSA over GQA
with paged KV caches): every query token is a row that routes to the top-k
of its causal prefix; K/V and index keys live in paged caches addressed
through per-request page tables.

Draw order for every workload (each tensor gets its own child seed, so the
order fixes the stream): lengths -> page permutation -> q_idx -> w ->
index keys (-> scales) -> q -> K -> V.  Large tensors are drawn in fixed
chunks, each from its own child seed, so the values do not depend on the
number of threads used to draw them.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

KEY_BF16 = 0
KEY_FP8_E4M3 = 1

_CHUNK = 1 << 22  # elements per independently seeded chunk


@dataclasses.dataclass(frozen=True)
class Workload:
    """Static shape of one workload (mirrors the library's config struct)."""

    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    idx_heads: int
    idx_dim: int
    page_size: int
    topk: int
    num_splits: int
    max_rows: int
    max_reqs: int
    max_pages_per_req: int
    score_width: int
    block_rows: int
    idx_key_dtype: int
    # request mix: per request, (cache length after this step, new tokens)
    kind: str  # "decode" | "mixed"

    @property
    def sm_scale(self) -> float:
        return float(1.0 / np.sqrt(self.head_dim))


def _wl(name, seed, **kw) -> Workload:
    return Workload(name=name, seed=seed, **kw)


# num_splits: what dsa_suggest_num_splits gives on a 152-SM GB300 (the
# tiny case keeps 2 so the merge of split partials runs on it too)
WORKLOADS = [
    _wl("tiny_decode_b2", 0, num_q_heads=4, num_kv_heads=1, head_dim=64,
        idx_heads=4, idx_dim=32, page_size=16, topk=16, num_splits=2,
        max_rows=2, max_reqs=2, max_pages_per_req=16, score_width=256,
        block_rows=1, idx_key_dtype=KEY_BF16, kind="decode"),
    _wl("decode_b8_l512_4096", 1, num_q_heads=64, num_kv_heads=8, head_dim=128,
        idx_heads=64, idx_dim=128, page_size=64, topk=512, num_splits=16,
        max_rows=8, max_reqs=8, max_pages_per_req=64, score_width=4096,
        block_rows=1, idx_key_dtype=KEY_BF16, kind="decode"),
    _wl("decode_b64_l32768_topk2048", 2, num_q_heads=64, num_kv_heads=8,
        head_dim=128, idx_heads=64, idx_dim=128, page_size=64, topk=2048,
        num_splits=19, max_rows=64, max_reqs=64, max_pages_per_req=512,
        score_width=32768, block_rows=1, idx_key_dtype=KEY_BF16, kind="decode"),
    _wl("mixed_48dec_512prefill", 3, num_q_heads=64, num_kv_heads=8,
        head_dim=128, idx_heads=64, idx_dim=128, page_size=64, topk=2048,
        num_splits=4, max_rows=1024, max_reqs=49, max_pages_per_req=512,
        score_width=32768, block_rows=4, idx_key_dtype=KEY_BF16, kind="mixed"),
    _wl("long_fp8_b16_l1024_131072", 4, num_q_heads=64, num_kv_heads=8,
        head_dim=128, idx_heads=64, idx_dim=128, page_size=64, topk=2048,
        num_splits=19, max_rows=16, max_reqs=16, max_pages_per_req=2048,
        score_width=131072, block_rows=1, idx_key_dtype=KEY_FP8_E4M3,
        kind="decode"),
    _wl("prefill64_at_1m", 5, num_q_heads=8, num_kv_heads=1, head_dim=128,
        idx_heads=64, idx_dim=128, page_size=64, topk=2048, num_splits=4,
        max_rows=80, max_reqs=3, max_pages_per_req=16384, score_width=1 << 20,
        block_rows=4, idx_key_dtype=KEY_BF16, kind="mixed"),
    _wl("mixed_correlated_48dec_512prefill", 6, num_q_heads=64, num_kv_heads=8,
        head_dim=128, idx_heads=64, idx_dim=128, page_size=64, topk=2048,
        num_splits=4, max_rows=1024, max_reqs=49, max_pages_per_req=512,
        score_width=32768, block_rows=4, idx_key_dtype=KEY_BF16, kind="mixed"),
    # the largest row count the library takes: a fresh 4095-token prompt
    # (row j sees j + 1 keys) and one decode row; 8 query heads per KV head
    # at head dim 128, so the prompt's 16-row slots form prefill groups
    _wl("prompt4095_plus_decode_max_rows", 7, num_q_heads=8, num_kv_heads=1,
        head_dim=128, idx_heads=16, idx_dim=64, page_size=64, topk=256,
        num_splits=2, max_rows=4096, max_reqs=2, max_pages_per_req=128,
        score_width=8192, block_rows=4, idx_key_dtype=KEY_BF16, kind="mixed"),
]


def workload(i: int) -> Workload:
    return WORKLOADS[i]


# ----------------------------------------------------------------------------
# random streams
# ----------------------------------------------------------------------------
_TENSOR_IDS = {
    "lengths": 0, "pages": 1, "q_idx": 2, "w": 3, "idx_keys": 4,
    "idx_scale": 5, "q": 6, "k": 7, "v": 8, "extra": 9,
}


def _rng(seed: int, name: str, chunk: int | None = None) -> np.random.Generator:
    key = (_TENSOR_IDS[name],) if chunk is None else (_TENSOR_IDS[name], chunk)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _chunked_fill(seed: int, name: str, n: int, fill) -> np.ndarray:
    """Draw n values in fixed chunks; fill(rng, out_slice) writes one chunk."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        fill(_rng(seed, name, c), out[lo:hi])

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _normal_f32(seed, name, n, scale=1.0):
    def fill(rng, out):
        rng.standard_normal(out=out, dtype=np.float32)
        if scale != 1.0:
            out *= np.float32(scale)
    return _chunked_fill(seed, name, n, fill)


def _uniform_f32(seed, name, n):
    def fill(rng, out):
        rng.random(out=out, dtype=np.float32)
    return _chunked_fill(seed, name, n, fill)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even.

    Input generation only: the synthetic tensors are "fp32 drawn, stored in
    bf16".  No NaN or inf is ever drawn here.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    flat_in = x.reshape(-1).view(np.uint32)
    flat_out = out.reshape(-1)
    n = flat_in.size
    step = 1 << 24

    def work(lo):
        b = flat_in[lo:lo + step].astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
        flat_out[lo:lo + step] = b.astype(np.uint16)

    starts = range(0, n, step)
    if n > step:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, starts))
    else:
        for lo in starts:
            work(lo)
    return out


def quantize_e4m3_per_token(k: np.ndarray):
    """Per-token fp8 e4m3 keys: scale = amax/448, code = RNE cast of k/scale.

    k: float32 [..., D].  Returns (codes uint8 [..., D], scale float32 [...]).
    Input generation only (the cache writer upstream of the method).  Uses
    torch's float8_e4m3fn cast; |k/scale| <= 448 so nothing saturates.
    """
    import torch

    amax = np.abs(k).max(axis=-1)
    scale = (np.maximum(amax, np.float32(1e-12)) / np.float32(448.0)).astype(np.float32)
    ratio = (k / scale[..., None]).astype(np.float32)
    codes = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes.copy(), scale


# ----------------------------------------------------------------------------
# request mixes
# ----------------------------------------------------------------------------
def request_mix(wl: Workload):
    """Per-request (cache length after this step, new tokens this step)."""
    rng = _rng(wl.seed, "lengths")
    if wl.seed == 0:
        cache_len = np.array([37, 200], dtype=np.int32)
        new = np.ones(2, dtype=np.int32)
    elif wl.seed == 1:
        cache_len = rng.integers(512, 4096, size=8, endpoint=True).astype(np.int32)
        new = np.ones(8, dtype=np.int32)
    elif wl.seed == 2:
        cache_len = np.full(wl.max_reqs, 32768, dtype=np.int32)
        new = np.ones(wl.max_reqs, dtype=np.int32)
    elif wl.seed in (3, 6):
        dec = rng.integers(1024, 32768, size=48, endpoint=True).astype(np.int32)
        cache_len = np.concatenate([dec, np.array([8192 + 512], dtype=np.int32)])
        new = np.concatenate([np.ones(48, dtype=np.int32), np.array([512], dtype=np.int32)])
    elif wl.seed == 4:
        cache_len = rng.integers(1024, 131072, size=16, endpoint=True).astype(np.int32)
        new = np.ones(16, dtype=np.int32)
    elif wl.seed == 7:
        dec = int(rng.integers(4096, 8192, endpoint=True))
        cache_len = np.array([4095, dec], dtype=np.int32)
        new = np.array([4095, 1], dtype=np.int32)
    elif wl.seed == 5:
        near = int(rng.integers((1 << 20) - 4096, 1 << 20, endpoint=True))
        short = int(rng.integers(4096, 65536, endpoint=True))
        cache_len = np.array([near, 1 << 20, short], dtype=np.int32)
        new = np.array([1, 64, 1], dtype=np.int32)
    else:
        raise ValueError(wl.seed)
    return cache_len, new


def page_tables(wl: Workload, cache_len: np.ndarray):
    """Random physical page permutation; unused table entries are -1.

    Returns (page_table int32 [max_reqs, max_pages_per_req], num_pages).
    Request b owns ceil(cache_len[b]/P) pages taken in order from one
    random permutation of the whole pool, so the pool is exactly full.
    """
    P = wl.page_size
    npages = (cache_len.astype(np.int64) + P - 1) // P
    total = int(npages.sum())
    perm = _rng(wl.seed, "pages").permutation(total).astype(np.int32)
    pt = np.full((wl.max_reqs, wl.max_pages_per_req), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n]
        off += int(n)
    return pt, total


def generate(wl: Workload | int, *, with_kv: bool = True):
    """All inputs of one step as host numpy arrays (bf16 as uint16 bits).

    Keys of the dict:
      cache_len, new_tokens  int32 [B]
      page_table             int32 [max_reqs, max_pages_per_req]
      num_pages              int
      q_idx                  uint16 (bf16) [max_rows, idx_heads, idx_dim]
      w                      float32 [max_rows, idx_heads]
      idx_cache              uint16 (bf16) or uint8 (e4m3) [NP, P, idx_dim]
      idx_scale              float32 [NP, P] (fp8 keys) or None
      q                      uint16 (bf16) [max_rows, Hq, D]
      k_cache, v_cache       uint16 (bf16) [NP, P, Hkv, D]  (if with_kv)
    """
    if isinstance(wl, int):
        wl = workload(wl)
    s = wl.seed
    cache_len, new = request_mix(wl)
    pt, npool = page_tables(wl, cache_len)
    R, HI, DI = wl.max_rows, wl.idx_heads, wl.idx_dim
    P = wl.page_size
    out = dict(workload=wl, cache_len=cache_len, new_tokens=new,
               page_table=pt, num_pages=npool)
    qi = _normal_f32(s, "q_idx", R * HI * DI).reshape(R, HI, DI)
    if s == 6:  # each 16-row slot's queries around one shared base vector
        base = _normal_f32(s, "extra", (R + 15) // 16 * HI * DI).reshape(-1, HI, DI)
        qi = np.repeat(base, 16, axis=0)[:R] + np.float32(0.25) * qi
    out["q_idx"] = round_to_bf16_bits(qi).reshape(R, HI, DI)
    if s == 0:
        out["w"] = _uniform_f32(s, "w", R * HI).reshape(R, HI)
    else:
        out["w"] = _normal_f32(s, "w", R * HI, scale=1.0 / 8.0).reshape(R, HI)
    nkey = npool * P * DI
    kf = _normal_f32(s, "idx_keys", nkey).reshape(npool, P, DI)
    if wl.idx_key_dtype == KEY_BF16:
        out["idx_cache"] = round_to_bf16_bits(kf)
        out["idx_scale"] = None
    else:
        codes, scale = quantize_e4m3_per_token(kf)
        out["idx_cache"] = codes
        out["idx_scale"] = scale
    del kf
    Hq, Hkv, D = wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    out["q"] = round_to_bf16_bits(_normal_f32(s, "q", R * Hq * D)).reshape(R, Hq, D)
    if with_kv:
        n = npool * P * Hkv * D
        out["k_cache"] = round_to_bf16_bits(_normal_f32(s, "k", n)).reshape(npool, P, Hkv, D)
        out["v_cache"] = round_to_bf16_bits(_normal_f32(s, "v", n)).reshape(npool, P, Hkv, D)
    return out
