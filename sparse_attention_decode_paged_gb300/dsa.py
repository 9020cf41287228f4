"""Python binding of libdsa.so (include/dsa.h): argument marshalling only.

Every function has the name of the C entry point it calls and takes torch
tensors where the C call takes device pointers.  Each checks device,
dtype, shape and contiguity, passes raw pointers and the current CUDA stream
(or the one given), and raises DsaError on a non-OK status.  All arithmetic
of the step runs in the library's CUDA kernels; there is no fallback: if
libdsa.so cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa.so")

DSA_OK = 0
DSA_ERR_INVALID_ARG = 1
DSA_ERR_UNSUPPORTED = 2
DSA_ERR_CAPACITY = 3
DSA_ERR_CUDA = 4
DSA_ERR_DEVICE_BOUNDS = 5

DSA_DEV_BAD_ROW = 1 << 0
DSA_DEV_BAD_PAGE = 1 << 1
DSA_DEV_BAD_INDEX = 1 << 2
DSA_DEV_BAD_BLOCK = 1 << 3
DSA_DEV_TIMEOUT = 1 << 4
DSA_DEV_BAD_HIST = 1 << 5

DSA_KEY_BF16 = 0
DSA_KEY_FP8_E4M3 = 1

DSA_FLAG_TOPK_HISTOGRAM = 1 << 0
DSA_FLAG_KV_INTERLEAVED = 1 << 1
DSA_FLAG_TEST_WAIT_TIMEOUT = 1 << 2  # test only: one indexer wait runs out (see dsa.h)
DSA_FLAG_NO_PREFILL_GROUPS = 1 << 3  # every row takes the per-row attention

EXPORTED = (
    "dsa_validate_config", "dsa_workspace_size", "dsa_workspace_layout",
    "dsa_reset_device_status", "dsa_read_device_status", "dsa_build_rows", "dsa_score_windows",
    "dsa_suggest_num_splits",
    "dsa_indexer_scores", "dsa_indexer_scores_window", "dsa_topk", "dsa_topk_window",
    "dsa_sparse_attn", "dsa_merge", "dsa_step",
    "dsa_step_noalloc", "dsa_last_error", "dsa_version",
)


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dsa status {status}: {message}")
        self.status = status


class dsa_config_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "idx_heads", "idx_dim", "page_size",
        "topk", "num_splits", "max_rows", "max_reqs", "max_pages_per_req", "score_width",
        "num_pages", "block_rows", "idx_key_dtype")] + [("sm_scale", ctypes.c_float),
                                                        ("flags", ctypes.c_int32),
                                                        ("score_buffer_bytes", ctypes.c_int64)]


class dsa_step_args_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "page_table", "row_req", "row_len", "block_first", "block_nrows", "q_idx", "w",
        "idx_cache", "idx_scale", "q", "k_cache", "v_cache", "out", "lse")]


class dsa_workspace_layout_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "scores", "topk_idx", "part_m", "part_l", "part_acc", "group", "key_hist", "total")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m sparse_attention_decode_paged_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    cfgp = ctypes.POINTER(dsa_config_t)
    i32p = ctypes.POINTER(ctypes.c_int32)
    proto = {
        "dsa_validate_config": [cfgp],
        "dsa_workspace_size": [cfgp, ctypes.POINTER(sz)],
        "dsa_workspace_layout": [cfgp, ctypes.POINTER(dsa_workspace_layout_t)],
        "dsa_reset_device_status": [vp, vp],
        "dsa_read_device_status": [vp, ctypes.POINTER(ctypes.c_uint32), vp],
        "dsa_build_rows": [cfgp, i32] + [vp] * 7 + [i32p, i32p],
        "dsa_score_windows": [cfgp, i32p, i32p],
        "dsa_suggest_num_splits": [cfgp, i32, i32p],
        "dsa_indexer_scores": [cfgp] + [vp] * 12,
        "dsa_indexer_scores_window": [cfgp, i32, i32] + [vp] * 12,
        "dsa_topk": [cfgp] + [vp] * 5,
        "dsa_topk_window": [cfgp, i32, i32] + [vp] * 5,
        "dsa_sparse_attn": [cfgp] + [vp] * 12,
        "dsa_merge": [cfgp] + [vp] * 6,
        "dsa_step": [cfgp, ctypes.POINTER(dsa_step_args_t), vp, vp],
        "dsa_step_noalloc": [cfgp, ctypes.POINTER(dsa_step_args_t), vp, vp],
    }
    for name, args in proto.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    for name in ("dsa_last_error", "dsa_version"):
        fn = getattr(lib, name)
        fn.argtypes = []
        fn.restype = ctypes.c_char_p
    return lib


_lib = _load()


def _check(status: int):
    if status != DSA_OK:
        raise DsaError(status, _lib.dsa_last_error().decode())


def version() -> str:
    """The library's version string."""
    return _lib.dsa_version().decode()


# ----------------------------------------------------------------------------
# config
# ----------------------------------------------------------------------------
def make_config(*, num_q_heads, num_kv_heads, head_dim, idx_heads, idx_dim, page_size, topk,
                num_splits, max_rows, max_reqs, max_pages_per_req, score_width, num_pages,
                block_rows=1, idx_key_dtype=DSA_KEY_BF16, sm_scale=None, flags=0,
                score_buffer_bytes=0) -> dsa_config_t:
    """A dsa_config_t (fields as in include/dsa.h); sm_scale defaults to
    1/sqrt(head_dim).  Not validated here: see dsa_validate_config."""
    if sm_scale is None:
        sm_scale = 1.0 / float(np.sqrt(head_dim))
    return dsa_config_t(num_q_heads, num_kv_heads, head_dim, idx_heads, idx_dim, page_size, topk,
                        num_splits, max_rows, max_reqs, max_pages_per_req, score_width,
                        num_pages, block_rows, idx_key_dtype, float(sm_scale), int(flags),
                        int(score_buffer_bytes))


def config_from_workload(wl, num_pages: int, **override) -> dsa_config_t:
    """The config of a generated workload (workloads.Workload) over a pool
    of num_pages pages; keyword arguments override single fields."""
    kw = dict(num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
              idx_heads=wl.idx_heads, idx_dim=wl.idx_dim, page_size=wl.page_size,
              topk=wl.topk, num_splits=wl.num_splits, max_rows=wl.max_rows,
              max_reqs=wl.max_reqs, max_pages_per_req=wl.max_pages_per_req,
              score_width=wl.score_width, num_pages=num_pages, block_rows=wl.block_rows,
              idx_key_dtype=wl.idx_key_dtype, sm_scale=wl.sm_scale)
    kw.update(override)
    return make_config(**kw)


def dsa_validate_config(cfg: dsa_config_t) -> None:
    """Raises DsaError if the library has no kernel for this config."""
    _check(_lib.dsa_validate_config(ctypes.byref(cfg)))


def dsa_workspace_size(cfg: dsa_config_t) -> int:
    """Bytes of device workspace dsa_step needs for this config."""
    n = ctypes.c_size_t(0)
    _check(_lib.dsa_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return int(n.value)


def dsa_workspace_layout(cfg: dsa_config_t) -> dict:
    """Byte offsets of the step's intermediates inside the workspace."""
    lay = dsa_workspace_layout_t()
    _check(_lib.dsa_workspace_layout(ctypes.byref(cfg), ctypes.byref(lay)))
    return {name: int(getattr(lay, name)) for name, _ in lay._fields_}


# ----------------------------------------------------------------------------
# pointer marshalling
# ----------------------------------------------------------------------------
_BF16 = (torch.bfloat16, torch.int16)
_FP8 = (torch.float8_e4m3fn, torch.uint8)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, name, dtypes, numel=None):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name}: {t.numel()} elements < {numel} required")
    return ctypes.c_void_p(t.data_ptr())


def _ws(workspace):
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda:
        raise TypeError("workspace: expected a CUDA tensor")
    return ctypes.c_void_p(workspace.data_ptr())


def alloc_workspace(cfg: dsa_config_t, device=None) -> torch.Tensor:
    """A zeroed uint8 device buffer of dsa_workspace_size(cfg) bytes."""
    return torch.zeros(dsa_workspace_size(cfg), dtype=torch.uint8, device=device or "cuda")


def workspace_views(cfg: dsa_config_t, workspace: torch.Tensor) -> dict:
    """Typed views of the step intermediates inside a workspace (the score
    buffer holds one window of rows, all max_rows without a budget)."""
    lay = dsa_workspace_layout(cfg)
    R, W, K = cfg.max_rows, cfg.score_width, cfg.topk
    WR = dsa_score_windows(cfg)[0]
    HS = cfg.num_q_heads * cfg.num_splits

    def view(off, n, dtype, shape):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return workspace[off:off + nbytes].view(dtype).view(*shape)

    return dict(
        status=view(lay["status"], 1, torch.int32, (1,)),
        scores=view(lay["scores"], WR * W, torch.float32, (WR, W)),
        topk_idx=view(lay["topk_idx"], R * K, torch.int32, (R, K)),
        part_m=view(lay["part_m"], R * HS, torch.float32, (R, cfg.num_q_heads, cfg.num_splits)),
        part_l=view(lay["part_l"], R * HS, torch.float32, (R, cfg.num_q_heads, cfg.num_splits)),
        part_acc=view(lay["part_acc"], R * HS * cfg.head_dim, torch.float32,
                      (R, cfg.num_q_heads, cfg.num_splits, cfg.head_dim)),
    )


# ----------------------------------------------------------------------------
# entry points
# ----------------------------------------------------------------------------
def dsa_reset_device_status(workspace, stream=None) -> None:
    """Clears the workspace's sticky device status word (async on stream)."""
    _check(_lib.dsa_reset_device_status(_ws(workspace), _stream(stream)))


def dsa_read_device_status(workspace, stream=None) -> int:
    """The sticky device status word (synchronizes the stream)."""
    v = ctypes.c_uint32(0)
    st = _lib.dsa_read_device_status(_ws(workspace), ctypes.byref(v), _stream(stream))
    if st not in (DSA_OK, DSA_ERR_DEVICE_BOUNDS):
        _check(st)
    return int(v.value)


_ROW_KEYS = ("row_req", "row_len", "row_pos", "block_first", "block_nrows")


def _host_i32(a, name, n):
    """Address of a contiguous int32 host buffer of at least n elements (a
    numpy array, or a CPU torch tensor such as a pinned staging buffer)."""
    if isinstance(a, torch.Tensor):
        if a.is_cuda or a.dtype != torch.int32 or not a.is_contiguous() or a.numel() < n:
            raise ValueError(f"{name}: expected a contiguous CPU int32 tensor of >= {n} elements")
        return a.data_ptr()
    if not isinstance(a, np.ndarray) or a.dtype != np.int32 or not a.flags.c_contiguous or a.size < n:
        raise ValueError(f"{name}: expected a contiguous int32 numpy array of >= {n} elements")
    return a.ctypes.data


def dsa_build_rows(cfg: dsa_config_t, req_cache_len, req_new_tokens, out=None) -> dict:
    """Host row builder.  Inputs: int sequences.  Outputs: numpy int32 arrays
    [max_rows] keyed row_req, row_len, row_pos, block_first, block_nrows, plus
    num_rows and num_blocks.  With out = a dict of five such host buffers
    (numpy arrays or CPU torch tensors, e.g. pinned staging for the copy to
    the device) the rows are written there in place and the dict is returned
    with the two counts added."""
    cl = np.ascontiguousarray(req_cache_len, dtype=np.int32)
    nt = np.ascontiguousarray(req_new_tokens, dtype=np.int32)
    if cl.shape != nt.shape or cl.ndim != 1:
        raise ValueError("req_cache_len and req_new_tokens must be 1-D and equal in length")
    R = cfg.max_rows
    outs = {k: np.zeros(R, np.int32) for k in _ROW_KEYS} if out is None else out
    nr, nb = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(_lib.dsa_build_rows(ctypes.byref(cfg), int(cl.size), cl.ctypes.data, nt.ctypes.data,
                               *(_host_i32(outs[k], k, R) for k in _ROW_KEYS),
                               ctypes.byref(nr), ctypes.byref(nb)))
    outs["num_rows"] = int(nr.value)
    outs["num_blocks"] = int(nb.value)
    return outs


def dsa_suggest_num_splits(cfg, num_sms: int = 0) -> int:
    """A num_splits for cfg's rows and top-k on num_sms SMs (0: the current
    device's); a tuning aid, see include/dsa.h."""
    s = ctypes.c_int32()
    _check(_lib.dsa_suggest_num_splits(ctypes.byref(cfg), int(num_sms), ctypes.byref(s)))
    return int(s.value)


def dsa_score_windows(cfg) -> tuple:
    """(window_rows, num_windows) of the step's score windows."""
    wr, nw = ctypes.c_int32(), ctypes.c_int32()
    _check(_lib.dsa_score_windows(ctypes.byref(cfg), ctypes.byref(wr), ctypes.byref(nw)))
    return int(wr.value), int(nw.value)


def dsa_indexer_scores(cfg, q_idx, w, idx_cache, idx_scale, page_table, row_req, row_len,
                       block_first, block_nrows, scores, workspace, stream=None, window=None) -> None:
    """Scores of every row into scores [max_rows, score_width], or with
    window=(row_begin, row_end) of those rows only, into scores
    [row_end - row_begin, score_width] (dsa_indexer_scores_window)."""
    R = cfg.max_rows
    keyt = _FP8 if cfg.idx_key_dtype == DSA_KEY_FP8_E4M3 else _BF16
    lo, hi = (0, R) if window is None else (int(window[0]), int(window[1]))
    args = (_dev(q_idx, "q_idx", _BF16, R * cfg.idx_heads * cfg.idx_dim),
            _dev(w, "w", (torch.float32,), R * cfg.idx_heads),
            _dev(idx_cache, "idx_cache", keyt, cfg.num_pages * cfg.page_size * cfg.idx_dim),
            _dev(idx_scale, "idx_scale", (torch.float32,), cfg.num_pages * cfg.page_size),
            _dev(page_table, "page_table", (torch.int32,), cfg.max_reqs * cfg.max_pages_per_req),
            _dev(row_req, "row_req", (torch.int32,), R), _dev(row_len, "row_len", (torch.int32,), R),
            _dev(block_first, "block_first", (torch.int32,), R),
            _dev(block_nrows, "block_nrows", (torch.int32,), R),
            _dev(scores, "scores", (torch.float32,), max(hi - lo, 0) * cfg.score_width),
            _ws(workspace), _stream(stream))
    if window is None:
        _check(_lib.dsa_indexer_scores(ctypes.byref(cfg), *args))
    else:
        _check(_lib.dsa_indexer_scores_window(ctypes.byref(cfg), lo, hi, *args))


def dsa_topk(cfg, scores, row_len, topk_idx, workspace, stream=None, window=None) -> None:
    """Top-k of every row from scores [max_rows, score_width], or with
    window=(row_begin, row_end) of those rows only, from scores
    [row_end - row_begin, score_width] (dsa_topk_window)."""
    R = cfg.max_rows
    lo, hi = (0, R) if window is None else (int(window[0]), int(window[1]))
    args = (_dev(scores, "scores", (torch.float32,), max(hi - lo, 0) * cfg.score_width),
            _dev(row_len, "row_len", (torch.int32,), R),
            _dev(topk_idx, "topk_idx", (torch.int32,), R * cfg.topk), _ws(workspace), _stream(stream))
    if window is None:
        _check(_lib.dsa_topk(ctypes.byref(cfg), *args))
    else:
        _check(_lib.dsa_topk_window(ctypes.byref(cfg), lo, hi, *args))


def _kv_ptrs(cfg, k_cache, v_cache):
    """K and V cache pointers.  With DSA_FLAG_KV_INTERLEAVED, k_cache is the
    one [num_pages, P, 2, Hkv, D] cache and the V pointer is derived from it
    (v_cache may be None, or a view whose first element is the first V row)."""
    kv = cfg.num_pages * cfg.page_size * cfg.num_kv_heads * cfg.head_dim
    if cfg.flags & DSA_FLAG_KV_INTERLEAVED:
        k = _dev(k_cache, "k_cache", _BF16, 2 * kv)
        v = ctypes.c_void_p(k.value + cfg.num_kv_heads * cfg.head_dim * 2)
        if v_cache is not None and v_cache.data_ptr() != v.value:
            raise ValueError("v_cache: with DSA_FLAG_KV_INTERLEAVED it must start at k_cache's first V row")
        return k, v
    return _dev(k_cache, "k_cache", _BF16, kv), _dev(v_cache, "v_cache", _BF16, kv)


def dsa_sparse_attn(cfg, q, k_cache, v_cache, page_table, row_req, row_len, topk_idx, part_m,
                    part_l, part_acc, workspace, stream=None) -> None:
    """Split sparse GQA attention over topk_idx: partial m, l [R, Hq, S] and
    acc [R, Hq, S, D] (fp32).  With DSA_FLAG_KV_INTERLEAVED, k_cache is the
    one interleaved cache and v_cache may be None."""
    R, Hq, S, D = cfg.max_rows, cfg.num_q_heads, cfg.num_splits, cfg.head_dim
    k_ptr, v_ptr = _kv_ptrs(cfg, k_cache, v_cache)
    _check(_lib.dsa_sparse_attn(
        ctypes.byref(cfg), _dev(q, "q", _BF16, R * Hq * D), k_ptr, v_ptr,
        _dev(page_table, "page_table", (torch.int32,), cfg.max_reqs * cfg.max_pages_per_req),
        _dev(row_req, "row_req", (torch.int32,), R), _dev(row_len, "row_len", (torch.int32,), R),
        _dev(topk_idx, "topk_idx", (torch.int32,), R * cfg.topk),
        _dev(part_m, "part_m", (torch.float32,), R * Hq * S),
        _dev(part_l, "part_l", (torch.float32,), R * Hq * S),
        _dev(part_acc, "part_acc", (torch.float32,), R * Hq * S * D),
        _ws(workspace), _stream(stream)))


def dsa_merge(cfg, part_m, part_l, part_acc, out, lse=None, stream=None) -> None:
    """Merges the split partials into out (bf16 [R, Hq, D]) and, if given,
    lse (fp32 [R, Hq])."""
    R, Hq, S, D = cfg.max_rows, cfg.num_q_heads, cfg.num_splits, cfg.head_dim
    _check(_lib.dsa_merge(
        ctypes.byref(cfg), _dev(part_m, "part_m", (torch.float32,), R * Hq * S),
        _dev(part_l, "part_l", (torch.float32,), R * Hq * S),
        _dev(part_acc, "part_acc", (torch.float32,), R * Hq * S * D),
        _dev(out, "out", _BF16, R * Hq * D), _dev(lse, "lse", (torch.float32,), R * Hq),
        _stream(stream)))


STEP_FIELDS = ("page_table", "row_req", "row_len", "block_first", "block_nrows", "q_idx", "w",
               "idx_cache", "idx_scale", "q", "k_cache", "v_cache", "out", "lse")


def make_step_args(cfg, t: dict) -> dsa_step_args_t:
    """Pack a dict of device tensors (keys = STEP_FIELDS) into dsa_step_args_t."""
    R, Hq, D = cfg.max_rows, cfg.num_q_heads, cfg.head_dim
    keyt = _FP8 if cfg.idx_key_dtype == DSA_KEY_FP8_E4M3 else _BF16
    kv = cfg.num_pages * cfg.page_size * cfg.num_kv_heads * D
    i32 = (torch.int32,)
    f32 = (torch.float32,)
    spec = dict(page_table=(i32, cfg.max_reqs * cfg.max_pages_per_req), row_req=(i32, R),
                row_len=(i32, R), block_first=(i32, R), block_nrows=(i32, R),
                q_idx=(_BF16, R * cfg.idx_heads * cfg.idx_dim), w=(f32, R * cfg.idx_heads),
                idx_cache=(keyt, cfg.num_pages * cfg.page_size * cfg.idx_dim),
                idx_scale=(f32, cfg.num_pages * cfg.page_size), q=(_BF16, R * Hq * D),
                k_cache=(_BF16, kv), v_cache=(_BF16, kv), out=(_BF16, R * Hq * D),
                lse=(f32, R * Hq))
    a = dsa_step_args_t()
    for name in STEP_FIELDS:
        if name in ("k_cache", "v_cache"):
            continue
        dt, n = spec[name]
        p = _dev(t.get(name), name, dt, n)
        setattr(a, name, p.value if p is not None else None)
    k_ptr, v_ptr = _kv_ptrs(cfg, t.get("k_cache"), t.get("v_cache"))
    a.k_cache = k_ptr.value if k_ptr is not None else None
    a.v_cache = v_ptr.value if v_ptr is not None else None
    return a


def dsa_step(cfg, args, workspace, stream=None) -> None:
    """args: a dsa_step_args_t (see make_step_args) or a dict of tensors."""
    if isinstance(args, dict):
        args = make_step_args(cfg, args)
    _check(_lib.dsa_step(ctypes.byref(cfg), ctypes.byref(args), _ws(workspace), _stream(stream)))


def dsa_step_noalloc(cfg, args, status=None, stream=None) -> None:
    """dsa_step with the library's built-in scratch array instead of a
    caller workspace (for callers that cannot allocate device memory).
    status: optional CUDA int32 tensor of >= 1 element that receives the
    step's device status word."""
    if isinstance(args, dict):
        args = make_step_args(cfg, args)
    st = _dev(status, "status", (torch.int32,), 1)
    _check(_lib.dsa_step_noalloc(ctypes.byref(cfg), ctypes.byref(args), st, _stream(stream)))
