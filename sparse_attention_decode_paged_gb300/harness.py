"""Device-side plumbing around the C-ABI: upload one step's inputs, build the
rows through the library, hold the outputs and workspace, run or capture a
step.  PyTorch is used here only for device memory, streams and CUDA graphs.
"""
from __future__ import annotations

import numpy as np
import torch

from . import dsa


def to_device(a: np.ndarray | None, device="cuda", kind: str = "raw"):
    """numpy -> CUDA tensor; kind 'bf16' reinterprets uint16 bits as bfloat16."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if kind == "bf16":
        t = torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a).to(device)
    return t


DEVICE_ROW_KEYS = ("row_req", "row_len", "block_first", "block_nrows")


def _arena(parts, device):
    """One byte buffer holding several tensors, each at a 256-byte aligned
    offset: parts = [(name, dtype, shape)] -> (buffer, {name: view})."""
    off, spans = 0, []
    for name, dtype, shape in parts:
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        spans.append((name, dtype, shape, off, n))
        off = (off + n + 255) // 256 * 256
    buf = torch.zeros(max(off, 256), dtype=torch.uint8, device=device)
    return buf, {name: buf[o:o + n].view(dtype).view(*shape) for name, dtype, shape, o, n in spans}


class DeviceStep:
    """All device buffers of one DSA layer-step for a generated workload.

    The per-step inputs that change from step to step (row maps, page table,
    q_idx, w, q) live in one device arena, `inputs`, and the outputs (out,
    lse) in another, `outputs`, so a serving loop moves them with one copy
    each way; t[...] are views into them."""

    def __init__(self, inp: dict, device="cuda", **cfg_override):
        wl = inp["workload"]
        self.inp = inp
        self.cfg = dsa.config_from_workload(wl, inp["num_pages"], **cfg_override)
        dsa.dsa_validate_config(self.cfg)
        self.rows = dsa.dsa_build_rows(self.cfg, inp["cache_len"], inp["new_tokens"])
        R, Hq, D = wl.max_rows, wl.num_q_heads, wl.head_dim
        pt = np.ascontiguousarray(inp["page_table"])
        self.inputs, t = _arena(
            [(k, torch.int32, (R,)) for k in DEVICE_ROW_KEYS]
            + [("page_table", torch.int32, pt.shape),
               ("q_idx", torch.bfloat16, inp["q_idx"].shape),
               ("w", torch.float32, inp["w"].shape),
               ("q", torch.bfloat16, inp["q"].shape)], device)
        for k in DEVICE_ROW_KEYS:
            t[k].copy_(torch.from_numpy(self.rows[k]))
        t["page_table"].copy_(torch.from_numpy(pt))
        for k, kind in (("q_idx", "bf16"), ("w", "raw"), ("q", "bf16")):
            t[k].copy_(to_device(inp[k], device, kind))
        if inp["idx_scale"] is None:
            t["idx_cache"] = to_device(inp["idx_cache"], device, "bf16")
            t["idx_scale"] = None
        else:
            t["idx_cache"] = to_device(inp["idx_cache"], device)
            t["idx_scale"] = to_device(inp["idx_scale"], device)
        t["k_cache"] = to_device(inp["k_cache"], device, "bf16")
        t["v_cache"] = to_device(inp["v_cache"], device, "bf16")
        if self.cfg.flags & dsa.DSA_FLAG_KV_INTERLEAVED:
            # one cache [NP, P, 2, Hkv, D]: each token's K row, then its V row
            kv = torch.stack((t["k_cache"], t["v_cache"]), dim=2).contiguous()
            t["k_cache"], t["v_cache"] = kv, kv[:, :, 1]
        self.outputs, outs = _arena([("out", torch.bfloat16, (R, Hq, D)), ("lse", torch.float32, (R, Hq))], device)
        t.update(outs)
        self.t = t
        self.workspace = dsa.alloc_workspace(self.cfg, device)
        self.views = dsa.workspace_views(self.cfg, self.workspace)
        self.args = dsa.make_step_args(self.cfg, t)

    def step(self, stream=None):
        dsa.dsa_step(self.cfg, self.args, self.workspace, stream)

    def status(self) -> int:
        return dsa.dsa_read_device_status(self.workspace)

    def capture(self, stream: torch.cuda.Stream | None = None) -> torch.cuda.CUDAGraph:
        """Warm up once eagerly, then capture one step into a CUDA graph."""
        stream = stream or torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            self.step(stream)
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return g

    def set_rows(self, cache_len, new_tokens, page_table=None):
        """Rebuild rows on the host and copy them into the static buffers."""
        self.rows = dsa.dsa_build_rows(self.cfg, cache_len, new_tokens)
        for k in ("row_req", "row_len", "block_first", "block_nrows"):
            self.t[k].copy_(torch.from_numpy(self.rows[k]))
        if page_table is not None:
            self.t["page_table"].copy_(torch.from_numpy(np.ascontiguousarray(page_table)))
