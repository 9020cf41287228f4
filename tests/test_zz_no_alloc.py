"""dsa_step_noalloc: the step with the library's built-in scratch array.

Callers that cannot allocate device memory (inside stream capture, under a
foreign allocator, C hosts without one) use this entry point.  It runs the
same kernels on the same inputs as dsa_step with a caller workspace, so its
outputs must be bit-identical to that call's.  Collected last so that a
stop-at-first-failure run has already run every other test; it also passes
alone in a fresh process.
"""
import pytest
import torch

from sparse_attention_decode_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _reference(i):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    dev = DeviceStep(W.generate(i))
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    return dev, dev.t["out"].clone(), dev.t["lse"].clone()


def _noalloc(dsa_lib, dev):
    out = torch.full_like(dev.t["out"], float("nan"))
    lse = torch.full_like(dev.t["lse"], float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dsa_lib.dsa_step_noalloc(dev.cfg, dict(dev.t, out=out, lse=lse), status)
    torch.cuda.synchronize()
    return int(status.item()), out, lse


def test_noalloc_step_matches_workspace_step(dsa_lib, cuda_ok):
    """Bit-identical to dsa_step on two calls in a row, and again after a
    call with another config has reused the array (A, A, B, A): the
    histogram region a layout change moves onto is cleared first."""
    refs = {i: _reference(i) for i in (0, 1)}
    for n, i in enumerate((0, 0, 1, 0)):
        dev, ref_out, ref_lse = refs[i]
        status, out, lse = _noalloc(dsa_lib, dev)
        assert status == 0, (n, i)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), (n, i)
        assert torch.equal(lse, ref_lse), (n, i)


def test_noalloc_rejects_configs_beyond_the_array(dsa_lib, cuda_ok):
    wl = W.workload(3)  # mixed step: 1024 row slots x 32768 scores, far above 32 MiB
    cfg = dsa_lib.config_from_workload(wl, 100000)
    assert dsa_lib.dsa_workspace_size(cfg) > (32 << 20)
    with pytest.raises(dsa_lib.DsaError) as e:
        dsa_lib.dsa_step_noalloc(cfg, dsa_lib.dsa_step_args_t())
    assert e.value.status == dsa_lib.DSA_ERR_CAPACITY
