"""dsa_step_noalloc: the step with the library's built-in scratch array.

Callers that cannot allocate device memory (inside stream capture, under a
foreign allocator, C hosts without one) use this entry point; it must give
the same result as dsa_step with a caller workspace.  Collected last so that
a stop-at-first-failure run has already run every other test; it also passes
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from sparse_attention_decode_paged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("i", [0, 1])
def test_noalloc_step_matches_workspace_step(i, dsa_lib, cuda_ok):
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    dev = DeviceStep(W.generate(i))
    dev.step()
    torch.cuda.synchronize()
    assert dev.status() == 0
    ref_out = dev.t["out"].float().cpu().numpy()
    ref_lse = dev.t["lse"].cpu().numpy()
    out = torch.empty_like(dev.t["out"])
    lse = torch.empty_like(dev.t["lse"])
    tensors = dict(dev.t, out=out, lse=lse)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):  # two calls in a row share the array
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        dsa_lib.dsa_step_noalloc(dev.cfg, tensors, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        got = out.float().cpu().numpy()
        np.testing.assert_allclose(got, ref_out, atol=1e-2, rtol=2e-2, err_msg=f"call {call}")
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse.cpu().numpy()))
        np.testing.assert_allclose(lse.cpu().numpy()[fin], ref_lse[fin], atol=1e-2, rtol=2e-2)


def test_noalloc_rejects_configs_beyond_the_array(dsa_lib, cuda_ok):
    wl = W.workload(3)  # mixed step: 1024 row slots x 32768 scores, far above 32 MiB
    cfg = dsa_lib.config_from_workload(wl, 100000)
    assert dsa_lib.dsa_workspace_size(cfg) > (32 << 20)
    with pytest.raises(dsa_lib.DsaError) as e:
        dsa_lib.dsa_step_noalloc(cfg, dsa_lib.dsa_step_args_t())
    assert e.value.status == dsa_lib.DSA_ERR_CAPACITY
