"""The device-side failure path, exercised without a GPU fault: a bounded
wait that runs out is recorded in the workspace's status word, the kernel
returns, msa_check_device_status reports MSA_ERR_TIMEOUT with the site, and
the context stays usable (the status word is cleared and later calls work)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_is_reported():
    import torch
    from block_sparse_gqa_causal_gb300 import api
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.selftest_wait_timeout(ws, spin_limit=4096)
    torch.cuda.synchronize()
    assert int(ws[128:132].view(torch.int32).item()) == 1      # the wait gave up and the kernel went on
    with pytest.raises(api.MsaError) as ei:
        api.check_device_status(ws)
    assert ei.value.code == 5 and "site 901" in str(ei.value)
    api.check_device_status(ws)                                # cleared after the report
    # the context is still usable: a real call on the same stream succeeds
    sh = api.Shape(B=1, Nq=512, Nk=512, Hq=4, Hkv=2, d=64, d_idx=64, topk=2)
    qi = torch.randn(1, 512, 2, 64, device="cuda").bfloat16()
    ki = torch.randn(1, 512, 64, device="cuda").bfloat16()
    ws2 = api.new_workspace(sh, api.OP_INDEX_SELECT)
    sel = api.index_select(sh, qi, ki, workspace=ws2)
    torch.cuda.synchronize()
    api.check_device_status(ws2)
    s = sel.cpu().numpy()
    assert np.all(s.max(axis=-1) == (np.arange(512) // 128)[None, None, :])
