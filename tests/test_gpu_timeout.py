"""The bounded waits of the tensor-core kernels, made to run out on purpose:
k3moe_selftest_bounded_wait waits, with the production iteration bound, on an
mbarrier phase that nothing completes (no copy or MMA in flight), so the wait
gives up, the kernel reports K3MOE_DEV_TIMEOUT and returns, and the context stays
usable for the next call."""
import numpy as np
import pytest
import torch

import mxfp4_expert_ffn_router_gb300 as k3
import gen


@pytest.mark.gpu
def test_bounded_wait_runs_out_and_reports_timeout():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    k3.k3moe_selftest_bounded_wait(st, el)
    torch.cuda.synchronize()
    assert int(st.item()) & k3.K3MOE_DEV_TIMEOUT
    ns = int(el.item())
    assert 0 < ns < 10e9, ns  # the bound ends the wait (about a second)
    # the context is still usable: a routing call runs and reports nothing
    s = gen.Shape(2, 256, 128, 8, 2)
    logits = torch.from_numpy(np.random.default_rng(5).standard_normal((2, 8)).astype(np.float32)).cuda()
    idx = torch.empty((2, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((2, 2), dtype=torch.float32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    k3.k3moe_route(s, logits, idx, w, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = np.argsort(-logits.cpu().numpy(), axis=1, kind="stable")[:, :2]
    assert (idx.cpu().numpy() == ref).all()


def test_selftest_refuses_null_pointers():
    """On the host, before any device call."""
    L = k3.lib()
    assert L.k3moe_selftest_bounded_wait(None, None, None) == k3.K3MOE_ERR_ARG
