"""Failure detection of the persistent kernels' grid barrier, without faulting the GPU.

moe_route_arm_barrier_timeout makes one CTA of the next persistent launch leave before
the first grid barrier and limits that launch's barrier waits to 1 ms.  The other CTAs'
waits run out; every wait is bounded, so every CTA returns.  The call must be reported
through moe_route_device_status() as MOE_ROUTE_E_DEVICE_TIMEOUT, and the next call must
be exact again (the last CTA out restores the barrier words)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    import serving_moe_route_02_gb300 as mr
    mr.load()
    mr.reserve()
    return mr


@pytest.mark.parametrize("path", [2, 3])
@pytest.mark.parametrize("cta", [0, 1])
def test_barrier_timeout_reported_then_next_call_exact(mr, path, cta):
    lib = mr.load()
    cfg = gen.cfg3(3000, off=784, cnt=112)
    dev = torch.device("cuda")
    lg = torch.from_numpy(cfg["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    assert mr.device_status() == 0
    prev = mr.set_path(path)
    try:
        assert lib.moe_route_arm_barrier_timeout(cta, 1000) == mr.OK
        mr.route(lg, bias, local_offset=784, local_count=112)
        torch.cuda.synchronize()
        assert mr.device_status() == mr.E_DEVICE_TIMEOUT
        out = mr.route(lg, bias, local_offset=784, local_count=112, want_ids=True)
        torch.cuda.synchronize()
        assert mr.device_status() == 0
    finally:
        lib.moe_route_arm_barrier_timeout(-1, 0)
        mr.set_path(prev)
    parity.compare({k: v.cpu().numpy() for k, v in out.items()}, oracle.route_cfg(cfg), cfg, exact=True)


def test_arming_is_consumed_by_one_launch(mr):
    lib = mr.load()
    cfg = gen.cfg3(1000)
    dev = torch.device("cuda")
    lg = torch.from_numpy(cfg["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    assert lib.moe_route_arm_barrier_timeout(2, 1000) == mr.OK
    assert lib.moe_route_arm_barrier_timeout(-1, 0) == mr.OK  # disarmed before any launch
    out = mr.route(lg, bias, want_ids=True)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    parity.compare({k: v.cpu().numpy() for k, v in out.items()}, oracle.route_cfg(cfg), cfg, exact=True)
