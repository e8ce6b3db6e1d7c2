"""Failure path of the kernels' waits, on the GPU without a fault: a wait on an mbarrier
that nothing completes gives up after its bound, reports CSA2_DEV_PIPELINE_TIMEOUT
through the workspace status word, and the context stays usable."""
import numpy as np
import pytest
import torch

import sparse_attention_kv_decode_b300 as csa2
from oracle import fp4

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_ms", [2, 30])
def test_a_wait_nothing_completes_gives_up_and_reports(limit_ms):
    dev = "cuda"
    ws = csa2.csa2_workspace(1, 1, 1, 0, 1, device=dev)
    s = torch.cuda.Stream(device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        csa2.csa2_check_bounded_wait(limit_ms * 1_000_000, ws, stream=s)
        e1.record(s)
    s.synchronize()
    ms = e0.elapsed_time(e1)
    # the bound is checked every 256 polls of try_wait, which may itself suspend a while
    assert limit_ms * 0.9 <= ms < limit_ms + 1000, ms
    st, flags = csa2.csa2_read_device_status(ws, s)
    assert st == 5 and flags == csa2.DEV_PIPELINE_TIMEOUT      # CSA2_ERR_TIMEOUT
    # the context still works: a quantise call right after matches the oracle bit for bit
    x = torch.randn((8, 576), device=dev)
    codes, scales = csa2.csa2_encode_kv(x)
    torch.cuda.synchronize()
    c, sc = fp4.encode(x.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), c) and np.array_equal(scales.cpu().numpy(), sc)
    assert csa2.csa2_read_device_status(ws) == (0, 0)
