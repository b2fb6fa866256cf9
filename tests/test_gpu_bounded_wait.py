"""GPU: the bounded device wait gives up, reports and returns.

Every wait of the streaming kernels on a bulk-copy barrier is bounded in SM
cycles; when it runs out the kernel records SPLITZIP_ERR_TIMEOUT and finishes
instead of spinning.  splitzip_selftest_bounded_wait runs that path on
purpose with no copy in flight (a warp waits on an mbarrier that nothing
arrives on, with a short limit), so the status word, the time the wait took
and the state of the GPU afterwards can be checked.  Nothing here faults or
waits without a bound.
"""
import numpy as np
import pytest
import torch

import oracle
import lossless_kv_cache_gb300 as sz
from lossless_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit", [10_000, 1_000_000])
def test_wait_runs_out_and_reports_timeout(splitzip_lib, limit):
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    cycles = torch.full((2,), -7, dtype=torch.int64, device="cuda")
    st = sz.splitzip_selftest_bounded_wait(limit, status.data_ptr(), cycles.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
    assert st == sz.OK
    torch.cuda.synchronize()
    assert int(status[0]) == sz.ERR_TIMEOUT
    waited, control = (int(v) for v in cycles.cpu())
    assert limit < waited < limit + 1_000_000  # gave up just after the limit
    assert 0 <= control < limit                # the completed barrier did not wait


def test_gpu_still_usable_after_a_timeout(splitzip_lib):
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert sz.splitzip_selftest_bounded_wait(50_000, status.data_ptr(), None,
                                             torch.cuda.current_stream().cuda_stream) == sz.OK
    torch.cuda.synchronize()
    assert int(status[0]) == sz.ERR_TIMEOUT
    # an ordinary encode + decode on the same context afterwards
    x = W.escape_stress(4, chunks=3)
    bits = x.numpy().view(np.uint16)
    cb = oracle.calibrate(oracle.histogram(bits, 0), 0)
    blob = sz.encode(x.to("cuda"), sz.Codebook.make(sz.BF16, cb), sz.BF16)
    np.testing.assert_array_equal(blob.cpu().numpy(), oracle.encode(bits, 0, cb))
    assert torch.equal(sz.decode(blob, x.numel(), sz.BF16).cpu(), x)

