"""Failure detection on the GPU without a GPU fault.

Every wait in the library's kernels is bounded by a time limit; the
self-test kernel makes one run out on purpose (an mbarrier nothing completes)
and checks that the status word reports it, that the other waiters in the CTA
stop as soon as the first gives up, and that the context is still usable.
"""
import math

import numpy as np
import pytest
import torch

import prefix_kv_gb300 as bca
from prefix_kv_gb300 import _native
from gpu_cases import DEV, assert_close, ragged_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()


def test_bounded_wait_times_out_and_reports():
    lib = _native.load()
    status = bca.new_status(DEV)
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    limit = 20_000_000   # 20 ms; the other waiters would wait 1 s without the abort flag
    code = lib.bca_selftest_wait_timeout(limit, status.data_ptr(), elapsed.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert code == 0
    assert bca.read_status(status) == 7          # BCA_ERR_TIMEOUT
    ns = int(elapsed.item())
    assert limit <= ns < 500_000_000, ns
    # the context is still usable: a normal call afterwards matches the oracle
    case = ragged_case(91, [300, 129])
    st = bca.new_status(DEV)
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="after timeout")


def test_selftest_rejects_bad_limits():
    lib = _native.load()
    status = bca.new_status(DEV)
    assert lib.bca_selftest_wait_timeout(0, status.data_ptr(), None, None) == 1
    assert lib.bca_selftest_wait_timeout(2_000_000_000, status.data_ptr(), None, None) == 1
    assert lib.bca_selftest_wait_timeout(1000, None, None, None) == 1
