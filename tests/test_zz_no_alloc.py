"""bca_prefill_noalloc: the prefill entry point for callers that cannot allocate.

Callers such as a plugin inside a runtime that owns all GPU memory, or a loop
that must not pay cudaMalloc's synchronisation, can neither allocate nor pass a
workspace.  This entry point keeps its scratch in a fixed array inside the
library.  Here it is called through the C ABI twice in a row, on two different
problems (the larger first, so the second runs over the first one's leftover
scratch), and each result is compared with bca_prefill's on the same inputs at
the parity tolerances.  The file is named so that pytest collects it last.
"""
import math

import pytest
import torch

from gpu_cases import DEV, ragged_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from prefix_kv_gb300 import _native, build_native
    build_native.build()
    assert torch.cuda.is_available()
    return _native.load()


def _noalloc(lib, case, status):
    d = lambda t: t.to(DEV)
    ti = lambda a: torch.from_numpy(a).to(DEV)
    q, k, v = d(case.q), d(case.k), d(case.v)
    bid, cq, ck = ti(case.block_id), ti(case.cu_q), ti(case.cu_k)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), dtype=torch.float32, device=DEV)
    code = lib.bca_prefill_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), bid.data_ptr(), cq.data_ptr(), ck.data_ptr(),
        len(case.cu_q) - 1, q.shape[1], 128, q.shape[0], k.shape[0], case.max_q, case.max_k,
        1.0 / math.sqrt(128), out.data_ptr(), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert code == 0, code
    return out, lse


def test_noalloc_matches_prefill_on_two_calls(lib):
    import prefix_kv_gb300 as bca
    cases = [ragged_case(81, [700, 129, 1300], [700, 100, 1300]),   # larger first ...
             ragged_case(82, [260, 33], [200, 33])]                  # ... then smaller
    for case in cases:
        status = bca.new_status(DEV)
        out, lse = _noalloc(lib, case, status)
        ref_out, ref_lse = case.run()
        assert bca.read_status(status) == 0
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        err = (out.float() - ref_out.float()).abs()
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
        rel = (lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)
        assert rel.max().item() <= 1e-3


def test_noalloc_rejects_oversized(lib):
    # more query rows than the fixed scratch holds: refused before any launch
    code = lib.bca_prefill_noalloc(16, 16, 16, 16, 16, 16, 1, 1, 128, 262145, 262145, 262145,
                                   262145, 0.1, 16, 16, None, None)
    assert code == 4
