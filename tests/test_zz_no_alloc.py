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


def _noalloc(lib, case, status, block_id=None, total_q=None, guard=0):
    """One call through the C ABI.  out/lse start as NaN; with `guard`, out is the
    head of a buffer `guard` rows longer whose tail must stay NaN.  `total_q` may
    claim fewer query rows than the case's offsets reach."""
    d = lambda t: t.to(DEV)
    ti = lambda a: torch.from_numpy(a).to(DEV)
    q, k, v = d(case.q), d(case.k), d(case.v)
    bid = ti(case.block_id if block_id is None else block_id)
    cq, ck = ti(case.cu_q), ti(case.cu_k)
    tq = q.shape[0] if total_q is None else total_q
    buf = torch.full((tq + guard,) + tuple(q.shape[1:]), float("nan"), dtype=q.dtype, device=DEV)
    out = buf[:tq]
    lse_buf = torch.full((q.shape[1] * tq + guard,), float("nan"), dtype=torch.float32,
                         device=DEV)
    lse = lse_buf[:q.shape[1] * tq].view(q.shape[1], tq)
    code = lib.bca_prefill_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), bid.data_ptr(), cq.data_ptr(), ck.data_ptr(),
        len(case.cu_q) - 1, q.shape[1], 128, tq, k.shape[0], case.max_q, case.max_k,
        1.0 / math.sqrt(128), out.data_ptr(), lse.data_ptr(), status.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert code == 0, code
    return out, lse, (buf[tq:], lse_buf[q.shape[1] * tq:])


def _close(out, lse, ref_out, ref_lse):
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    err = (out.float() - ref_out.float()).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    rel = (lse - ref_lse).abs() / ref_lse.abs().clamp(min=1.0)
    assert rel.max().item() <= 1e-3


def test_noalloc_matches_prefill_on_two_calls(lib):
    import prefix_kv_gb300 as bca
    cases = [ragged_case(81, [700, 129, 1300], [700, 100, 1300]),   # larger first ...
             ragged_case(82, [260, 33], [200, 33])]                  # ... then smaller
    for case in cases:
        status = bca.new_status(DEV)
        out, lse, _ = _noalloc(lib, case, status)
        ref_out, ref_lse = case.run()
        assert bca.read_status(status) == 0
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_failed_sequence_does_not_reuse_stale_scratch(lib):
    """A sequence that fails its device-side check must not run on the tile
    records a previous, larger call left in the shared scratch: its rows keep
    their NaN fill, and the other sequences match bca_prefill."""
    import prefix_kv_gb300 as bca
    big = ragged_case(83, [900, 1100, 640], [900, 1100, 640])
    status = bca.new_status(DEV)
    _noalloc(lib, big, status)                      # leaves valid records for all three
    assert bca.read_status(status) == 0
    case = ragged_case(83, [900, 1100, 640], [900, 1100, 640])
    bid = case.block_id.copy()
    a, e = int(case.cu_k[1]), int(case.cu_k[2])
    bid[a:e] = -1
    bid[a + 5:a + 9] = 7                            # id 7 in two separate runs of sequence 1
    bid[a + 20:a + 30] = 7
    status = bca.new_status(DEV)
    out, lse, _ = _noalloc(lib, case, status, block_id=bid)
    assert bca.read_status(status) == 3             # BCA_ERR_BLOCK_ID
    q0, q1 = int(case.cu_q[1]), int(case.cu_q[2])
    assert torch.isnan(out[q0:q1].float()).all() and torch.isnan(lse[:, q0:q1]).all()
    ref_out, ref_lse = case.run()                   # the sequences that passed are unaffected
    keep = torch.cat([torch.arange(0, q0), torch.arange(q1, out.shape[0])]).to(DEV)
    _close(out[keep], lse[:, keep], ref_out[keep], ref_lse[:, keep])


def test_noalloc_rejects_offsets_past_the_arrays(lib):
    """cu_seqlens_q whose last entry lies 128 rows past total_q: that sequence fails
    with BCA_ERR_SEQLENS before any of its rows is touched, nothing is written past
    the output or the LSE (NaN guard regions behind them stay NaN), and the other
    sequence matches bca_prefill."""
    import prefix_kv_gb300 as bca
    case = ragged_case(84, [300, 500], [300, 500])
    tq = int(case.cu_q[-1]) - 128
    status = bca.new_status(DEV)
    out, lse, (guard, lse_guard) = _noalloc(lib, case, status, total_q=tq, guard=256)
    assert bca.read_status(status) == 8             # BCA_ERR_SEQLENS
    assert torch.isnan(guard.float()).all() and torch.isnan(lse_guard).all()
    q0 = int(case.cu_q[1])
    assert torch.isnan(out[q0:].float()).all() and torch.isnan(lse[:, q0:]).all()
    ref_out, ref_lse = case.run()
    _close(out[:q0], lse[:, :q0], ref_out[:q0], ref_lse[:, :q0])


def test_noalloc_rejects_oversized(lib):
    # more query rows than the fixed scratch holds: refused before any launch
    code = lib.bca_prefill_noalloc(16, 16, 16, 16, 16, 16, 1, 1, 128, 262145, 262145, 262145,
                                   262145, 0.1, 16, 16, None, None)
    assert code == 4
