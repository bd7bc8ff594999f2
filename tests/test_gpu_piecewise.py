"""The piecewise prefill baseline (one attention call per segment) on the GPU:
against the oracle, and against the single-launch prefill, at the tolerances of
the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W
from gpu_cases import (DEV, OUT_MAX, OUT_MEAN, SCALE, PrefillCase, assert_close, ragged_case,
                       tile_boundary_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()


def _run_piecewise(case, status=None):
    d = lambda t: t.to(DEV)
    return bca.prefill_piecewise(d(case.q), d(case.k), d(case.v),
                                 torch.from_numpy(case.block_id).to(DEV), case.block_id,
                                 case.cu_k, SCALE, status=status)


def test_piecewise_tiny_all_rows():
    case = PrefillCase.from_workload(W.tiny_mixed())
    st = bca.new_status(DEV)
    out, lse = _run_piecewise(case, st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="piecewise tiny")


@pytest.mark.parametrize("seed,kv", [(81, [300, 5, 1000]), (82, [129, 128, 1, 700])])
def test_piecewise_ragged_varlen(seed, kv):
    case = ragged_case(seed, kv)
    st = bca.new_status(DEV)
    out, lse = _run_piecewise(case, st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what=f"piecewise {seed}")


def test_piecewise_edit_matches_oracle_and_single_launch():
    case = PrefillCase.from_workload(W.edit_two_ref())
    out_p, lse_p = _run_piecewise(case)
    out_s, lse_s = case.run()
    rows = tile_boundary_rows(case.cu_q, extra=64, seed=4)
    heads = np.array([6])
    assert_close(out_p, lse_p, *case.reference(rows=rows, heads=heads), rows=rows, heads=heads,
                 what="piecewise edit")
    d = (out_p.float() - out_s.float()).abs()
    assert d.max().item() <= OUT_MAX and d.mean().item() <= OUT_MEAN / 4
    assert ((lse_p - lse_s).abs() / lse_s.abs().clamp(min=1)).max().item() <= 1e-3


def test_piecewise_workspace_checked():
    case = PrefillCase.from_workload(W.tiny_mixed())
    need = bca.prefill_piecewise_workspace_bytes(case.block_id, case.cu_k, 2)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    d = lambda t: t.to(DEV)
    with pytest.raises(RuntimeError, match="status 4 "):
        bca.prefill_piecewise(d(case.q), d(case.k), d(case.v),
                              torch.from_numpy(case.block_id).to(DEV), case.block_id, case.cu_k,
                              SCALE, workspace=ws)
