"""The decode's balanced tail, against the CPU oracle.

The query-tile pairs of a last, partly filled wave (all pairs, when there are
fewer than SMs) are cut into one equal key range per SM; a range that crosses a
pair boundary is two pieces.  Each piece leaves unnormalised rows, row maxima
and row sums in the workspace, and a merge grid combines the pieces of each
pair.  Covered here: ranges that cross pair boundaries, ragged target and prefix
lengths, a pair whose second tile is empty, a sequence without prefix, a tail
behind a full pair grid, a workspace reused across calls (including after a
call that failed validation), the key-split tail that runs without a workspace,
and the errors: a workspace too small, a prefix longer than max_prefix, a
cache too small for the prefixes.
"""
import numpy as np
import pytest
import torch

import prefix_kv_gb300 as bca
from prefix_kv_gb300 import _native
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV, DecodeCase, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()
    assert torch.cuda.is_available()


def _case(seed, H, pre, tgt, **kw):
    kp = W.randn_bf16((sum(pre), H, 128), seed)
    vp = W.randn_bf16((sum(pre), H, 128), seed + 100)
    qt = W.randn_bf16((sum(tgt), H, 128), seed + 200)
    kt = W.randn_bf16((sum(tgt), H, 128), seed + 300)
    vt = W.randn_bf16((sum(tgt), H, 128), seed + 400)
    cu_p = np.concatenate([[0], np.cumsum(pre)])
    cu_q = np.concatenate([[0], np.cumsum(tgt)])
    # unused cache capacity holds NaN: only the prefix may be read
    return DecodeCase(qt, kt, vt, kp, vp, cu_q, cu_p, layers=2, layer=1,
                      cache_fill=float("nan"), **kw)


def _tail_bytes(case, max_pre=None):
    return bca.prefix_decode_workspace_bytes(len(case.cu_q) - 1, case.q_tgt.shape[1], case.max_q,
                                             case.max_pre if max_pre is None else max_pre)


def _nan_outputs(case):
    out = torch.full(tuple(case.q_tgt.shape), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((case.q_tgt.shape[1], case.q_tgt.shape[0]), float("nan"),
                     dtype=torch.float32, device=DEV)
    return out, lse


CASES = {
    # one sequence, 16 pairs of 55 key tiles: 110 ranges of 8 tiles, many crossing a pair edge
    "one_seq": (11, 4, [6000], [1000]),
    # ragged: an odd target tile count (the last pair's second tile empty), a sequence with
    # no prefix and two target tiles (its later pairs empty), prefixes ending inside tiles
    "ragged": (12, 2, [5000, 0, 6500], [1000, 130, 777]),
    # tile-aligned lengths: pieces start and end on tile edges only
    "aligned": (13, 3, [6144, 4096], [1024, 768]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_balanced_tail_matches_oracle(name):
    seed, H, pre, tgt = CASES[name]
    case = _case(seed, H, pre, tgt)
    if _tail_bytes(case) == 0:
        pytest.skip("no balanced tail for this shape on this device")
    st = bca.new_status(DEV)
    out, lse = _nan_outputs(case)
    case.run(status=st, out=out, lse=lse)
    assert bca.read_status(st) == 0
    ref = case.reference()
    assert_close(out, lse, *ref, what=f"balanced tail {name}")
    # the key-split tail (no workspace) computes the same attention
    out2, lse2 = case.run(status=st, balanced_tail=False)
    assert bca.read_status(st) == 0
    assert_close(out2, lse2, *ref, what=f"key-split tail {name}")


def test_balanced_tail_behind_a_full_pair_grid():
    # 8 heads x 5 sequences x 4 pairs = 160 pairs: one full wave of 152 in the pair grid,
    # 8 pairs in the balanced tail (63 key tiles each)
    H = 8
    case = _case(81, H, [6000, 0, 333, 7000, 128], [1000, 700, 1024, 5, 257])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if not (160 > sms and _tail_bytes(case) > 0):
        pytest.skip(f"{sms} SMs: this shape does not give both grids")
    st = bca.new_status(DEV)
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="pair grid + balanced tail")


def test_balanced_tail_full_size_edit_against_key_split():
    # the edit workload's decode: 512 pairs, 56 of them in the tail; every row of one head
    # that has tail pairs against the oracle, and all heads against the key-split tail
    wl = W.edit_two_ref()
    case = DecodeCase.from_workload(wl)
    assert _tail_bytes(case) > 0
    out, lse = case.run()
    out2, lse2 = case.run(balanced_tail=False)
    assert_close(out, lse, out2.float().cpu().numpy(), lse2.cpu().numpy(), what="balanced vs split")
    heads = np.array([31])
    assert_close(out, lse, *case.reference(heads=heads), heads=heads, what=wl.name)


def test_workspace_reused_across_calls_and_after_a_failed_call():
    a = _case(21, 4, [6000], [1000])
    b = _case(22, 2, [5000, 0, 6500], [1000, 130, 777])
    if _tail_bytes(a) == 0 or _tail_bytes(b) == 0:
        pytest.skip("no balanced tail for these shapes on this device")
    ws = torch.empty(max(_tail_bytes(a), _tail_bytes(b)), dtype=torch.uint8, device=DEV)
    st = bca.new_status(DEV)
    for case in (a, b, a):
        out, lse = case.run(status=st, workspace=ws)
        assert bca.read_status(st) == 0
        assert_close(out, lse, *case.reference(), what="reused workspace")
    # a call whose cache is too small fails validation (the pieces mark their slots);
    # the next valid call over the same workspace is unaffected
    small = _case(21, 4, [6000], [1000])
    small.cache_k = small.cache_k[:, :, :5000].contiguous()
    small.cache_v = small.cache_v[:, :, :5000].contiguous()
    st = bca.new_status(DEV)
    out, lse = _nan_outputs(small)
    small.run(status=st, workspace=ws, out=out, lse=lse)
    assert bca.read_status(st) == 5                     # BCA_ERR_CAPACITY
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    st = bca.new_status(DEV)
    out, lse = a.run(status=st, workspace=ws)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *a.reference(), what="after a failed call")


def test_prefix_longer_than_max_prefix_is_reported():
    case = _case(31, 4, [6000], [1000])
    if _tail_bytes(case, max_pre=5800) == 0:
        pytest.skip("no balanced tail for this shape on this device")
    st = bca.new_status(DEV)
    out, lse = _nan_outputs(case)
    case.run(status=st, max_pre=5800, out=out, lse=lse)
    assert bca.read_status(st) == 8                      # BCA_ERR_SEQLENS
    assert torch.isnan(out.float()).all()                # every pair is in the tail


def test_workspace_too_small_is_rejected():
    case = _case(41, 4, [6000], [1000])
    need = _tail_bytes(case)
    if need == 0:
        pytest.skip("no balanced tail for this shape on this device")
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(_native.BcaError) as e:
        case.run(workspace=ws)
    assert e.value.code == 4                             # BCA_ERR_WORKSPACE
