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


# ------------------------------------------------ the paged and FP8 decodes use it too

def _ti(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a, dtype=np.int32))).to(DEV)


def test_balanced_tail_paged_ragged():
    """Paged decode of the ragged batch through a shuffled page table over a pool 1.5x the
    prefix pages: against the oracle, and bit-identical to the contiguous decode (the
    pieces read the same rows in the same order)."""
    seed, H, pre, tgt = CASES["ragged"]
    case = _case(seed, H, pre, tgt)
    if _tail_bytes(case) == 0:
        pytest.skip("no balanced tail for this shape on this device")
    need = [(p + 127) // 128 for p in pre]
    n_pages = sum(need) + sum(need) // 2
    perm = np.random.default_rng(seed).permutation(n_pages).astype(np.int32)
    pt = np.full((len(pre), max(need)), -1, np.int32)
    at = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[at:at + n]
        at += n
    ck = torch.full((2, H, n_pages * 128, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    cv = torch.full_like(ck, float("nan"))
    st = bca.new_status(DEV)
    bca.prefix_cache_append_paged(case.k_pre.to(DEV), case.v_pre.to(DEV), _ti(case.cu_pre),
                                  _ti(case.cu_pre), _ti(pt), ck, cv, 1, status=st)
    out, lse = bca.prefix_decode_paged(case.q_tgt.to(DEV), ck, cv, 1, _ti(case.cu_pre), _ti(pt),
                                       case.k_tgt.to(DEV), case.v_tgt.to(DEV), _ti(case.cu_q),
                                       case.max_q, case.max_pre, status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="paged balanced tail")
    out_c, lse_c = case.run(status=st)
    assert bca.read_status(st) == 0
    assert torch.equal(out.view(torch.int16), out_c.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_c.view(torch.int32))


@pytest.mark.parametrize("mode", ["v", "kv"])
def test_balanced_tail_fp8_ragged(mode):
    """FP8 decode of the ragged batch, the tail's slots after the expanded layers in the
    workspace: against the oracle over the dequantised cache, and against the FP8 decode
    that runs the key-split tail (a workspace without room for the slots)."""
    from oracle import fp8 as ofp8
    import oracle
    seed, H, pre, tgt = CASES["ragged"]
    case = _case(seed, H, pre, tgt)
    if _tail_bytes(case) == 0:
        pytest.skip("no balanced tail for this shape on this device")
    cap = int(case.cu_pre[-1]) + 64
    kdt = torch.uint8 if mode == "kv" else torch.bfloat16
    ck = torch.zeros((1, H, cap, 128), dtype=kdt, device=DEV)
    cv = torch.zeros((1, H, cap, 128), dtype=torch.uint8, device=DEV)
    sk = torch.zeros((1, H, cap), dtype=torch.float32, device=DEV)
    sv = torch.zeros_like(sk)
    st = bca.new_status(DEV)
    cp, cq = _ti(case.cu_pre), _ti(case.cu_q)
    bca.prefix_cache_append_fp8(case.k_pre.to(DEV), case.v_pre.to(DEV), cp, cp, ck, cv,
                                sk if mode == "kv" else None, sv, 0, mode=mode, status=st)
    qt, kt, vt = case.q_tgt.to(DEV), case.k_tgt.to(DEV), case.v_tgt.to(DEV)
    args = (qt, ck, cv, sk if mode == "kv" else None, sv, 0, cp, kt, vt, cq, case.max_q,
            case.max_pre)
    out, lse = bca.prefix_decode_fp8(*args, mode=mode, status=st)
    assert bca.read_status(st) == 0
    vc, vs = ofp8.quantize_rows(case.v_pre)
    vh = torch.from_numpy(ofp8.dequantize_rows(vc, vs)).to(torch.bfloat16)
    if mode == "kv":
        kc, ks = ofp8.quantize_rows(case.k_pre)
        kh = torch.from_numpy(ofp8.dequantize_rows(kc, ks)).to(torch.bfloat16)
    else:
        kh = case.k_pre
    ref = oracle.prefix_decode(case.q_tgt, kh, vh, case.cu_pre, case.k_tgt, case.v_tgt,
                               case.cu_q, 1.0 / np.sqrt(128))
    assert_close(out, lse, *ref, what=f"fp8 {mode} balanced tail")
    layers = torch.empty(bca.prefix_decode_fp8_workspace_bytes(mode, H, cap), dtype=torch.uint8,
                         device=DEV)
    out2, lse2 = bca.prefix_decode_fp8(*args, mode=mode, status=st, workspace=layers)
    assert bca.read_status(st) == 0
    assert_close(out2, lse2, *ref, what=f"fp8 {mode} key-split tail")


@pytest.mark.parametrize("H,tgt", [
    (3, [200, 0, 129]),   # a small batch with a zero-length target: pair grid only
    (1, [8000]),          # 32 pairs of 63 key tiles: the balanced tail
])
def test_decode_over_an_empty_cache(H, tgt):
    """No sequence has a prefix and the cache has capacity 0: the decode is plain
    attention of the targets over their own keys."""
    import oracle
    qt, kt, vt = (W.randn_bf16((sum(tgt), H, 128), s) for s in (51, 52, 53))
    cq = np.concatenate([[0], np.cumsum(tgt)]).astype(np.int32)
    cp = np.zeros(len(tgt) + 1, np.int32)
    empty = torch.empty((1, H, 0, 128), dtype=torch.bfloat16, device=DEV)
    if H == 1:
        assert bca.prefix_decode_workspace_bytes(len(tgt), H, max(tgt), 0) > 0
    st = bca.new_status(DEV)
    out, lse = bca.prefix_decode(qt.to(DEV), empty, empty, 0, _ti(cp), kt.to(DEV), vt.to(DEV),
                                 _ti(cq), max(tgt), 0, status=st)
    assert bca.read_status(st) == 0
    kp = torch.empty((0, H, 128), dtype=torch.bfloat16)
    ref = oracle.prefix_decode(qt, kp, kp, cp, kt, vt, cq, 1.0 / np.sqrt(128))
    assert_close(out, lse, *ref, what=f"empty cache {tgt}")


def test_workspace_bytes_follow_the_tail_plan():
    """Two 133,120-byte slots per key range, one range per SM, when the last wave is worth
    balancing (the edit decode's 56 pairs of 98 key tiles); none for a last wave whose
    ranges would be too short (the text-to-image decode: 56 pairs of 34 tiles), for a
    decode of whole waves, or for arguments out of range."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    items = 32 * 16                           # 32 heads x 16 pairs of 4096 target rows
    if not (0 < items % sms and items % sms < sms // 2 and sms <= 256):
        pytest.skip(f"{sms} SMs: the edit decode has no short last wave")
    assert bca.prefix_decode_workspace_bytes(1, 32, 4096, 8384) == 2 * sms * 133120
    assert bca.prefix_decode_workspace_bytes(1, 32, 4096, 256) == 0
    assert bca.prefix_decode_workspace_bytes(sms, 2, 256, 8384) == 0     # 2 x sms pairs
    assert bca.prefix_decode_workspace_bytes(0, 32, 4096, 8384) == 0
    assert bca.prefix_decode_workspace_bytes(1, 32, 4096, -1) == 0
    assert bca.prefix_decode_workspace_bytes(1, 32, 4096, 8384, head_dim=64) == 0
