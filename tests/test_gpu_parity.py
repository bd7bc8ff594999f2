"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Small cases compare every output; the full-size workloads compare every row of
sampled heads, or a seeded row sample that always holds every row of the first
and last tile of each sequence and the rows on each tile edge.
"""
import numpy as np
import pytest
import torch

import oracle
import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W
from gpu_cases import (DEV, SCALE, DecodeCase, PrefillCase, assert_close, ragged_case,
                       tile_boundary_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()
    assert torch.cuda.is_available()


def _status():
    return bca.new_status(DEV)


# ---------------------------------------------------------------- schedule prep

def _check_schedule(case, rows_per_seq=None):
    st = _status()
    row_end, tiles = bca.schedule_prep(torch.from_numpy(case.block_id).to(DEV),
                                       torch.from_numpy(case.cu_q).to(DEV),
                                       torch.from_numpy(case.cu_k).to(DEV), case.max_q,
                                       status=st)
    assert bca.read_status(st) == 0
    row_end, tiles = row_end.cpu().numpy(), tiles.cpu().numpy()
    for b in range(len(case.cu_q) - 1):
        q0, q1 = case.cu_q[b], case.cu_q[b + 1]
        k0, k1 = case.cu_k[b], case.cu_k[b + 1]
        local = np.arange(q1 - q0) if rows_per_seq is None else np.unique(
            np.concatenate([np.arange(min(q1 - q0, 130)),
                            np.random.default_rng(b).integers(0, max(1, q1 - q0),
                                                              size=rows_per_seq)]))
        local = local[local < q1 - q0]
        m = oracle.visibility(case.block_id[k0:k1], q1 - q0, local)
        e = row_end[q0 + local]
        # every row sees exactly the key prefix [0, e)
        assert (m == (np.arange(k1 - k0)[None, :] < e[:, None])).all(), b
        # tile records: max / min / count over the tile's rows
        for t in range((q1 - q0 + 127) // 128):
            er = row_end[q0 + t * 128: min(q1, q0 + t * 128 + 128)]
            assert tuple(tiles[b, t, :3]) == (er.max(), er.min(), er.size)
        assert (tiles[b, (q1 - q0 + 127) // 128:] == 0).all()


def test_schedule_tiny():
    _check_schedule(PrefillCase.from_workload(W.tiny_mixed()))


def test_schedule_ragged_bottom_right():
    _check_schedule(ragged_case(5, [1, 129, 300, 517, 256], [1, 100, 300, 260, 256]))


def test_schedule_many_runs():
    # many short spans, adjacent spans with distinct ids
    _check_schedule(ragged_case(6, [2000, 777], max_spans=200, max_span=9))


@pytest.mark.parametrize("wl", [W.edit_two_ref(), W.cfg_large_edit(), W.neo_mixed()],
                         ids=lambda w: w.name)
def test_schedule_full_size(wl):
    cu = wl.cu_seqlens()
    case = PrefillCase(torch.zeros(0), torch.zeros(0), torch.zeros(0), wl.block_id(), cu, cu)
    _check_schedule(case, rows_per_seq=400)


def test_schedule_rejects_split_id():
    bid = np.array([-1, 0, 0, -1, 0, 1, 1, -1], np.int32)      # id 0 in two runs
    cu = np.array([0, 8], np.int32)
    st = _status()
    _, tiles = bca.schedule_prep(torch.from_numpy(bid).to(DEV), torch.from_numpy(cu).to(DEV),
                                 torch.from_numpy(cu).to(DEV), 8, status=st)
    assert bca.read_status(st) == 3
    assert (tiles.cpu() == 0).all()


def test_schedule_rejects_bad_id_and_lengths():
    cu = np.array([0, 4], np.int32)
    st = _status()
    bca.schedule_prep(torch.tensor([-1, -2, 0, 0], dtype=torch.int32, device=DEV),
                      torch.from_numpy(cu).to(DEV), torch.from_numpy(cu).to(DEV), 4, status=st)
    assert bca.read_status(st) == 3
    st = _status()
    bca.schedule_prep(torch.tensor([-1, -1, 0, 0], dtype=torch.int32, device=DEV),
                      torch.tensor([0, 5], dtype=torch.int32, device=DEV),
                      torch.from_numpy(cu).to(DEV), 5, status=st)      # q_len > kv_len
    assert bca.read_status(st) == 8


def test_schedule_rejects_offsets_past_the_arrays():
    """A sequence whose offsets run past total_q (or total_k) fails with
    BCA_ERR_SEQLENS before any row end is written: a guard region behind row_end
    keeps its fill, and the sequence's tile records are zero."""
    from prefix_kv_gb300 import _native
    lib = _native.load()
    bid = torch.full((400,), -1, dtype=torch.int32, device=DEV)
    for cu_q, cu_k, total_q, total_k in (
            ([0, 200, 400], [0, 200, 400], 272, 400),     # cu_q[2] = total_q + 128
            ([0, 200, 400], [0, 200, 400], 400, 272),     # cu_k[2] past total_k
            ([0, -8, 400], [0, 200, 400], 400, 400)):     # negative offset
        cq = torch.tensor(cu_q, dtype=torch.int32, device=DEV)
        ck = torch.tensor(cu_k, dtype=torch.int32, device=DEV)
        row_end = torch.full((total_q + 256,), -5, dtype=torch.int32, device=DEV)
        tiles = torch.full((2, 2, 4), -5, dtype=torch.int32, device=DEV)
        st = _status()
        code = lib.bca_schedule_prep(bid.data_ptr(), cq.data_ptr(), ck.data_ptr(), 2, total_q,
                                     total_k, 256, row_end.data_ptr(), tiles.data_ptr(),
                                     st.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert code == 0
        assert bca.read_status(st) == 8, (cu_q, cu_k, total_q, total_k)
        assert (row_end[total_q:] == -5).all()
        assert (tiles[1] == 0).all()


def _ids(*runs):
    """Block ids from (id, length) runs."""
    return np.concatenate([np.full(n, i, np.int32) for i, n in runs])


def _raw_prep(bid, cu_q, cu_k, max_q):
    """bca_schedule_prep into buffers filled with -5 (so that zeroed records are the
    kernel's writes): (status, row_end, tiles) on the host."""
    from prefix_kv_gb300 import _native
    ti = lambda a: torch.from_numpy(np.asarray(a, np.int32)).to(DEV)
    bid_d, cq, ck = ti(bid), ti(cu_q), ti(cu_k)
    batch, tps = len(cu_q) - 1, (max_q + 127) // 128
    row_end = torch.full((int(cu_q[-1]),), -5, dtype=torch.int32, device=DEV)
    tiles = torch.full((batch, tps, 4), -5, dtype=torch.int32, device=DEV)
    st = _status()
    code = _native.load().bca_schedule_prep(
        bid_d.data_ptr(), cq.data_ptr(), ck.data_ptr(), batch, int(cu_q[-1]), len(bid), max_q,
        row_end.data_ptr(), tiles.data_ptr(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 0
    return bca.read_status(st), row_end.cpu().numpy(), tiles.cpu().numpy()


def _packed_case(seqs):
    """(block ids, q_len or None for q_len = kv_len) per sequence -> a schedule-only case."""
    kv = [len(s) for s, _ in seqs]
    ql = [len(s) if q is None else q for s, q in seqs]
    cu_k = np.concatenate([[0], np.cumsum(kv)]).astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return PrefillCase(torch.zeros(0), torch.zeros(0), torch.zeros(0),
                       np.concatenate([s for s, _ in seqs]), cu_q, cu_k)


def test_schedule_rows_over_several_chunks():
    """The prep works in 1024-row chunks of a sequence: image runs crossing chunk
    edges, a sequence whose last chunk holds one row, bottom-right rows whose first
    row lies inside an image, and shorter sequences whose last chunks have no rows
    (their tile records stay zero)."""
    case = _packed_case([
        (_ids((-1, 100), (0, 1900), (-1, 30), (1, 1019)), None),     # run 0 spans rows 100..1999
        (_ids((-1, 1), (0, 1024)), None),                            # 1025 rows
        (_ids((-1, 5), (3, 4000), (-1, 7), (4, 1300)), 2500),        # rows = keys 2812..5311
        (_ids((2, 1023)), None),                                     # one image, one chunk
        (_ids((-1, 700)), None),                                     # text only
    ])
    _check_schedule(case)
    # the same into buffers filled with -5: every row end and every record (zeroed
    # ones included) is written by the kernel
    code, row_end, tiles = _raw_prep(case.block_id, case.cu_q, case.cu_k, case.max_q)
    assert code == 0 and (row_end >= 1).all()
    for b in range(len(case.cu_q) - 1):
        n_t = (int(case.cu_q[b + 1] - case.cu_q[b]) + 127) // 128
        assert (tiles[b, :n_t, :3] > 0).all() and (tiles[b, n_t:] == 0).all()


def test_schedule_split_id_past_the_first_chunks():
    """An id split into two runs beyond the first 8192 positions fails its whole
    sequence (every chunk's tile records zero); the other sequence of the batch
    is scheduled as usual."""
    good = _ids((-1, 64), (0, 2000), (-1, 16))
    bad = _ids((-1, 9000), (7, 50), (-1, 200), (7, 10), (-1, 40))
    case = _packed_case([(good, None), (bad, None)])
    code, row_end, tiles = _raw_prep(case.block_id, case.cu_q, case.cu_k, case.max_q)
    assert code == 3
    assert (tiles[1] == 0).all()
    n = len(good)
    m = oracle.visibility(good, n, np.arange(n))
    assert (m == (np.arange(n)[None, :] < row_end[:n, None])).all()
    for t in range((n + 127) // 128):
        er = row_end[t * 128: min(n, t * 128 + 128)]
        assert tuple(tiles[0, t, :3]) == (er.max(), er.min(), er.size)
    assert (tiles[0, (n + 127) // 128:] == 0).all()


def test_schedule_run_count_limit():
    """1024 image runs in a sequence are scheduled; 1025 give BCA_ERR_UNSUPPORTED
    with zeroed tile records."""
    at_limit = np.repeat(np.arange(1024, dtype=np.int32), 2)      # 1024 two-token images
    _check_schedule(_packed_case([(at_limit, None)]))
    over = np.arange(1025, dtype=np.int32)                         # 1025 one-token images
    cu = np.array([0, 1025], np.int32)
    code, _, tiles = _raw_prep(over, cu, cu, 1025)
    assert code == 2
    assert (tiles == 0).all()


# ---------------------------------------------------------------- prefill

def test_prefill_tiny_all_outputs():
    case = PrefillCase.from_workload(W.tiny_mixed())
    st = _status()
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="tiny")


@pytest.mark.parametrize("seed,kv,ql", [
    (11, [1, 129, 300, 517], None),
    (12, [640, 200, 1000], [640, 33, 999]),       # bottom-right rows
    (13, [128, 256, 384], [1, 128, 2]),
    (14, [1537], None),
])
def test_prefill_ragged_varlen(seed, kv, ql):
    case = ragged_case(seed, kv, ql)
    st = _status()
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what=f"ragged{seed}")


@pytest.mark.parametrize("heads", [12, 16, 20])
def test_prefill_head_groups(heads):
    # the grid runs the heads in groups (6 x 2, 8 x 2, 5 x 4 here): every head's rows
    case = ragged_case(30 + heads, [700, 260], heads=heads)
    out, lse = case.run()
    assert_close(out, lse, *case.reference(), what=f"heads{heads}")


def test_prefill_adjacent_spans_and_many_runs():
    case = ragged_case(21, [1200, 333], max_spans=40, max_span=40)
    out, lse = case.run()
    assert_close(out, lse, *case.reference(), what="many runs")


def test_prefill_all_text_and_single_block():
    for bid_val in (-1, 0):
        case = ragged_case(31, [700])
        case.block_id[:] = bid_val
        out, lse = case.run()
        assert_close(out, lse, *case.reference(), what=f"uniform id {bid_val}")


def test_prefill_large_scores():
    case = ragged_case(41, [300, 260])
    case.q = (case.q.float() * 8).to(torch.bfloat16)
    out, lse = case.run()
    assert_close(out, lse, *case.reference(), what="large scores")


def test_prefill_prefix_rows_ignore_target():
    """The prefix cannot read the target: changing target q/k/v leaves every prefix row
    bit-identical on the GPU too (target keys lie outside every prefix row's range)."""
    wl = W.tiny_mixed()
    case = PrefillCase.from_workload(wl)
    out1, lse1 = case.run()
    tr = torch.from_numpy(wl.target_rows())
    case.q[tr] = W.randn_bf16((len(tr), 2, 128), 99)
    case.k[tr] = W.randn_bf16((len(tr), 2, 128), 98)
    case.v[tr] = W.randn_bf16((len(tr), 2, 128), 97)
    out2, lse2 = case.run()
    P = wl.prefix_lens()[0]
    assert torch.equal(out1[:P], out2[:P]) and torch.equal(lse1[:, :P], lse2[:, :P])
    assert not torch.equal(out1[P:], out2[P:])


def test_prefill_invalid_sequence_left_untouched():
    case = ragged_case(51, [200, 300])
    case.block_id[10:20] = 5
    case.block_id[30:40] = 5          # id 5 split into two runs in sequence 0
    sentinel = torch.full((500, 3, 128), 7.0, dtype=torch.bfloat16, device=DEV)
    st = _status()
    out, lse = case.run(status=st, out=sentinel)
    assert bca.read_status(st) == 3
    assert (out[:200].float() == 7.0).all()
    ref_out, ref_lse = case.reference(rows=np.arange(200, 500))
    assert_close(out, lse, ref_out, ref_lse, rows=np.arange(200, 500), what="valid seq")


@pytest.mark.parametrize("wl,heads", [(W.t2i_1024(), [0, 13, 31]),
                                      (W.edit_two_ref(), [5, 30])], ids=lambda x: getattr(x, "name", ""))
def test_prefill_full_size_all_rows(wl, heads):
    case = PrefillCase.from_workload(wl)
    out, lse = case.run()
    assert_close(out, lse, *case.reference(heads=np.array(heads)), heads=heads, what=wl.name)


@pytest.mark.parametrize("wl", [W.cfg_large_edit(), W.neo_mixed()], ids=lambda w: w.name)
def test_prefill_full_size_sampled_rows(wl):
    case = PrefillCase.from_workload(wl)
    out, lse = case.run()
    rows = tile_boundary_rows(case.cu_q, extra=256, seed=1)
    heads = np.array([3, 28])
    ref = case.reference(rows=rows, heads=heads)
    assert_close(out, lse, *ref, rows=rows, heads=heads, what=wl.name)


@pytest.mark.parametrize("kv,ql", [([2300, 2400], [2300, 1900]), ([2300, 260], [2300, 200])],
                         ids=["long", "short-second"])
def test_prefill_key_split_tail_ragged(kv, ql):
    """32 heads, a sequence of 2300 and a bottom-right one: a pair grid of 8 x 9 x 8 =
    576 CTAs, whose 120 cheapest pairs (the first two tile pairs of every sequence and
    head) run as key-split single tiles: rows that see no key of warpgroup 1's half,
    random layouts.  With a 200-row second sequence its only pair (a ragged second
    tile of 72 rows) is among them, and so are items past that sequence's end."""
    case = ragged_case(31, kv, ql, heads=32, max_spans=6, max_span=700)
    out, lse = case.run()
    rows = np.unique(np.concatenate([tile_boundary_rows(case.cu_q[:2], extra=64, seed=2),
                                     np.arange(2300, 2300 + ql[1])]))   # every row of sequence 1
    heads = np.array([0, 17, 24, 31])
    ref = case.reference(rows=rows, heads=heads)
    assert_close(out, lse, *ref, rows=rows, heads=heads, what="key-split tail")


# ---------------------------------------------------------------- decode

def test_decode_tiny():
    case = DecodeCase.from_workload(W.tiny_mixed())
    st = _status()
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="decode tiny")


@pytest.mark.parametrize("seed,pre,tgt", [
    (61, [24, 0, 300, 129], [16, 200, 1, 256]),
    (62, [1000], [130]),
    (63, [128, 256], [128, 384]),
    (64, [0, 5, 0], [100, 3, 128]),   # a single key tile: nothing to split
])
def test_decode_ragged(seed, pre, tgt):
    H = 3
    kp = W.randn_bf16((sum(pre), H, 128), seed)
    vp = W.randn_bf16((sum(pre), H, 128), seed + 100)
    qt = W.randn_bf16((sum(tgt), H, 128), seed + 200)
    kt = W.randn_bf16((sum(tgt), H, 128), seed + 300)
    vt = W.randn_bf16((sum(tgt), H, 128), seed + 400)
    cu_p = np.concatenate([[0], np.cumsum(pre)])
    cu_q = np.concatenate([[0], np.cumsum(tgt)])
    # unused cache capacity holds NaN: only the prefix may be read
    case = DecodeCase(qt, kt, vt, kp, vp, cu_q, cu_p, layers=2, layer=1, cache_fill=float("nan"))
    st = _status()
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what=f"decode{seed}")


def test_decode_pair_grid_and_tail_ragged():
    # 8 heads x 5 sequences x 4 pairs = 160 items on a 152-SM GB300: 152 run in the pair
    # grid and 8 as 16 key-split tail CTAs; ragged lengths leave some pairs half or wholly
    # empty, and one sequence has no prefix
    H = 8
    pre, tgt = [900, 0, 333, 1500, 128], [1000, 700, 1024, 5, 257]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    items = H * 4 * len(tgt)
    if not (items > sms and 0 < items % sms <= sms // 2):
        pytest.skip(f"{sms} SMs: this shape does not give both decode grids")
    kp = W.randn_bf16((sum(pre), H, 128), 81)
    vp = W.randn_bf16((sum(pre), H, 128), 82)
    qt = W.randn_bf16((sum(tgt), H, 128), 83)
    kt = W.randn_bf16((sum(tgt), H, 128), 84)
    vt = W.randn_bf16((sum(tgt), H, 128), 85)
    cu_p = np.concatenate([[0], np.cumsum(pre)])
    cu_q = np.concatenate([[0], np.cumsum(tgt)])
    case = DecodeCase(qt, kt, vt, kp, vp, cu_q, cu_p, layers=1, layer=0, cache_fill=float("nan"))
    st = _status()
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what="pairs+tail")


# heads 28-31 hold the last 56 tile pairs, the decode's last partial wave: the balanced
# tail's pieces and merge on the edit workload, key-split tiles on text-to-image
@pytest.mark.parametrize("wl,heads", [(W.t2i_1024(), [1, 30]), (W.edit_two_ref(), [2, 17, 31])],
                         ids=lambda x: getattr(x, "name", ""))
def test_decode_full_size(wl, heads):
    case = DecodeCase.from_workload(wl)
    out, lse = case.run()
    assert_close(out, lse, *case.reference(heads=np.array(heads)), heads=heads, what=wl.name)


def test_decode_cfg_sampled_rows():
    wl = W.cfg_large_edit()
    case = DecodeCase.from_workload(wl)
    out, lse = case.run()
    rows = tile_boundary_rows(case.cu_q, extra=128, seed=2)
    heads = np.array([9])
    assert_close(out, lse, *case.reference(rows=rows, heads=heads), rows=rows, heads=heads,
                 what=wl.name)


def test_decode_capacity_overflow_reported():
    case = DecodeCase.from_workload(W.tiny_mixed())
    st = _status()
    bca.prefix_decode(case.q_tgt.to(DEV), case.cache_k[:, :, :20].contiguous().to(DEV),
                      case.cache_v[:, :, :20].contiguous().to(DEV), 0,
                      torch.from_numpy(case.cu_pre).to(DEV), case.k_tgt.to(DEV),
                      case.v_tgt.to(DEV), torch.from_numpy(case.cu_q).to(DEV), 16, 24,
                      status=st)
    assert bca.read_status(st) == 5


def test_decode_rejects_query_offsets_past_total_q():
    """Target offsets that run past total_q: that sequence fails with BCA_ERR_SEQLENS
    and nothing is written behind the output or the LSE; the first sequence is
    still computed."""
    from prefix_kv_gb300 import _native
    lib = _native.load()
    H, P = 2, 200
    tq_all = 300
    q = W.randn_bf16((tq_all, H, 128), 91).to(DEV)
    kt = W.randn_bf16((tq_all, H, 128), 92).to(DEV)
    vt = W.randn_bf16((tq_all, H, 128), 93).to(DEV)
    ck = W.randn_bf16((1, H, 2 * P, 128), 94).to(DEV)
    cv = W.randn_bf16((1, H, 2 * P, 128), 95).to(DEV)
    cu_q = torch.tensor([0, 100, 300], dtype=torch.int32, device=DEV)
    cu_p = torch.tensor([0, P, 2 * P], dtype=torch.int32, device=DEV)
    total_q = 172                                   # cu_q[2] = total_q + 128
    out_buf = torch.full((total_q + 256, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse_buf = torch.full((H * total_q + 256,), float("nan"), dtype=torch.float32, device=DEV)
    st = _status()
    code = lib.bca_prefix_decode(q.data_ptr(), ck.data_ptr(), cv.data_ptr(), 0, 1, 2 * P,
                                 cu_p.data_ptr(), kt.data_ptr(), vt.data_ptr(), cu_q.data_ptr(),
                                 2, H, 128, total_q, 200, P, SCALE, out_buf.data_ptr(),
                                 lse_buf.data_ptr(), None, 0, st.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
    assert code == 0
    assert bca.read_status(st) == 8
    assert torch.isnan(out_buf[100:].float()).all() and torch.isnan(lse_buf[H * total_q:]).all()
    lse = lse_buf[:H * total_q].view(H, total_q)
    ref_out, ref_lse = oracle.prefix_decode(
        q[:100].cpu(), ck[0, :, :P].permute(1, 0, 2).cpu(), cv[0, :, :P].permute(1, 0, 2).cpu(),
        np.array([0, P]), kt[:100].cpu(), vt[:100].cpu(), np.array([0, 100]), SCALE)
    assert_close(out_buf[:100], lse[:, :100], ref_out, ref_lse, what="first sequence")


# ---------------------------------------------------------------- cache append

def _append_expected(k, v, cu_k, cu_p, layers, layer, cap):
    H = k.shape[1]
    ek = np.full((layers, H, cap, 128), -1, dtype=np.int16)
    ev = ek.copy()
    oracle.cache_append(k.view(torch.int16).numpy(), v.view(torch.int16).numpy(), cu_k, cu_p,
                        ek, ev, layer)
    return ek, ev


@pytest.mark.parametrize("seed,kv,pre", [(71, [40], [24]), (72, [300, 5, 129], [299, 0, 128])])
def test_append_bit_exact(seed, kv, pre):
    H, layers, layer = 3, 3, 2
    k = W.randn_bf16((sum(kv), H, 128), seed)
    v = W.randn_bf16((sum(kv), H, 128), seed + 1)
    cu_k = np.concatenate([[0], np.cumsum(kv)]).astype(np.int32)
    cu_p = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cap = int(cu_p[-1]) + 7
    ck = torch.full((layers, H, cap, 128), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    cv = ck.clone()
    st = _status()
    bca.prefix_cache_append(k.to(DEV), v.to(DEV), torch.from_numpy(cu_k).to(DEV),
                            torch.from_numpy(cu_p).to(DEV), ck, cv, layer, status=st)
    assert bca.read_status(st) == 0
    ek, ev = _append_expected(k, v, cu_k, cu_p, layers, layer, cap)
    assert np.array_equal(ck.view(torch.int16).cpu().numpy(), ek)
    assert np.array_equal(cv.view(torch.int16).cpu().numpy(), ev)


def test_append_full_size_edit():
    wl = W.edit_two_ref()
    _, k, v = W.make_qkv(wl)
    cu_k, cu_p = wl.cu_seqlens(), wl.cu_prefix()
    cap = int(cu_p[-1])
    ck = torch.zeros((2, 32, cap, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    bca.prefix_cache_append(k.to(DEV), v.to(DEV), torch.from_numpy(cu_k).to(DEV),
                            torch.from_numpy(cu_p).to(DEV), ck, cv, 1)
    P = wl.prefix_lens()[0]
    assert torch.equal(ck[1].cpu(), k[:P].permute(1, 0, 2))
    assert torch.equal(cv[1].cpu(), v[:P].permute(1, 0, 2))
    assert (ck[0] == 0).all()


def test_append_rejects_overflow_and_long_prefix():
    k = W.randn_bf16((10, 2, 128), 1).to(DEV)
    ck = torch.zeros((1, 2, 8, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    st = _status()
    bca.prefix_cache_append(k, k, torch.tensor([0, 10], dtype=torch.int32, device=DEV),
                            torch.tensor([0, 9], dtype=torch.int32, device=DEV), ck, cv, 0,
                            status=st)
    assert bca.read_status(st) == 5 and (ck == 0).all()
    st = _status()
    bca.prefix_cache_append(k, k, torch.tensor([0, 4, 10], dtype=torch.int32, device=DEV),
                            torch.tensor([0, 5, 6], dtype=torch.int32, device=DEV), ck, cv, 0,
                            status=st)
    assert bca.read_status(st) == 8 and (ck == 0).all()


# ---------------------------------------------------------------- the whole path

@pytest.mark.parametrize("wl", [W.tiny_mixed(), W.edit_two_ref()], ids=lambda w: w.name)
def test_prefill_append_decode_pipeline(wl):
    """extract step (prefill + append) then a cached step (decode) over the cache:
    decode equals the oracle, and equals the prefill's target rows within tolerance."""
    q, k, v = W.make_qkv(wl)
    cu = torch.from_numpy(wl.cu_seqlens()).to(DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    st = _status()
    S = wl.seq_lens[0]
    out, lse = bca.prefill(qd, kd, vd, torch.from_numpy(wl.block_id()).to(DEV), cu, cu, S, S,
                           status=st)
    cu_p = torch.from_numpy(wl.cu_prefix()).to(DEV)
    cap = int(wl.cu_prefix()[-1])
    ck = torch.empty((1, wl.num_heads, cap, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.empty_like(ck)
    bca.prefix_cache_append(kd, vd, cu, cu_p, ck, cv, 0, status=st)
    tr = torch.from_numpy(wl.target_rows()).to(DEV)
    cu_t = torch.from_numpy(wl.cu_target()).to(DEV)
    dout, dlse = bca.prefix_decode(qd[tr].contiguous(), ck, cv, 0, cu_p, kd[tr].contiguous(),
                                   vd[tr].contiguous(), cu_t, wl.target_lens()[0],
                                   wl.prefix_lens()[0], status=st)
    assert bca.read_status(st) == 0
    # cached == uncached within the output tolerance
    d = (dout.float() - out[tr].float()).abs()
    assert d.max().item() <= 2e-2 and d.mean().item() <= 2e-3
    heads = np.array([0, wl.num_heads - 1])
    P = wl.prefix_lens()[0]
    ref = oracle.prefix_decode(q[wl.target_rows()], k[:P], v[:P], wl.cu_prefix(),
                               k[wl.target_rows()], v[wl.target_rows()], wl.cu_target(),
                               1.0 / np.sqrt(128), heads=heads)
    assert_close(dout, dlse, *ref, heads=heads, what="pipeline decode")
