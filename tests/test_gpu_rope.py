"""Q/K prologue on the GPU (RoPE coordinates, rotation table, fused RMS norm +
three-axis RoPE + cache append) against the CPU oracle.

Tolerances: coordinates bit-exact (integer work); table |cos, sin - ref| <= 1e-6
(fp32 rounding of double-precision values); q_out / k_out per element
|gpu - ref| <= 2^-8 |ref| + 2^-16 max|row| (one bf16 rounding of an fp32 result
whose own error is ~1e-6 of the row's scale).  The cache K row must equal the
k_out row bit for bit and the cache V row the input v row.
"""
import numpy as np
import pytest
import torch

import prefix_kv_gb300 as bca
from oracle import rope
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()


def _ti(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _positions(bid, cu, gw, status=None):
    return bca.rope_positions(_ti(bid.astype(np.int32)), _ti(cu.astype(np.int32)),
                              _ti(gw.astype(np.int32)), status=status)


@pytest.mark.parametrize("wl", W.all_workloads(), ids=lambda w: w.name)
def test_positions_bit_exact(wl):
    bid, cu, gw = wl.block_id(), wl.cu_seqlens(), wl.grid_widths()
    st = bca.new_status(DEV)
    got = _positions(bid, cu, gw, st).cpu().numpy()
    assert bca.read_status(st) == 0
    assert np.array_equal(got, rope.rope_positions(bid, cu, gw))


def test_positions_ragged_layouts():
    rng = np.random.default_rng(3)
    for trial in range(6):
        segs_all, bids = [], []
        for _ in range(int(rng.integers(1, 5))):
            L = int(rng.integers(1, 3000))
            segs = W.random_layout(rng, L, max_span=300)
            segs_all.append(segs)
            bids.append(np.concatenate([np.full(s.length, s.block, np.int32) for s in segs]))
        n_ids = 1 + max([s.block for segs in segs_all for s in segs] + [0])
        gw = np.zeros((len(segs_all), n_ids), np.int32)
        for b, segs in enumerate(segs_all):
            for s in segs:
                if s.is_image:
                    divs = [d for d in range(1, s.length + 1) if s.length % d == 0]
                    gw[b, s.block] = divs[int(rng.integers(0, len(divs)))]
        bid = np.concatenate(bids)
        cu = np.concatenate([[0], np.cumsum([len(x) for x in bids])]).astype(np.int32)
        st = bca.new_status(DEV)
        got = _positions(bid, cu, gw, st).cpu().numpy()
        assert bca.read_status(st) == 0
        assert np.array_equal(got, rope.rope_positions(bid, cu, gw)), trial


@pytest.mark.parametrize("bad", ["width", "id_range", "split_id"])
def test_positions_rejects_bad_layout(bad):
    bid = np.array([-1, 0, 0, 0, 0, 0, 0, -1, 1, 1], np.int32)
    gw = np.array([[3, 2]], np.int32)
    if bad == "width":
        gw[0, 0] = 4                      # 6 tokens are not rows of 4
    elif bad == "id_range":
        bid[8:] = 2
    else:
        bid[8:] = 0                       # id 0 in two runs
    st = bca.new_status(DEV)
    out = _positions(bid, np.array([0, 10]), gw, st)
    torch.cuda.synchronize()
    assert bca.read_status(st) == 3


def test_table_matches_angles():
    wl = W.cfg_large_edit()
    pos = rope.rope_positions(wl.block_id(), wl.cu_seqlens(), wl.grid_widths())
    tab = bca.rope_table(_ti(pos.astype(np.int32))).cpu().numpy().astype(np.float64)
    th = rope.rope_angles(pos)
    assert np.abs(tab[..., 0] - np.cos(th)).max() <= 1e-6
    assert np.abs(tab[..., 1] - np.sin(th)).max() <= 1e-6


def _assert_rot_close(got, ref, what):
    g = got.float().cpu().numpy().astype(np.float64)
    rowmax = np.abs(ref).max(axis=-1, keepdims=True)
    err = np.abs(g - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -16 * rowmax
    assert np.all(np.isfinite(g)), what
    assert np.all(err <= bound), f"{what}: worst excess {(err - bound).max():.3e}"


class PrologueCase:
    def __init__(self, wl, layers=2, layer=1, with_gamma=True, seed=7):
        self.wl = wl
        g = torch.Generator("cpu")
        g.manual_seed(seed)
        shape = (wl.total, wl.num_heads, 128)
        self.q = (torch.randn(shape, generator=g) * 3).to(torch.bfloat16)
        self.k = (torch.randn(shape, generator=g) * 0.2).to(torch.bfloat16)
        self.v = torch.randn(shape, generator=g).to(torch.bfloat16)
        self.gq = (1 + 0.5 * torch.randn(128, generator=g)).float() if with_gamma else None
        self.gk = (1 + 0.5 * torch.randn(128, generator=g)).float() if with_gamma else None
        self.pos = rope.rope_positions(wl.block_id(), wl.cu_seqlens(), wl.grid_widths())
        self.cu, self.cp = wl.cu_seqlens(), wl.cu_prefix()
        self.layers, self.layer = layers, layer
        self.cap = int(self.cp[-1]) + 40

    def run(self, append=True, in_place=False, cap=None, status=None):
        cap = self.cap if cap is None else cap
        d = lambda t: None if t is None else t.to(DEV)
        q, k, v = d(self.q), d(self.k), d(self.v)
        table = bca.rope_table(_ti(self.pos.astype(np.int32)))
        ck = torch.full((self.layers, self.wl.num_heads, cap, 128), 7.0, dtype=torch.bfloat16,
                        device=DEV)
        cv = torch.full_like(ck, 7.0)
        kw = dict(q_out=q, k_out=k) if in_place else {}
        qo, ko = bca.qk_norm_rope_append(
            q, k, table, _ti(self.cu), v=v if append else None,
            cu_prefix=_ti(self.cp) if append else None, cache_k=ck if append else None,
            cache_v=cv if append else None, layer=self.layer, gamma_q=d(self.gq),
            gamma_k=d(self.gk), status=status, **kw)
        return qo, ko, ck, cv

    def reference(self):
        return rope.qk_norm_rope(self.q, self.k, self.gq, self.gk, self.pos)


@pytest.mark.parametrize("wl", [W.tiny_mixed(), W.t2i_1024(), W.edit_two_ref()],
                         ids=lambda w: w.name)
def test_fused_against_oracle(wl):
    case = PrologueCase(wl)
    st = bca.new_status(DEV)
    qo, ko, ck, cv = case.run(status=st)
    assert bca.read_status(st) == 0
    rq, rk = case.reference()
    _assert_rot_close(qo, rq, "q")
    _assert_rot_close(ko, rk, "k")
    # the cache: prefix rows are the k_out rows bit for bit and the v rows; the rest untouched
    ck_, cv_ = ck[case.layer].cpu(), cv[case.layer].cpu()
    for b in range(wl.batch):
        n = int(case.cp[b + 1] - case.cp[b])
        src = slice(int(case.cu[b]), int(case.cu[b]) + n)
        dst = slice(int(case.cp[b]), int(case.cp[b]) + n)
        assert torch.equal(ck_[:, dst].view(torch.int16), ko.cpu()[src].transpose(0, 1).view(torch.int16))
        assert torch.equal(cv_[:, dst].view(torch.int16), case.v[src].transpose(0, 1).view(torch.int16))
    assert bool((ck[0] == 7).all()) and bool((ck_[:, int(case.cp[-1]):] == 7).all())
    assert bool((cv_[:, int(case.cp[-1]):] == 7).all())


def test_fused_varlen_batch_and_no_gamma():
    case = PrologueCase(W.neo_mixed(n_seqs=6, lo=200, hi=900, image_total=120), with_gamma=False)
    qo, ko, ck, _ = case.run()
    rq, rk = case.reference()
    _assert_rot_close(qo, rq, "q")
    _assert_rot_close(ko, rk, "k")


def test_in_place_and_no_append_give_the_same_bits():
    case = PrologueCase(W.tiny_mixed())
    qo, ko, _, _ = case.run()
    qi, ki, _, _ = case.run(in_place=True)
    qn, kn, ckn, _ = case.run(append=False)
    for a, b in ((qo, qi), (ko, ki), (qo, qn), (ko, kn)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert bool((ckn == 7).all())


def test_fused_capacity_overflow_writes_nothing():
    case = PrologueCase(W.tiny_mixed())
    st = bca.new_status(DEV)
    qo, ko, ck, cv = case.run(cap=int(case.cp[-1]) - 1, status=st)
    assert bca.read_status(st) == 5
    assert bool((ck == 7).all()) and bool((cv == 7).all())
