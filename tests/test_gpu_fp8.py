"""FP8 E4M3 prefix cache on the GPU: quantising append (codes and scales bit-exact
against the oracle) and prefix decode over the quantised cache (against the oracle
run on the dequantised cache, and more accurate with V-only than K+V quantisation)."""
import numpy as np
import pytest
import torch

import oracle
import prefix_kv_gb300 as bca
from oracle import fp8
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV, SCALE, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()


def _fp8_caches(layers, H, cap, mode, dev):
    kdt = torch.uint8 if mode == "kv" else torch.bfloat16
    ck = torch.zeros((layers, H, cap, 128), dtype=kdt, device=dev)
    cv = torch.zeros((layers, H, cap, 128), dtype=torch.uint8, device=dev)
    sk = torch.full((layers, H, cap), -1.0, dtype=torch.float32, device=dev)
    sv = torch.full((layers, H, cap), -1.0, dtype=torch.float32, device=dev)
    return ck, cv, sk, sv


@pytest.mark.parametrize("mode", ["v", "kv"])
@pytest.mark.parametrize("seed,kv,pre", [(101, [40], [24]), (102, [300, 5, 1000], [299, 0, 871])])
def test_append_fp8_bit_exact(mode, seed, kv, pre):
    H, layers, layer = 3, 2, 1
    k = (W.randn_bf16((sum(kv), H, 128), seed).float() * 3).to(torch.bfloat16)
    v = W.randn_bf16((sum(kv), H, 128), seed + 1)
    v[2, 1] = 0                                        # an all-zero row
    cu_k = np.concatenate([[0], np.cumsum(kv)]).astype(np.int32)
    cu_p = np.concatenate([[0], np.cumsum(pre)]).astype(np.int32)
    cap = int(cu_p[-1]) + 5
    ck, cv, sk, sv = _fp8_caches(layers, H, cap, mode, DEV)
    st = bca.new_status(DEV)
    bca.prefix_cache_append_fp8(k.to(DEV), v.to(DEV), torch.from_numpy(cu_k).to(DEV),
                                torch.from_numpy(cu_p).to(DEV), ck, cv,
                                sk if mode == "kv" else None, sv, layer, mode=mode, status=st)
    assert bca.read_status(st) == 0
    exp = {"k": np.zeros(tuple(ck.shape), np.uint8 if mode == "kv" else np.uint16),
           "v": np.zeros(tuple(cv.shape), np.uint8),
           "sk": np.full(tuple(sk.shape), -1.0, np.float32), "sv": np.full(tuple(sv.shape), -1.0, np.float32)}
    fp8.cache_append_fp8(k, v, cu_k, cu_p, mode, layer, exp)
    assert np.array_equal(cv.cpu().numpy(), exp["v"])
    assert np.array_equal(sv.cpu().numpy().view(np.uint32), exp["sv"].view(np.uint32))
    if mode == "kv":
        assert np.array_equal(ck.cpu().numpy(), exp["k"])
        assert np.array_equal(sk.cpu().numpy().view(np.uint32), exp["sk"].view(np.uint32))
    else:
        assert np.array_equal(ck.cpu().view(torch.int16).numpy().view(np.uint16), exp["k"])


def test_append_fp8_rejects_overflow():
    k = W.randn_bf16((10, 2, 128), 1).to(DEV)
    ck, cv, sk, sv = _fp8_caches(1, 2, 8, "kv", DEV)
    st = bca.new_status(DEV)
    bca.prefix_cache_append_fp8(k, k, torch.tensor([0, 10], dtype=torch.int32, device=DEV),
                                torch.tensor([0, 9], dtype=torch.int32, device=DEV),
                                ck, cv, sk, sv, 0, mode="kv", status=st)
    assert bca.read_status(st) == 5 and (cv == 0).all()


# ---------------------------------------------------------------- expansion back to bf16

def test_dequant_fp8_bit_exact_all_codes():
    """Every code under scales from 0 through subnormal to 1e30: bf16(value * scale)
    bit-exact against the oracle (NaN codes stay NaN); rows outside the prefix
    range are not written."""
    rng = np.random.default_rng(5)
    L, H, cap, layer = 2, 3, 700, 1
    codes = rng.integers(0, 256, size=(L, H, cap, 128), dtype=np.uint8)
    codes[layer, 0, 10, :] = np.arange(128, dtype=np.uint8)
    codes[layer, 0, 11, :] = np.arange(128, 256, dtype=np.uint8)
    scales = (np.exp(rng.uniform(np.log(1e-30), np.log(1e30), size=(L, H, cap)))).astype(np.float32)
    scales[layer, :, 10:12] = 1.0
    scales[layer, 1, 20] = 0.0
    scales[layer, 2, 21] = np.float32(1e-40)                     # subnormal scale
    cu_p = np.array([7, 300, 300, 650], dtype=np.int32)          # starts past token 0
    out = torch.full((H, cap, 128), 1.5, dtype=torch.bfloat16, device=DEV)
    st = bca.new_status(DEV)
    bca.prefix_cache_dequant_fp8(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV),
                                 torch.from_numpy(cu_p).to(DEV), layer, out=out, status=st)
    assert bca.read_status(st) == 0
    got = out.float().cpu().numpy()
    exp = fp8.dequantize_rows(codes[layer], scales[layer])           # [H, cap, 128] float32
    rows = slice(int(cu_p[0]), int(cu_p[-1]))
    g, e = got[:, rows], exp[:, rows]
    nan = np.isnan(e)
    assert np.array_equal(np.isnan(g), nan)
    assert np.array_equal(g[~nan].view(np.uint32), e[~nan].view(np.uint32))
    assert (got[:, :cu_p[0]] == 1.5).all() and (got[:, cu_p[-1]:] == 1.5).all()


def test_dequant_fp8_rejects_overflow():
    codes = torch.zeros((1, 2, 8, 128), dtype=torch.uint8, device=DEV)
    scales = torch.ones((1, 2, 8), dtype=torch.float32, device=DEV)
    out = torch.full((2, 8, 128), 1.5, dtype=torch.bfloat16, device=DEV)
    st = bca.new_status(DEV)
    bca.prefix_cache_dequant_fp8(codes, scales, torch.tensor([0, 9], dtype=torch.int32, device=DEV),
                                 0, out=out, status=st)
    assert bca.read_status(st) == 5 and (out == 1.5).all()


# ---------------------------------------------------------------- decode over the FP8 cache

def _dequantized(x):
    """The oracle's dequantised copy of packed bf16 rows [n, H, 128]."""
    codes, scales = fp8.quantize_rows(x)
    return torch.from_numpy(fp8.dequantize_rows(codes, scales)).to(torch.bfloat16)


class Fp8DecodeCase:
    """Prefix decode inputs with the prefix held in an FP8 cache that the oracle's
    quantising append wrote.  Capacity past the last prefix holds NaN codes and
    NaN scales: only the prefix rows may be read."""

    def __init__(self, qt, kt, vt, kp, vp, cu_q, cu_p, mode, layers=2, layer=1):
        self.qt, self.kt, self.vt, self.kp, self.vp = qt, kt, vt, kp, vp
        self.cu_q = np.asarray(cu_q, np.int32)
        self.cu_p = np.asarray(cu_p, np.int32)
        self.mode, self.layer = mode, layer
        H = qt.shape[1]
        cap = int(self.cu_p[-1]) + 64
        kshape = (layers, H, cap, 128)
        caches = {"k": np.full(kshape, 0x7F if mode == "kv" else 0x7FC0,
                               np.uint8 if mode == "kv" else np.uint16),
                  "v": np.full(kshape, 0x7F, np.uint8),
                  "sk": np.full(kshape[:3], np.nan, np.float32),
                  "sv": np.full(kshape[:3], np.nan, np.float32)}
        fp8.cache_append_fp8(kp, vp, self.cu_p, self.cu_p, mode, layer, caches)
        self.caches = caches
        self.max_q = int(np.diff(self.cu_q).max())
        self.max_pre = int(np.diff(self.cu_p).max())

    @classmethod
    def from_workload(cls, wl, mode):
        q, k, v = W.make_qkv(wl)
        tr, pr = wl.target_rows(), wl.prefix_rows()
        return cls(q[tr].contiguous(), k[tr].contiguous(), v[tr].contiguous(), k[pr].contiguous(),
                   v[pr].contiguous(), wl.cu_target(), wl.cu_prefix(), mode)

    def run(self, status=None, workspace=None):
        c = self.caches
        ck = torch.from_numpy(c["k"]) if self.mode == "kv" else \
            torch.from_numpy(c["k"].view(np.int16)).view(torch.bfloat16)
        d = lambda t: t.to(DEV)
        ti = lambda a: torch.from_numpy(a).to(DEV)
        return bca.prefix_decode_fp8(
            d(self.qt), d(ck), ti(c["v"]), ti(c["sk"]) if self.mode == "kv" else None, ti(c["sv"]),
            self.layer, ti(self.cu_p), d(self.kt), d(self.vt), ti(self.cu_q), self.max_q,
            self.max_pre, SCALE, mode=self.mode, workspace=workspace, status=status)

    def reference(self, quantised=True, rows=None, heads=None):
        kp, vp = self.kp, self.vp
        if quantised:
            vp = _dequantized(vp)
            if self.mode == "kv":
                kp = _dequantized(kp)
        return oracle.prefix_decode(self.qt, kp, vp, self.cu_p, self.kt, self.vt, self.cu_q, SCALE,
                                    rows=rows, heads=heads)


def _ragged(seed, pre, tgt, mode, H=3):
    kp = (W.randn_bf16((sum(pre), H, 128), seed).float() * 2).to(torch.bfloat16)
    vp = W.randn_bf16((sum(pre), H, 128), seed + 100)
    if sum(pre) > 3:
        vp[3, 0] = 0                                   # an all-zero row (scale 0)
    qt = W.randn_bf16((sum(tgt), H, 128), seed + 200)
    kt = W.randn_bf16((sum(tgt), H, 128), seed + 300)
    vt = W.randn_bf16((sum(tgt), H, 128), seed + 400)
    cu_p = np.concatenate([[0], np.cumsum(pre)])
    cu_q = np.concatenate([[0], np.cumsum(tgt)])
    return Fp8DecodeCase(qt, kt, vt, kp, vp, cu_q, cu_p, mode)


@pytest.mark.parametrize("mode", ["v", "kv"])
@pytest.mark.parametrize("seed,pre,tgt", [
    (71, [24, 0, 300, 129], [16, 200, 1, 256]),
    (72, [1000], [130]),
    (73, [128, 256], [128, 384]),
])
def test_decode_fp8_ragged(mode, seed, pre, tgt):
    case = _ragged(seed, pre, tgt, mode)
    st = bca.new_status(DEV)
    out, lse = case.run(status=st)
    assert bca.read_status(st) == 0
    assert_close(out, lse, *case.reference(), what=f"fp8 {mode} decode{seed}")


@pytest.mark.parametrize("mode", ["v", "kv"])
def test_decode_fp8_full_size_edit(mode):
    wl = W.edit_two_ref()
    case = Fp8DecodeCase.from_workload(wl, mode)
    out, lse = case.run()
    heads = np.array([3, 20])
    assert_close(out, lse, *case.reference(heads=heads), heads=heads, what=f"{wl.name} fp8 {mode}")


def test_decode_fp8_workspace_checked():
    case = _ragged(75, [200], [64], "kv")
    ws = torch.empty(bca.prefix_decode_fp8_workspace_bytes("kv", 3, case.caches["v"].shape[2]) - 256,
                     dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError, match="status 4 "):
        case.run(workspace=ws)


def test_decode_fp8_v_only_closer_than_kv():
    """Quantising V alone perturbs the output less than quantising K and V
    (both measured against the unquantised cache)."""
    heads = np.array([1])
    errs = {}
    for mode in ("v", "kv"):
        case = _ragged(74, [700, 333], [256, 100], mode)
        out, _ = case.run()
        ref, _ = case.reference(quantised=False, heads=heads)
        errs[mode] = float(np.abs(out.float().cpu().numpy()[:, heads] - ref).mean())
    assert 0 < errs["v"] < errs["kv"]
