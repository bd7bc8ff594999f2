"""FP8 E4M3 prefix cache on the GPU: quantising append (codes and scales bit-exact
against the oracle) and prefix decode over the quantised cache (against the oracle
run on the dequantised cache, and more accurate with V-only than K+V quantisation)."""
import numpy as np
import pytest
import torch

import prefix_kv_gb300 as bca
from oracle import fp8
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV

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
