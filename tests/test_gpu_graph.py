"""The whole step (prefill with the prefix cache append, then prefix decode) captured
into a CUDA graph and replayed: the replay's outputs, LSE and cache rows are
bit-identical to the eager calls'.  Every kernel launches on the caller's stream; the
prefill's attention grid (a programmatic dependent of the schedule prep), its key-split
grid and the decode's balanced-tail grids (the pieces, then their merge) are captured as
programmatic edges."""
import pytest
import torch

import prefix_kv_gb300 as bca
from prefix_kv_gb300 import workloads as W
from gpu_cases import DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from prefix_kv_gb300 import build_native
    build_native.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("wl", [W.t2i_1024(), W.edit_two_ref()], ids=lambda w: w.name)
def test_step_captured_in_a_cuda_graph(wl):
    q, k, v = [t.to(DEV) for t in W.make_qkv(wl)]
    bid = torch.from_numpy(wl.block_id()).to(DEV)
    cu = torch.from_numpy(wl.cu_seqlens()).to(DEV)
    S, H = wl.seq_lens[0], wl.num_heads
    P, N = wl.prefix_lens()[0], wl.target_lens()[0]
    tr = torch.from_numpy(wl.target_rows()).to(DEV)
    qt, kt, vt = q[tr].contiguous(), k[tr].contiguous(), v[tr].contiguous()
    cup = torch.tensor([0, P], dtype=torch.int32, device=DEV)
    cut = torch.tensor([0, N], dtype=torch.int32, device=DEV)
    ck = torch.zeros((1, H, P, 128), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    out, dout = torch.empty_like(q), torch.empty_like(qt)
    lse = torch.empty((H, S), dtype=torch.float32, device=DEV)
    dlse = torch.empty((H, N), dtype=torch.float32, device=DEV)
    ws = torch.empty(bca.prefill_workspace_bytes(1, S, S), dtype=torch.uint8, device=DEV)
    dws = torch.empty(bca.prefix_decode_workspace_bytes(1, H, N, P), dtype=torch.uint8,
                      device=DEV)
    st = bca.new_status(DEV)
    results = (out, lse, dout, dlse, ck, cv)

    def step():
        bca.prefill_append(q, k, v, bid, cu, cu, S, S, cup, ck, cv, 0, out=out, lse=lse,
                           workspace=ws, status=st)
        bca.prefix_decode(qt, ck, cv, 0, cup, kt, vt, cut, N, P, out=dout, lse=dlse, status=st,
                          workspace=dws)

    step()
    torch.cuda.synchronize()
    assert bca.read_status(st) == 0
    ref = [t.clone() for t in results]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):       # warm-up off the default stream before capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in results:
        t.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert bca.read_status(st) == 0
    for name, a, b in zip(("out", "lse", "dout", "dlse", "cache_k", "cache_v"), results, ref):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
