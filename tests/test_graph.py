"""A forward + backward captured into a CUDA graph replays to the same bits as
the same calls run eagerly.  The deterministic backward forks its dQ pass onto
a second stream and joins it again; capture must follow that fork."""
import pytest
import torch

from bwd_tcgen05_tma_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_tcgen05_tma_gb300 import build

    build.build()


@pytest.mark.parametrize("metadata_from_forward", [False, True])
def test_graph_replay_matches_eager(metadata_from_forward):
    from gpu_util import DevCase

    from bwd_tcgen05_tma_gb300 import attn as A

    case = I.synth("thd", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
                   fmt="THD_SEGMENTS", causal=True, seed=41, seg=(40, 400), pad_frac=0.05)
    d = DevCase(case, dq_mode="deterministic")
    d.params.metadata_from_forward = 1 if metadata_from_forward else 0
    ws = d.ws_bwd  # large enough for both passes
    o = torch.empty((case.B * case.Sq, case.Hq, case.d_v), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((case.B, case.Hq, case.Sq), dtype=torch.float32, device="cuda")
    g, (dq, dk, dv) = d.grad_buffers()

    def step():
        A.attn_fwd(d.params, o, lse, ws)
        A.attn_bwd(d.params, o, d.do, lse, dq, dk, dv, None, ws)

    step()  # eager (also makes the library's second stream outside capture)
    st, _ = A.attn_read_status(ws)
    assert st == 0
    ref_o, ref_lse = o.clone(), lse.clone()
    ref_g = {k: v.clone() for k, v in g.items()}

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            step()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        for v in g.values():
            v.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        st, _ = A.attn_read_status(ws)
        assert st == 0
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(lse, ref_lse)
        for k in ref_g:
            assert torch.equal(g[k].view(torch.int16), ref_g[k].view(torch.int16)), k
