"""Failure detection without a GPU fault: every wait inside the kernels is
bounded.  A test-only parameter makes the forward's work scheduler hand out
nothing; every other role's wait for work then runs out (about 2 s), the
kernel records ATTN_ERR_DEVICE_TIMEOUT with the wait that ran out first, frees
its tensor memory and returns.  The host reads that status, and the next
normal call on the same workspace (and the backward after it) is correct."""
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


def test_bounded_wait_runs_out_and_the_next_call_is_clean():
    from conftest import oracle_full
    from gpu_util import DevCase, check_backward, check_forward

    from bwd_tcgen05_tma_gb300 import attn as A

    # query heads in pairs over one KV head: the forward that has the knob
    case = I.synth("wt", B=1, Sq=400, Skv=400, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
                   fmt="THD_SEGMENTS", causal=True, seed=71, seg=(40, 300), pad_frac=0.05)
    d = DevCase(case)
    d.params.test_wait_timeout = 1
    o = torch.full((case.B * case.Sq, case.Hq, case.d_v), 7.0, dtype=torch.bfloat16,
                   device="cuda")
    lse = torch.full((case.B, case.Hq, case.Sq), 7.0, dtype=torch.float32, device="cuda")
    A.attn_fwd(d.params, o, lse, d.ws_fwd)
    st, stats = A.attn_read_status(d.ws_fwd)
    assert st == 6, f"expected ATTN_ERR_DEVICE_TIMEOUT, got {st}"
    assert stats.status == 6
    # the producer, the MMA issuer or a softmax warp of the forward
    assert stats.wait_site in {0x610, 0x620} | set(range(0x630, 0x638)), hex(stats.wait_site)
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)  # nothing was written
    # the context is usable and a normal call on the same workspace is correct
    d.params.test_wait_timeout = 0
    ref = oracle_full(case)
    o2, lse2 = d.forward()
    assert d.fwd_stats.status == 0 and d.fwd_stats.wait_site == 0
    check_forward(case, ref, o2, lse2)
    g, db = d.backward()
    check_backward(case, ref, g, db)
