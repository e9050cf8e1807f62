"""The forward entry point that allocates nothing (attn_fwd_noalloc).

Some callers cannot allocate device memory when they run attention (plugin
hosts that pass only inputs and outputs, runtimes that forbid allocation after
start-up, loops that cannot take cudaMalloc's implicit synchronisation).  The
no-allocation forward uses the library's fixed device scratch array instead of
a caller workspace.  This test checks, through the C ABI, that two calls in a
row on different problems (so stale scratch contents from the first call would
show up in the second) give bit for bit the O, LSE and max-logit of the
regular attn_fwd, and that a problem too large for the fixed scratch is
rejected without a launch.

It sits in its own file named to be collected last, so that a run stopping at
the first failure has already run every other test.
"""
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


def _cases():
    a = I.synth("na", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
                fmt="THD_SEGMENTS", causal=True, seed=41, seg=(40, 400), pad_frac=0.05)
    b = I.synth("nb", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192, d_v=128, layout="HD_HD_HD",
                fmt="THD_SEGMENTS", causal=False, seed=42, seg=(60, 200), kv_seg=(60, 300),
                bias_shape=(1, 2, 300, 520))
    return a, b


def test_noalloc_forward_matches_workspace_forward_twice():
    import ctypes

    from gpu_util import DevCase

    from bwd_tcgen05_tma_gb300 import attn as A

    for case in _cases():  # two calls in a row, different problems
        d = DevCase(case)
        # max-logit too: its -inf initialisation runs in the metadata kernel,
        # on the shared scratch's path
        ml_ref = torch.full((case.B, case.Hq), float("nan"), dtype=torch.float32, device="cuda")
        d.params.max_logit = ctypes.c_void_p(ml_ref.data_ptr())
        o_ref, lse_ref = d.forward()
        o_ref, lse_ref = o_ref.clone(), lse_ref.clone()
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        ml = torch.full_like(ml_ref, float("nan"))
        d.params.max_logit = ctypes.c_void_p(ml.data_ptr())
        A.attn_fwd_noalloc(d.params, o, lse)
        torch.cuda.synchronize()
        # the forward is deterministic: the same bits as the workspace call
        # (stale scratch contents from the previous call would show here)
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)
        assert torch.equal(ml, ml_ref)
        assert torch.isfinite(ml_ref).any()


def test_noalloc_rejects_problems_beyond_the_scratch():
    from bwd_tcgen05_tma_gb300 import attn as A

    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    # 300k query tokens + 300k key tokens need more than the fixed scratch
    p = A.make_params(layout="HD_HD_HD", fmt="BSHD", mask="CAUSAL", B=1, Sq=300000, Skv=300000,
                      Hq=1, Hkv=1, d_qk=128, d_v=128, scale=0.1, q=t, k=t, v=t)
    assert A.attn_fwd_workspace_size(p) > A.FWD_NOALLOC_SCRATCH_BYTES
    with pytest.raises(A.AttnError) as e:
        A.attn_fwd_noalloc(p, t, torch.empty(1, device="cuda"))
    assert e.value.code == 4  # ATTN_ERR_WORKSPACE_TOO_SMALL
