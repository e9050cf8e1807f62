"""GPU parity of the fp16 element type (an adjacent precision of the same
path: the same oracle on inputs rounded to fp16 instead of bf16; the kernels
take fp16 MMA operands, accumulate in fp32 and round P, dS and the outputs to
fp16).  Both metadata paths, both dQ modes, every layout, 192-wide heads with
a bias and its gradient; the same tolerances as bf16."""
import numpy as np
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


CASES = {
    "thd_gqa_3hd": lambda: I.synth(
        "h1", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
        fmt="THD_SEGMENTS", causal=True, seed=61, seg=(40, 400), pad_frac=0.05, dtype="fp16"),
    "bshd_mha_causal": lambda: I.synth(
        "h2", B=2, Sq=300, Skv=300, Hq=2, Hkv=2, d_qk=64, d_v=128, layout="HD_HD_HD",
        fmt="BSHD", causal=True, seed=62, dtype="fp16"),
    "kvpacked_gqa": lambda: I.synth(
        "h3", B=1, Sq=700, Skv=700, Hq=4, Hkv=1, d_qk=128, d_v=128, layout="HD_2HD",
        fmt="BSHD", causal=True, seed=63, dtype="fp16"),
    "cross_bias_192": lambda: I.synth(
        "h4", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192, d_v=128, layout="HD_HD_HD",
        fmt="THD_SEGMENTS", causal=False, seed=64, seg=(60, 200), kv_seg=(60, 300),
        bias_shape=(1, 2, 300, 520), dtype="fp16"),
}


def _ref(case):
    from conftest import oracle_full

    return oracle_full(case)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("force_general", [False, True])
def test_fp16_forward(name, force_general):
    from gpu_util import DevCase, check_forward

    case = CASES[name]()
    d = DevCase(case, force_general=force_general)
    o, lse = d.forward()
    assert o.dtype == torch.float16
    check_forward(case, _ref(case), o, lse)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("dq_mode", ["deterministic", "atomic"])
def test_fp16_backward(name, dq_mode):
    from gpu_util import DevCase, check_backward

    case = CASES[name]()
    d = DevCase(case, dq_mode=dq_mode)
    d.forward()
    g, db = d.backward()
    check_backward(case, _ref(case), g, db)


def test_fp16_deterministic_bits_and_differs_from_bf16():
    """Deterministic mode reproduces itself bit for bit in fp16 too; and the
    fp16 call really computes in fp16 (the bf16 call on the same values, which
    are not all bf16-representable, would not read them)."""
    from gpu_util import DevCase

    case = CASES["thd_gqa_3hd"]()
    d = DevCase(case)
    d.forward()
    g1, _ = d.backward()
    g1 = {k: v.clone() for k, v in g1.items()}
    d.forward()
    g2, _ = d.backward()
    for k in g1:
        assert torch.equal(g1[k].view(torch.int16), g2[k].view(torch.int16))
    q = case.buffers["qkv"]
    assert not np.array_equal(I.bf16_round(q), q)  # fp16 values, not bf16 ones
