"""GPU parity: the CUDA library (through the C ABI) against the float64 oracle
on the same seeded inputs, element by element (relative Frobenius error over
valid elements, exact zeros / -inf where the definition gives them)."""
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


def small_cases():
    """Sizes the oracle finishes in seconds that still span several tiles and
    end in a ragged tail."""
    return {
        "tiny": lambda: I.workload("tiny"),
        "bshd_causal_ragged": lambda: I.synth(
            "bshd", B=2, Sq=300, Skv=300, Hq=2, Hkv=2, d_qk=128, d_v=128, layout="HD_HD_HD",
            fmt="BSHD", causal=True, seed=11),
        "bshd_noncausal_cross": lambda: I.synth(
            "bshd_x", B=2, Sq=200, Skv=333, Hq=2, Hkv=1, d_qk=64, d_v=64, layout="HD_HD_HD",
            fmt="BSHD", causal=False, seed=12),
        "thd_gqa_3hd": lambda: I.synth(
            "thd", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
            fmt="THD_SEGMENTS", causal=True, seed=13, seg=(40, 400), pad_frac=0.05),
        "cross_bias_192": lambda: I.synth(
            "xb", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192, d_v=128, layout="HD_HD_HD",
            fmt="THD_SEGMENTS", causal=False, seed=14, seg=(60, 200), kv_seg=(60, 300),
            bias_shape=(1, 2, 300, 520)),
        "kvpacked_gqa": lambda: I.synth(
            "kvp", B=1, Sq=700, Skv=700, Hq=4, Hkv=1, d_qk=128, d_v=128, layout="HD_2HD",
            fmt="BSHD", causal=True, seed=15),
        "qk192_v64": lambda: I.synth(
            "q192", B=1, Sq=260, Skv=260, Hq=2, Hkv=2, d_qk=192, d_v=64, layout="HD_HD_HD",
            fmt="THD_SEGMENTS", causal=True, seed=16, seg=(30, 140), pad_frac=0.1),
    }


CASES = small_cases()


def _ref(case):
    from conftest import oracle_full

    return oracle_full(case)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("force_general", [False, True])
def test_forward_matches_oracle(name, force_general):
    from gpu_util import DevCase, check_forward

    case = CASES[name]()
    ref = _ref(case)
    d = DevCase(case, force_general=force_general)
    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    if force_general:
        assert d.fwd_stats.path == 1


def test_fast_path_taken_for_matching_metadata():
    from gpu_util import DevCase

    d = DevCase(CASES["thd_gqa_3hd"]())
    d.forward()
    assert d.fwd_stats.path == 0 and d.fwd_stats.reason == 1
    d = DevCase(CASES["bshd_causal_ragged"]())
    d.forward()
    assert d.fwd_stats.path == 0 and d.fwd_stats.reason == 0
    d = DevCase(CASES["cross_bias_192"]())
    d.forward()
    assert d.fwd_stats.path == 1 and d.fwd_stats.reason == 3


def test_equal_length_cross_attention_takes_general_path():
    """Sq == Skv but Q and KV segments drawn independently: the general path."""
    from gpu_util import DevCase, check_forward

    case = I.synth("eqx", B=2, Sq=512, Skv=512, Hq=2, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="THD_SEGMENTS", causal=True, seed=21, seg=(50, 300),
                   kv_seg=(50, 300))
    d = DevCase(case)
    o, lse = d.forward()
    assert d.fwd_stats.path == 1 and d.fwd_stats.reason in (4, 5)
    check_forward(case, _ref(case), o, lse)


def test_derived_positions():
    """Missing segment positions are derived on the device from the ids."""
    from gpu_util import DevCase, check_forward

    case = CASES["thd_gqa_3hd"]()
    d = DevCase(case, with_pos=False)
    o, lse = d.forward()
    assert d.fwd_stats.path == 0
    check_forward(case, _ref(case), o, lse)


def test_cu_seqlens_format():
    from gpu_util import DevCase, check_forward

    base = I.synth("cu", B=1, Sq=900, Skv=900, Hq=2, Hkv=2, d_qk=128, d_v=128,
                   layout="HD_HD_HD", fmt="BSHD", causal=True, seed=22)
    base.fmt = "THD_CU_SEQLENS"
    base.cu_seqlens_q = np.array([0, 130, 130, 500, 777, 860], dtype=np.int32)  # empty segment
    base.cu_seqlens_kv = base.cu_seqlens_q.copy()
    d = DevCase(base)
    o, lse = d.forward()
    assert d.fwd_stats.path == 0
    check_forward(base, _ref(base), o, lse)
