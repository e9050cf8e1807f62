"""GPU parity of the band masks (sliding windows, two-sided bands, bottom-right
alignment) against the oracle's Window, on both metadata paths and both dQ
modes, at sizes that span several tiles and end in a ragged tail.

The pages define no windows; the band is read as: key j is kept for query i
(in the same nonzero segment) when -left <= pos_kv[j] - (pos_q[i] + shift) <=
right, with shift = Skv - Sq under bottom-right alignment."""
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


def _with(case, window=None, bottom_right=False):
    case.window = window
    case.bottom_right = bottom_right
    return case


CASES = {
    # packed THD GQA, causal sliding window of 101 keys (fast path)
    "thd_causal_window": lambda: _with(I.synth(
        "bw1", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
        fmt="THD_SEGMENTS", causal=True, seed=51, seg=(40, 400), pad_frac=0.05), (100, None)),
    # dense rows, two-sided band, not causal (fast path), odd GQA group
    "bshd_two_sided": lambda: _with(I.synth(
        "bw2", B=2, Sq=300, Skv=300, Hq=3, Hkv=1, d_qk=64, d_v=128, layout="HD_HD_HD",
        fmt="BSHD", causal=False, seed=52), (70, 45)),
    # dense rows of unequal lengths, causal aligned bottom-right (general path)
    "bshd_bottom_right_causal": lambda: _with(I.synth(
        "bw3", B=2, Sq=200, Skv=333, Hq=2, Hkv=2, d_qk=128, d_v=128, layout="HD_HD_HD",
        fmt="BSHD", causal=True, seed=53), None, True),
    # the same with a causal window of 64 keys
    "bshd_bottom_right_window": lambda: _with(I.synth(
        "bw4", B=1, Sq=250, Skv=600, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="HD_HD_HD",
        fmt="BSHD", causal=True, seed=54), (63, 0), True),
    # cross attention with independent segments and a band (general path,
    # 192-wide heads, bias with its gradient)
    "cross_band_192": lambda: _with(I.synth(
        "bw5", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192, d_v=128, layout="HD_HD_HD",
        fmt="THD_SEGMENTS", causal=False, seed=55, seg=(60, 200), kv_seg=(60, 300),
        bias_shape=(1, 2, 300, 520)), (40, 25)),
    # long dense rows with a causal window: packed KV, several tiles per row
    "kvpacked_window": lambda: _with(I.synth(
        "bw6", B=1, Sq=1100, Skv=1100, Hq=4, Hkv=1, d_qk=128, d_v=128, layout="HD_2HD",
        fmt="BSHD", causal=True, seed=56), (200, 0)),
}


def _ref(case):
    from conftest import oracle_full

    return oracle_full(case)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("force_general", [False, True])
def test_band_forward(name, force_general):
    from gpu_util import DevCase, check_forward

    case = CASES[name]()
    d = DevCase(case, force_general=force_general)
    o, lse = d.forward()
    check_forward(case, _ref(case), o, lse)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("dq_mode", ["deterministic", "atomic"])
def test_band_backward(name, dq_mode):
    from gpu_util import DevCase, check_backward, check_forward

    case = CASES[name]()
    ref = _ref(case)
    d = DevCase(case, dq_mode=dq_mode)
    o, lse = d.forward()
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)


def test_band_backward_general_path():
    from gpu_util import DevCase, check_backward

    case = CASES["thd_causal_window"]()
    d = DevCase(case, dq_mode="deterministic", force_general=True)
    d.forward()
    g, db = d.backward()
    assert d.bwd_stats.path == 1
    check_backward(case, _ref(case), g, db)


def test_window_narrows_the_scheduled_tiles():
    """A causal window of 201 keys over 1100-token rows: each 128-row query
    tile meets at most three 128-key tiles, on both paths, instead of the
    growing causal triangle."""
    from gpu_util import DevCase

    case = CASES["kvpacked_window"]()
    n_qt = (case.Sq + 127) // 128
    for general in (False, True):
        d = DevCase(case, force_general=general)
        d.forward()
        assert d.fwd_stats.tile_pairs <= 3 * n_qt * case.B
    plain = _with(CASES["kvpacked_window"](), None)
    d = DevCase(plain)
    d.forward()
    assert d.fwd_stats.tile_pairs == n_qt * (n_qt + 1) // 2
