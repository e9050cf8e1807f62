"""The checking build (libattn_sm103_debug.so, compiled with -DATTN_DEBUG)
stands in for a memory checker: every tensor-map copy and global store of
every kernel is preceded by a bounds check that would record
ATTN_ERR_DEVICE_BOUNDS and skip the access.  Run over odd and edge-case sizes
(one query, tile boundaries +-1, ragged tails, empty segments, 192-wide heads,
bias, bands, fp16, both metadata paths and both dQ modes), no check may fire
and every output must still match the oracle."""
import pytest
import torch

from bwd_tcgen05_tma_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_tcgen05_tma_gb300 import attn as A
    from bwd_tcgen05_tma_gb300 import build

    build.build()
    path = build.build(debug=True)
    with A.library_scope(path) as lib:
        assert lib.attn_build_flags() & A.BUILD_DEVICE_CHECKS
        yield lib


def _case(name, **kw):
    base = dict(layout="HD_HD_HD", fmt="BSHD", causal=True, d_qk=128, d_v=128)
    base.update(kw)
    return I.synth(name, **base)


CASES = {
    # one query over five keys (with one key, P = 1 and dQ = dK = 0 exactly,
    # which a relative error cannot compare)
    "one_query": lambda: _case("c1", B=1, Sq=1, Skv=5, Hq=2, Hkv=1, causal=False, seed=81),
    "tile_minus_one": lambda: _case("c127", B=2, Sq=127, Skv=127, Hq=2, Hkv=2, seed=82),
    "tile_plus_one": lambda: _case("c129", B=1, Sq=129, Skv=129, Hq=4, Hkv=2, d_qk=64, d_v=64,
                                   seed=83),
    "thd_ragged_3hd": lambda: _case("c1350", B=1, Sq=1350, Skv=1350, Hq=4, Hkv=2, layout="3HD",
                                    fmt="THD_SEGMENTS", seed=84, seg=(1, 500), pad_frac=0.07),
    "cross_bias_192": lambda: _case("cx", B=2, Sq=300, Skv=520, Hq=2, Hkv=2, d_qk=192,
                                    fmt="THD_SEGMENTS", causal=False, seed=85, seg=(60, 200),
                                    kv_seg=(60, 300), bias_shape=(1, 2, 300, 520)),
    "kvpacked_odd": lambda: _case("ckv", B=1, Sq=777, Skv=777, Hq=3, Hkv=1, layout="HD_2HD",
                                  seed=86),
}


def _run(case, dq_mode, force_general):
    from conftest import oracle_full
    from gpu_util import DevCase, check_backward, check_forward

    ref = oracle_full(case)
    d = DevCase(case, dq_mode=dq_mode, force_general=force_general)
    o, lse = d.forward()  # asserts the device status is ATTN_OK
    check_forward(case, ref, o, lse)
    g, db = d.backward()
    check_backward(case, ref, g, db)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("dq_mode,force_general", [("deterministic", False), ("atomic", True)])
def test_no_check_fires(debug_lib, name, dq_mode, force_general):
    _run(CASES[name](), dq_mode, force_general)


def test_no_check_fires_with_a_band(debug_lib):
    case = CASES["thd_ragged_3hd"]()
    case.window = (100, None)
    _run(case, "deterministic", False)


def test_no_check_fires_fp16(debug_lib):
    case = _case("c129h", B=1, Sq=129, Skv=129, Hq=4, Hkv=2, d_qk=64, d_v=64, seed=87,
                 dtype="fp16")
    _run(case, "atomic", False)


def test_no_check_fires_fp8(debug_lib):
    """The E4M3 forward on segments whose starts are not 16-aligned, packed
    QKV, GQA, causal: every copy (keys are the innermost coordinate of the
    transposed-V copies) and store passes its check."""
    from test_fp8 import CASES as FP8_CASES, _run as fp8_run

    fp8_run(FP8_CASES["thd_gqa_3hd"]())
