"""GPU parity of the FP8 (E4M3) forward against the oracle's
attention_forward_fp8 (reading stated there and in attn.h): packed and
separate layouts, GQA, segments with padding, causal and cross attention,
both metadata paths, a band, the max-logit output, and descale factors other
than 1.  Q / K / V are E4M3 codes; O comes back in bf16."""
import numpy as np
import pytest
import torch

from bwd_tcgen05_tma_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = 5e-3  # relative Frobenius error on O and LSE, as for the 16-bit forward
DESCALE = (0.75, 1.5, 0.5)


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_tcgen05_tma_gb300 import build

    build.build()


def _case(name, **kw):
    base = dict(d_qk=128, d_v=128, dtype="fp8_e4m3")
    base.update(kw)
    return I.synth(name, **base)


CASES = {
    "thd_gqa_3hd": lambda: _case("f1", B=2, Sq=1000, Skv=1000, Hq=4, Hkv=2, layout="3HD",
                                 fmt="THD_SEGMENTS", causal=True, seed=91, seg=(40, 400),
                                 pad_frac=0.05),
    "bshd_cross": lambda: _case("f2", B=2, Sq=200, Skv=333, Hq=2, Hkv=1, layout="HD_HD_HD",
                                fmt="BSHD", causal=False, seed=92),
    "kvpacked_causal": lambda: _case("f3", B=1, Sq=700, Skv=700, Hq=4, Hkv=1, layout="HD_2HD",
                                     fmt="BSHD", causal=True, seed=93),
}


def _dev_codes(x):
    return torch.from_numpy(I.e4m3_codes(x)).cuda()


def _run(case, force_general=False, with_max_logit=False):
    from conftest import oracle_mask, oracle_metadata, oracle_qkv
    from gpu_util import int_dev, rel
    from oracle import attn_ref as R

    from bwd_tcgen05_tma_gb300 import attn as A

    c = case
    t = {k: _dev_codes(v) for k, v in c.buffers.items()}
    q, k, v = {"3HD": (t.get("qkv"), None, None), "HD_2HD": (t.get("q"), t.get("kv"), None),
               "HD_HD_HD": (t.get("q"), t.get("k"), t.get("v"))}[c.layout]
    ml = torch.full((c.B, c.Hq), float("nan"), dtype=torch.float32, device="cuda") \
        if with_max_logit else None
    # the parameter block holds bare addresses: keep the metadata tensors alive
    meta = [int_dev(c.q_ids), int_dev(c.q_pos), int_dev(c.kv_ids), int_dev(c.kv_pos)]
    p = A.make_params(layout=c.layout, fmt=c.fmt, mask=c.mask, B=c.B, Sq=c.Sq, Skv=c.Skv,
                      Hq=c.Hq, Hkv=c.Hkv, d_qk=c.d_qk, d_v=c.d_v, scale=c.scale, q=q, k=k, v=v,
                      q_seg_ids=meta[0], q_seg_pos=meta[1], kv_seg_ids=meta[2], kv_seg_pos=meta[3],
                      force_general_path=force_general, window=c.window,
                      bottom_right=c.bottom_right, dtype="fp8_e4m3", descale=DESCALE,
                      max_logit=ml)
    ws = torch.zeros(A.attn_fwd_workspace_size(p), dtype=torch.uint8, device="cuda")
    o = torch.full((c.B * c.Sq, c.Hq, c.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.B, c.Hq, c.Sq), float("nan"), dtype=torch.float32, device="cuda")
    A.attn_fwd(p, o, lse, ws)
    st, stats = A.attn_read_status(ws)
    del meta
    assert st == 0, f"device status {st}"
    # the oracle on the same E4M3 values
    q8, k8, v8 = oracle_qkv(c)
    qi, qp, ki, kp = oracle_metadata(c)
    ro, rl = R.attention_forward_fp8(q8, k8, v8, *DESCALE, qi, qp, ki, kp, oracle_mask(c),
                                     c.scale)
    og = o.float().cpu().numpy().reshape(c.B, c.Sq, c.Hq, c.d_v)
    lg = lse.cpu().numpy()
    has = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lg), has)
    has_o = has.transpose(0, 2, 1)
    assert np.all(og[~has_o] == 0.0)
    eo, el = rel(og[has_o], ro[has_o]), rel(lg[has], rl[has])
    assert eo <= TOL, f"O rel err {eo}"
    assert el <= TOL, f"LSE rel err {el}"
    if with_max_logit:
        rm = R.max_logit(q8 * DESCALE[0], k8 * DESCALE[1], qi, qp, ki, kp, oracle_mask(c), c.scale)
        mg = ml.cpu().numpy()
        fin = np.isfinite(rm)
        assert np.array_equal(np.isfinite(mg), fin)
        np.testing.assert_allclose(mg[fin], rm[fin], rtol=1e-4, atol=1e-4)
    return stats, og, has_o


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("force_general", [False, True])
def test_fp8_forward_matches_oracle(name, force_general):
    stats, _, _ = _run(CASES[name](), force_general=force_general)
    assert stats.path == (1 if force_general or name == "bshd_cross" else 0)


def test_fp8_forward_band_and_max_logit():
    c = CASES["thd_gqa_3hd"]()
    c.window = (100, None)
    _run(c, with_max_logit=True)


def test_fp8_forward_is_the_quantised_result():
    """The kernel reproduces the rounding of P, not the exact attention: its O
    is as far from the float64 attention of the descaled inputs as the
    oracle's FP8 result is (the two distances agree to within a tenth)."""
    from conftest import oracle_mask, oracle_metadata, oracle_qkv
    from gpu_util import rel
    from oracle import attn_ref as R

    c = CASES["bshd_cross"]()
    q8, k8, v8 = oracle_qkv(c)
    qi, qp, ki, kp = oracle_metadata(c)
    ro8, _ = R.attention_forward_fp8(q8, k8, v8, *DESCALE, qi, qp, ki, kp, oracle_mask(c), c.scale)
    ro, _ = R.attention_forward(q8 * DESCALE[0], k8 * DESCALE[1], v8 * DESCALE[2], qi, qp, ki, kp,
                                oracle_mask(c), c.scale)
    _, og, has = _run(c)  # parity with the quantised oracle is asserted inside
    gap_oracle = rel(ro8[has], ro[has])
    gap_kernel = rel(og[has], ro[has])
    assert gap_oracle > 1e-3  # E4M3 rounding of P is visible at this size
    assert abs(gap_kernel - gap_oracle) <= 0.1 * gap_oracle
