"""Pins of the oracle's FP8 forward (reading stated in oracle.attn_ref.
attention_forward_fp8) to things other than itself: the E4M3 rounding against
PyTorch's float8_e4m3fn conversion and against the format's own code table, a
case worked by hand, a closed form, and the bound the quantisation of P puts
on the distance to the exact float64 attention of the same inputs."""
import numpy as np
import pytest

from oracle import attn_ref as R

torch = pytest.importorskip("torch")


def _e4m3_table():
    """Every finite E4M3 value, decoded by PyTorch from all 256 codes."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).double().numpy()
    return np.unique(vals[np.isfinite(vals)])


def test_e4m3_round_matches_torch():
    rng = np.random.default_rng(5)
    x = rng.normal(size=100000) * np.exp2(rng.uniform(-12, 9, 100000))
    x = np.clip(x, -R.E4M3_MAX, R.E4M3_MAX)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(R.e4m3_round(x), ref)


def test_e4m3_round_lands_on_the_code_table_and_is_nearest():
    table = _e4m3_table()
    assert table.max() == R.E4M3_MAX and np.min(table[table > 0]) == 2.0 ** -9
    rng = np.random.default_rng(6)
    x = rng.uniform(-R.E4M3_MAX, R.E4M3_MAX, 20000) * np.exp2(rng.integers(-14, 1, 20000))
    r = R.e4m3_round(x)
    assert np.all(np.isin(r, table))
    # nearest: no table value is strictly closer
    idx = np.searchsorted(table, x)
    lo = table[np.clip(idx - 1, 0, table.size - 1)]
    hi = table[np.clip(idx, 0, table.size - 1)]
    best = np.minimum(np.abs(x - lo), np.abs(x - hi))
    assert np.all(np.abs(r - x) <= best + 1e-300)
    assert np.array_equal(R.e4m3_round(table), table)  # idempotent


def test_e4m3_round_ties_and_saturation():
    # halfway cases go to the even code; beyond 448 saturates
    assert R.e4m3_round(2.0 ** -10) == 0.0           # between 0 and 2^-9
    assert R.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8  # between 2^-9 (odd) and 2^-8 (even)
    assert R.e4m3_round(1.0 + 1 / 16) == 1.0          # between 1 and 1.125
    assert R.e4m3_round(1.0 + 3 / 16) == 1.25         # between 1.125 and 1.25
    assert R.e4m3_round(500.0) == R.E4M3_MAX and R.e4m3_round(-1e9) == -R.E4M3_MAX


def _one_row_case(scores, v_rows):
    """q, k realising the given scores for one query over len(scores) keys
    with scale 1: q = e_0 * 1, k_j = scores_j * e_0 (d = 4)."""
    n = len(scores)
    q = np.zeros((1, 1, 1, 4))
    q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, n, 1, 4))
    k[0, :, 0, 0] = scores
    v = np.asarray(v_rows, dtype=np.float64).reshape(1, n, 1, -1)
    ids_q = np.ones((1, 1), np.int32)
    ids_k = np.ones((1, n), np.int32)
    pos_q = np.zeros((1, 1), np.int32)
    pos_k = np.zeros((1, n), np.int32)
    return q, k, v, ids_q, pos_q, ids_k, pos_k


def test_hand_worked_case():
    """One query, two keys, scores 0 and ln 0.7: p = (1, 0.7), l = 1.7;
    256 * 0.7 = 179.2 lies in [128, 256) where E4M3 steps by 16, so it
    rounds to 176 (11 * 16); with v = (1, 0) and (0, 1):
    O = (256 * (1, 0) + 176 * (0, 1)) / (256 * 1.7) = (1/1.7, 0.6875/1.7)."""
    q, k, v, iq, pq, ik, pk = _one_row_case([0.0, np.log(0.7)], [[1.0, 0.0], [0.0, 1.0]])
    o, lse = R.attention_forward_fp8(q, k, v, 1.0, 1.0, 1.0, iq, pq, ik, pk, False, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], [1 / 1.7, 0.6875 / 1.7], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], np.log(1.7), rtol=1e-14)
    # the descale factors multiply exactly where the reading puts them
    o2, lse2 = R.attention_forward_fp8(q, k * 0.5, v, 2.0, 1.0, 3.0, iq, pq, ik, pk, False, 1.0)
    np.testing.assert_allclose(o2, 3 * o, rtol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)


def _random_case(seed, B=2, Sq=70, Skv=90, Hq=4, Hkv=2, d=16, causal=False):
    rng = np.random.default_rng(seed)
    q8 = R.e4m3_round(rng.normal(size=(B, Sq, Hq, d)) * 2)
    k8 = R.e4m3_round(rng.normal(size=(B, Skv, Hkv, d)) * 2)
    v8 = R.e4m3_round(rng.normal(size=(B, Skv, Hkv, d)) * 2)
    iq = np.ones((B, Sq), np.int32)
    ik = np.ones((B, Skv), np.int32)
    iq[:, -5:] = 0  # padding rows
    pq = np.tile(np.arange(Sq, dtype=np.int32), (B, 1))
    pk = np.tile(np.arange(Skv, dtype=np.int32), (B, 1))
    return q8, k8, v8, iq, pq, ik, pk


def test_closed_form_equal_scores():
    """q = 0: every valid score is 0, p = 1, 256 p = 256 is exact, so O is the
    mean of the valid value rows times descale_v and LSE = ln(count)."""
    q8, k8, v8, iq, pq, ik, pk = _random_case(7, causal=True)
    q8 = np.zeros_like(q8)
    o, lse = R.attention_forward_fp8(q8, k8, v8, 0.5, 2.0, 1.5, iq, pq, ik, pk, True, 0.3)
    B, Sq, Hq, _ = q8.shape
    for b in range(B):
        for i in range(Sq):
            if iq[b, i] == 0:
                assert np.all(o[b, i] == 0) and np.all(np.isneginf(lse[b, :, i]))
                continue
            n = min(i + 1, k8.shape[1])
            for h in range(Hq):
                g = h // 2
                np.testing.assert_allclose(o[b, i, h], 1.5 * v8[b, :n, g].mean(axis=0), rtol=1e-12,
                                           atol=1e-14)
                np.testing.assert_allclose(lse[b, h, i], np.log(n), rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_quantisation_bound_against_exact_attention(causal):
    """|O8 - O| <= descale_v * sum_j |P8_j / 256 - p_j| |v_j| / l, and since
    E4M3 rounding of 256 p is within 2^-4 relative for values >= 2^-6 and
    within 2^-10 absolute below, O8 - O is at most 2^-4 max|v| + 2^-18 n max|v| / l
    per element, against the float64 oracle on the descaled inputs; LSE does
    not see the rounding at all."""
    q8, k8, v8, iq, pq, ik, pk = _random_case(8)
    dq_, dk_, dv_, scale = 0.7, 1.3, 0.9, 0.25
    o8, lse8 = R.attention_forward_fp8(q8, k8, v8, dq_, dk_, dv_, iq, pq, ik, pk, causal, scale)
    o, lse = R.attention_forward(q8 * dq_, k8 * dk_, v8 * dv_, iq, pq, ik, pk, causal, scale)
    np.testing.assert_allclose(lse8, lse, rtol=1e-12)
    vmax = np.abs(v8 * dv_).max()
    n = k8.shape[1]
    bound = 2.0 ** -4 * vmax + 2.0 ** -18 * n * vmax
    assert np.max(np.abs(o8 - o)) <= bound
    # and the rounding is really there: O8 is not the exact result
    assert np.max(np.abs(o8 - o)) > 1e-6


def test_planted_mistakes_are_caught():
    """Mistakes a kernel or an oracle could plausibly make, each caught by a
    hand-worked case: normalising by the sum of the rounded P (case above);
    rounding p itself instead of 256 p (a small p: 256 p = 1.3 rounds to
    1.25, while p = 1.3 / 256 < 2^-6 would round on the subnormal grid, to
    3 * 2^-9 = 1.5 / 256); dropping descale_v."""
    q, k, v, iq, pq, ik, pk = _one_row_case([0.0, np.log(0.7)], [[1.0, 0.0], [0.0, 1.0]])
    o, _ = R.attention_forward_fp8(q, k, v, 1.0, 1.0, 3.0, iq, pq, ik, pk, False, 1.0)
    want = 3.0 * np.array([1 / 1.7, 0.6875 / 1.7])
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-14)
    p = np.array([1.0, 0.7])
    p8 = R.e4m3_round(256 * p)
    assert not np.allclose(3.0 * (p8 @ v[0, :, 0]) / p8.sum(), want, rtol=1e-6)  # self-normalised
    assert not np.allclose((p8 @ v[0, :, 0]) / (256 * p.sum()), want, rtol=1e-6)  # no descale_v

    q, k, v, iq, pq, ik, pk = _one_row_case([0.0, np.log(1.3 / 256)], [[1.0, 0.0], [0.0, 1.0]])
    o, _ = R.attention_forward_fp8(q, k, v, 1.0, 1.0, 1.0, iq, pq, ik, pk, False, 1.0)
    l = 1.0 + 1.3 / 256
    want = np.array([1.0, 1.25 / 256]) / l
    np.testing.assert_allclose(o[0, 0, 0], want, rtol=1e-14)
    p = np.array([1.0, 1.3 / 256])
    assert not np.allclose(R.e4m3_round(p) @ v[0, :, 0] / l, want, rtol=1e-6)  # no 256 scale


def test_fp8_forward_rows_are_independent():
    """The full-size GPU test runs the E4M3 oracle on sampled query rows only:
    a row's O and LSE depend on that row alone (P is quantised against the
    row's own maximum), so the oracle on a subset of rows gives the full run's
    values for them, up to float64 summation order."""
    import sys
    import os

    sys.path.insert(0, os.path.dirname(__file__))
    from conftest import oracle_mask, oracle_metadata

    from bwd_tcgen05_tma_gb300 import inputs as I

    case = I.synth("rows", B=2, Sq=300, Skv=300, Hq=4, Hkv=2, d_qk=128, d_v=128, layout="3HD",
                   fmt="THD_SEGMENTS", causal=True, seed=5, seg=(30, 160), pad_frac=0.05)
    vals = {k: I.e4m3_value(I.e4m3_codes(x)) for k, x in case.buffers.items()}
    q8, k8, v8 = R.unpack_layout(case.layout, vals, case.B, case.Sq, case.Skv, case.Hq,
                                 case.Hkv, 128, 128)
    qi, qp, ki, kp = oracle_metadata(case)
    fo, fl = R.attention_forward_fp8(q8, k8, v8, 1.0, 1.0, 1.0, qi, qp, ki, kp,
                                     oracle_mask(case), case.scale)
    rows = [0, 7, 61, 150, 299]
    for b in range(case.B):
        ro, rl = R.attention_forward_fp8(q8[b:b + 1, rows], k8[b:b + 1], v8[b:b + 1], 1.0, 1.0,
                                         1.0, qi[b:b + 1, rows], qp[b:b + 1, rows], ki[b:b + 1],
                                         kp[b:b + 1], oracle_mask(case), case.scale)
        np.testing.assert_allclose(ro[0], fo[b, rows], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isfinite(rl[0]), np.isfinite(fl[b][:, rows]))
        fin = np.isfinite(rl[0])
        np.testing.assert_allclose(rl[0][fin], fl[b][:, rows][fin], rtol=0, atol=1e-12)
