"""Full-size parity: every named workload at its full size, run through the
C ABI exactly as the bench runs it (one workspace, forward then backward
reusing the forward's metadata), checked against the float64 oracle on
sampled outputs the oracle computes one by one: O, LSE and dQ rows of sampled
(batch row, query head) pairs, dK and dV rows of sampled (batch row, KV head)
key positions.  Each sampled output is exact in the oracle (a query row needs
only its own softmax row; a key row recomputes every query row that attends to
it), so the tolerances are the same as at reduced sizes."""
import numpy as np
import pytest
import torch

from bwd_tcgen05_tma_gb300 import inputs as I

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL_O = 5e-3
TOL_LSE = 5e-3
TOL_GRAD = 1.5e-2

CASES = [("tiny", "deterministic"), ("bshd", "deterministic"), ("thd_gqa", "deterministic"),
         ("thd_gqa", "atomic"), ("cross_bias", "deterministic"), ("long_kv", "deterministic"),
         ("long_kv", "atomic")]


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_tcgen05_tma_gb300 import build

    build.build()


def sample_query_rows(ids, rng, n_random=4):
    """First and last valid rows, the first row of a later segment, a padded
    row when there is one, and a few random valid rows."""
    S = ids.shape[0]
    valid = np.nonzero(ids != 0)[0]
    rows = {int(valid[0]), int(valid[-1])}
    starts = [t for t in valid[1:] if ids[t] != ids[t - 1]]
    if starts:
        rows.add(int(starts[len(starts) // 2]))
    pad = np.nonzero(ids == 0)[0]
    if pad.size:
        rows.add(int(pad[0]))
    rows.update(int(x) for x in rng.choice(valid, size=min(n_random, valid.size), replace=False))
    return sorted(r for r in rows if 0 <= r < S)


def sample_key_rows(kv_ids, q_ids, causal):
    """Key positions whose attending query rows the oracle can recompute in a
    few seconds, among segments that some query row attends to: with a causal
    mask the last keys of segments (few rows attend to them), keys 64 and 127
    before the end of the last one, and the first key of the shortest segment;
    without one, three keys of the shortest segment."""
    valid = np.nonzero(kv_ids != 0)[0]
    seen = set(np.unique(q_ids[q_ids != 0]).tolist())
    n = kv_ids.shape[0]
    ends = [int(t) for t in valid if (t + 1 == n or kv_ids[t + 1] != kv_ids[t])
            and int(kv_ids[t]) in seen]
    starts = [int(t) for t in valid if (t == 0 or kv_ids[t - 1] != kv_ids[t])
              and int(kv_ids[t]) in seen]
    seg = sorted(zip(starts, ends), key=lambda se: se[1] - se[0])
    if causal:
        cols = set(ends[:2] + ends[-2:])
        s1, e1 = max(zip(starts, ends), key=lambda se: se[1])
        cols.update(t for t in (e1 - 64, e1 - 127) if t >= s1)
        s0, e0 = seg[0]
        if e0 - s0 < 2048:
            cols.add(s0)
    else:
        s0, e0 = seg[0]
        cols = {s0, (s0 + e0) // 2, e0}
    return sorted(cols)


def rel(x, ref):
    from oracle import attn_ref as R

    return R.rel_frobenius(np.asarray(x, np.float64), np.asarray(ref, np.float64))


@pytest.mark.parametrize("name,dq_mode", CASES)
def test_full_size_sampled(name, dq_mode):
    import bench
    from conftest import oracle_metadata, oracle_qkv
    from gpu_util import unpack_grads
    from oracle import attn_ref as R

    case = I.workload(name)
    prob = bench.Problem(case, dq_mode)
    prob.step()
    st, stats = prob.A.attn_read_status(prob.ws)
    assert st == 0, f"device status {st}"
    torch.cuda.synchronize()

    q, k, v = oracle_qkv(case)
    qi, qp, ki, kp = oracle_metadata(case)
    do = case.do.astype(np.float64)
    bias = case.bias  # float32 holding bf16 values; promoted row by row
    B, Sq, Hq, Hkv = case.B, case.Sq, case.Hq, case.Hkv
    rng = np.random.default_rng(7)
    o_dev = prob.o.view(B, Sq, Hq, case.d_v)
    lse_dev = prob.lse
    dq_dev, dk_dev, dv_dev = unpack_grads(case, prob.grads)

    heads = sorted({0, min(Hq - 1, Hq // 2 + 1), Hq - 1})
    got = {"o": [], "lse": [], "dq": [], "dk": [], "dv": []}
    ref = {key: [] for key in got}
    for b in sorted({0, B - 1}):
        rows = sample_query_rows(qi[b], rng)
        for h in heads:
            ro, rl = R.forward_rows(q, k, v, qi, qp, ki, kp, case.causal, case.scale, b, h, rows,
                                    bias)
            rd = R.backward_dq_rows(q, k, v, do, qi, qp, ki, kp, case.causal, case.scale, b, h,
                                    rows, bias)
            go = o_dev[b, rows, h].float().cpu().numpy()
            gl = lse_dev[b, h, rows].cpu().numpy()
            fin = np.isfinite(rl)
            assert np.array_equal(np.isfinite(gl), fin), (b, h, "LSE finiteness")
            assert np.all(go[~fin] == 0.0), (b, h, "rows without keys give O = 0")
            assert np.all(dq_dev[b, rows, h][~fin] == 0.0), (b, h, "and dQ = 0")
            got["o"].append(go[fin])
            ref["o"].append(ro[fin])
            got["lse"].append(gl[fin])
            ref["lse"].append(rl[fin])
            got["dq"].append(dq_dev[b, rows, h])
            ref["dq"].append(rd)
        cols = sample_key_rows(ki[b], qi[b], case.causal)
        for g in sorted({0, Hkv - 1}):
            rk, rv = R.backward_dkdv_cols(q, k, v, do, qi, qp, ki, kp, case.causal, case.scale, b,
                                          g, cols, bias)
            got["dk"].append(dk_dev[b, cols, g])
            ref["dk"].append(rk)
            got["dv"].append(dv_dev[b, cols, g])
            ref["dv"].append(rv)
    tol = {"o": TOL_O, "lse": TOL_LSE, "dq": TOL_GRAD, "dk": TOL_GRAD, "dv": TOL_GRAD}
    for key in got:
        e = rel(np.concatenate([x.ravel() for x in got[key]]),
                np.concatenate([x.ravel() for x in ref[key]]))
        assert e <= tol[key], f"{name} {dq_mode}: {key} rel err {e}"


def test_full_size_fp8_forward_sampled():
    """The E4M3 forward on the full packed THD GQA workload (E4M3 codes of its
    inputs, descale factors 1), as the bench runs it, against the oracle's
    E4M3 forward on sampled query rows of every head.  A row's O and LSE
    depend only on that row (P is quantised against the row's own final
    maximum), so the oracle run on the sampled rows alone is exact."""
    import bench
    from conftest import oracle_mask, oracle_metadata
    from oracle import attn_ref as R

    case = I.workload("thd_gqa")
    prob = bench.Problem(case, "deterministic")
    f8 = bench.Fp8Forward(case, prob)
    f8.fwd()
    f8.check_status()
    torch.cuda.synchronize()

    B, Sq, Skv, Hq, Hkv = case.B, case.Sq, case.Skv, case.Hq, case.Hkv
    vals = {key: I.e4m3_value(I.e4m3_codes(x)) for key, x in case.buffers.items()}
    q8, k8, v8 = R.unpack_layout(case.layout, vals, B, Sq, Skv, Hq, Hkv, case.d_qk, case.d_v)
    qi, qp, ki, kp = oracle_metadata(case)
    o_dev = f8.o.view(B, Sq, Hq, case.d_v)
    rng = np.random.default_rng(11)
    got = {"o": [], "lse": []}
    ref = {"o": [], "lse": []}
    for b in sorted({0, B - 1}):
        rows = sample_query_rows(qi[b], rng)
        ro, rl = R.attention_forward_fp8(q8[b:b + 1, rows], k8[b:b + 1], v8[b:b + 1], 1.0, 1.0,
                                         1.0, qi[b:b + 1, rows], qp[b:b + 1, rows], ki[b:b + 1],
                                         kp[b:b + 1], oracle_mask(case), case.scale)
        go = o_dev[b, rows].float().cpu().numpy()        # [rows, Hq, d_v]
        gl = f8.lse[b][:, rows].cpu().numpy()            # [Hq, rows]
        fin = np.isfinite(rl[0])                         # [Hq, rows]
        assert np.array_equal(np.isfinite(gl), fin), "LSE finiteness"
        fin_o = fin.T                                    # [rows, Hq]
        assert np.all(go[~fin_o] == 0.0), "rows without keys give O = 0"
        got["o"].append(go[fin_o])
        ref["o"].append(ro[0][fin_o])
        got["lse"].append(gl[fin])
        ref["lse"].append(rl[0][fin])
    for key, tol in (("o", TOL_O), ("lse", TOL_LSE)):
        e = rel(np.concatenate([x.ravel() for x in got[key]]),
                np.concatenate([x.ravel() for x in ref[key]]))
        assert e <= tol, f"E4M3 forward: {key} rel err {e}"
