"""The bench's FLOP numerator: the exact count of unmasked (query, key) pairs
from the segment metadata, against the oracle's own mask summed element by
element (CPU only)."""
import numpy as np
import pytest

from bwd_tcgen05_tma_gb300 import flops as F
from bwd_tcgen05_tma_gb300 import inputs as I
from oracle import attn_ref as R


def oracle_pairs(case):
    from conftest import oracle_metadata

    qi, qp, ki, kp = oracle_metadata(case)
    return R.count_valid_pairs(qi, qp, ki, kp, case.causal)


@pytest.mark.parametrize("name", ["tiny", "bshd", "thd_gqa", "cross_bias"])
def test_pair_count_matches_oracle_mask(name):
    case = I.workload(name)
    assert F.valid_pairs_per_head(case) == oracle_pairs(case)


def test_headline_pair_count_and_flops():
    """The THD GQA workload: 293,369,728 unmasked pairs over its 32 query
    heads; forward 2 P (d_qk + d_v), backward 2 P (3 d_qk + 2 d_v)."""
    case = I.workload("thd_gqa")
    fwd, bwd, P = F.attention_flops(case)
    assert P == 293_369_728 == oracle_pairs(case) * case.Hq
    assert fwd == 2.0 * P * 256 and bwd == 2.0 * P * (3 * 128 + 2 * 128)


def test_pair_count_other_formats():
    """Dense non-causal rows, cu_seqlens with an empty segment, and segments
    without positions (derived from the ids)."""
    case = I.synth("d", B=2, Sq=70, Skv=90, Hq=2, Hkv=1, d_qk=64, d_v=64, layout="HD_HD_HD",
                   fmt="BSHD", causal=False, seed=1)
    assert F.valid_pairs_per_head(case) == 2 * 70 * 90 == oracle_pairs(case)
    case = I.synth("c", B=1, Sq=300, Skv=300, Hq=2, Hkv=2, d_qk=64, d_v=64, layout="HD_HD_HD",
                   fmt="BSHD", causal=True, seed=2)
    case.fmt = "THD_CU_SEQLENS"
    case.cu_seqlens_q = np.array([0, 40, 40, 170, 290], dtype=np.int32)
    case.cu_seqlens_kv = case.cu_seqlens_q.copy()
    assert F.valid_pairs_per_head(case) == oracle_pairs(case)
    case = I.synth("s", B=2, Sq=200, Skv=200, Hq=2, Hkv=2, d_qk=64, d_v=64, layout="HD_HD_HD",
                   fmt="THD_SEGMENTS", causal=True, seed=3, seg=(10, 60), pad_frac=0.1)
    case.q_pos = case.kv_pos = None
    assert F.valid_pairs_per_head(case) == oracle_pairs(case)
