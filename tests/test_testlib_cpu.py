"""CPU self-checks of the test plumbing used by the GPU parity tests."""
import numpy as np

import workloads as W
from sa_testlib import compact_decode_case, oracle_decode


def test_compact_helper_matches_full_oracle(oracle):
    """The sampled-sequence helper used at full sizes must hand the oracle the
    same bytes as the full case."""
    for layout in ("HND", "NHD"):
        case = W.make_decode_case([20, 50, 90], page_size=16, poison_pages=2, seed=113, layout=layout)
        full_o, full_l = oracle_decode(oracle, case)
        sub = compact_decode_case(case, [2, 0])
        o, l = oracle_decode(oracle, sub)
        assert np.array_equal(o, full_o[[2, 0]]) and np.array_equal(l, full_l[[2, 0]])
    case = W.make_decode_case([256, 3], page_size=256, paged=False, seed=3)
    full_o, full_l = oracle_decode(oracle, case)
    o, l = oracle_decode(oracle, compact_decode_case(case, [1]))
    assert np.array_equal(o, full_o[[1]])


def test_oracle_selected_rows_match_full(oracle):
    case = W.make_decode_case([20, 50, 90], page_size=16, seed=114)
    full_o, full_l = oracle_decode(oracle, case)
    o, l = oracle_decode(oracle, case, sel_rows=[1, 2])
    assert np.array_equal(o, full_o[1:]) and np.array_equal(l, full_l[1:])
