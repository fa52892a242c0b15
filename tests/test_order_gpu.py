"""Unsplit decode calls on ragged batches of up to 128 sequences run the
longest sequences first: block z serves the sequence of rank z in decreasing
length, ties by index.  The results must not depend on that mapping.  Cases
at the edges of the rule: ties among the lengths, exactly 128 sequences (the
largest ordered batch), 129 (given order), a window (given order), and the
multi-token kernel under the same rule.  Every output row is checked against
the fp64 oracle."""
import numpy as np
import pytest

import workloads as W
from sa_testlib import check_close, decode_gpu, oracle_decode, oracle_prefill
from test_decode_multi_gpu import case_of, multi_gpu

pytestmark = pytest.mark.gpu


def ragged_with_ties(B, seed):
    """Lengths in [1, 300], a third of them repeated (ties), one empty slot."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 301, B)
    lens[rng.choice(B, B // 3, replace=False)] = 96
    lens[0] = 0
    return [int(x) for x in lens]


@pytest.mark.parametrize("B,window", [(7, 0), (128, 0), (129, 0), (128, 37)])
def test_one_token_unsplit_ordering(sa, oracle, B, window):
    case = W.make_decode_case(ragged_with_ties(B, 500 + B), page_size=16, window=window, poison_pages=5,
                              seed=510 + B)
    out, lse = decode_gpu(sa, case.to("cuda"), num_splits=1)
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "B=%d w=%d unsplit" % (B, window))
    assert sa.sa_device_status() == 0


@pytest.mark.parametrize("B,q_len", [(128, 4), (129, 4), (128, 7)])
def test_multi_token_unsplit_ordering(sa, oracle, B, q_len):
    lens = [max(L, q_len) for L in ragged_with_ties(B, 600 + B)]
    case = case_of(q_len, lens, seed=620 + B)
    out, lse = multi_gpu(sa, case.to("cuda"), q_len, num_splits=1)
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out, lse, ref_o, ref_l, "B=%d q_len=%d unsplit" % (B, q_len))
    assert sa.sa_device_status() == 0
