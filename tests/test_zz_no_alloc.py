"""sa_decode_static_workspace: the decode entry point for callers that cannot
allocate device memory (a plugin whose host owns all device allocations, or a
latency-critical caller that must not call cudaMalloc).  Its split scratch is
the library's own fixed device array.  It must give what sa_decode gives, call
after call, and refuse a split that does not fit the array before launching.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test.  It must pass on its own in a fresh
process too."""
import pytest
import torch

import workloads as W
from sa_testlib import check_close, oracle_decode

pytestmark = pytest.mark.gpu


def _both(sa, case, splits):
    B, Hq, D = case.q.shape
    maxlen = int(case.seqlens.max())
    ref_out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(B, Hq, device="cuda")
    need = sa.sa_decode_workspace_size(B, Hq, case.kv.num_kv_heads, D, maxlen, case.window, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    sa.sa_decode(case.q, case.kv, case.seqlens, case.sinks, case.window, case.sm_scale, ref_out, ref_lse,
                 max_kv_len=maxlen, workspace=ws, num_splits=splits)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    sa.sa_decode_static_workspace(case.q, case.kv, case.seqlens, case.sinks, case.window, case.sm_scale, out, lse,
                                  max_kv_len=maxlen, num_splits=splits)
    torch.cuda.synchronize()
    return out, lse, ref_out, ref_lse, need


def test_static_workspace_matches_sa_decode_twice_in_a_row(sa, oracle):
    # different calls back to back: a later call must not see an earlier one's leftovers
    cases = [W.make_decode_case([1, 300, 1500, 4000], page_size=16, window=0, poison_pages=3, seed=300),
             W.make_decode_case([2000, 17, 900], page_size=16, window=128, kv_dtype="e4m3", seed=301),
             W.make_decode_case([5000, 64, 3333, 1, 777, 2048], page_size=16, window=0, seed=302)]
    refs = [oracle_decode(oracle, c) for c in cases]
    gpu = [c.to("cuda") for c in cases]
    for i, splits in [(0, 7), (1, 3), (2, 0), (0, 7), (2, 5)]:
        out, lse, ref_out, ref_lse, need = _both(sa, gpu[i], splits)
        assert 0 < need <= sa.SA_STATIC_WORKSPACE_BYTES or splits == 0
        # the same kernels with the same split: bit for bit what sa_decode gives
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), "out differs from sa_decode"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), "lse differs from sa_decode"
        check_close(out, lse, refs[i][0], refs[i][1], "static workspace vs oracle, case %d splits=%d" % (i, splits))
    assert sa.sa_device_status() == 0


def test_static_workspace_refuses_a_split_that_does_not_fit(sa):
    case = W.make_decode_case([64] * 256, page_size=16, seed=303).to("cuda")
    B, Hq, D = case.q.shape
    assert sa.sa_decode_workspace_size(B, Hq, 8, D, 64, 0, 4) > sa.SA_STATIC_WORKSPACE_BYTES
    out = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sa.SinkAttnError) as ei:
        sa.sa_decode_static_workspace(case.q, case.kv, case.seqlens, case.sinks, 0, 0.125, out, None,
                                      max_kv_len=64, num_splits=4)
    assert ei.value.status == sa.SA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0  # nothing was launched
