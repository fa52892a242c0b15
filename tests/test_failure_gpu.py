"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes gives up after its limit, sets SA_DEVICE_TIMEOUT and returns, and
the context keeps working.  Out-of-range writes are caught by canary regions
around every output and workspace buffer (bit-exact after each call)."""
import time

import numpy as np
import pytest
import torch

import workloads as W
from sa_testlib import check_close, decode_gpu, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu

SA_DEVICE_TIMEOUT = 0x4
GUARD = 4096  # bytes of canary on each side


def test_bounded_wait_times_out_and_the_context_survives(sa, oracle):
    sa.sa_device_status()  # clear
    t0 = time.time()
    sa.sa_selftest_wait_timeout()
    flags = sa.sa_device_status()  # synchronises
    dt = time.time() - t0
    assert flags & SA_DEVICE_TIMEOUT
    assert not flags & 0x80000000, "a wait on a barrier nobody completes returned success"
    assert 0.5 < dt < 30.0
    case = W.make_decode_case([100, 300], page_size=16, seed=600)
    out, lse = decode_gpu(sa, case.to("cuda"), num_splits=2)
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out, lse, ref_o, ref_l, "decode after the timeout")
    assert sa.sa_device_status() == 0


class Guarded:
    """A device buffer with random canary bytes before and after the view the
    library writes."""

    def __init__(self, shape, dtype, seed):
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        g = torch.Generator(device="cpu").manual_seed(seed)
        self.raw = torch.randint(0, 256, (GUARD + n + GUARD,), generator=g, dtype=torch.uint8).cuda()
        self.before = self.raw.clone()
        self.n = n
        self.view = self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self, what):
        torch.cuda.synchronize()
        assert torch.equal(self.raw[:GUARD], self.before[:GUARD]), what + ": write before the buffer"
        assert torch.equal(self.raw[GUARD + self.n:], self.before[GUARD + self.n:]), what + ": write past the buffer"


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_writes_stay_inside_out_lse_workspace(sa, oracle, splits):
    case = W.make_decode_case([1, 77, 300, 1500], page_size=16, window=0, poison_pages=3, seed=601)
    g = case.to("cuda")
    B, Hq, D = case.q.shape
    out = Guarded((B, Hq, D), torch.bfloat16, 1)
    lse = Guarded((B, Hq), torch.float32, 2)
    wsb = sa.sa_decode_workspace_size(B, Hq, 8, D, 1500, 0, splits)
    ws = Guarded((max(wsb, 16),), torch.uint8, 3)
    sa.sa_decode(g.q, g.kv, g.seqlens, g.sinks, 0, g.sm_scale, out.view, lse.view, max_kv_len=1500, workspace=ws.view,
                 num_splits=splits)
    for buf, name in [(out, "out"), (lse, "lse"), (ws, "workspace")]:
        buf.check("decode S=%d %s" % (splits, name))
    ref_o, ref_l = oracle_decode(oracle, case)
    check_close(out.view, lse.view, ref_o, ref_l, "guarded decode")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_prefill_writes_stay_inside_out_lse(sa, oracle, kv_dtype):
    case = W.make_prefill_case([130, 7, 129], [300, 7, 129], paged=True, page_size=16, kv_dtype=kv_dtype, seed=602)
    g = case.to("cuda")
    T, Hq, D = case.q.shape
    out = Guarded((T, Hq, D), torch.bfloat16, 4)
    lse = Guarded((T, Hq), torch.float32, 5)
    sa.sa_prefill(g.q, g.cu_seqlens_q, g.kv, g.seqlens, g.sinks, 0, g.sm_scale, out.view, lse.view, max_q_len=130,
                  max_kv_len=300)
    out.check("prefill out")
    lse.check("prefill lse")
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out.view, lse.view, ref_o, ref_l, "guarded prefill")


def test_multi_token_decode_writes_stay_inside(sa, oracle):
    case = W.make_prefill_case([5, 5], [9, 700], paged=True, page_size=16, layout="HND", seed=603)
    g = case.to("cuda")
    R, Hq, D = case.q.shape
    out = Guarded((R, Hq, D), torch.bfloat16, 6)
    lse = Guarded((R, Hq), torch.float32, 7)
    wsb = sa.sa_decode_multi_workspace_size(2, 5, Hq, 8, D, 700, 0, 3)
    ws = Guarded((max(wsb, 16),), torch.uint8, 8)
    sa.sa_decode_multi(g.q, 5, g.kv, g.seqlens, g.sinks, 0, g.sm_scale, out.view, lse.view, max_kv_len=700,
                       workspace=ws.view, num_splits=3)
    for buf, name in [(out, "out"), (lse, "lse"), (ws, "workspace")]:
        buf.check("multi " + name)
    ref_o, ref_l = oracle_prefill(oracle, case)
    check_close(out.view, lse.view, ref_o, ref_l, "guarded multi-token decode")


def test_rope_append_q_out_stays_inside(sa):
    kv = W.make_kv([40], 8, 64, 16, paged=True, seed=604, layout="HND").to("cuda")
    gen = torch.Generator().manual_seed(605)
    q = torch.randn(40, 64, 64, generator=gen).to(torch.bfloat16).cuda()
    k = torch.randn(40, 8, 64, generator=gen).to(torch.bfloat16).cuda()
    v = torch.randn(40, 8, 64, generator=gen).to(torch.bfloat16).cuda()
    table = sa.sa_rope_yarn_table(64, theta=1e4, factor=1.0, original_max_position=4096, beta_fast=32.0,
                                  beta_slow=1.0).cuda()
    for scale, dtype in [(0.0, torch.bfloat16), (0.05, torch.uint8)]:
        q_out = Guarded((40, 64, 64), dtype, 9)
        sa.sa_rope_append(q, k, v, torch.zeros(40, dtype=torch.int32, device="cuda"),
                          torch.arange(40, dtype=torch.int32, device="cuda"), table, kv, 1, q_out.view,
                          q_out_scale=scale)
        q_out.check("rope q_out (%s)" % dtype)
    assert sa.sa_device_status() == 0
