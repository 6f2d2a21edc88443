"""The device-side failure path, exercised without a GPU fault: a bounded wait (both forms the
kernels use) that runs out records a code in the plan's error word and returns instead of
hanging, the host reads the code, the context stays usable, and kernels started after a
recorded error skip their work."""
import time

import pytest
import torch

import workloads as W
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(fcp):
    d_plan = torch.zeros(256, dtype=torch.uint8, device="cuda")
    t0 = time.perf_counter()
    fcp.selftest_bounded_wait(d_plan)
    code = fcp.device_error(d_plan)  # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert code == 0x40
    # the backward's poll-then-suspend wait gave up too, recording its code in the next word
    assert int(d_plan[4:8].view(torch.int32).item()) == 0x41
    assert 1.5 < elapsed < 60  # the waits' limit is 2 s
    assert fcp.device_error(d_plan) == 0  # reading clears the word
    # the context still runs the whole path correctly
    w = W.tiny_causal()
    r = U.run_path(fcp, w)
    ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
    U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, "after the self-test")


def test_kernels_skip_work_after_a_recorded_error(fcp):
    """With the error word already set, every forward and backward CTA skips its work: the
    partial and gradient buffers keep their contents and the code is reported unchanged."""
    w = W.Workload("skip", [700, 1300], 256, 8, 2, 128, 3, True)
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim)
    q, k, v = W.make_qkv(w, device="cuda")
    do = W.make_dout(w, device="cuda")
    att.part_o.fill_(7.0)
    att.d_plan[:4].copy_(torch.tensor([9, 0, 0, 0], dtype=torch.uint8))  # error word = 9
    fcp.block_attn_fwd(att.plan, att.d_plan, q, k, v, att.part_o, att.part_lse)
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    dq_acc = torch.zeros((w.hq, w.total_tokens, w.head_dim), dtype=torch.float32, device="cuda")
    di = torch.zeros((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    lse = torch.zeros((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    fcp.block_attn_bwd_tiles(att.plan, att.d_plan, q, k, v, do, lse, di, dq_acc, dk, dv)
    torch.cuda.synchronize()
    assert torch.all(att.part_o == 7.0)
    assert torch.all(dk == 3.0) and torch.all(dv == 3.0) and torch.all(dq_acc == 0.0)
    assert fcp.device_error(att.d_plan) == 9
