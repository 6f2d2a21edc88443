"""FcpAttention.replan: a training loop plans every batch anew. A second batch with other
sequence lengths and the same total tokens runs through the buffers allocated for the first
(the plan is rebuilt on the host and its device image uploaded in stream order) and matches
the float64 oracle; a batch that does not fit the buffers is refused on the host."""
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _check(att, w, seed):
    dev = torch.device("cuda")
    q, k, v = W.make_qkv(w, device=dev, seed=seed)
    do = W.make_dout(w, device=dev, seed=seed)
    o, lse = att.forward(q, k, v)
    grads = att.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    att.check_device_error()
    ro, rl = A.attention_forward(q, k, v, w.seqlens, w.causal)
    U.check_forward(U.np64(o), U.np64(lse), ro, rl, w.name)
    rdq, rdk, rdv = A.attention_backward(q, k, v, do, w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, w.name)


def test_replan_runs_a_new_batch_in_the_same_buffers(fcp):
    first = W.Workload("replan first", [1500, 700, 1896], 512, 8, 2, 128, 4, True)
    att = fcp.FcpAttention(first.seqlens, first.block_size, first.causal, first.n_workers, first.hq, first.hkv,
                           first.head_dim, coalesce=16)
    _check(att, first, seed=1)
    buffers = (att.d_plan.data_ptr(), att.part_o.data_ptr(), att.workspace.data_ptr())
    for i, lens in enumerate(([300, 3000, 796], [64] * 64, [4096])):
        w = W.Workload(f"replan {i}", lens, 512, 8, 2, 128, 4, True)
        att.replan(lens)
        assert att.plan.seqlens == lens
        assert (att.d_plan.data_ptr(), att.part_o.data_ptr(), att.workspace.data_ptr()) == buffers
        _check(att, w, seed=2 + i)


def test_replan_refuses_a_batch_that_does_not_fit(fcp):
    att = fcp.FcpAttention([1000, 1000], 512, True, 2, 4, 2, 64)
    with pytest.raises(ValueError):
        att.replan([1000, 1001])  # a different total
    with pytest.raises(RuntimeError):
        fcp.FcpAttention.from_plan(fcp.Plan.ring([1000, 1000], 2, True), 4, 2, 64).replan()
