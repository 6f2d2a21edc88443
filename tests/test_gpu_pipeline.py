"""GPU parity of the block-level pipeline ("Unleashing Scalable Context Parallelism for
Foundation Models Pre-Training via FCP", Section 4.2, Figure 7): the forward launched one
execution stage at a time (fcp_block_attn_fwd_stage), then merged, against the float64
oracle; the stages together write exactly the partials of one whole launch; the backward
over the scheduled work list."""
import pytest
import torch

import workloads as W
from oracle import attention as A
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _sync():
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", W.small_cases(), ids=lambda w: w.name)
@pytest.mark.parametrize("degree", [1, 2, 16])
def test_staged_forward_and_backward_small(fcp, w, degree):
    r = U.run_path(fcp, w, pipeline=degree)
    assert r["att"].n_stages == r["att"].plan.view()["n_exec_stages"]
    ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
    U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, f"{w.name} c={degree}")
    rdq, rdk, rdv = A.attention_backward(r["q"], r["k"], r["v"], r["do"], w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), r["grads"], (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, f"{w.name} c={degree}")


@pytest.mark.parametrize("degree", [1, 4])
def test_stages_write_the_partials_of_one_launch(fcp, degree):
    """Each forward unit is computed the same way whichever launch holds it, so the stage
    launches and one whole launch give bit-identical partial buffers."""
    w = W.Workload("staged", [1500, 40, 700, 2600, 3000], 256, 8, 2, 128, 6, True)
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim,
                           pipeline=degree, backward=False)
    assert att.n_stages > 2
    q, k, v = W.make_qkv(w, device="cuda")
    att.part_o.fill_(float("nan"))
    att.part_lse.fill_(float("nan"))
    for st in range(att.n_stages):
        fcp.block_attn_fwd_stage(att.plan, att.d_plan, st, q, k, v, att.part_o, att.part_lse)
    staged_o, staged_l = att.part_o.clone(), att.part_lse.clone()
    rows = att.plan.view()["partial_rows"]
    assert not torch.isnan(staged_o[:, :rows]).any() and not torch.isnan(staged_l[:, :rows]).any()
    att.part_o.fill_(float("nan"))
    att.part_lse.fill_(float("nan"))
    fcp.block_attn_fwd(att.plan, att.d_plan, q, k, v, att.part_o, att.part_lse)
    assert torch.equal(att.part_o[:, :rows], staged_o[:, :rows])
    assert torch.equal(att.part_lse[:, :rows], staged_l[:, :rows])
    with pytest.raises(fcp.FcpError) as e:
        fcp.block_attn_fwd_stage(att.plan, att.d_plan, att.n_stages, q, k, v, att.part_o, att.part_lse)
    assert e.value.status == 1
    att.check_device_error()


def test_causal_mixed_pipelined_sampled(fcp):
    """The full-size mixed workload, pipelined with the pages' default coalesce degree 16."""
    w = W.causal_mixed()
    r = U.run_path(fcp, w, pipeline=16)
    assert r["att"].n_stages > 1
    U.sampled_forward(r, w, rows_per_seq=24)
    U.sampled_backward(r, w, rows_per_seq=12, kv_tail=64)


def test_full_mask_pipelined_sampled(fcp):
    """The full-mask batch (16 lognormal sequences, 65536 tokens, 1024-token blocks, 8 workers),
    forward only, pipelined at coalesce degree 4, on sampled rows."""
    w = W.full_mask()
    r = U.run_path(fcp, w, pipeline=4)
    assert r["att"].n_stages > 2
    U.sampled_forward(r, w, rows_per_seq=24)


@pytest.mark.parametrize("causal", [True, False])
def test_ring_plan_pipelined(fcp, causal):
    """The ring baseline's plan also runs through the pipeline (many small blocks, many stages)."""
    w = W.Workload("ring pipe", [1500, 40, 700, 2600], 256, 8, 2, 128, 4, causal)
    plan = fcp.Plan.ring(w.seqlens, w.n_workers, w.causal)
    n = plan.schedule(2)
    assert n > 2
    att = fcp.FcpAttention.from_plan(plan, w.hq, w.hkv, w.head_dim, backward=True)
    assert att.n_stages == n
    q, k, v = W.make_qkv(w, device="cuda")
    do = W.make_dout(w, device="cuda")
    o, lse = att.forward(q, k, v)
    dq, dk, dv = att.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    att.check_device_error()
    Q, K, V, dO = (U.np64(t) for t in (q, k, v, do))
    ro, rl = A.attention_forward(Q, K, V, w.seqlens, causal)
    U.check_forward(U.np64(o), U.np64(lse), ro, rl, "ring pipelined")
    rdq, rdk, rdv = A.attention_backward(Q, K, V, dO, w.seqlens, causal)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, "ring pipelined")
