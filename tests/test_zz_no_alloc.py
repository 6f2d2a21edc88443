"""The allocation-free backward (fcp_block_attn_bwd_static_scratch) against the regular one.

The variant is for callers that cannot allocate device memory: it keeps its scratch in a
fixed array inside the library. Here it is called through the C ABI twice in a row (the
second call sees the array exactly as the first left it) and each result is compared with
fcp_block_attn_bwd given a caller-allocated workspace, within the backward tolerance of the
parity tests. This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import workloads as W
from tests import parity_util as U

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("w", [W.tiny_causal(),
                               W.Workload("small full d128", [700, 129, 1500, 64], 512, 8, 2, 128, 3, False)],
                         ids=lambda w: w.name)
def test_static_scratch_backward_matches_regular(fcp, w):
    L = fcp.lib()
    dev = torch.device("cuda")
    q, k, v = W.make_qkv(w, device=dev)
    do = W.make_dout(w, device=dev)
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim,
                           coalesce=w.coalesce, device=dev)
    assert att.plan.workspace_bytes(w.hq, w.head_dim) <= L.fcp_bwd_static_scratch_bytes()
    o, lse = att.forward(q, k, v)
    ref = att.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
        st = L.fcp_block_attn_bwd_static_scratch(att.plan.handle, _p(att.d_plan), _p(q), _p(k), _p(v), _p(o),
                                                 _p(do), _p(lse), w.hq, w.hkv, w.head_dim, _p(dq), _p(dk), _p(dv),
                                                 stream)
        assert st == 0, L.fcp_last_error()
        torch.cuda.synchronize()
        att.check_device_error()
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            U.check_grad(name, U.np64(got), U.np64(want), f"{w.name} call {call}")


def test_static_scratch_rejects_oversize(fcp):
    L = fcp.lib()
    w = W.causal_mixed()  # 64 heads x 65536 tokens x 129 floats: far beyond the array
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers)
    assert plan.workspace_bytes(w.hq, w.head_dim) > L.fcp_bwd_static_scratch_bytes()
    # null device pointers: the size check comes first, and if it ever did not, the call would
    # stop at the pointer checks instead of launching anything
    st = L.fcp_block_attn_bwd_static_scratch(plan.handle, None, None, None, None, None, None, None, w.hq, w.hkv,
                                             w.head_dim, None, None, None, None)
    assert st == 3
    assert b"exceeds" in L.fcp_last_error()
