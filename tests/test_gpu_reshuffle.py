"""GPU parity of the transparent reshuffle (permutation between the user's and the workers'
token layouts) against the oracle's worker order: bit-exact gather and round trip."""
import pytest
import torch

import workloads as W
from oracle import plan as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [W.tiny_causal(), W.causal_mixed(), W.full_mask()], ids=lambda w: w.name)
@pytest.mark.parametrize("dtype,width", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 128),
                                         (torch.bfloat16, 48)])
@pytest.mark.parametrize("heads", [3, 19])
def test_reshuffle_matches_oracle_order(fcp, w, dtype, width, heads):
    """Heads 3 take only the per-head tail of the copy loop, 19 two groups of eight and a tail;
    width 48 in bf16 is a 96-byte row, six 16-byte chunks (not a power of two)."""
    part = P.partition(w.seqlens, w.block_size, w.causal)
    dist = P.distribute(part, w.n_workers, w.token_cap)
    order = torch.tensor(P.worker_order(part, dist, w.n_workers), dtype=torch.long)
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers, w.token_cap)
    d_plan = torch.empty(plan.device_bytes(), dtype=torch.uint8, device="cuda")
    plan.upload(d_plan)
    g = torch.Generator(device="cuda").manual_seed(7)
    x = torch.randn((heads, w.total_tokens, width), generator=g, device="cuda").to(dtype)
    y = torch.empty_like(x)
    fcp.reshuffle(plan, d_plan, x, y, to_workers=True)
    z = torch.empty_like(x)
    fcp.reshuffle(plan, d_plan, y, z, to_workers=False)
    torch.cuda.synchronize()
    xc, yc = x.cpu(), y.cpu()
    assert torch.equal(yc, xc[:, order])
    assert torch.equal(z.cpu(), xc)


def test_reshuffle_more_head_groups_than_grid_rows(fcp):
    """524291 heads = 65537 groups of eight plus three: more head groups than the launch's
    65535 grid rows, so some CTAs take a second group (and the three-head tail)."""
    w = W.Workload("many heads", [5, 3], 2, 2, 1, 8, 2, True)
    part = P.partition(w.seqlens, w.block_size, w.causal)
    dist = P.distribute(part, w.n_workers, w.token_cap)
    order = torch.tensor(P.worker_order(part, dist, w.n_workers), dtype=torch.long)
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers, w.token_cap)
    d_plan = torch.empty(plan.device_bytes(), dtype=torch.uint8, device="cuda")
    plan.upload(d_plan)
    heads = 8 * 65537 + 3
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn((heads, w.total_tokens, 8), generator=g, device="cuda").to(torch.bfloat16)
    y = torch.empty_like(x)
    fcp.reshuffle(plan, d_plan, x, y, to_workers=True)
    z = torch.empty_like(x)
    fcp.reshuffle(plan, d_plan, y, z, to_workers=False)
    torch.cuda.synchronize()
    xc = x.cpu()
    assert torch.equal(y.cpu(), xc[:, order])
    assert torch.equal(z.cpu(), xc)
