"""The backward's query bands in the host plan (no GPU): the default choice, explicit band
sizes, refusals, and the plan validator's check that every (backward unit, band) pair with a
64-row query step starting in the band is listed exactly once."""
import pytest

import workloads as W


def _plan(fcp, w, band=None, coalesce=16):
    p = fcp.Plan(w.seqlens, w.block_size, w.causal)
    if band is not None:
        p.set_bwd_band(band)
    p.distribute(w.n_workers, w.token_cap)
    p.coalesce(coalesce)
    return p


def test_default_bands_only_for_long_batches(fcp):
    assert _plan(fcp, W.block_sweep(4096)).bwd_bands() == (0, 0)  # 32768 tokens
    p = _plan(fcp, W.long_causal())  # 524288 tokens
    assert p.bwd_bands() == (524288 // 16384, 16384)
    p.validate()


@pytest.mark.parametrize("band", [64, 192, 1024])
@pytest.mark.parametrize("w", W.small_cases(), ids=lambda w: w.name)
def test_explicit_bands_validate(fcp, w, band):
    p = _plan(fcp, w, band)
    n, rows = p.bwd_bands()
    assert rows == band and n == -(-w.total_tokens // band)
    p.validate()
    assert p.band_workspace_bytes(w.hkv, w.head_dim) >= 2 * w.hkv * w.total_tokens * w.head_dim * 4


def test_bands_set_after_distribution_and_removed(fcp):
    w = W.tiny_causal()
    p = _plan(fcp, w)
    assert p.bwd_bands() == (0, 0)
    size0 = p.device_bytes()
    p.set_bwd_band(256).validate()
    assert p.bwd_bands()[1] == 256 and p.device_bytes() > size0
    assert p.band_workspace_bytes(w.hkv, w.head_dim) > 0
    p.set_bwd_band(0).validate()
    assert p.bwd_bands() == (0, 0) and p.band_workspace_bytes(w.hkv, w.head_dim) == 0


@pytest.mark.parametrize("bad", [-2, 1, 100])
def test_band_size_must_be_whole_steps(fcp, bad):
    p = fcp.Plan([1000], 256, True)
    with pytest.raises(fcp.FcpError):
        p.set_bwd_band(bad)


def test_bands_of_a_pipelined_and_a_ring_plan(fcp):
    w = W.Workload("mixed", [1500, 40, 700, 2600], 512, 8, 2, 128, 3, True)
    p = fcp.Plan(w.seqlens, w.block_size, w.causal).set_bwd_band(128).distribute(w.n_workers)
    p.schedule(2)
    p.validate()
    assert p.bwd_bands()[0] == -(-w.total_tokens // 128)
    r = fcp.Plan.ring(w.seqlens, w.n_workers, w.causal)
    r.set_bwd_band(64).validate()
    assert r.bwd_bands()[0] == -(-w.total_tokens // 64)
