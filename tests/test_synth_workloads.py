"""The five standard workloads against the recipe they are stated to follow: layer
counts, device counts and units, tier sizes, candidate and strategy counts, batch
sizes, budgets, and the transformer-block sizes (sequence 2048, microbatch 1):
dense block fl = 24 s h^2 flops, 12 h^2 bf16 parameters, output 2 s h bytes,
working activations 17x the output; MoE block with 64 experts of 8 h^2 parameters,
top-2 routing.  The pages' own models and clusters (Nest §5) are not available;
these stand in for them."""
import numpy as np
import pytest

from memory_aware_device_gb300 import synth

S_, GB = 2048, 10**9

RECIPE = {   # cfg: (layers, D, unit, tier sizes, candidates, strategies, batch)
    1: (8, 8, 1, [8], 1, 8, 1),
    2: (32, 64, 1, [8, 32, 64], 2, 12, 16),
    3: (96, 1024, 8, [8, 256, 512, 1024], 4, 36, 64),
    4: (48, 512, 8, [8, 128, 512], 3, 56, 256),
    5: (128, 4096, 8, [8, 128, 1024, 4096], 4, 672, 1024),
}


@pytest.mark.parametrize("cfg", sorted(RECIPE))
def test_workload_shapes(cfg):
    L, D, unit, G, C, S, B = RECIPE[cfg]
    assert synth.CONFIG_BATCH[cfg] == B
    for b in sorted({0, 1, B - 1}):
        x = synth.config_instance(cfg, b)
        assert (x.L, x.D, x.unit, x.tierG.tolist(), x.C, x.S) == (L, D, unit, G, C, S)
        assert (x.M, x.R, x.opt_factor) == (4096, 10**6, 6)
        if cfg == 5 or (cfg == 2 and b > 0):   # drawn uniformly in [40, 180] GB
            assert 40 * GB <= x.budget <= 180 * GB
        else:
            assert x.budget == 80 * GB


def test_nominal_tiers():
    x = synth.config_instance(2, 0)
    # 900 / 50 / 25 GB/s as bytes per microsecond, 2 / 5 / 10 us as nanoseconds
    assert x.tierBw.tolist() == [900000, 50000, 25000]
    assert x.tierLat.tolist() == [2000, 5000, 10000]


def test_dense_block_sizes():
    x = synth.config_instance(2, 0)
    h = 4096
    assert (x.fl == 24 * S_ * h * h).all()
    assert (x.pd == 2 * 12 * h * h).all()
    assert (x.ao == 2 * S_ * h).all()
    assert (x.aw == 17 * x.ao).all()
    assert not x.moe.any() and not x.pe.any() and not x.a2a.any()


def test_moe_blocks_alternate():
    x = synth.config_instance(4, 0)
    h = 4096
    assert x.moe.tolist() == [0, 1] * 24
    m = np.flatnonzero(x.moe)
    assert (x.pe[m] == 64 * 8 * h * h * 2).all()          # 64 experts of 8 h^2 bf16 parameters
    assert (x.fl[m] == (8 + 16 * 2) * S_ * h * h).all()   # attention + two routed FFNs
    assert (x.pd[m] == 4 * h * h * 2).all()               # the attention block stays dense
    assert (x.a2a[m] > 0).all() and not x.a2a[x.moe == 0].any()
    y = synth.config_instance(5, 0)
    assert int(y.moe.sum()) == 64
