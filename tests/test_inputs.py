"""The seeded synthetic inputs: the workloads have the shapes, sizes and value
ranges their recipe states, and the same seed draws the same problem (so the
benchmark's configuration cannot drift while the parity tests stay green)."""

import math

import pytest
import torch

import kda_inputs as ki

# sizes of the five named configurations: (token·heads, (sequence, value head) units)
SIZES = {
    "fixed_b1_t64_h2": (128, 2),
    "fixed_b2_t1024_h32": (65_536, 64),
    "fixed_b4_t2048_hqk16_hv32": (262_144, 128),
    "packed_8x1024_h96": (786_432, 768),
    "packed_24mixed_hqk8_hv64": (3_532_544, 1536),
}

# lengths the recipe gives for the mixed workload (24 draws of U[1, 4000], seed 4)
MIXED = [1531, 3695, 632, 774, 3490, 3977, 3320, 3977, 2483, 362, 1339, 3997, 2856, 1614, 2751, 88,
         2968, 2234, 3401, 3813, 179, 2381, 2919, 415]


def test_mixed_workload_lengths():
    assert ki.mixed_lengths(4, 24, 4000) == MIXED
    assert sum(MIXED) == 55_196 and min(MIXED) == 88 and max(MIXED) == 3997
    assert all(n % 16 for n in MIXED)  # every sequence ends on a ragged sub-chunk


@pytest.mark.parametrize("name", sorted(SIZES))
def test_workload_sizes(name):
    w = ki.WORKLOADS[name]
    token_heads, units = SIZES[name]
    assert w.token_heads == token_heads
    n_seq = (w.mixed_n or len(w.lengths)) if w.packed else w.B
    assert n_seq * w.hv == units
    assert w.hv % w.hqk == 0


def test_draws_are_seeded_and_follow_the_recipe():
    a = ki.make_inputs(1, 0, 2, 4, seed=7, lengths=[5, 19])
    b = ki.make_inputs(1, 0, 2, 4, seed=7, lengths=[5, 19])
    c = ki.make_inputs(1, 0, 2, 4, seed=8, lengths=[5, 19])
    for k, v in a.items():
        assert torch.equal(v, b[k]), k
    assert not torch.equal(a["q"], c["q"])
    assert a["cu_seqlens"].tolist() == [0, 5, 24] and a["cu_seqlens"].dtype == torch.int64
    for k in ("q", "k", "v", "g", "beta", "do"):
        assert a[k].dtype == torch.bfloat16, k
    assert a["q"].shape == (1, 24, 2, 128) and a["v"].shape == (1, 24, 4, 128) and a["beta"].shape == (1, 24, 4)
    for k in ("A_log", "dt_bias", "h0", "dfinal_state"):
        assert a[k].dtype == torch.float32, k
    assert a["h0"].shape == (2, 4, 128, 128) and a["dt_bias"].shape == (4, 128)
    assert (a["A_log"] >= 0).all() and (a["A_log"] < math.log(16.0)).all()


def test_precomputed_gate_inputs_ranges():
    x = ki.precomputed_gate_inputs(ki.make_inputs(2, 33, 1, 2, seed=9), seed=10)
    g, beta = x["g"].float(), x["beta"].float()
    assert (g <= 0).all() and (g >= -5).all()
    assert (beta >= 0).all() and (beta <= 1).all()
