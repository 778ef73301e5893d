"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Small shapes are compared element by element over every output; the five
named workloads run at full size in the launch configuration the benchmark
times, and are compared on every output of a sample of heads (all sequences,
so the per-head parameter gradients are complete). Also: structural checks on
the GPU path itself (packed = fixed, GQA = repeated heads, determinism), a
property that holds at any size (beta = 1 with q = k returns scale * v), and
the context rules (reuse, modified inputs, aliasing, wrong stream).
"""

import json
import os

import numpy as np
import pytest
import torch

import kda_inputs as ki
from kda_test_utils import compare, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu

REPORT = os.environ.get("KDA_PARITY_REPORT")


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from linear_attention_gated_gb300 import build
    build.build()
    from linear_attention_gated_gb300 import kda
    kda.load_library()


def _log(name, report):
    if REPORT:
        with open(REPORT, "a") as f:
            f.write(json.dumps({"case": name, "rel_l2": {k: v[0] for k, v in report.items()},
                                "max_abs": {k: v[1] for k, v in report.items()}}) + "\n")


SMALL = [
    ("fixed_b1_t1_h1", dict(B=1, T=1, hqk=1, hv=1, seed=100)),
    ("fixed_b2_t17_h2", dict(B=2, T=17, hqk=2, hv=2, seed=101)),
    ("fixed_b1_t300_h1", dict(B=1, T=300, hqk=1, hv=1, seed=102)),
    ("packed_ragged_gqa2", dict(B=1, T=0, hqk=1, hv=2, seed=103, lengths=[1, 15, 16, 17, 33, 64, 100])),
    ("packed_gqa4", dict(B=1, T=0, hqk=2, hv=8, seed=104, lengths=[5, 40, 129])),
    ("fixed_b3_t48_gqa3", dict(B=3, T=48, hqk=2, hv=6, seed=105)),
]


@pytest.mark.parametrize("name,cfg", SMALL, ids=[s[0] for s in SMALL])
def test_parity_small(name, cfg):
    x = ki.make_inputs(**cfg)
    gpu, _ = run_gpu(x)
    ref = run_oracle(x)
    _log(name, compare(gpu, ref))


def test_extreme_gates_and_betas():
    """Half of the key dimensions near the strongest decay the gate allows (g = 4: a in [-5, -4.9]
    for every token, so one 16-token sub-chunk spans a factor of about e^-80, near the end of
    FP32's normal range), the other half near none (g = -4: a in [-0.09, 0]), and beta logits of
    -12 or +12: the chunked form's decay factors and their inverses reach their extremes and must
    still match the oracle."""
    x = ki.make_inputs(1, 0, 2, 2, seed=106, lengths=[70, 33])
    dims = torch.arange(ki.DIM)
    x["g"] = torch.where(dims % 2 == 0, 4.0, -4.0).expand_as(x["g"]).to(torch.bfloat16).contiguous()
    tok = torch.arange(x["beta"].shape[1]).view(1, -1, 1)
    x["beta"] = torch.where(tok % 3 == 0, -12.0, 12.0).expand_as(x["beta"]).to(torch.bfloat16).contiguous()
    gpu, _ = run_gpu(x)
    _log("extreme_gates_and_betas", compare(gpu, run_oracle(x)))


def test_long_sequence():
    """One 32763-token sequence and a 21-token one, GQA 1:2: 2048 sub-chunks of FP32 state and
    adjoint accumulation in one unit. The decay gradient's per-sub-chunk anchor, the parameter
    gradients summed over the whole sequence and the initial-state gradient carried back through
    it must still meet the bars."""
    x = ki.make_inputs(1, 0, 1, 2, seed=107, lengths=[32763, 21])
    gpu, _ = run_gpu(x)
    _log("long_sequence", compare(gpu, run_oracle(x)))


def test_zero_and_scaled_rows():
    """Padding-like tokens with all-zero q or k (the norm's eps takes over: q^ = 0 and the norm
    backward scales by 1/sqrt(1e-6) = 1000), a query row scaled by 1000 (normalised away) and value
    rows scaled by 50 (outputs and state grow in proportion) still match the oracle."""
    x = ki.make_inputs(1, 0, 2, 4, seed=108, lengths=[50, 29])
    x["q"][0, 5:9] = 0
    x["k"][0, 12:14] = 0
    x["k"][0, 60] = 0
    x["q"][0, 20] = (x["q"][0, 20].float() * 1000).to(torch.bfloat16)
    x["v"][0, 30:40] = (x["v"][0, 30:40].float() * 50).to(torch.bfloat16)
    gpu, _ = run_gpu(x)
    _log("zero_and_scaled_rows", compare(gpu, run_oracle(x)))


def _random_case(seed):
    """A seeded random small problem: layout, sequence count and lengths (ragged, 1..159 tokens),
    query/key heads and GQA ratio."""
    rng = np.random.default_rng(seed)
    hqk = int(rng.integers(1, 4))
    hv = hqk * int(rng.choice([1, 2, 4]))
    if rng.random() < 0.5:
        lengths = [int(t) for t in rng.integers(1, 160, int(rng.integers(1, 5)))]
        return dict(B=1, T=0, hqk=hqk, hv=hv, seed=seed, lengths=lengths)
    return dict(B=int(rng.integers(1, 4)), T=int(rng.integers(1, 120)), hqk=hqk, hv=hv, seed=seed)


@pytest.mark.parametrize("seed", range(300, 316))
def test_parity_random_shapes(seed):
    x = ki.make_inputs(**_random_case(seed))
    gpu, _ = run_gpu(x)
    _log(f"random_{seed}", compare(gpu, run_oracle(x)))


# full-size workloads: sampled query/key heads (None = all)
WORKLOADS = [
    ("fixed_b1_t64_h2", None),
    ("fixed_b2_t1024_h32", None),
    ("fixed_b4_t2048_hqk16_hv32", [0, 9, 15]),
    ("packed_8x1024_h96", [0, 47, 95]),
    ("packed_24mixed_hqk8_hv64", [5]),
]


@pytest.mark.parametrize("name,heads", WORKLOADS, ids=[w[0] for w in WORKLOADS])
def test_parity_workload(name, heads):
    w = ki.WORKLOADS[name]
    x = ki.workload_inputs(name)
    gpu, _ = run_gpu(x)
    r = w.hv // w.hqk
    ref = run_oracle(x, heads=heads, r=r)
    _log(name, compare(gpu, ref, heads=heads, r=r))


def test_packed_equals_fixed():
    x = ki.make_inputs(2, 100, 2, 4, seed=7)
    fixed, _ = run_gpu(x)
    p = {k: (v.reshape(1, 200, *v.shape[2:]) if k in ("q", "k", "v", "g", "do") else v)
         for k, v in x.items()}
    p["beta"] = x["beta"].reshape(1, 200, -1)
    p["cu_seqlens"] = torch.tensor([0, 100, 200], dtype=torch.int64)
    packed, _ = run_gpu(p)
    for name in fixed:
        a, b = fixed[name], packed[name]
        assert torch.equal(a.reshape(b.shape), b), name


def test_gqa_equals_repeated_heads():
    r = 2
    x = ki.make_inputs(1, 0, 2, 4, seed=8, lengths=[70, 33])
    gqa, _ = run_gpu(x)
    rep = dict(x, q=x["q"].repeat_interleave(r, dim=2), k=x["k"].repeat_interleave(r, dim=2))
    eq, _ = run_gpu(rep)
    for name in ("o", "final_state", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state"):
        assert torch.equal(gqa[name], eq[name]), name
    for name in ("dq", "dk"):
        summed = eq[name].float().reshape(1, 103, 2, r, 128).sum(3)
        err = (gqa[name].float() - summed).norm() / summed.norm()
        assert err < 5e-3, (name, float(err))


def test_deterministic():
    x = ki.make_inputs(1, 0, 2, 8, seed=9, lengths=[50, 200, 17])
    a, _ = run_gpu(x)
    b, _ = run_gpu(x)
    for name in a:
        assert torch.equal(a[name], b[name]), name


def test_context_reuse_matches_fresh_context():
    x1 = ki.make_inputs(2, 40, 2, 2, seed=10)
    x2 = ki.make_inputs(2, 40, 2, 2, seed=11)
    _, ctx = run_gpu(x1)
    reused, _ = run_gpu(x2, ctx=ctx)
    fresh, _ = run_gpu(x2)
    for name in fresh:
        assert torch.equal(reused[name], fresh[name]), name


def test_two_contexts_on_two_streams_at_once():
    """Two problems enqueued on two streams before either is waited for (their kernels may
    share the GPU) give bit for bit what each gives alone: a context shares no device state
    with another."""
    from linear_attention_gated_gb300 import kda_bwd, kda_fwd
    xs = [to_device(ki.make_inputs(1, 0, 2, 4, seed=16, lengths=[300, 47, 129])),
          to_device(ki.make_inputs(3, 200, 1, 2, seed=17))]
    alone = [run_gpu(ki.make_inputs(1, 0, 2, 4, seed=16, lengths=[300, 47, 129]))[0],
             run_gpu(ki.make_inputs(3, 200, 1, 2, seed=17))[0]]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = []
    for x, s in zip(xs, streams):
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            o, hT, ctx = kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["h0"],
                                 cu_seqlens=x.get("cu_seqlens"), cu_seqlens_cpu=x.get("cu_seqlens_cpu"))
            grads = kda_bwd(ctx, x["do"], x["dfinal_state"])
        results.append((o, hT) + tuple(grads))
    torch.cuda.synchronize()
    for want, got in zip(alone, results):
        for name, t in zip(["o", "final_state", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias",
                            "dinitial_state"], got):
            assert torch.equal(t.cpu(), want[name]), name


def test_step_captured_in_a_cuda_graph():
    """With a context made beforehand on the capturing stream, kda_fwd + kda_bwd only enqueue
    kernels, so a whole step can be captured into a CUDA graph; replayed on new input values
    copied into the captured tensors it gives bit for bit what the eager calls give."""
    from linear_attention_gated_gb300 import kda_bwd, kda_fwd
    shape = dict(B=1, T=0, hqk=2, hv=4, lengths=[100, 37])
    x = to_device(ki.make_inputs(seed=18, **shape))
    keys = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o, hT, ctx = kda_fwd(*[x[k_] for k_ in keys], cu_seqlens=x["cu_seqlens"], cu_seqlens_cpu=x["cu_seqlens_cpu"])
        grads = kda_bwd(ctx, x["do"], x["dfinal_state"])
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda_fwd(*[x[k_] for k_ in keys], cu_seqlens=x["cu_seqlens"], cu_seqlens_cpu=x["cu_seqlens_cpu"],
                out=o, final_state_out=hT, context_out=ctx)
        kda_bwd(ctx, x["do"], x["dfinal_state"], out=grads)
    y = ki.make_inputs(seed=19, **shape)
    for k_ in keys + ["do", "dfinal_state"]:
        x[k_].copy_(y[k_].to("cuda"))
    graph.replay()
    torch.cuda.synchronize()
    want, _ = run_gpu(y)
    for name, got in zip(["o", "final_state", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias",
                          "dinitial_state"], (o, hT) + tuple(grads)):
        assert torch.equal(got.cpu(), want[name]), name


def test_every_output_element_written():
    """Outputs pre-filled with NaN come back finite (no unwritten region)."""
    from linear_attention_gated_gb300 import kda_bwd, kda_fwd
    x = to_device(ki.make_inputs(1, 0, 1, 3, seed=12, lengths=[3, 31, 18]))
    o = torch.full(x["v"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    hT = torch.full(x["h0"].shape, float("nan"), device="cuda")
    o, hT, ctx = kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["h0"],
                         cu_seqlens=x["cu_seqlens"], cu_seqlens_cpu=x["cu_seqlens_cpu"], out=o,
                         final_state_out=hT)
    shapes = [(x["q"].shape, torch.bfloat16)] * 2 + [(x["v"].shape, torch.bfloat16)] * 2 + [
        (x["beta"].shape, torch.bfloat16), (x["A_log"].shape, torch.float32),
        (x["dt_bias"].shape, torch.float32), (x["h0"].shape, torch.float32)]
    out = tuple(torch.full(s, float("nan"), dtype=dt, device="cuda") for s, dt in shapes)
    grads = kda_bwd(ctx, x["do"], x["dfinal_state"], out=out)
    torch.cuda.synchronize()
    for t in (o, hT) + tuple(grads):
        assert torch.isfinite(t.float()).all()


def test_beta_one_query_equal_key_returns_scaled_value():
    """Property at a full-size shape: with beta = sigmoid(+inf) = 1 and q = k the
    updated state maps k^ to v exactly, so o = v / sqrt(128) (to BF16 rounding)."""
    from linear_attention_gated_gb300 import kda_fwd
    x = to_device(ki.workload_inputs("packed_8x1024_h96"))
    beta = torch.full_like(x["beta"], float("inf"))
    o, _, _ = kda_fwd(x["k"], x["k"], x["v"], x["g"], beta, x["A_log"], x["dt_bias"], x["h0"],
                      cu_seqlens=x["cu_seqlens"], cu_seqlens_cpu=x["cu_seqlens_cpu"])
    want = x["v"].double() / np.sqrt(128.0)
    err = (o.double() - want).norm() / want.norm()
    assert err < 5e-3, float(err)


def test_modified_input_is_rejected():
    from linear_attention_gated_gb300 import KdaError, kda_bwd, kda_fwd
    x = to_device(ki.make_inputs(1, 32, 1, 1, seed=13))
    o, hT, ctx = kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["h0"])
    x["v"].add_(1.0)
    with pytest.raises(KdaError) as e:
        kda_bwd(ctx, x["do"], x["dfinal_state"])
    assert e.value.name == "KDA_ERR_CONTEXT"


def test_overlapping_output_is_rejected():
    from linear_attention_gated_gb300 import KdaError, kda_fwd
    x = to_device(ki.make_inputs(1, 32, 1, 1, seed=14))
    with pytest.raises(KdaError) as e:
        kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["h0"], out=x["v"])
    assert e.value.name == "KDA_ERR_ALIASING"


def test_backward_on_another_stream_is_rejected():
    from linear_attention_gated_gb300 import KdaError, kda_bwd, kda_fwd
    x = to_device(ki.make_inputs(1, 32, 1, 1, seed=15))
    o, hT, ctx = kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["h0"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with pytest.raises(KdaError) as e:
            kda_bwd(ctx, x["do"], x["dfinal_state"])
    assert e.value.name == "KDA_ERR_CONTEXT"
