"""Decode (T = 1) through the C ABI, against the FP64 oracle.

One decode step is the recurrence for a single token from a given state, so the
oracle's forward over one token per sequence (with the state as h0) gives its
output and new state. A run of decode steps must also reproduce the oracle's
forward over the whole run. Bars: BF16 outputs and BF16 states as in the parity
tests (|x - ref| <= 1e-2 + 1e-2 |ref|, relative L2 <= 5e-3); FP32 states
relative L2 <= 1e-3.
"""

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_test_utils import BF16_ATOL, BF16_REL_L2, BF16_RTOL, FP32_REL_L2, rel_l2

pytestmark = pytest.mark.gpu

LOGITS = dict(use_gate_in_kernel=True, beta_is_logit=True)  # the training-style inputs of make_inputs


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from linear_attention_gated_gb300 import build
    build.build()
    from linear_attention_gated_gb300 import kda
    kda.load_library()


def _bf16_check(name, x, ref):
    x = np.asarray(x, dtype=np.float64)
    bad = np.abs(x - ref) > BF16_ATOL + BF16_RTOL * np.abs(ref)
    assert not bad.any(), f"{name}: {int(bad.sum())} elements outside atol/rtol 1e-2"
    assert rel_l2(x, ref) <= BF16_REL_L2, (name, rel_l2(x, ref))


def _oracle_forward(x, h0):
    f = {k: v.double().numpy() for k, v in x.items() if isinstance(v, torch.Tensor)}
    return oracle.forward(f["q"], f["k"], f["v"], f["g"], f["beta"], f["A_log"], f["dt_bias"],
                          h0.double().numpy(), cu_seqlens=None)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16], ids=["fp32_state", "bf16_state"])
def test_decode_step_matches_oracle(state_dtype):
    from linear_attention_gated_gb300 import kda
    x = ki.make_inputs(5, 1, 2, 4, seed=31)  # 5 sequences, one token each, GQA 2 -> 4
    state = x["h0"].to(state_dtype)
    o_ref, s_ref = _oracle_forward(x, state.float())
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    st = state.cuda()
    o = kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], st, **LOGITS)
    torch.cuda.synchronize()
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    got = st.float().cpu().numpy()
    if state_dtype == torch.float32:
        assert rel_l2(got, s_ref) <= FP32_REL_L2, rel_l2(got, s_ref)
    else:
        _bf16_check("state", got, s_ref)


def test_decode_steps_reproduce_forward():
    """Six decode steps from h0 give the oracle's forward over the six tokens."""
    from linear_attention_gated_gb300 import kda
    T = 6
    x = ki.make_inputs(3, T, 1, 2, seed=32)
    o_ref, s_ref = _oracle_forward(x, x["h0"])
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    st = d["h0"].clone()
    outs = []
    for t in range(T):
        tok = {k: d[k][:, t:t + 1].contiguous() for k in ("q", "k", "v", "g", "beta")}
        outs.append(kda.kda_decode(tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"], d["A_log"],
                                   d["dt_bias"], st, **LOGITS))
    torch.cuda.synchronize()
    _bf16_check("o", torch.cat(outs, dim=1).float().cpu().numpy(), o_ref)
    assert rel_l2(st.cpu().numpy(), s_ref) <= FP32_REL_L2


def test_decode_state_indices():
    """Sequences read and write their own pool slots; other slots are untouched."""
    from linear_attention_gated_gb300 import kda
    x = ki.make_inputs(3, 1, 2, 2, seed=33)
    pool = 0.05 * torch.randn((7, 2, 128, 128), generator=torch.Generator().manual_seed(34))
    slots = torch.tensor([5, 0, 3], dtype=torch.int32)
    o_ref, s_ref = _oracle_forward(x, pool[slots.long()])
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    p = pool.cuda()
    o = kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], p,
                       state_indices=slots.cuda(), **LOGITS)
    torch.cuda.synchronize()
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    got = p.cpu()
    assert rel_l2(got[slots.long()].numpy(), s_ref) <= FP32_REL_L2
    untouched = [i for i in range(7) if i not in slots.tolist()]
    assert torch.equal(got[untouched], pool[untouched])


def test_decode_rejections():
    from linear_attention_gated_gb300 import kda
    x = ki.make_inputs(2, 1, 1, 1, seed=35)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool = torch.zeros((4, 1, 128, 128), device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], pool)
    with pytest.raises(kda.KdaError, match="share a state slot"):
        kda.kda_decode(*args, state_indices=torch.tensor([1, 1], dtype=torch.int32, device="cuda"), **LOGITS)
    with pytest.raises(kda.KdaError, match="out of range"):
        kda.kda_decode(*args, state_indices=torch.tensor([0, 4], dtype=torch.int32, device="cuda"), **LOGITS)
    small = torch.zeros((1, 1, 128, 128), device="cuda")
    with pytest.raises(kda.KdaError, match="slot per sequence"):
        kda.kda_decode(*args[:7], small, **LOGITS)
    with pytest.raises(kda.KdaError, match="overlaps"):
        kda.kda_decode(*args, out=d["v"], **LOGITS)
    with pytest.raises(kda.KdaError, match="lower_bound"):
        kda.kda_decode(*args, lower_bound=-3.0, **LOGITS)
    with pytest.raises(TypeError, match="A_log"):
        kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, pool, **LOGITS)


@pytest.mark.parametrize("use_gate_in_kernel,beta_is_logit", [(False, False), (False, True), (True, False)],
                         ids=["log_g_sigmoided_beta", "log_g_beta_logit", "gate_in_kernel_sigmoided_beta"])
def test_decode_gate_modes(use_gate_in_kernel, beta_is_logit):
    """The recurrent_kda page's gate modes: g already the log decay (A_log and
    dt_bias then not needed), beta already sigmoided."""
    from linear_attention_gated_gb300 import kda
    x = ki.make_inputs(4, 1, 2, 4, seed=36)
    y = ki.precomputed_gate_inputs(x, seed=37)
    if use_gate_in_kernel:
        y["g"] = x["g"]
    if beta_is_logit:
        y["beta"] = x["beta"]
    f = {k: v.double().numpy() for k, v in y.items() if isinstance(v, torch.Tensor)}
    o_ref, s_ref = oracle.forward(f["q"], f["k"], f["v"], f["g"], f["beta"], f["A_log"], f["dt_bias"],
                                  f["h0"], log_space_g=not use_gate_in_kernel,
                                  presigmoid_beta=not beta_is_logit)
    d = {k: v.cuda() for k, v in y.items() if isinstance(v, torch.Tensor)}
    st = d["h0"].clone()
    gate = (d["A_log"], d["dt_bias"]) if use_gate_in_kernel else (None, None)
    o = kda.kda_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], *gate, st,
                       use_gate_in_kernel=use_gate_in_kernel, beta_is_logit=beta_is_logit)
    torch.cuda.synchronize()
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    assert rel_l2(st.cpu().numpy(), s_ref) <= FP32_REL_L2


def test_decode_graph_replay_with_rewritten_indices():
    """A decode step with device slot indices, captured into a CUDA graph (the host mirror is
    checked once, when the call is captured): a replay reads the device indices as they are
    then. Rewritten to other distinct slots, it updates those slots exactly as an eager call
    does; an index rewritten outside the pool leaves the pool alone and gives NaN for that
    sequence, while the others are unaffected."""
    from linear_attention_gated_gb300 import kda
    x = ki.make_inputs(3, 1, 2, 2, seed=36)
    pool0 = (0.05 * torch.randn((6, 2, 128, 128), generator=torch.Generator().manual_seed(37))).cuda()
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    toks = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"])
    idx_cpu = torch.tensor([0, 1, 2], dtype=torch.int32)
    idx = idx_cpu.cuda()
    pool = pool0.clone()
    out = torch.empty_like(d["v"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda.kda_decode(*toks, pool, state_indices=idx, state_indices_cpu=idx_cpu, out=out, **LOGITS)

    new = torch.tensor([4, 2, 5], dtype=torch.int32)
    pool.copy_(pool0)
    idx.copy_(new.cuda())
    graph.replay()
    ref_pool = pool0.clone()
    ref_o = kda.kda_decode(*toks, ref_pool, state_indices=new.cuda(), state_indices_cpu=new, **LOGITS)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(pool, ref_pool)

    pool.copy_(pool0)
    idx.copy_(torch.tensor([4, 6, 5], dtype=torch.int32).cuda())  # 6 is outside the 6-slot pool
    graph.replay()
    torch.cuda.synchronize()
    assert torch.isnan(out[1].float()).all()
    assert torch.equal(out[0], ref_o[0]) and torch.equal(out[2], ref_o[2])
    want = pool0.clone()
    want[4], want[5] = ref_pool[4], ref_pool[5]
    assert torch.equal(pool, want)
