"""Inference prefill (kda_prefill) through the C ABI, against the FP64 oracle
and against the training forward.

Prefill is the forward recurrence from a pool slot's state, with the final
state written back to the slot, optionally with BF16 state checkpoints every N
tokens (row 0 of each sequence: its initial state; row j: the state before
token j N). The oracle's forward over each sequence gives o and the final
state; its forward over each prefix gives the checkpoint rows. Bars as in the
parity tests (BF16 tensors: |x - ref| <= 1e-2 + 1e-2 |ref| and relative L2 <=
5e-3; FP32 states: relative L2 <= 1e-3).
"""

import numpy as np
import pytest
import torch

import kda_inputs as ki
import oracle
from kda_test_utils import BF16_ATOL, BF16_REL_L2, BF16_RTOL, FP32_REL_L2, rel_l2, run_gpu

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


def _oracle(x, h0, lengths, **modes):
    f = {k: v.double().numpy() for k, v in x.items() if isinstance(v, torch.Tensor) and k != "cu_seqlens"}
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return oracle.forward(f["q"], f["k"], f["v"], f["g"], f["beta"], f["A_log"], f["dt_bias"],
                          h0.double().numpy(), cu_seqlens=cu, **modes)


def _prefix_state(x, h0, lengths, n, upto):
    """Oracle state of sequence n after its first `upto` tokens."""
    if upto == 0:
        return h0[n].double().numpy()
    t0 = int(sum(lengths[:n]))
    y = {k: (v[:, t0:t0 + upto].contiguous() if k in ("q", "k", "v", "g", "beta") else v)
         for k, v in x.items() if isinstance(v, torch.Tensor) and k != "cu_seqlens"}
    _, s = _oracle(y, h0[n:n + 1], [upto])
    return s[0]


def test_prefill_matches_oracle_and_training_forward():
    from linear_attention_gated_gb300 import kda
    lengths = [40, 17, 70]
    x = ki.make_inputs(1, 0, 2, 4, seed=41, lengths=lengths)
    o_ref, s_ref = _oracle(x, x["h0"], lengths)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool = d["h0"].clone()
    o = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], pool,
                        cu_seqlens=d["cu_seqlens"], **LOGITS)
    torch.cuda.synchronize()
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    assert rel_l2(pool.cpu().numpy(), s_ref) <= FP32_REL_L2
    # the same kernel arithmetic as the training forward: identical results
    gpu, _ = run_gpu(x)
    assert torch.equal(o.cpu(), torch.as_tensor(gpu["o"]).cpu())
    assert torch.equal(pool.cpu(), torch.as_tensor(gpu["final_state"]).cpu())


def test_prefill_bf16_pool_slots_and_checkpoints():
    from linear_attention_gated_gb300 import kda
    lengths = [33, 64, 5]
    every = 32
    x = ki.make_inputs(1, 0, 1, 2, seed=42, lengths=lengths)
    slots = torch.tensor([4, 1, 2], dtype=torch.int32)
    pool0 = (0.05 * torch.randn((6, 2, 128, 128), generator=torch.Generator().manual_seed(43))).to(torch.bfloat16)
    h0 = pool0[slots.long()].float()
    o_ref, s_ref = _oracle(x, h0, lengths)
    counts = [(n + every - 1) // every for n in lengths]
    starts = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool = pool0.cuda()
    ck = torch.full((int(starts[-1]), 2, 128, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], pool,
                        cu_seqlens=d["cu_seqlens"], state_indices=slots.cuda(), checkpoints=ck,
                        checkpoint_cu_starts=starts.cuda(), checkpoint_every_n_tokens=every, **LOGITS)
    torch.cuda.synchronize()
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    got = pool.float().cpu()
    _bf16_check("final state", got[slots.long()].numpy(), s_ref)
    assert torch.equal(pool.cpu()[[0, 3, 5]], pool0[[0, 3, 5]])  # slots no sequence uses
    ckc = ck.float().cpu().numpy()
    for n in range(len(lengths)):
        for j in range(counts[n]):
            _bf16_check(f"checkpoint {n},{j}", ckc[int(starts[n]) + j], _prefix_state(x, h0, lengths, n, j * every))


def test_prefill_rejections():
    from linear_attention_gated_gb300 import kda
    lengths = [20, 12]
    x = ki.make_inputs(1, 0, 1, 1, seed=44, lengths=lengths)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool = torch.zeros((2, 1, 128, 128), device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], pool)
    ck = torch.zeros((2, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([0, 1, 3], dtype=torch.int64, device="cuda")  # sequence 1 needs 1 row, not 2
    with pytest.raises(kda.KdaError, match="ceil"):
        kda.kda_prefill(*args, cu_seqlens=d["cu_seqlens"], checkpoints=ck, checkpoint_cu_starts=bad,
                        checkpoint_every_n_tokens=32, **LOGITS)
    with pytest.raises(kda.KdaError, match="multiple of 16"):
        kda.kda_prefill(*args, cu_seqlens=d["cu_seqlens"], checkpoints=ck,
                        checkpoint_cu_starts=torch.tensor([0, 1, 2], dtype=torch.int64, device="cuda"),
                        checkpoint_every_n_tokens=24, **LOGITS)
    with pytest.raises(kda.KdaError, match="share a state slot"):
        kda.kda_prefill(*args, cu_seqlens=d["cu_seqlens"],
                        state_indices=torch.tensor([1, 1], dtype=torch.int32, device="cuda"), **LOGITS)


@pytest.mark.parametrize("use_gate_in_kernel,beta_is_logit", [(False, False), (False, True), (True, False)],
                         ids=["log_g_sigmoided_beta", "log_g_beta_logit", "gate_in_kernel_sigmoided_beta"])
def test_prefill_gate_modes(use_gate_in_kernel, beta_is_logit):
    """The recurrent_kda page's gate modes over packed sequences with ragged
    tails: g already the log decay (in [-5, 0]; A_log and dt_bias not needed),
    beta already sigmoided. The status word stays clear."""
    from linear_attention_gated_gb300 import kda
    lengths = [37, 16, 90]
    x = ki.make_inputs(1, 0, 2, 4, seed=45, lengths=lengths)
    y = ki.precomputed_gate_inputs(x, seed=46)
    if use_gate_in_kernel:
        y["g"] = x["g"]
    if beta_is_logit:
        y["beta"] = x["beta"]
    o_ref, s_ref = _oracle(y, y["h0"], lengths, log_space_g=not use_gate_in_kernel,
                           presigmoid_beta=not beta_is_logit)
    d = {k: v.cuda() for k, v in y.items() if isinstance(v, torch.Tensor)}
    pool = d["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gate = (d["A_log"], d["dt_bias"]) if use_gate_in_kernel else (None, None)
    o = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], *gate, pool, cu_seqlens=d["cu_seqlens"],
                        device_status=status, use_gate_in_kernel=use_gate_in_kernel,
                        beta_is_logit=beta_is_logit)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _bf16_check("o", o.float().cpu().numpy(), o_ref)
    assert rel_l2(pool.cpu().numpy(), s_ref) <= FP32_REL_L2


def test_prefill_log_gate_out_of_range_sets_status():
    """A log-space gate value above 0 (a decay above 1) is outside the range
    the chunked evaluation accepts: bit 1 of the status word is set. The value
    used (0.25) keeps every intermediate finite."""
    from linear_attention_gated_gb300 import kda
    lengths = [20]
    x = ki.precomputed_gate_inputs(ki.make_inputs(1, 0, 1, 1, seed=47, lengths=lengths), seed=48)
    x["g"][0, 7, 0, 3] = 0.25
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool = d["h0"].clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], None, None, pool, cu_seqlens=d["cu_seqlens"],
                    device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2


def test_prefill_device_index_outside_pool_sets_status():
    """The kernel checks the device slot indices again (they are what a replayed CUDA graph
    reads): an index outside the pool, behind a host mirror that was in range, sets bit 2 of the
    status word and leaves the pool alone; the other sequence is computed as usual."""
    from linear_attention_gated_gb300 import kda
    lengths = [40, 23]
    x = ki.make_inputs(1, 0, 1, 2, seed=49, lengths=lengths)
    d = {k: v.cuda() for k, v in x.items() if isinstance(v, torch.Tensor)}
    pool0 = (0.05 * torch.randn((3, 2, 128, 128), generator=torch.Generator().manual_seed(50))).cuda()
    cu_cpu = x["cu_seqlens"].clone()
    mirror = torch.tensor([2, 0], dtype=torch.int32)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"])
    ref_pool = pool0.clone()
    ref_o = kda.kda_prefill(*args, ref_pool, cu_seqlens=d["cu_seqlens"], cu_seqlens_cpu=cu_cpu,
                            state_indices=mirror.cuda(), state_indices_cpu=mirror, **LOGITS)
    pool = pool0.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.kda_prefill(*args, pool, cu_seqlens=d["cu_seqlens"], cu_seqlens_cpu=cu_cpu,
                        state_indices=torch.tensor([2, 3], dtype=torch.int32, device="cuda"),
                        state_indices_cpu=mirror, device_status=status, **LOGITS)
    torch.cuda.synchronize()
    assert int(status.item()) == 4
    assert torch.equal(o[:, :lengths[0]], ref_o[:, :lengths[0]])
    want = pool0.clone()
    want[2] = ref_pool[2]
    assert torch.equal(pool, want)
