"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding, run the FP64 oracle on the same inputs, compare with the stated bars.

Tolerances (taken from the requirement on this path):
  BF16 tensors (o, dq, dk, dv, dg, dbeta): elementwise |x - ref| <= 1e-2 + 1e-2 |ref|
    and relative L2 error <= 5e-3;
  FP32 tensors (final state, dinitial_state, dA_log, ddt_bias): relative L2 <= 1e-3.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

BF16_ATOL = 1e-2
BF16_RTOL = 1e-2
BF16_REL_L2 = 5e-3
FP32_REL_L2 = 1e-3

FWD_KEYS = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0"]
OUT_NAMES = ["o", "final_state", "dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state"]
BF16_OUTS = {"o", "dq", "dk", "dv", "dg", "dbeta"}


def to_device(x: dict, device="cuda") -> dict:
    d = {}
    for k, v in x.items():
        d[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    if x.get("cu_seqlens") is not None:
        d["cu_seqlens_cpu"] = x["cu_seqlens"].clone()
    return d


def run_gpu(x: dict, ctx=None, device="cuda"):
    """Forward + backward through the C ABI. Returns (outputs dict of CPU tensors, ctx)."""
    from linear_attention_gated_gb300 import kda_bwd, kda_fwd
    d = to_device(x, device)
    o, hT, ctx = kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["h0"],
                         cu_seqlens=d.get("cu_seqlens"), context_out=ctx,
                         cu_seqlens_cpu=d.get("cu_seqlens_cpu"))
    grads = kda_bwd(ctx, d["do"], d["dfinal_state"])
    torch.cuda.synchronize()
    outs = dict(zip(OUT_NAMES, (o, hT) + tuple(grads)))
    return {k: v.cpu() for k, v in outs.items()}, ctx


def slice_heads(x: dict, heads, r: int) -> dict:
    """Inputs restricted to the given query/key heads and their r value heads each
    (the recurrence never mixes heads, so this is the same problem, smaller)."""
    heads = list(heads)
    vheads = [qh * r + j for qh in heads for j in range(r)]
    y = dict(x)
    for k in ("q", "k"):
        y[k] = x[k][:, :, heads]
    for k in ("v", "g", "do"):
        y[k] = x[k][:, :, vheads]
    y["beta"] = x["beta"][:, :, vheads]
    y["A_log"] = x["A_log"][vheads]
    y["dt_bias"] = x["dt_bias"][vheads]
    y["h0"] = x["h0"][:, vheads]
    y["dfinal_state"] = x["dfinal_state"][:, vheads]
    return y


def run_oracle(x: dict, heads=None, r: int = 1) -> dict:
    """FP64 oracle outputs; with ``heads`` only for those query/key heads."""
    if heads is not None:
        x = slice_heads(x, heads, r)
    f = {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    cu = f.get("cu_seqlens")
    o, hT = oracle.forward(*[f[k] for k in FWD_KEYS], cu_seqlens=cu)
    grads = oracle.backward(*[f[k] for k in FWD_KEYS], f["do"], f["dfinal_state"], cu_seqlens=cu)
    return dict(zip(OUT_NAMES, (o, hT) + tuple(grads)))


def _select(name, arr, heads, r):
    """Restrict a tensor to the sampled query/key heads (and their value heads)."""
    if heads is None:
        return arr
    heads = list(heads)
    vheads = [qh * r + j for qh in heads for j in range(r)]
    if name in ("dq", "dk"):
        return arr[:, :, heads]
    if name in ("o", "dv", "dg"):
        return arr[:, :, vheads]
    if name == "dbeta":
        return arr[:, :, vheads]
    if name in ("final_state", "dinitial_state"):
        return arr[:, vheads]
    if name in ("dA_log", "ddt_bias"):
        return arr[vheads]
    raise KeyError(name)


def rel_l2(x, ref):
    num = np.linalg.norm((x - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    return float(num / den) if den > 0 else float(num)


def compare(gpu: dict, ref: dict, heads=None, r=1, names=OUT_NAMES):
    """Assert the bars for every output (``ref`` from run_oracle with the same
    ``heads``); returns {name: (rel_l2, max_abs_err)}."""
    report = {}
    for name in names:
        x = _select(name, gpu[name].double().numpy(), heads, r)
        y = ref[name]
        assert x.shape == y.shape, (name, x.shape, y.shape)
        assert np.all(np.isfinite(x)), f"{name}: non-finite values"
        rl = rel_l2(x, y)
        err = np.abs(x - y)
        report[name] = (rl, float(err.max()) if err.size else 0.0)
        if name in BF16_OUTS:
            bad = err > BF16_ATOL + BF16_RTOL * np.abs(y)
            assert not bad.any(), f"{name}: {int(bad.sum())} elements outside atol/rtol 1e-2"
            assert rl <= BF16_REL_L2, f"{name}: relative L2 {rl:.3e} > {BF16_REL_L2}"
        else:
            assert rl <= FP32_REL_L2, f"{name}: relative L2 {rl:.3e} > {FP32_REL_L2}"
    return report
