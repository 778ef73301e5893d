"""Python binding of the KDA training C ABI (include/kda.h).

Argument marshalling only: torch provides device memory and the current CUDA
stream; every step of the forward and backward runs in libkda.so's kernels.
There is no CPU fallback: if the library cannot be loaded the calls raise.

Names follow the C ABI (``kda_fwd``, ``kda_bwd``); the documented training pair
(flashinfer.kda_training.recurrent_kda_training_forward / _backward) is exposed
under those names too.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")
DIM = 128
SCALE = 1.0 / math.sqrt(DIM)

_STATUS = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARGUMENT", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_ALIASING",
    4: "KDA_ERR_CONTEXT", 5: "KDA_ERR_CUDA", 6: "KDA_ERR_DEVICE_TIMEOUT",
    7: "KDA_ERR_WORKSPACE_TOO_SMALL",
}

EXPORTED = ("kda_ctx_workspace_bytes", "kda_fwd", "kda_bwd", "kda_ctx_status", "kda_ctx_destroy",
            "kda_status_string", "kda_last_error_message", "kda_chunk_tokens",
            "kda_checkpoint_tokens", "kda_bwd_noalloc", "kda_decode", "kda_prefill",
            "kda_selftest_device_timeout", "kda_step_arena_bytes", "kda_step_host",
            "kda_bwd_standalone_workspace_bytes", "kda_bwd_standalone", "kda_noalloc_status")


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = _STATUS.get(status, str(status))


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libkda.so and declare the C signatures. Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run __graft_entry__.build() "
                           "(or python linear_attention_gated_gb300/build.py)")
    lib = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kda_ctx_workspace_bytes.argtypes = [I, I, I, I, P, I, ctypes.POINTER(S)]
    lib.kda_ctx_workspace_bytes.restype = ctypes.c_int
    lib.kda_fwd.argtypes = [P] * 8 + [P, P, I, I, I, I, I, I, F, F, P, P, P, S, ctypes.POINTER(P), P]
    lib.kda_fwd.restype = ctypes.c_int
    lib.kda_bwd.argtypes = [P] * 12
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_ctx_status.argtypes = [P]
    lib.kda_ctx_status.restype = ctypes.c_int
    lib.kda_ctx_destroy.argtypes = [P]
    lib.kda_step_arena_bytes.argtypes = [I, I, I, I, P, I, ctypes.POINTER(S)]
    lib.kda_step_arena_bytes.restype = ctypes.c_int
    lib.kda_step_host.argtypes = [P] * 8 + [P, I, I, I, I, I, I, F, F] + [P] * 12 + [P, S, ctypes.POINTER(P), P, P, P]
    lib.kda_step_host.restype = ctypes.c_int
    lib.kda_ctx_destroy.restype = None
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_error_message.argtypes = []
    lib.kda_last_error_message.restype = ctypes.c_char_p
    lib.kda_bwd_noalloc.argtypes = [P] * 8 + [P, P, I, I, I, I, I, I, F, F] + [P] * 10 + [P]
    lib.kda_bwd_noalloc.restype = ctypes.c_int
    lib.kda_noalloc_status.argtypes = [P]
    lib.kda_noalloc_status.restype = ctypes.c_int
    lib.kda_bwd_standalone_workspace_bytes.argtypes = [I, I, I, I, P, I, ctypes.POINTER(S)]
    lib.kda_bwd_standalone_workspace_bytes.restype = ctypes.c_int
    lib.kda_bwd_standalone.argtypes = ([P] * 8 + [P, P, I, I, I, I, I, I, F, F] + [P] * 10
                                       + [P, S, ctypes.POINTER(P), P])
    lib.kda_bwd_standalone.restype = ctypes.c_int
    lib.kda_decode.argtypes = [P] * 8 + [ctypes.c_int32, P, P, I, I, I, I, I, F, F, ctypes.c_int32,
                                         ctypes.c_int32, P, P]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_prefill.argtypes = [P] * 7 + [P, P, I, I, I, I, I, I, F, F, ctypes.c_int32, ctypes.c_int32, P,
                                          ctypes.c_int32, P, P, I, P, P, I, P, P, I, P, P]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_selftest_device_timeout.argtypes = [P]
    lib.kda_selftest_device_timeout.restype = ctypes.c_int
    lib.kda_chunk_tokens.argtypes = []
    lib.kda_chunk_tokens.restype = ctypes.c_int32
    lib.kda_checkpoint_tokens.argtypes = []
    lib.kda_checkpoint_tokens.restype = ctypes.c_int32
    _lib = lib
    return lib


def _check(rc: int):
    if rc != 0:
        msg = load_library().kda_last_error_message().decode()
        raise KdaError(rc, msg)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _want(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")


def workspace_bytes(B, T, Hqk, Hv, cu_seqlens_cpu=None) -> int:
    lib = load_library()
    out = ctypes.c_size_t(0)
    if cu_seqlens_cpu is not None:
        cu = cu_seqlens_cpu.to(torch.int64).contiguous()
        rc = lib.kda_ctx_workspace_bytes(B, T, Hqk, Hv, _ptr(cu), cu.numel() - 1, ctypes.byref(out))
    else:
        rc = lib.kda_ctx_workspace_bytes(B, T, Hqk, Hv, None, 0, ctypes.byref(out))
    _check(rc)
    return int(out.value)


class KdaContext:
    """Saved forward context: the C handle, the device workspace it owns and the
    borrowed inputs with their tensor versions (inputs must not change between
    the forward and the backward)."""

    def __init__(self):
        self.handle = ctypes.c_void_p(None)
        self.workspace = None
        self.inputs = ()
        self.versions = ()
        self.shape_key = None
        self.device = None
        self.stream = None

    def _snapshot(self, inputs):
        self.inputs = tuple(inputs)
        self.versions = tuple(t._version for t in inputs)
        self.ws_version = self.workspace._version

    def check_unchanged(self):
        for t, v in zip(self.inputs, self.versions):
            if t._version != v:
                raise KdaError(4, "an input of the forward was modified before the backward")
        if self.workspace._version != self.ws_version:
            raise KdaError(4, "the context workspace was modified before the backward")

    def status(self):
        _check(load_library().kda_ctx_status(self.handle))

    def __del__(self):
        try:
            if self.handle and self.handle.value:
                load_library().kda_ctx_destroy(self.handle)
                self.handle = ctypes.c_void_p(None)
        except Exception:
            pass


def _check_forward_inputs(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens, cu_seqlens_cpu):
    """Dtype, shape, contiguity and device checks of the forward's inputs (the C ABI
    repeats the shape rules on the host). Returns (B, T, Hqk, Hv, D, N)."""
    for name, t in (("q", q), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dim() != 4:
            raise ValueError(f"{name} must be a [B, T, H, 128] tensor")
    B, T, Hqk, D = q.shape
    Hv = v.shape[2]
    bf, f32 = torch.bfloat16, torch.float32
    _want(q, "q", bf); _want(k, "k", bf, q.shape); _want(v, "v", bf, (B, T, Hv, D))
    _want(g, "g", bf, (B, T, Hv, D)); _want(beta, "beta", bf, (B, T, Hv))
    _want(A_log, "A_log", f32, (Hv,)); _want(dt_bias, "dt_bias", f32, (Hv, D))
    if q.device.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    for name, t in (("k", k), ("v", v), ("g", g), ("beta", beta), ("A_log", A_log), ("dt_bias", dt_bias),
                    ("initial_state", initial_state)):
        if t.device != q.device:
            raise ValueError(f"{name} must be on {q.device}")
    if cu_seqlens is not None:
        if cu_seqlens_cpu is None:
            raise ValueError("packed input requires cu_seqlens_cpu, a trusted CPU mirror of cu_seqlens")
        _want(cu_seqlens, "cu_seqlens", torch.int64)
        if cu_seqlens.dim() != 1 or cu_seqlens.device != q.device:
            raise ValueError(f"cu_seqlens must be a 1-D tensor on {q.device}")
        _want(cu_seqlens_cpu, "cu_seqlens_cpu", torch.int64, cu_seqlens.shape)
        if cu_seqlens_cpu.device.type != "cpu":
            raise ValueError("cu_seqlens_cpu must be a CPU tensor")
        N = cu_seqlens.numel() - 1
    else:
        if cu_seqlens_cpu is not None:
            raise ValueError("cu_seqlens_cpu must be omitted for fixed-length input")
        N = B
    _want(initial_state, "initial_state", f32, (N, Hv, D, D))
    return B, T, Hqk, Hv, D, N


def kda_fwd(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens=None, scale=None,
            lower_bound=-5.0, out=None, final_state_out=None, context_out=None, *,
            cu_seqlens_cpu=None):
    """Training forward (flashinfer.kda_training.recurrent_kda_training_forward, parameters; the
    recurrence of flashinfer.kda_backward.recurrent_kda_backward, description). Returns
    (o BF16 [B,T,Hv,128], final_state FP32 [N,Hv,128,128], ctx); ctx holds the state checkpoints
    and tapes the backward consumes (flashinfer.kda_training, module description)."""
    lib = load_library()
    B, T, Hqk, Hv, D, N = _check_forward_inputs(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens,
                                                cu_seqlens_cpu)
    bf, f32 = torch.bfloat16, torch.float32
    dev = q.device
    o = out if out is not None else torch.empty((B, T, Hv, D), dtype=bf, device=dev)
    hT = final_state_out if final_state_out is not None else torch.empty((N, Hv, D, D), dtype=f32, device=dev)
    _want(o, "out", bf, (B, T, Hv, D)); _want(hT, "final_state_out", f32, (N, Hv, D, D))
    key = (B, T, Hqk, Hv, None if cu_seqlens_cpu is None else tuple(cu_seqlens_cpu.tolist()))
    stream = torch.cuda.current_stream(dev)
    ctx = context_out
    if ctx is None:
        ctx = KdaContext()
        nbytes = workspace_bytes(B, T, Hqk, Hv, cu_seqlens_cpu)
        ctx.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        ctx.shape_key, ctx.device, ctx.stream = key, dev, stream.cuda_stream
    elif ctx.shape_key != key or ctx.device != dev or ctx.stream != stream.cuda_stream:
        raise KdaError(4, "context reuse needs the same shapes, device and stream")
    ws = ctx.workspace
    rc = lib.kda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                     _ptr(initial_state), _ptr(cu_seqlens),
                     _ptr(cu_seqlens_cpu) if cu_seqlens_cpu is not None else None,
                     N if cu_seqlens is not None else 0, B, T, Hqk, Hv, D,
                     float("nan") if scale is None else float(scale), float(lower_bound),
                     _ptr(o), _ptr(hT), _ptr(ws), ws.numel(), ctypes.byref(ctx.handle),
                     ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    ctx._snapshot((q, k, v, g, beta, A_log, dt_bias, initial_state)
                  + ((cu_seqlens,) if cu_seqlens is not None else ()))
    ctx.out_shapes = dict(q=tuple(q.shape), v=tuple(v.shape), beta=tuple(beta.shape),
                          A_log=tuple(A_log.shape), dt_bias=tuple(dt_bias.shape),
                          h0=tuple(initial_state.shape))
    return o, hT, ctx


GRAD_NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state")


def kda_bwd(ctx: KdaContext, do, dfinal_state, out=None):
    """Training backward from a saved context, without rerunning the forward
    (flashinfer.kda_training.recurrent_kda_training_backward; gradient list and order of
    flashinfer.kda_backward.recurrent_kda_backward, description). Returns
    (dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dinitial_state); dg and dbeta are with respect to
    the raw gate and the raw beta logits."""
    lib = load_library()
    if not isinstance(ctx, KdaContext) or not ctx.handle.value:
        raise KdaError(4, "not a forward context")
    ctx.check_unchanged()
    s = ctx.out_shapes
    _want(do, "do", torch.bfloat16, s["v"])
    _want(dfinal_state, "dfinal_state", torch.float32, s["h0"])
    dev = ctx.device
    if out is None:
        bf, f32 = torch.bfloat16, torch.float32
        out = (torch.empty(s["q"], dtype=bf, device=dev), torch.empty(s["q"], dtype=bf, device=dev),
               torch.empty(s["v"], dtype=bf, device=dev), torch.empty(s["v"], dtype=bf, device=dev),
               torch.empty(s["beta"], dtype=bf, device=dev), torch.empty(s["A_log"], dtype=f32, device=dev),
               torch.empty(s["dt_bias"], dtype=f32, device=dev), torch.empty(s["h0"], dtype=f32, device=dev))
    if len(out) != 8:
        raise ValueError("out must hold eight gradient tensors in return order")
    shapes = (s["q"], s["q"], s["v"], s["v"], s["beta"], s["A_log"], s["dt_bias"], s["h0"])
    dtypes = (torch.bfloat16,) * 5 + (torch.float32,) * 3
    for t, name, shp, dt in zip(out, GRAD_NAMES, shapes, dtypes):
        _want(t, name, dt, shp)
    stream = torch.cuda.current_stream(dev)
    rc = lib.kda_bwd(ctx.handle, _ptr(do), _ptr(dfinal_state), *[_ptr(t) for t in out],
                     ctypes.c_void_p(stream.cuda_stream))
    _check(rc)
    return tuple(out)


def _grad_buffers(out, shapes, dev):
    dtypes = (torch.bfloat16,) * 5 + (torch.float32,) * 3
    if out is None:
        out = tuple(torch.empty(s_, dtype=dt, device=dev) for s_, dt in zip(shapes, dtypes))
    if len(out) != 8:
        raise ValueError("out must hold eight gradient tensors in return order")
    for t, name, s_, dt in zip(out, GRAD_NAMES, shapes, dtypes):
        _want(t, name, dt, s_)
        if t.device != dev:
            raise ValueError(f"{name} must be on {dev}")
    return tuple(out)


def _check_adjoints(do, dfinal_state, B, T, Hv, D, N, dev):
    _want(do, "do", torch.bfloat16, (B, T, Hv, D))
    _want(dfinal_state, "dfinal_state", torch.float32, (N, Hv, D, D))
    if do.device != dev or dfinal_state.device != dev:
        raise ValueError(f"do and dfinal_state must be on {dev}")


def kda_bwd_noalloc(q, k, v, g, beta, A_log, dt_bias, initial_state, do, dfinal_state,
                    cu_seqlens=None, scale=None, lower_bound=-5.0, out=None, *, cu_seqlens_cpu=None):
    """Standalone backward that allocates no device memory in the library (for
    callers that cannot call cudaMalloc; scratch is a fixed array compiled into
    libkda.so). The pages have no counterpart for this entry point; it computes
    what recurrent_kda_training_forward followed by _backward computes
    (flashinfer.kda_training). Returns the eight gradients of kda_bwd. ``out`` (eight tensors in
    return order) lets the caller own every output buffer as well. ``noalloc_status()`` reads
    back the call's device status word."""
    lib = load_library()
    B, T, Hqk, Hv, D, N = _check_forward_inputs(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens,
                                                cu_seqlens_cpu)
    dev = q.device
    _check_adjoints(do, dfinal_state, B, T, Hv, D, N, dev)
    shapes = ((B, T, Hqk, D), (B, T, Hqk, D), (B, T, Hv, D), (B, T, Hv, D), (B, T, Hv), (Hv,), (Hv, D),
              (N, Hv, D, D))
    out = _grad_buffers(out, shapes, dev)
    with torch.cuda.device(dev):
        rc = lib.kda_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                                 _ptr(initial_state), _ptr(cu_seqlens),
                                 _ptr(cu_seqlens_cpu) if cu_seqlens_cpu is not None else None,
                                 N if cu_seqlens is not None else 0, B, T, Hqk, Hv, D,
                                 float("nan") if scale is None else float(scale), float(lower_bound),
                                 _ptr(do), _ptr(dfinal_state), *[_ptr(t) for t in out], _stream_handle(dev))
    _check(rc)
    return out


def noalloc_status(device=None):
    """Synchronise the current stream of ``device`` and read back the status word of the
    last kda_bwd_noalloc call there; raises KdaError on a device-side error."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(load_library().kda_noalloc_status(_stream_handle(dev)))


class RecurrentKDABackwardWorkspace:
    """Reusable scratch of ``recurrent_kda_backward`` (flashinfer.kda_backward.recurrent_kda_backward,
    parameter ``workspace``): one device buffer of kda_bwd_standalone_workspace_bytes and the
    handle bound to it. The first call that uses it (eager) uploads the launch plan, built from
    the host copy of cu_seqlens, which the workspace keeps; later calls with the same shapes,
    device and stream only launch kernels, so they can be captured into a CUDA graph."""

    def __init__(self, B, T, Hqk, Hv, cu_seqlens_cpu=None, device=None):
        lib = load_library()
        dev = torch.device(device if device is not None else "cuda")
        if dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.dev = dev
        self.cu_cpu = None if cu_seqlens_cpu is None else cu_seqlens_cpu.to(torch.int64).contiguous().cpu()
        n = ctypes.c_size_t(0)
        _check(lib.kda_bwd_standalone_workspace_bytes(
            B, T, Hqk, Hv, _ptr(self.cu_cpu), self.cu_cpu.numel() - 1 if self.cu_cpu is not None else 0,
            ctypes.byref(n)))
        self.buffer = torch.empty(int(n.value), dtype=torch.uint8, device=self.dev)
        self.key = (B, T, Hqk, Hv, None if self.cu_cpu is None else tuple(self.cu_cpu.tolist()))
        self.handle = ctypes.c_void_p(None)

    def status(self):
        _check(load_library().kda_ctx_status(self.handle))

    def __del__(self):
        try:
            if self.handle and self.handle.value:
                load_library().kda_ctx_destroy(self.handle)
                self.handle = ctypes.c_void_p(None)
        except Exception:
            pass


def recurrent_kda_backward(q, k, v, g, beta, A_log, dt_bias, initial_state, do, dfinal_state, cu_seqlens=None,
                           scale=None, lower_bound=-5.0, workspace=None, out=None, *, cu_seqlens_cpu=None):
    """All gradients of the recurrent KDA training recurrence from the forward's inputs, the
    initial state and the adjoints (flashinfer.kda_backward.recurrent_kda_backward: signature,
    description, parameters ``workspace`` and ``out``). Returns (dq, dk, dv, dg, dbeta, dA_log,
    ddt_bias, dinitial_state). ``workspace`` (RecurrentKDABackwardWorkspace) and ``out`` (eight
    tensors in return order) make every buffer caller-owned; with both, a call after the first
    one only launches kernels (CUDA-graph capturable). Packed input: the host copy of
    cu_seqlens comes from ``cu_seqlens_cpu``, else from the workspace, else from a copy of the
    device tensor (which waits for the device)."""
    lib = load_library()
    if cu_seqlens is not None and cu_seqlens_cpu is None:
        if workspace is not None and workspace.cu_cpu is not None:
            cu_seqlens_cpu = workspace.cu_cpu
        else:
            cu_seqlens_cpu = cu_seqlens.cpu()
    B, T, Hqk, Hv, D, N = _check_forward_inputs(q, k, v, g, beta, A_log, dt_bias, initial_state, cu_seqlens,
                                                cu_seqlens_cpu)
    dev = q.device
    _check_adjoints(do, dfinal_state, B, T, Hv, D, N, dev)
    shapes = ((B, T, Hqk, D), (B, T, Hqk, D), (B, T, Hv, D), (B, T, Hv, D), (B, T, Hv), (Hv,), (Hv, D),
              (N, Hv, D, D))
    out = _grad_buffers(out, shapes, dev)
    if workspace is None:
        workspace = RecurrentKDABackwardWorkspace(B, T, Hqk, Hv, cu_seqlens_cpu, device=dev)
    key = (B, T, Hqk, Hv, None if cu_seqlens_cpu is None else tuple(cu_seqlens_cpu.tolist()))
    if workspace.key != key or workspace.dev != dev:
        raise KdaError(4, "the workspace was made for other shapes or another device")
    ws = workspace.buffer
    with torch.cuda.device(dev):
        rc = lib.kda_bwd_standalone(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                                    _ptr(initial_state), _ptr(cu_seqlens),
                                    _ptr(cu_seqlens_cpu) if cu_seqlens_cpu is not None else None,
                                    N if cu_seqlens is not None else 0, B, T, Hqk, Hv, D,
                                    float("nan") if scale is None else float(scale), float(lower_bound),
                                    _ptr(do), _ptr(dfinal_state), *[_ptr(t) for t in out], _ptr(ws), ws.numel(),
                                    ctypes.byref(workspace.handle), _stream_handle(dev))
    _check(rc)
    return out


def _want_gate_params(A_log, dt_bias, Hv, K, use_gate_in_kernel):
    if use_gate_in_kernel or A_log is not None:
        _want(A_log, "A_log", torch.float32, (Hv,))
    if use_gate_in_kernel or dt_bias is not None:
        _want(dt_bias, "dt_bias", torch.float32, (Hv, K))


def kda_decode(q, k, v, g, beta, A_log, dt_bias, state, state_indices=None, scale=None, lower_bound=-5.0,
               out=None, use_gate_in_kernel=False, beta_is_logit=False, *, state_indices_cpu=None):
    """One decode step (T = 1; flashinfer.kda.recurrent_kda, description and parameters q,
    initial_state, ssm_state_indices): updates ``state`` in place and returns o.

    q, k [N, 1, Hqk, 128] and v, g [N, 1, Hv, 128] BF16, beta [N, 1, Hv] BF16,
    A_log [Hv] and dt_bias [Hv, 128] FP32 (None allowed unless
    use_gate_in_kernel); state [num_slots, Hv, 128, 128] BF16 or FP32
    (value-first), read and written at slot state_indices[n] (int32 [N], on the
    device; slot n when None). ``state_indices_cpu``, a trusted CPU copy of
    state_indices, is what the library validates; without it the indices are
    copied to the host, which waits for the device. Gate modes and their
    defaults as on the recurrent_kda page: g is the log decay unless
    ``use_gate_in_kernel``, beta is already sigmoided unless ``beta_is_logit``.
    Argument marshalling only: the step is one launch of the library's decode
    kernel."""
    lib = load_library()
    N, T, Hqk, K = q.shape
    Hv = v.shape[2]
    if T != 1:
        raise ValueError("decode takes one token per sequence (T = 1)")
    _want(q, "q", torch.bfloat16); _want(k, "k", torch.bfloat16, q.shape)
    _want(v, "v", torch.bfloat16); _want(g, "g", torch.bfloat16, v.shape)
    _want(beta, "beta", torch.bfloat16, (N, 1, Hv))
    _want_gate_params(A_log, dt_bias, Hv, K, use_gate_in_kernel)
    if state.dtype == torch.bfloat16:
        sdt = 0
    elif state.dtype == torch.float32:
        sdt = 1
    else:
        raise TypeError("state must be bfloat16 or float32")
    if state.dim() != 4 or tuple(state.shape[1:]) != (Hv, K, K) or not state.is_contiguous():
        raise ValueError(f"state must be contiguous [num_slots, {Hv}, {K}, {K}]")
    if out is None:
        out = torch.empty_like(v)
    _want(out, "out", torch.bfloat16, v.shape)
    idx_dev = idx_host = None
    if state_indices is not None:
        if state_indices.dtype != torch.int32 or state_indices.shape != (N,):
            raise ValueError("state_indices must be int32 [N]")
        idx_dev = state_indices.contiguous()
        if state_indices_cpu is None:
            idx_host = idx_dev.cpu()
        else:
            if (state_indices_cpu.dtype != torch.int32 or state_indices_cpu.shape != (N,)
                    or state_indices_cpu.device.type != "cpu"):
                raise ValueError("state_indices_cpu must be a CPU int32 [N] tensor")
            idx_host = state_indices_cpu.contiguous()
    elif state_indices_cpu is not None:
        raise ValueError("state_indices_cpu given without state_indices")
    dev = q.device
    with torch.cuda.device(dev):
        rc = lib.kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                            _ptr(state), sdt, _ptr(idx_dev) if idx_dev is not None else None,
                            ctypes.c_void_p(idx_host.data_ptr()) if idx_host is not None else None,
                            state.shape[0], N, Hqk, Hv, K, float("nan") if scale is None else float(scale),
                            float(lower_bound), int(bool(use_gate_in_kernel)), int(bool(beta_is_logit)),
                            _ptr(out), _stream_handle(dev))
    _check(rc)
    return out


def kda_prefill(q, k, v, g, beta, A_log, dt_bias, state, cu_seqlens=None, state_indices=None, checkpoints=None,
                checkpoint_cu_starts=None, checkpoint_every_n_tokens=0, scale=None, lower_bound=-5.0, out=None,
                device_status=None, use_gate_in_kernel=False, beta_is_logit=False, *, cu_seqlens_cpu=None,
                state_indices_cpu=None, checkpoint_cu_starts_cpu=None):
    """Inference prefill from a state pool (flashinfer.kda.recurrent_kda, parameters
    initial_state, ssm_state_indices, state_checkpoints, checkpoint_cu_starts and
    checkpoint_every_n_tokens): returns o; the final state of every
    sequence is written back to its slot of ``state`` (BF16 or FP32, [num_slots,
    Hv, 128, 128]); optional BF16 ``checkpoints`` [C, Hv, 128, 128] every
    ``checkpoint_every_n_tokens`` tokens, counted by the int64 device tensor
    ``checkpoint_cu_starts`` [N + 1]. Layouts as for kda_fwd. Gate modes as
    for kda_decode; with the gate precomputed (use_gate_in_kernel False) every
    g must lie in [-5, 0], else bit 1 of ``device_status`` (int32 device
    tensor) is set. Argument marshalling only: one launch of the library's
    forward kernel. The ``*_cpu`` keywords pass trusted CPU mirrors of the
    device index tensors; without them the mirrors are copied from the device
    (a synchronising copy)."""
    lib = load_library()
    B, T, Hqk, K = q.shape
    Hv = v.shape[2]
    _want(q, "q", torch.bfloat16); _want(k, "k", torch.bfloat16, q.shape)
    _want(v, "v", torch.bfloat16); _want(g, "g", torch.bfloat16, v.shape)
    _want(beta, "beta", torch.bfloat16, (B, T, Hv))
    _want_gate_params(A_log, dt_bias, Hv, K, use_gate_in_kernel)
    sdt = {torch.bfloat16: 0, torch.float32: 1}.get(state.dtype)
    if sdt is None:
        raise TypeError("state must be bfloat16 or float32")
    if state.dim() != 4 or tuple(state.shape[1:]) != (Hv, K, K) or not state.is_contiguous():
        raise ValueError(f"state must be contiguous [num_slots, {Hv}, {K}, {K}]")
    if out is None:
        out = torch.empty_like(v)
    _want(out, "out", torch.bfloat16, v.shape)
    def mirror(t, given, name):
        if t is None:
            if given is not None:
                raise ValueError(f"{name}_cpu given without {name}")
            return None
        if given is None:
            return t.cpu()
        if given.device.type != "cpu" or given.shape != t.shape or given.dtype != t.dtype:
            raise ValueError(f"{name}_cpu must be a CPU tensor of the shape and dtype of {name}")
        return given
    cu_host = mirror(cu_seqlens, cu_seqlens_cpu, "cu_seqlens")
    N = (cu_host.numel() - 1) if cu_host is not None else B
    idx_host = mirror(state_indices, state_indices_cpu, "state_indices")
    cks_host = mirror(checkpoint_cu_starts, checkpoint_cu_starts_cpu, "checkpoint_cu_starts")
    n_ck = 0
    if checkpoints is not None:
        _want(checkpoints, "checkpoints", torch.bfloat16)
        n_ck = checkpoints.shape[0]
    def host(t):
        return ctypes.c_void_p(t.data_ptr()) if t is not None else None
    dev = q.device
    with torch.cuda.device(dev):
        rc = lib.kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                             _ptr(cu_seqlens), host(cu_host), N, B, T, Hqk, Hv, K,
                             float("nan") if scale is None else float(scale), float(lower_bound),
                             int(bool(use_gate_in_kernel)), int(bool(beta_is_logit)), _ptr(state), sdt,
                             _ptr(state_indices), host(idx_host), state.shape[0], _ptr(out), _ptr(checkpoints), n_ck,
                             _ptr(checkpoint_cu_starts), host(cks_host), int(checkpoint_every_n_tokens),
                             _ptr(device_status), _stream_handle(dev))
    _check(rc)
    return out


def selftest_device_timeout(device=None) -> int:
    """Run the device-side timeout self-test on the current stream of `device`:
    one CTA waits on an mbarrier nothing arrives at and must give up after
    about 1 ms. Returns the status code (KDA_ERR_DEVICE_TIMEOUT is the expected
    outcome) without raising."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib.kda_selftest_device_timeout(_stream_handle(dev)))


recurrent_kda_training_forward = kda_fwd


class HostStep:
    """Training steps (flashinfer.kda_training forward and backward) from and to
    host memory through kda_step_host: owns one
    device arena (kda_step_arena_bytes) and the context created in it. Each call
    enqueues the input copies on ``h2d_stream``, the forward and backward on
    ``stream`` and the output copies on ``d2h_stream`` (each defaults to a new
    stream of its own; pass the same streams to two HostStep objects and use
    them in turn to overlap one step's copies with the other's kernels) and
    returns; ``synchronize()`` waits for the output copies. Host tensors should
    be pinned (``pin_memory()``)."""

    IN_NAMES = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state", "do", "dfinal_state")

    def __init__(self, B, T, Hqk, Hv, cu_seqlens_cpu=None, device=None, stream=None, h2d_stream=None,
                 d2h_stream=None):
        lib = load_library()
        self.dev = torch.device(device if device is not None else "cuda")
        self.B, self.T, self.Hqk, self.Hv = B, T, Hqk, Hv
        self.cu = None if cu_seqlens_cpu is None else cu_seqlens_cpu.to(torch.int64).contiguous()
        self.N = B if self.cu is None else self.cu.numel() - 1
        n = ctypes.c_size_t(0)
        _check(lib.kda_step_arena_bytes(B, T, Hqk, Hv, _ptr(self.cu), self.N if self.cu is not None else 0,
                                        ctypes.byref(n)))
        self.arena = torch.empty(int(n.value), dtype=torch.uint8, device=self.dev)
        self.stream = stream if stream is not None else torch.cuda.Stream(self.dev)
        self.h2d_stream = h2d_stream if h2d_stream is not None else torch.cuda.Stream(self.dev)
        self.d2h_stream = d2h_stream if d2h_stream is not None else torch.cuda.Stream(self.dev)
        self.handle = ctypes.c_void_p(None)

    def shapes(self):
        B, T, Hqk, Hv, N, D = self.B, self.T, self.Hqk, self.Hv, self.N, DIM
        bf, f32 = torch.bfloat16, torch.float32
        ins = {"q": ((B, T, Hqk, D), bf), "k": ((B, T, Hqk, D), bf), "v": ((B, T, Hv, D), bf),
               "g": ((B, T, Hv, D), bf), "beta": ((B, T, Hv), bf), "A_log": ((Hv,), f32),
               "dt_bias": ((Hv, D), f32), "initial_state": ((N, Hv, D, D), f32), "do": ((B, T, Hv, D), bf),
               "dfinal_state": ((N, Hv, D, D), f32)}
        outs = (("o", (B, T, Hv, D), bf), ("final_state", (N, Hv, D, D), f32), ("dq", (B, T, Hqk, D), bf),
                ("dk", (B, T, Hqk, D), bf), ("dv", (B, T, Hv, D), bf), ("dg", (B, T, Hv, D), bf),
                ("dbeta", (B, T, Hv), bf), ("dA_log", (Hv,), f32), ("ddt_bias", (Hv, D), f32),
                ("dinitial_state", (N, Hv, D, D), f32))
        return ins, outs

    def empty_outputs(self, pin_memory=True):
        """Host output buffers in the order (o, final_state, dq, dk, dv, dg, dbeta,
        dA_log, ddt_bias, dinitial_state)."""
        _, outs = self.shapes()
        return tuple(torch.empty(shp, dtype=dt, pin_memory=pin_memory) for _, shp, dt in outs)

    def __call__(self, q, k, v, g, beta, A_log, dt_bias, initial_state, do, dfinal_state, out,
                 scale=None, lower_bound=-5.0):
        lib = load_library()
        ins, outs = self.shapes()
        args = dict(zip(self.IN_NAMES, (q, k, v, g, beta, A_log, dt_bias, initial_state, do, dfinal_state)))
        for name, t in args.items():
            _want(t, name, ins[name][1], ins[name][0])
            if t.device.type != "cpu":
                raise ValueError(f"{name} must be a host tensor")
        if len(out) != len(outs):
            raise ValueError("out must hold ten host tensors")
        for t, (name, shp, dt) in zip(out, outs):
            _want(t, name, dt, shp)
            if t.device.type != "cpu":
                raise ValueError(f"{name} must be a host tensor")
        with torch.cuda.device(self.dev):
            rc = lib.kda_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                                   _ptr(initial_state), _ptr(self.cu), self.N if self.cu is not None else 0,
                                   self.B, self.T, self.Hqk, self.Hv, DIM,
                                   float("nan") if scale is None else float(scale), float(lower_bound),
                                   _ptr(do), _ptr(dfinal_state), *[_ptr(t) for t in out], _ptr(self.arena),
                                   self.arena.numel(), ctypes.byref(self.handle),
                                   ctypes.c_void_p(self.stream.cuda_stream),
                                   ctypes.c_void_p(self.h2d_stream.cuda_stream),
                                   ctypes.c_void_p(self.d2h_stream.cuda_stream))
        _check(rc)
        return out

    def synchronize(self):
        self.d2h_stream.synchronize()

    def status(self):
        _check(load_library().kda_ctx_status(self.handle))

    def __del__(self):
        try:
            if self.handle and self.handle.value:
                load_library().kda_ctx_destroy(self.handle)
                self.handle = ctypes.c_void_p(None)
        except Exception:
            pass


def recurrent_kda_training_backward(context, do, dfinal_state, out=None):
    return kda_bwd(context, do, dfinal_state, out=out)
