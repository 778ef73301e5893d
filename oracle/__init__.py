"""FP64 CPU oracle of the recurrent KDA training recurrence (forward and backward).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. It shares no code with the CUDA path in ``linear_attention_gated_gb300``.

The arithmetic lives in ``kda_oracle.c`` (plain C, FP64, OpenMP over
independent (sequence, head) units); this module only marshals numpy arrays.
What the oracle computes, and the passages it follows, is stated in the header
of ``kda_oracle.c``:

* "flashinfer.kda_backward.recurrent_kda_backward", description: L2 norm of q
  and k with epsilon 1e-6, decay exp(lower_bound * sigmoid(exp(A_log) * (g +
  dt_bias))), sigmoid beta, adjoints ``do`` and ``dfinal_state``, gradient order.
* "flashinfer.kda_training.recurrent_kda_training_forward", parameters: shapes,
  value-first [N, Hv, V, K] state, Hv a multiple of Hqk.
* "flashinfer.kda_training", module description: fixed [B, T, H, 128] layout or
  packed B = 1 with int64 cu_seqlens; every sequence non-empty.

Inputs are numpy arrays holding the exact values the GPU path receives (BF16
or FP32 values upcast to float64). Fixed layout [B, T, H, D] is handled as B
packed sequences of length T (cu = 0, T, 2T, ...), which is the documented
meaning of a fixed-layout batch row.

Pins (tests/test_oracle_pins.py): finite differences of the forward for all
eight gradients, closed forms at special inputs (beta = 0, beta = 1 with q = k,
known gate values, a hand-worked two-token example), the chunked restatement
equal to the sequential form, and structural invariants (causality, value-first
orientation, GQA = repeated heads, packed = fixed). Every returned tensor is
covered by at least one pin.
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into libkda_oracle.so with gcc (FP64, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            D = ctypes.c_double
            lib.kda_oracle_forward.argtypes = [I, P, I, I, I, I] + [P] * 8 + [D, D, P, P, P]
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_forward_modes.argtypes = ([I, P, I, I, I, I] + [P] * 8 +
                                                     [D, D, ctypes.c_int, ctypes.c_int, P, P])
            lib.kda_oracle_forward_modes.restype = ctypes.c_int
            lib.kda_oracle_forward_chunked.argtypes = [I, P, I, I, I, I] + [P] * 8 + [D, D, I, P, P]
            lib.kda_oracle_forward_chunked.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = ([I, P, I, I, I, I] + [P] * 10 + [D, D, P] + [P] * 8)
            lib.kda_oracle_backward.restype = ctypes.c_int
            lib.kda_oracle_num_threads.argtypes = []
            lib.kda_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (OMP_NUM_THREADS, else all cores)."""
    return int(_load().kda_oracle_num_threads())


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


class _Problem:
    """Flatten fixed / packed layouts to the packed token axis the C code uses."""

    def __init__(self, q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens, scale, lower_bound, heads):
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        if q.ndim != 4 or v.ndim != 4 or beta.ndim != 3:
            raise ValueError("q/k/v/g must be [B,T,H,D] and beta [B,T,H]")
        B, T, hqk, dk = q.shape
        hv, dv = v.shape[2], v.shape[3]
        if k.shape != q.shape or g.shape != (B, T, hv, dk) or beta.shape != (B, T, hv):
            raise ValueError("inconsistent shapes")
        if hv % hqk:
            raise ValueError("Hv must be a multiple of Hqk")
        if cu_seqlens is None:
            cu = np.arange(0, (B + 1) * T, T, dtype=np.int64)
        else:
            if B != 1:
                raise ValueError("packed layout needs a batch dimension of one")
            cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
            if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) <= 0):
                raise ValueError("cu_seqlens must start at 0, end at T, with non-empty sequences")
        self.B, self.T = B, T
        self.nseq = len(cu) - 1
        self.cu = cu
        self.hqk, self.hv, self.dk, self.dv = hqk, hv, dk, dv
        self.q = q.reshape(B * T, hqk, dk)
        self.k = k.reshape(B * T, hqk, dk)
        self.v = v.reshape(B * T, hv, dv)
        self.g = g.reshape(B * T, hv, dk)
        self.beta = beta.reshape(B * T, hv)
        self.A_log = _f64(A_log).reshape(hv)
        self.dt_bias = _f64(dt_bias).reshape(hv, dk)
        self.h0 = _f64(h0).reshape(self.nseq, hv, dv, dk)
        self.scale = 1.0 / math.sqrt(dk) if scale is None else float(scale)
        self.lb = float(lower_bound)
        if heads is None:
            self.mask = None
        else:
            m = np.zeros(hqk, dtype=np.uint8)
            m[np.asarray(list(heads), dtype=np.int64)] = 1
            self.mask = m

    def common(self):
        return [self.nseq, _ptr(self.cu), self.hqk, self.hv, self.dk, self.dv,
                _ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(self.g), _ptr(self.beta),
                _ptr(self.A_log), _ptr(self.dt_bias), _ptr(self.h0)]

    def token_shape(self, h, d):
        return (self.B, self.T, h, d)


def _nan(shape):
    return np.full(shape, np.nan, dtype=np.float64)


def forward(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens=None, scale=None,
            lower_bound=-5.0, heads=None, log_space_g=False, presigmoid_beta=False):
    """Sequential FP64 forward. Returns (o [B,T,Hv,DV], final_state [N,Hv,DV,DK]).

    ``heads``: optional iterable of query/key heads to compute (with all their
    value heads); entries of other heads are NaN.

    Gate modes of "flashinfer.kda.recurrent_kda" (parameters g and beta):
    ``log_space_g`` takes g as the per-key log decay (decay exp(g); A_log,
    dt_bias and lower_bound unused); ``presigmoid_beta`` takes beta as the
    learning rate itself rather than its logit.
    """
    p = _Problem(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens, scale, lower_bound, heads)
    o = _nan((p.B * p.T, p.hv, p.dv))
    hT = _nan((p.nseq, p.hv, p.dv, p.dk))
    if log_space_g or presigmoid_beta:
        if heads is not None:
            raise ValueError("oracle forward: head selection is not offered with the gate modes")
        rc = _load().kda_oracle_forward_modes(*p.common(), p.scale, p.lb, int(bool(log_space_g)),
                                              int(bool(presigmoid_beta)), _ptr(o), _ptr(hT))
    else:
        rc = _load().kda_oracle_forward(*p.common(), p.scale, p.lb, _ptr(p.mask), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle forward rejected its arguments")
    return o.reshape(p.token_shape(p.hv, p.dv)), hT


def forward_chunked(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens=None, scale=None,
                    lower_bound=-5.0, chunk=16):
    """Chunked (WY / UT-transform) restatement of the same forward, FP64."""
    p = _Problem(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens, scale, lower_bound, None)
    o = _nan((p.B * p.T, p.hv, p.dv))
    hT = _nan((p.nseq, p.hv, p.dv, p.dk))
    rc = _load().kda_oracle_forward_chunked(*p.common(), p.scale, p.lb, int(chunk), _ptr(o), _ptr(hT))
    if rc:
        raise ValueError("oracle chunked forward rejected its arguments")
    return o.reshape(p.token_shape(p.hv, p.dv)), hT


def backward(q, k, v, g, beta, A_log, dt_bias, h0, do, dfinal_state, cu_seqlens=None,
             scale=None, lower_bound=-5.0, heads=None):
    """FP64 backward. Returns (dq, dk, dv, dg, dbeta, dA_log, ddt_bias, dinitial_state),
    the order of "flashinfer.kda_backward.recurrent_kda_backward"."""
    p = _Problem(q, k, v, g, beta, A_log, dt_bias, h0, cu_seqlens, scale, lower_bound, heads)
    do_ = _f64(do).reshape(p.B * p.T, p.hv, p.dv)
    dhT = _f64(dfinal_state).reshape(p.nseq, p.hv, p.dv, p.dk)
    dq = _nan((p.B * p.T, p.hqk, p.dk))
    dk = _nan((p.B * p.T, p.hqk, p.dk))
    dv = _nan((p.B * p.T, p.hv, p.dv))
    dg = _nan((p.B * p.T, p.hv, p.dk))
    dbeta = _nan((p.B * p.T, p.hv))
    dA_log = _nan((p.hv,))
    ddt_bias = _nan((p.hv, p.dk))
    dh0 = _nan((p.nseq, p.hv, p.dv, p.dk))
    rc = _load().kda_oracle_backward(*p.common(), _ptr(do_), _ptr(dhT), p.scale, p.lb,
                                     _ptr(p.mask), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg),
                                     _ptr(dbeta), _ptr(dA_log), _ptr(ddt_bias), _ptr(dh0))
    if rc:
        raise ValueError("oracle backward rejected its arguments")
    return (dq.reshape(p.token_shape(p.hqk, p.dk)), dk.reshape(p.token_shape(p.hqk, p.dk)),
            dv.reshape(p.token_shape(p.hv, p.dv)), dg.reshape(p.token_shape(p.hv, p.dk)),
            dbeta.reshape(p.B, p.T, p.hv), dA_log, ddt_bias, dh0)
