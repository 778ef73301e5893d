"""C-ABI checks that need no GPU: the library loads, exports every function
include/kda.h declares, sizes workspaces, and rejects bad arguments on the host
before any CUDA call (pointers below are fake addresses that are never read)."""

import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from linear_attention_gated_gb300 import build as b
    b.build()
    from linear_attention_gated_gb300 import kda
    return kda.load_library()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(kda_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for name in names:
        assert hasattr(lib, name), name
    from linear_attention_gated_gb300 import kda
    assert set(kda.EXPORTED) <= set(names)


def test_status_strings(lib):
    for st in range(8):
        assert lib.kda_status_string(st)
    assert lib.kda_last_error_message() == b""


def test_tiling_constants(lib):
    assert lib.kda_chunk_tokens() == 16
    assert lib.kda_checkpoint_tokens() % lib.kda_chunk_tokens() == 0


def ws_bytes(lib, B, T, hqk, hv, cu=None):
    out = ctypes.c_size_t()
    if cu is None:
        rc = lib.kda_ctx_workspace_bytes(B, T, hqk, hv, None, 0, ctypes.byref(out))
    else:
        arr = (ctypes.c_int64 * len(cu))(*cu)
        rc = lib.kda_ctx_workspace_bytes(B, T, hqk, hv, ctypes.cast(arr, ctypes.c_void_p),
                                         len(cu) - 1, ctypes.byref(out))
    return rc, out.value


def test_workspace_bytes_grows_with_problem(lib):
    rc, a = ws_bytes(lib, 1, 64, 2, 2)
    assert rc == 0 and a > 0 and a % 256 == 0
    rc, b = ws_bytes(lib, 2, 1024, 32, 32)
    assert rc == 0 and b > a
    # checkpoint storage: one 64 KiB state per (interval, head)
    ck = lib.kda_checkpoint_tokens()
    rc, c = ws_bytes(lib, 1, 8192, 96, 96, list(range(0, 8193, 1024)))
    assert rc == 0 and c >= 8 * math.ceil(1024 / ck) * 96 * 65536
    # GQA adds per-value-head scratch for the group sums
    rc, d1 = ws_bytes(lib, 4, 2048, 32, 32)
    rc, d2 = ws_bytes(lib, 4, 2048, 16, 32)
    assert d2 > d1


@pytest.mark.parametrize("args,status", [
    ((0, 64, 2, 2, None), 1),           # B = 0
    ((1, 0, 2, 2, None), 1),            # T = 0 (no tokens)
    ((1, 64, 2, 2, [0]), 1),            # packed with no sequences
    ((1, 64, 0, 2, None), 1),           # no query/key heads
    ((1, 64, 3, 4, None), 1),           # Hv not a multiple of Hqk
    ((2, 64, 2, 2, [0, 32, 64]), 1),    # packed with B != 1
    ((1, 64, 2, 2, [0, 32, 32, 64]), 1),  # empty sequence
    ((1, 64, 2, 2, [1, 32, 64]), 1),    # does not start at 0
    ((1, 64, 2, 2, [0, 32, 60]), 1),    # does not end at T
])
def test_workspace_bytes_rejects(lib, args, status):
    rc, _ = ws_bytes(lib, *args)
    assert rc == status


class FakeCall:
    """kda_fwd with fake, well-separated, aligned device addresses."""

    def __init__(self, lib, B=1, T=64, hqk=2, hv=2, cu=None):
        self.lib = lib
        self.B, self.T, self.hqk, self.hv, self.cu = B, T, hqk, hv, cu
        base = 1 << 40
        names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0", "cu_dev", "o", "hT", "ws"]
        self.addr = {n: base + i * (1 << 34) for i, n in enumerate(names)}
        rc, self.ws_bytes = ws_bytes(lib, B, T, hqk, hv, cu)
        assert rc == 0

    def __call__(self, head_dim=128, scale=float("nan"), lb=-5.0, ws_bytes=None, **override):
        a = dict(self.addr)
        a.update(override)
        P = ctypes.c_void_p
        cu_host = None
        nseq = 0
        if self.cu is not None:
            self._cu_arr = (ctypes.c_int64 * len(self.cu))(*self.cu)
            cu_host = ctypes.cast(self._cu_arr, P)
            nseq = len(self.cu) - 1
        else:
            a["cu_dev"] = None
        ctx = P(None)
        rc = self.lib.kda_fwd(*[P(a[n]) if a[n] is not None else None for n in
                                ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0"]],
                              P(a["cu_dev"]) if a["cu_dev"] is not None else None, cu_host, nseq,
                              self.B, self.T, self.hqk, self.hv, head_dim, scale, lb,
                              P(a["o"]) if a["o"] else None, P(a["hT"]), P(a["ws"]),
                              self.ws_bytes if ws_bytes is None else ws_bytes,
                              ctypes.byref(ctx), None)
        return rc, self.lib.kda_last_error_message().decode()


def test_fwd_rejects_unsupported_head_dim(lib):
    rc, msg = FakeCall(lib)(head_dim=64)
    assert rc == 2 and "128" in msg


def test_fwd_rejects_wrong_scale_and_lower_bound(lib):
    call = FakeCall(lib)
    assert call(scale=0.5)[0] == 2
    assert call(lb=-4.0)[0] == 2


def test_fwd_rejects_null_pointer(lib):
    rc, msg = FakeCall(lib)(o=None)
    assert rc == 1 and "NULL" in msg


def test_fwd_rejects_small_workspace(lib):
    call = FakeCall(lib)
    assert call(ws_bytes=call.ws_bytes - 256)[0] == 7


def test_fwd_rejects_unaligned_workspace_and_tensors(lib):
    call = FakeCall(lib)
    assert call(ws=call.addr["ws"] + 16)[0] == 1
    assert call(q=call.addr["q"] + 2)[0] == 1


def test_fwd_rejects_aliasing(lib):
    call = FakeCall(lib)
    rc, msg = call(o=call.addr["v"] + 1024)
    assert rc == 3 and "o" in msg
    rc, msg = call(hT=call.addr["ws"] + 4096)
    assert rc == 3
    rc, _ = call(ws=call.addr["h0"])
    assert rc == 3


def test_fwd_packed_rejects_missing_device_offsets(lib):
    call = FakeCall(lib, cu=[0, 10, 64])
    rc, msg = call(cu_dev=None)
    assert rc == 1


def test_fwd_reaches_device_check_when_arguments_are_valid(lib):
    """With valid arguments the only remaining failure here (no GPU) is the device query."""
    rc, msg = FakeCall(lib, cu=[0, 10, 64])()
    assert rc in (2, 5), msg


def test_bwd_rejects_null_context(lib):
    P = ctypes.c_void_p
    rc = lib.kda_bwd(None, *[P(1 << 40)] * 10, None)
    assert rc == 1


def test_ctx_destroy_accepts_null(lib):
    lib.kda_ctx_destroy(None)


@pytest.mark.parametrize("args", [
    (1 << 41, 64, 2, 2, None),          # more than 2^40 tokens
    (1, 1 << 36, 2, 1 << 8, None),      # more than 2^40 token-heads
    (1, 64, 1 << 12, 1 << 21, None),    # more than 2^20 value heads
    ((1 << 62), (1 << 62), 2, 2, None),  # B * T would overflow 64 bits
])
def test_workspace_bytes_rejects_absurd_sizes(lib, args):
    """Sizes that would overflow byte counts or build huge host tables are refused up front
    (no exception crosses the C ABI, no crash)."""
    rc, _ = ws_bytes(lib, *args)
    assert rc == 2
    assert "too large" in lib.kda_last_error_message().decode()


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_is_plain_c_and_cxx(tmp_path, lang, std):
    """include/kda.h compiles on its own as strict C99 and as C++11 (no torch or CUDA headers
    needed by a caller), with every warning an error."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / "use_kda.c"
    src.write_text('#include "kda.h"\n'
                   "int main(void) { size_t b = 0; kda_status s = kda_ctx_workspace_bytes(1, 64, 2, 2, 0, 0, &b);\n"
                   "  return (int)s + (int)(kda_status_string(s) == 0); }\n")
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror"] + (["-pedantic"] if lang == "c" else [])
                       + ["-I", inc, "-fsyntax-only", "-x", lang, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_standalone_workspace_bytes_covers_context(lib):
    out = ctypes.c_size_t()
    assert lib.kda_bwd_standalone_workspace_bytes(2, 1024, 32, 32, None, 0, ctypes.byref(out)) == 0
    rc, ctx = ws_bytes(lib, 2, 1024, 32, 32)
    # the context workspace plus room for o (BF16 [2, 1024, 32, 128]) and the final state
    assert out.value >= ctx + 2 * 2 * 1024 * 32 * 128 + 4 * 2 * 32 * 128 * 128
    assert out.value % 256 == 0
    assert lib.kda_bwd_standalone_workspace_bytes(1, 64, 3, 4, None, 0, ctypes.byref(out)) == 1


def _standalone(lib, ws_bytes_delta=0, **override):
    """kda_bwd_standalone with fake, well-separated, aligned device addresses."""
    P = ctypes.c_void_p
    base = 1 << 40
    names = ["q", "k", "v", "g", "beta", "A_log", "dt_bias", "h0", "do", "dhT", "dq", "dk", "dv", "dg",
             "dbeta", "dA_log", "ddt_bias", "dh0", "ws"]
    a = {n: base + i * (1 << 34) for i, n in enumerate(names)}
    a.update(override)
    need = ctypes.c_size_t()
    assert lib.kda_bwd_standalone_workspace_bytes(1, 64, 2, 2, None, 0, ctypes.byref(need)) == 0
    handle = P(None)
    rc = lib.kda_bwd_standalone(*[P(a[n]) for n in names[:8]], None, None, 0, 1, 64, 2, 2, 128,
                                float("nan"), -5.0, *[P(a[n]) for n in names[8:18]], P(a["ws"]),
                                need.value + ws_bytes_delta, ctypes.byref(handle), None)
    return rc, lib.kda_last_error_message().decode()


def test_standalone_rejects_small_workspace(lib):
    rc, msg = _standalone(lib, ws_bytes_delta=-256)
    assert rc == 7 and "workspace" in msg


def test_standalone_rejects_gradient_or_adjoint_in_workspace(lib):
    ws = (1 << 40) + 18 * (1 << 34)
    rc, msg = _standalone(lib, dk=ws + 4096)
    assert rc == 3 and "dk" in msg
    rc, msg = _standalone(lib, do=ws)
    assert rc == 3 and "do" in msg


def test_standalone_reaches_device_check_when_arguments_are_valid(lib):
    rc, msg = _standalone(lib)
    assert rc in (2, 5), msg
