"""Host-side tests of the C ABI (include/gdn.h): no GPU needed.

The library must load, export every function the header declares, and reject
bad arguments on the host before touching the device (the pointers passed
here are never dereferenced: each call fails its checks first).
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_mixer_delta_gb300 import build as b
    import gated_deltanet_mixer_delta_gb300 as gdn
    b.build()
    return gdn.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ["gdn_prefill", "gdn_prefill_varlen", "gdn_decode_step", "gdn_state_layout",
              "gdn_prefill_workspace_size", "gdn_workspace_status", "gdn_status_string",
              "gdn_gated_rmsnorm", "gdn_decode_step_gated"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from gated_deltanet_mixer_delta_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(gdn_\w+)", out))
    for n in header_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_state_layout(lib):
    import gated_deltanet_mixer_delta_gb300 as gdn
    lay = gdn.state_layout(256, 32, 128, 128)
    assert lay["shape"] == (256, 32, 128, 128)
    assert lay["stride"] == (32 * 128 * 128, 128 * 128, 128, 1)
    assert lay["bytes"] == 256 * 32 * 128 * 128 * 4 == 512 * 2 ** 20
    assert lay["bytes_per_head"] == 65536
    assert lay["alignment"] == 16
    with pytest.raises(gdn.GdnError):
        gdn.state_layout(1, 0, 128, 128)


def test_state_bytes_per_token_match_the_pages(lib):
    """tests/golden/state_bytes_per_token.txt: the pages give the float32 per-token
    state size (num_v_heads x 128 x 128) of each model: 1, 2 or 3 MiB per block."""
    import gated_deltanet_mixer_delta_gb300 as gdn
    rows = [l.split() for l in open(os.path.join(GOLDEN, "state_bytes_per_token.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 6
    for model, hv, dk, dv, mib in rows:
        lay = gdn.state_layout(1, int(hv), int(dk), int(dv))
        assert lay["bytes"] == int(mib) * 2 ** 20, model


def test_workspace_size(lib):
    import gated_deltanet_mixer_delta_gb300 as gdn
    a = gdn.workspace_size(4096, 1, 32, 128, 128)
    b = gdn.workspace_size(8192, 1, 32, 128, 128)
    assert 0 < a < b
    assert gdn.workspace_size(0, 0, 32, 128, 128) > 0
    assert gdn.workspace_size(10, 1, 32, 96, 96) == 0
    assert gdn.workspace_size(-1, 1, 32, 128, 128) == 0


def test_workspace_size_for_each_path(lib):
    """With a dtype the size is exactly what that path needs: 58 KiB records of operand
    images for 128 x 128 bf16 heads (tensor cores), fp32 records of 64 (Dk + Dv + 64) + 320
    floats otherwise; without one, the larger of the two."""
    import gated_deltanet_mixer_delta_gb300 as gdn
    T, N, HV = 4096, 1, 32
    bf = gdn.workspace_size(T, N, HV, 128, 128, dtype=torch.bfloat16)
    f32 = gdn.workspace_size(T, N, HV, 128, 128, dtype=torch.float32)
    both = gdn.workspace_size(T, N, HV, 128, 128)
    chunks = T // 64 + N                          # the packed bound on chunks
    assert f32 - bf == chunks * HV * (4 * (64 * (128 + 128 + 64) + 320) - 59392)
    assert both == max(bf, f32) == f32
    # 32 x 32 heads take the CUDA-core path whatever the dtype
    assert gdn.workspace_size(T, N, HV, 32, 32, dtype=torch.bfloat16) == \
        gdn.workspace_size(T, N, HV, 32, 32, dtype=torch.float32)
    assert lib.gdn_prefill_workspace_size_for(10, 1, 32, 128, 128, 7) == 0


def test_prefill_checks_the_workspace_of_its_own_path_on_host(lib):
    """The host check asks for the dtype's exact size: one byte less is rejected, and an
    fp32 call does not accept the smaller bf16 size."""
    import gated_deltanet_mixer_delta_gb300 as gdn
    bf = gdn.workspace_size(64, 1, 4, 128, 128, dtype=torch.bfloat16)
    assert _prefill(lib, wsb=bf - 1) == -4
    assert _prefill(lib, wsb=bf, dtype=1) == -4


def test_status_strings(lib):
    for s in [0, -1, -2, -3, -4, -5, -6, -7, 12345]:
        assert lib.gdn_status_string(s)
    assert lib.gdn_abi_version() >= 100


P = 0x10000          # fake, 16-byte aligned device address: never dereferenced
BIG = 1 << 40


def _prefill(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, b=P, s0=None, out=P, fin=P, st=None, B=1, T=64, HK=2, HV=4,
             Dk=128, Dv=128, dtype=0, scale=0.0, l2=1, ws=P, wsb=BIG, stream=None)
    a.update(kw)
    return lib.gdn_prefill(a["q"], a["k"], a["v"], a["g"], a["b"], a["s0"], a["out"], a["fin"],
                           a["st"], a["B"], a["T"], a["HK"], a["HV"], a["Dk"], a["Dv"],
                           a["dtype"], a["scale"], a["l2"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(HV=3), -1), (dict(HK=0), -1), (dict(B=-1), -1), (dict(T=-5), -1),
    (dict(Dk=96, Dv=96), -2), (dict(Dk=128, Dv=64), -2), (dict(dtype=7), -2),
    (dict(q=P + 4), -3), (dict(out=P + 8), -3), (dict(st=P + 2), -3),
    (dict(ws=None), -4), (dict(wsb=100), -4), (dict(ws=P + 16), -3),
    (dict(q=None), -1), (dict(fin=None), -1), (dict(scale=float("nan")), -1),
    # (sequence, value head, value slice) chains are numbered in 32 bits
    (dict(B=40000, T=1, HK=16000, HV=16000), -2),
])
def test_prefill_rejects_bad_arguments_on_host(lib, kw, code):
    assert _prefill(lib, **kw) == code


def _noalloc(lib, **kw):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.gdn_prefill_noalloc
    fn.restype = i
    fn.argtypes = [vp] * 9 + [i] * 7 + [f, i, vp]
    a = dict(q=P, k=P, v=P, g=P, b=P, s0=None, out=P, fin=P, st=None, B=1, T=64, HK=2, HV=4,
             Dk=128, Dv=128, dtype=0, scale=0.0, l2=1, stream=None)
    a.update(kw)
    return fn(a["q"], a["k"], a["v"], a["g"], a["b"], a["s0"], a["out"], a["fin"], a["st"],
              a["B"], a["T"], a["HK"], a["HV"], a["Dk"], a["Dv"], a["dtype"], a["scale"],
              a["l2"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(HV=3), -1), (dict(B=-1), -1), (dict(Dk=96, Dv=96), -2), (dict(dtype=5), -2),
    (dict(q=P + 4), -3), (dict(st=P + 8), -3), (dict(fin=None), -1),
    # the fixed scratch (64 MiB) holds 1129 records of 58 KiB after its header and chunk
    # table: 32 value heads x 35 chunks of 64 tokens fit, x 36 do not
    (dict(T=128 * 64, HK=16, HV=32), -4), (dict(B=4, T=36 * 64, HK=16, HV=32), -4),
    (dict(T=35 * 64 + 1, HK=16, HV=32), -4), (dict(B=40000, T=1, HK=16000, HV=16000), -2),
])
def test_noalloc_rejects_bad_arguments_and_oversized_shapes_on_host(lib, kw, code):
    """gdn_prefill_noalloc checks its arguments and its scratch limit before it looks up
    the scratch array or enqueues anything."""
    assert _noalloc(lib, **kw) == code


def test_noalloc_scratch_limit_boundary_on_host(lib):
    """B = 1, T = 2240 at 32 value heads (35 chunks, 1120 records) is the largest
    128 x 128 bf16 prompt the scratch takes: it passes the size check and only then
    needs a device (here none: GDN_ERR_CUDA); one token more is rejected with
    GDN_ERR_WORKSPACE before any device call."""
    assert _noalloc(lib, T=2240, HK=16, HV=32) not in (-4,)
    assert _noalloc(lib, T=2241, HK=16, HV=32) == -4


def test_noalloc_status_reader_arguments_on_host(lib):
    """gdn_prefill_noalloc_status rejects a null result pointer; without a device the
    copy itself fails with GDN_ERR_CUDA rather than returning a stale value."""
    fn = lib.gdn_prefill_noalloc_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert fn(None, None) == -1
    st = ctypes.c_int(12345)
    rc = fn(None, ctypes.byref(st))
    import torch
    if not torch.cuda.is_available():
        assert rc == -5 and st.value == 12345


def test_varlen_rejects_bad_arguments_on_host(lib):
    f = lib.gdn_prefill_varlen
    args = [P, P, P, P, P, None, P, P, None, P, 2, 100, 2, 4, 128, 128, 0, 0.0, 1, P, BIG, None]
    a = list(args); a[9] = None
    assert f(*a) == -1                           # cu_seqlens required
    a = list(args); a[10] = -1
    assert f(*a) == -1
    a = list(args); a[9] = P + 4
    assert f(*a) == -3
    a = list(args); a[20] = 10
    assert f(*a) == -4


def _decode(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, b=P, s=P, out=P, B=4, HK=2, HV=4, Dk=128, Dv=128, dtype=0,
             scale=0.0, l2=1, stream=None)
    a.update(kw)
    return lib.gdn_decode_step(a["q"], a["k"], a["v"], a["g"], a["b"], a["s"], a["out"], a["B"],
                               a["HK"], a["HV"], a["Dk"], a["Dv"], a["dtype"], a["scale"],
                               a["l2"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(HV=5), -1), (dict(B=-2), -1), (dict(Dk=48, Dv=48), -2), (dict(dtype=3), -2),
    (dict(s=None), -1), (dict(s=P + 4), -3), (dict(v=P + 2), -3), (dict(B=0), 0),
])
def test_decode_rejects_bad_arguments_on_host(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_selftest_wait_timeout_rejects_bad_arguments(lib):
    # host-side checks only: nothing is launched for these
    import ctypes
    f = lib.gdn_selftest_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
    assert f(None, 1000, None) == -1                      # GDN_ERR_INVALID_ARG
    assert f(ctypes.c_void_p(0x10000), 0, None) == -1     # zero limit
    assert f(ctypes.c_void_p(0x10000), 3_000_000_000, None) == -1   # above 2 s
    assert f(ctypes.c_void_p(0x10002), 1000, None) == -3  # GDN_ERR_MISALIGNED


def _norm(lib, **kw):
    a = dict(y=P, z=P, w=P, out=P, rows=10, Dv=128, dtype=0, eps=1e-6, stream=None)
    a.update(kw)
    return lib.gdn_gated_rmsnorm(a["y"], a["z"], a["w"], a["out"], a["rows"], a["Dv"], a["dtype"],
                                 a["eps"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(rows=-1), -1), (dict(eps=-1e-3), -1), (dict(eps=float("inf")), -1),
    (dict(eps=float("nan")), -1), (dict(y=None), -1), (dict(w=None), -1),
    (dict(Dv=48), -2), (dict(dtype=5), -2), (dict(z=P + 8), -3), (dict(out=P + 2), -3),
    (dict(rows=0, y=None, z=None, w=None, out=None), 0),
])
def test_gated_norm_rejects_bad_arguments_on_host(lib, kw, code):
    assert _norm(lib, **kw) == code


def _decode_gated(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, b=P, s=P, out=P, z=P, w=P, eps=1e-6, B=4, HK=2, HV=4, Dk=128,
             Dv=128, dtype=0, scale=0.0, l2=1, stream=None)
    a.update(kw)
    return lib.gdn_decode_step_gated(a["q"], a["k"], a["v"], a["g"], a["b"], a["s"], a["out"],
                                     a["z"], a["w"], a["eps"], a["B"], a["HK"], a["HV"], a["Dk"],
                                     a["Dv"], a["dtype"], a["scale"], a["l2"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(z=None), -1), (dict(w=None), -1), (dict(eps=-1.0), -1), (dict(HV=5), -1),
    (dict(z=P + 4), -3), (dict(w=P + 8), -3), (dict(Dk=48, Dv=48), -2), (dict(B=0), 0),
])
def test_gated_decode_rejects_bad_arguments_on_host(lib, kw, code):
    assert _decode_gated(lib, **kw) == code


def _prologue(lib, **kw):
    a = dict(proj=P, pb=P, pa=P, layout=0, w=P, al=P, db=P, sin=None, sout=None, cu=None, N=2,
             T=64, HK=2, HV=4, Dk=128, Dv=128, dtype=0, q=P, k=P, v=P, z=None, beta=P, g=P,
             stream=None)
    a.update(kw)
    return lib.gdn_conv_gate_prologue(a["proj"], a["pb"], a["pa"], a["layout"], a["w"], a["al"],
                                      a["db"], a["sin"], a["sout"], a["cu"], a["N"], a["T"], a["HK"],
                                      a["HV"], a["Dk"], a["Dv"], a["dtype"], a["q"], a["k"], a["v"],
                                      a["z"], a["beta"], a["g"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(layout=2), -1), (dict(N=-1), -1), (dict(T=-4), -1), (dict(T=63), -1),
    (dict(pa=None), -1), (dict(proj=None), -1), (dict(w=None), -1), (dict(g=None), -1),
    (dict(z=P), -1), (dict(HV=3), -1), (dict(Dk=96, Dv=96), -2), (dict(dtype=4), -2),
    (dict(N=70000, T=70000), -2), (dict(proj=P + 8), -3), (dict(sin=P + 4), -3),
    (dict(layout=1, pa=None, z=P + 2), -3),
])
def test_prologue_rejects_bad_arguments_on_host(lib, kw, code):
    assert _prologue(lib, **kw) == code


def test_gated_prefill_rejects_bad_arguments_on_host(lib):
    f = lib.gdn_prefill_gated
    base = [P, P, P, P, P, None, P, P, None, P, P, 1e-6, 1, 64, 2, 4, 128, 128, 0, 0.0, 1, P, BIG,
            None]
    a = list(base); a[9] = None
    assert f(*a) == -1                           # gate required
    a = list(base); a[10] = None
    assert f(*a) == -1                           # weight required
    a = list(base); a[11] = -1.0
    assert f(*a) == -1
    a = list(base); a[9] = P + 4
    assert f(*a) == -3
    g = lib.gdn_prefill_varlen_gated
    vbase = [P, P, P, P, P, None, P, P, None, P, P, 1e-6, None, 2, 100, 2, 4, 128, 128, 0, 0.0, 1,
             P, BIG, None]
    assert g(*vbase) == -1                       # cu_seqlens required
    a = list(vbase); a[12] = P; a[10] = P + 8
    assert g(*a) == -3
