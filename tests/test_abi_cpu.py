"""libpa.so loads and exports every entry point include/pa.h declares, and
its host-side argument checks answer without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from paged_kv_attention_16_gb300 import build as pbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pa.h")


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(pbuild.build())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pa_forward", "pa_mla_decode", "pa_reserve", "pa_get_device_status",
                 "pa_status_string", "pa_debug_gather"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_export():
    from paged_kv_attention_16_gb300 import pa
    assert sorted(pa.EXPORTS) == declared_functions()


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    assert lib.pa_status_string(0) == b"ok"
    assert b"unsupported" in lib.pa_status_string(2)


def _forward(lib, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, bt=1 << 20, sl=1 << 20, qsl=1 << 20, H=8, Hk=2,
                D=128, bs=16, scale=0.1, out=1 << 20, stream=None, dtype=1, S=1, T=1, mbps=4,
                nb=4, msl=64, kvs=0)
    args.update(kw)
    f = lib.pa_forward
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_float, vp, vp] + [ctypes.c_int] * 7
    a = args
    return f(a["q"], a["k"], a["v"], a["bt"], a["sl"], a["qsl"], a["H"], a["Hk"], a["D"], a["bs"],
             a["scale"], a["out"], a["stream"], a["dtype"], a["S"], a["T"], a["mbps"], a["nb"],
             a["msl"], a["kvs"])


@pytest.mark.parametrize("kw,want", [
    (dict(H=0), 1), (dict(Hk=3), 1), (dict(S=-1), 1), (dict(dtype=7), 1),
    (dict(D=96), 2), (dict(bs=8), 2), (dict(bs=512), 2), (dict(H=96, Hk=3), 2),
    (dict(kvs=100), 2), (dict(T=0), 0), (dict(q=0), 1), (dict(out=(1 << 20) + 4), 1),
])
def test_host_argument_checks(lib, kw, want):
    assert _forward(lib, **kw) == want


def test_workspace_bytes_grow_with_splits(lib):
    f = lib.pa_forward_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 8
    small = f(1, 64, 64, 32, 8, 128, 8192, 0)
    big = f(1, 64, 64, 32, 8, 128, 131072, 0)
    assert 0 < small < big


def test_workspace_holds_doubled_tile_splits(lib):
    """Extend / prefill rows on the tensor-core path are cut into up to twice
    the splits kv_split_tokens needs (equal splits, doubled when the batch's
    tile work is small against the grid): the workspace holds a split partial
    (head_dim fp32 + its log-sum-exp) per row, head and split for all of them."""
    f = lib.pa_forward_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 8
    T, H, Hk, D, msl, kvs = 4100, 8, 1, 128, 131072, 32768
    bf16 = 1
    auto = f(bf16, 6, T, H, Hk, D, msl, 0)
    chunked = f(bf16, 6, T, H, Hk, D, msl, kvs)
    splits = 2 * (-(-msl // kvs))
    assert chunked - auto >= T * H * splits * (D * 4 + 4)


def _cache_write(lib, **kw):
    args = dict(kn=1 << 20, vn=1 << 20, kc=1 << 20, vc=1 << 20, bt=1 << 20, sl=1 << 20,
                qsl=1 << 20, Hk=2, D=128, bs=16, stream=None, dtype=1, S=1, T=1, mbps=4, nb=4,
                layout=0)
    args.update(kw)
    f = lib.pa_cache_write
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp] * 7 + [ctypes.c_int] * 3 + [vp] + [ctypes.c_int] * 6
    a = args
    return f(a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["sl"], a["qsl"], a["Hk"], a["D"],
             a["bs"], a["stream"], a["dtype"], a["S"], a["T"], a["mbps"], a["nb"], a["layout"])


@pytest.mark.parametrize("kw,want", [
    (dict(Hk=0), 1), (dict(D=-1), 1), (dict(bs=0), 1), (dict(S=-1), 1), (dict(dtype=5), 1),
    (dict(D=4), 2), (dict(D=6, dtype=0), 2), (dict(T=0), 0), (dict(kn=0), 1), (dict(S=0), 1),
    (dict(kc=(1 << 20) + 8), 1), (dict(nb=0), 1), (dict(layout=2), 1), (dict(layout=-1), 1),
    (dict(layout=1, T=0), 0),
])
def test_cache_write_host_argument_checks(lib, kw, want):
    assert _cache_write(lib, **kw) == want


class _Options(ctypes.Structure):
    _fields_ = [("sinks", ctypes.c_void_p), ("kv_layout", ctypes.c_int),
                ("sliding_window", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("alibi_sqrt", ctypes.c_int), ("max_query_len", ctypes.c_int)]


def _forward_ex(lib, options, **kw):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, bt=1 << 20, sl=1 << 20, qsl=1 << 20, H=8, Hk=2,
                D=128, bs=16, scale=0.1, out=1 << 20, stream=None, dtype=1, S=1, T=1, mbps=4,
                nb=4, msl=64, kvs=0)
    args.update(kw)
    f = lib.pa_forward_ex
    f.restype = ctypes.c_int
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_float, vp, vp] + [ctypes.c_int] * 7 + [ctypes.POINTER(_Options)]
    a = args
    return f(a["q"], a["k"], a["v"], a["bt"], a["sl"], a["qsl"], a["H"], a["Hk"], a["D"], a["bs"],
             a["scale"], a["out"], a["stream"], a["dtype"], a["S"], a["T"], a["mbps"], a["nb"],
             a["msl"], a["kvs"], options)


@pytest.mark.parametrize("sinks,layout,kw,want", [
    (None, 0, dict(H=0), 1),              # the checks of pa_forward still apply
    (None, 0, dict(D=96), 2),
    (1 << 20, 0, dict(T=0), 0),           # nothing to do: no launch
    ((1 << 20) + 2, 0, dict(T=0), 1),     # a sinks array that is not 4-byte aligned
    ((1 << 20) + 2, 0, dict(), 1),
    (None, 1, dict(T=0), 0),              # HND
    (None, 2, dict(T=0), 1),              # no such layout
    (None, -1, dict(), 1),
])
def test_forward_ex_host_argument_checks(lib, sinks, layout, kw, want):
    opts = _Options(sinks, layout, 0, None, 0)
    assert _forward_ex(lib, ctypes.byref(opts), **kw) == want
    if sinks is None and layout == 0:
        assert _forward_ex(lib, None, **kw) == want  # null options: pa_forward


@pytest.mark.parametrize("window,slopes,use_sqrt,kw,want", [
    (128, 1 << 20, 1, dict(T=0), 0),
    (-1, None, 0, dict(T=0), 1),            # negative window
    (0, None, 2, dict(T=0), 1),             # alibi_sqrt neither 0 nor 1
    (0, (1 << 20) + 2, 0, dict(T=0), 1),    # slopes not 4-byte aligned
    (16, None, 0, dict(D=96), 2),           # the shape checks still apply
])
def test_forward_ex_variant_checks(lib, window, slopes, use_sqrt, kw, want):
    opts = _Options(None, 0, window, slopes, use_sqrt)
    assert _forward_ex(lib, ctypes.byref(opts), **kw) == want


def _mla_prefill(lib, **kw):
    args = dict(q=1 << 20, c=1 << 20, w=1 << 20, bt=1 << 20, sl=1 << 20, qsl=1 << 20, H=128,
                L=512, nope=128, R=64, dv=128, bs=64, scale=0.07, out=1 << 20, stream=None, S=1,
                T=1, mbps=4, nb=4, msl=64, tot=64, kvs=0)
    args.update(kw)
    f = lib.pa_mla_prefill
    f.restype = ctypes.c_int
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 6 + [ci] * 6 + [ctypes.c_float, vp, vp] + [ci] * 5 + [
        ctypes.c_longlong, ci]
    a = args
    return f(a["q"], a["c"], a["w"], a["bt"], a["sl"], a["qsl"], a["H"], a["L"], a["nope"],
             a["R"], a["dv"], a["bs"], a["scale"], a["out"], a["stream"], a["S"], a["T"],
             a["mbps"], a["nb"], a["msl"], a["tot"], a["kvs"])


@pytest.mark.parametrize("kw,want", [
    (dict(H=0), 1), (dict(S=-1), 1), (dict(tot=-1), 1), (dict(bs=0), 1),
    (dict(L=256), 2), (dict(R=32), 2), (dict(nope=64), 2), (dict(dv=64), 2), (dict(kvs=24), 2),
    (dict(T=0), 0), (dict(q=0), 1), (dict(w=0), 1), (dict(out=(1 << 20) + 2), 1),
])
def test_mla_prefill_host_argument_checks(lib, kw, want):
    assert _mla_prefill(lib, **kw) == want


def test_mla_prefill_workspace_grows_with_the_decompression_bound(lib):
    f = lib.pa_mla_prefill_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 4 + [ctypes.c_longlong, ctypes.c_int]
    small = f(8, 4096, 128, 4096, 8192, 0)
    big = f(8, 4096, 128, 4096, 16384, 0)
    # per position: 128 key and 128 value entries per head, plus the 64-wide
    # rotary key stored once, bf16
    assert big - small >= 8192 * (128 * (128 + 128) + 64) * 2
    assert f(-1, 1, 128, 64, 64, 0) == 0


def test_header_compiles_as_c_and_cxx(tmp_path):
    """include/pa.h is a plain C header (C99, pedantic) that C++ can include."""
    import shutil
    import subprocess
    src = tmp_path / "use_pa.c"
    src.write_text('#include "pa.h"\n'
                   "int main(void) {\n"
                   "  pa_forward_options o = {0};\n"
                   "  (void)o;\n"
                   "  return (int)PA_KV_HND - 1 + (int)PA_OK;\n"
                   "}\n")
    inc = os.path.dirname(HEADER)
    for cmd in (["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror"],
                ["g++", "-std=c++11", "-Wall", "-Werror", "-x", "c++"]):
        if shutil.which(cmd[0]) is None:
            continue
        subprocess.run(cmd + ["-I", inc, "-c", str(src), "-o", str(tmp_path / "o.o")],
                       check=True)


def test_binding_options_struct_matches_the_header(tmp_path):
    """ctypes' ForwardOptions has the size and field offsets the C compiler
    gives pa_forward_options."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        return
    from paged_kv_attention_16_gb300 import pa
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "pa.h"\n'
                   "int main(void) {\n"
                   '  printf("%zu %zu %zu %zu %zu %zu %zu\\n", sizeof(pa_forward_options),\n'
                   "         offsetof(pa_forward_options, sinks),\n"
                   "         offsetof(pa_forward_options, kv_layout),\n"
                   "         offsetof(pa_forward_options, sliding_window),\n"
                   "         offsetof(pa_forward_options, alibi_slopes),\n"
                   "         offsetof(pa_forward_options, alibi_sqrt),\n"
                   "         offsetof(pa_forward_options, max_query_len));\n"
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    O = pa.ForwardOptions
    want = [ctypes.sizeof(O)] + [getattr(O, f).offset for f, _ in O._fields_]
    assert got == want
