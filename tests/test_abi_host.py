"""Host-side checks of the C ABI: the library builds, loads and exports
every symbol include/pa.h declares, and invalid calls are rejected on the
host before anything is launched (no GPU needed: every pointer below is a
fake, and validation fails before any device access)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_74_gb300 as pa
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    pa.build()
    return pa.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert set(declared_functions()) == set(pa.ABI_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_abi_version_matches_header(lib):
    m = re.search(r"#define PA_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.pa_abi_version() == int(m.group(1))


def test_library_owns_no_stream_or_event():
    """Every call enqueues on the caller's stream only: the library creates
    no stream and no event (no hidden ordering between callers' streams, and
    nothing to create before a stream capture)."""
    csrc = os.path.join(ROOT, "paged_kv_cache_74_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, name), encoding="utf-8").read()
        for call in ("cudaStreamCreate", "cudaEventCreate", "cuStreamCreate", "cuEventCreate"):
            assert call not in text, f"{name} calls {call}"


def test_status_strings(lib):
    for s in range(5):
        assert lib.pa_status_string(s).decode().startswith("PA_")
    assert lib.pa_status_string(99) == b"unknown pa_status"


A = 0x10000  # a 256-byte-aligned fake device address (never dereferenced)


def decode_call(lib, **kw):
    args = dict(out=A, q=A, kc=A, vc=A, bt=A, mb=4, sl=A, ns=2, msl=64, hq=8, hkv=2, d=128, bs=16,
                nb=32, scale=0.125, pt=0, ws=A, wsb=1 << 20)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.pa_decode(vp(args["out"]), vp(args["q"]), vp(args["kc"]), vp(args["vc"]),
                         vp(args["bt"]), args["mb"], vp(args["sl"]), args["ns"], args["msl"],
                         args["hq"], args["hkv"], args["d"], args["bs"], args["nb"], args["scale"],
                         args["pt"], vp(args["ws"]), args["wsb"], vp(0))


@pytest.mark.parametrize("kw,expect", [
    (dict(out=0), 1), (dict(q=0), 1), (dict(kc=0), 1), (dict(bt=0), 1), (dict(sl=0), 1),
    (dict(q=A + 8), 1), (dict(out=A + 2), 1), (dict(bt=A + 2), 1),
    (dict(hq=6, hkv=4), 1), (dict(hkv=0), 1), (dict(ns=-1), 1), (dict(nb=0), 1),
    (dict(msl=65), 1), (dict(mb=0), 1), (dict(scale=float("inf")), 1), (dict(scale=float("nan")), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.125), 1),
    (dict(pt=24), 1), (dict(pt=-16), 1),
    (dict(d=96), 2), (dict(bs=48), 2), (dict(bs=128), 2), (dict(hq=34, hkv=2), 2), (dict(ns=70000), 2),
    (dict(ws=0), 3), (dict(wsb=16), 3),
    (dict(ws=A + 16), 1),
])
def test_decode_rejects_invalid_arguments(lib, kw, expect):
    assert decode_call(lib, **kw) == expect


def test_decode_empty_batch_is_a_no_op(lib):
    assert decode_call(lib, ns=0) == 0


def test_workspace_size(lib):
    small = lib.pa_decode_workspace_size(4, 4, 2, 64, 37, 0)
    assert small >= 256 and small % 256 == 0
    # forced 16-token partitions over 32K tokens need partials for 2048 partitions
    big = lib.pa_decode_workspace_size(8, 32, 8, 128, 32768, 16)
    assert big >= 8 * 32 * 2048 * (128 + 2) * 4
    assert lib.pa_decode_workspace_size(4, 6, 4, 64, 37, 0) == 0   # Hq % Hkv != 0
    assert lib.pa_decode_workspace_size(4, 4, 2, 80, 37, 0) == 0   # head_dim
    assert lib.pa_decode_workspace_size(4, 4, 2, 64, 37, 20) == 0  # not a block multiple


def test_reshape_and_cache_validation(lib):
    vp = ctypes.c_void_p
    call = lambda **k: lib.pa_reshape_and_cache(
        vp(k.get("key", A)), vp(k.get("value", A)), k.get("ks", 1024), k.get("vs", 1024),
        vp(k.get("kc", A)), vp(k.get("vc", A)), vp(k.get("sm", A)), k.get("n", 4), 8, 128, 16, 64,
        vp(0), vp(0))
    assert call(n=0) == 0                       # nothing to do, nothing launched
    assert call(key=0) == 1
    assert call(key=A + 4) == 1
    assert call(ks=1000) == 1                   # stride below one token row
    assert call(ks=1028) == 1                   # not a multiple of 8 elements
    assert call(sm=A + 4) == 1
    assert call(n=-1) == 1


def test_slot_mapping_validation(lib):
    vp = ctypes.c_void_p
    call = lambda **k: lib.pa_compute_slot_mapping(
        vp(k.get("out", A)), k.get("n", 4), vp(k.get("bt", A)), 4, vp(k.get("qsl", A)),
        vp(k.get("sl", A)), k.get("ns", 2), 16, 32, vp(0), vp(0))
    assert call(ns=0) == 0
    assert call(out=0) == 1
    assert call(out=A + 4) == 1
    assert call(qsl=A + 2) == 1
    assert call(n=-3) == 1


def test_prefill_validation(lib):
    vp = ctypes.c_void_p
    call = lambda **k: lib.pa_prefill_varlen(
        vp(A), vp(A), vp(A), vp(A), vp(k.get("qsl", A)), vp(A), 2, k.get("tq", 9),
        k.get("mql", 8), k.get("msl", 64), vp(A), 4, 8, 2, k.get("d", 128), 16, 32, 0.1, vp(A),
        1 << 20, vp(0))
    assert call(qsl=0) == 1
    assert call(mql=65) == 1
    assert call(d=80) == 2
    assert call(tq=0) == 0


@pytest.mark.parametrize("args,expect", [
    ((A, A, 2, 4, 0), 1), ((0, A, 2, 4, 2), 1), ((A, 0, 2, 4, 2), 1), ((A + 2, A, 2, 4, 2), 1),
    ((A, A, -1, 4, 2), 1), ((A, A, 2, -4, 2), 1), ((A, A, 0, 4, 2), 0), ((A, A, 2, 0, 2), 0),
])
def test_map_to_kernel_blocks_validation(lib, args, expect):
    out, src, rows, cols, k = args
    vp = ctypes.c_void_p
    assert lib.pa_map_to_kernel_blocks(vp(out), vp(src), rows, cols, k, vp(0), vp(0)) == expect


def decode_fp8_call(lib, **kw):
    args = dict(out=A, q=A, kc=A, vc=A, bt=A, mb=4, sl=A, ns=2, msl=64, hq=8, hkv=2, d=128, bs=16,
                nb=32, scale=0.125, ks=1.0, vs=1.0, pt=0, ws=A, wsb=1 << 20)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.pa_decode_fp8(vp(args["out"]), vp(args["q"]), vp(args["kc"]), vp(args["vc"]),
                             vp(args["bt"]), args["mb"], vp(args["sl"]), args["ns"], args["msl"],
                             args["hq"], args["hkv"], args["d"], args["bs"], args["nb"],
                             args["scale"], args["ks"], args["vs"], args["pt"], vp(args["ws"]),
                             args["wsb"], vp(0))


@pytest.mark.parametrize("kw,expect", [
    (dict(ks=0.0), 1), (dict(vs=-1.0), 1), (dict(ks=float("nan")), 1), (dict(vs=float("inf")), 1),
    (dict(q=0), 1), (dict(hq=68, hkv=4), 2), (dict(d=96), 2), (dict(ws=0), 3),
])
def test_decode_fp8_rejects_invalid_arguments(lib, kw, expect):
    assert decode_fp8_call(lib, **kw) == expect


def test_reshape_and_cache_fp8_rejects_bad_scales(lib):
    vp = ctypes.c_void_p
    for ks, vs in ((0.0, 1.0), (1.0, float("nan")), (-2.0, 1.0)):
        assert lib.pa_reshape_and_cache_fp8(vp(A), vp(A), 256, 256, vp(A), vp(A), vp(A), 4, 2, 128,
                                            16, 32, ks, vs, vp(0), vp(0)) == 1
    # num_tokens == 0 is a no-op even with null pointers
    assert lib.pa_reshape_and_cache_fp8(vp(0), vp(0), 256, 256, vp(0), vp(0), vp(0), 0, 2, 128, 16,
                                        32, 1.0, 1.0, vp(0), vp(0)) == 0


def prefill_fp8_call(lib, **kw):
    args = dict(out=A, q=A, kc=A, vc=A, qsl=A, sl=A, ns=2, tq=10, mql=9, msl=64, bt=A, mb=4, hq=8,
                hkv=2, d=128, bs=16, nb=32, scale=0.125, ks=1.0, vs=1.0, ws=A, wsb=1 << 30)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.pa_prefill_varlen_fp8(vp(args["out"]), vp(args["q"]), vp(args["kc"]), vp(args["vc"]),
                                     vp(args["qsl"]), vp(args["sl"]), args["ns"], args["tq"],
                                     args["mql"], args["msl"], vp(args["bt"]), args["mb"],
                                     args["hq"], args["hkv"], args["d"], args["bs"], args["nb"],
                                     args["scale"], args["ks"], args["vs"], vp(args["ws"]),
                                     args["wsb"], vp(0))


@pytest.mark.parametrize("kw,expect", [
    (dict(ks=0.0), 1), (dict(vs=-1.0), 1), (dict(ks=float("inf")), 1), (dict(vs=float("nan")), 1),
    (dict(qsl=0), 1), (dict(mql=65), 1), (dict(scale=0.0), 1), (dict(d=96), 2), (dict(ws=0), 3),
])
def test_prefill_fp8_rejects_invalid_arguments(lib, kw, expect):
    """Checked on the host before any launch (no GPU needed)."""
    assert prefill_fp8_call(lib, **kw) == expect


def decode_xsplit_call(lib, **kw):
    args = dict(out=A, q=A, kc=A, vc=A, bt=A, mb=4, sl=A, ns=2, msl=64, hq=8, hkv=2, d=128, bs=16,
                nb=32, scale=0.125, pt=0, ws=A, wsb=1 << 20)
    args.update(kw)
    vp = ctypes.c_void_p
    return lib.pa_decode_xsplit(vp(args["out"]), vp(args["q"]), vp(args["kc"]), vp(args["vc"]),
                                vp(args["bt"]), args["mb"], vp(args["sl"]), args["ns"],
                                args["msl"], args["hq"], args["hkv"], args["d"], args["bs"],
                                args["nb"], args["scale"], args["pt"], vp(args["ws"]),
                                args["wsb"], vp(0))


@pytest.mark.parametrize("kw,expect", [
    (dict(out=0), 1), (dict(kc=A + 8), 1), (dict(hq=6, hkv=4), 1), (dict(msl=65), 1),
    (dict(scale=float("nan")), 1), (dict(pt=24), 1), (dict(ws=A + 16), 1),
    (dict(d=96), 2), (dict(bs=8), 2), (dict(hq=34, hkv=2), 2),
    (dict(ws=0), 3), (dict(wsb=16), 3),
])
def test_decode_xsplit_rejects_invalid_arguments(lib, kw, expect):
    assert decode_xsplit_call(lib, **kw) == expect


def test_decode_xsplit_empty_batch_is_a_no_op(lib):
    assert decode_xsplit_call(lib, ns=0) == 0


def test_workspace_size_covers_the_xsplit_units(lib):
    """Groups above 4 q heads run as several work units per kv head in the
    x-split decode: the workspace must hold a pair counter per unit."""
    for hq, hkv in ((64, 8), (40, 8), (16, 1)):
        ws = lib.pa_decode_workspace_size(1000, hq, hkv, 128, 4096, 0)
        g = hq // hkv
        units = hkv * (g // max(x for x in (1, 2, 3, 4) if g % x == 0))
        assert ws >= 1000 * units * 8


def test_reshape_and_cache_xsplit_validation(lib):
    vp = ctypes.c_void_p
    call = lambda **k: lib.pa_reshape_and_cache_xsplit(
        vp(k.get("key", A)), vp(k.get("value", A)), k.get("ks", 1024), k.get("vs", 1024),
        vp(k.get("kc", A)), vp(k.get("vc", A)), vp(k.get("sm", A)), k.get("n", 4), 8,
        k.get("d", 128), 16, 64, vp(0), vp(0))
    assert call(n=0) == 0
    assert call(key=0) == 1
    assert call(vc=A + 2) == 1
    assert call(ks=1000) == 1
    assert call(vs=1028) == 1
    assert call(n=-1) == 1
    assert call(d=12) == 2


def test_append_tokens_validation(lib):
    vp = ctypes.c_void_p
    call = lambda **k: lib.pa_append_tokens(
        vp(k.get("key", A)), vp(k.get("value", A)), k.get("ks", 1024), k.get("vs", 1024),
        vp(k.get("kc", A)), vp(k.get("vc", A)), vp(k.get("bt", A)), k.get("mb", 4),
        vp(k.get("qsl", A)), vp(k.get("sl", A)), k.get("ns", 4), k.get("n", 4), 8,
        k.get("d", 128), 16, 64, vp(k.get("sm", 0)), vp(0), vp(0))
    assert call(n=0) == 0 and call(ns=0) == 0      # nothing to do, nothing launched
    assert call(key=0) == 1
    assert call(bt=0) == 1
    assert call(qsl=A + 2) == 1
    assert call(sm=A + 4) == 1
    assert call(ks=1000) == 1
    assert call(ns=-1) == 1
    assert call(mb=0) == 1
    assert call(d=12) == 2
