"""The C ABI library: it loads, exports every declared entry point, and rejects
bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verification_45_gb300 import _native

HEADER = os.path.join(_native.INCLUDE, "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    _native.build()
    return _native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_debug", "spec_verify_ex", "spec_sample", "spec_ngram_propose",
              "spec_tree_verify", "spec_device_pointer", "spec_verify_launch_shape", "spec_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(4):
        assert lib.spec_status_string(code)
    assert lib.spec_status_string(99) == b"unknown status"


def _call(lib, **over):
    # Never dereferenced: every case below fails validation (or is B = 0) before
    # anything is launched; a case that passes validation must not be added here.
    fake = 0x10000
    args = dict(target=fake, draft=fake, tokens=fake, num_draft=fake, uniforms=fake, temperature=fake,
                out_tokens=fake, out_num=fake, B=4, gmax=4, V=1024, dtype=1, status=None, stream=None)
    args.update(over)
    vp = ctypes.c_void_p
    return lib.spec_verify(vp(args["target"]), vp(args["draft"]), vp(args["tokens"]), vp(args["num_draft"]),
                           vp(args["uniforms"]), vp(args["temperature"]), vp(args["out_tokens"]),
                           vp(args["out_num"]), args["B"], args["gmax"], args["V"], args["dtype"],
                           vp(args["status"]) if args["status"] else None, None)


@pytest.mark.parametrize("over,code", [
    (dict(target=0), 1), (dict(num_draft=0), 1), (dict(uniforms=0), 1), (dict(temperature=0), 1),
    (dict(out_tokens=0), 1), (dict(out_num=0), 1), (dict(tokens=0), 1),
    (dict(B=-1), 1), (dict(gmax=17), 1), (dict(gmax=-1), 1), (dict(V=0), 1), (dict(V=(1 << 24) + 1), 1),
    (dict(dtype=7), 2), (dict(target=0x10001), 1), (dict(tokens=0x10002), 1), (dict(status=0x10003), 1),
    (dict(B=0), 0),
])
def test_host_argument_checks(lib, over, code):
    assert _call(lib, **over) == code


@pytest.mark.parametrize("cluster,kernel", [(17, 0), (32, 0), (-1, 0), (0, 4), (0, -1), (0, 1)])
def test_launch_options_checked(lib, cluster, kernel):
    vp = ctypes.c_void_p
    f = vp(0x10000)
    opts = _native.Options(cluster, kernel)
    rc = lib.spec_verify_ex(f, f, f, f, f, f, f, f, 4, 4, 1024, 1, None, None, ctypes.byref(opts))
    assert rc == 1


@pytest.mark.parametrize("which,code", [("logits", 1), ("uniforms", 1), ("temperature", 1), ("out", 1),
                                        ("V", 1), ("dtype", 2), ("B0", 0), ("kernel1", 1)])
def test_sampler_argument_checks(lib, which, code):
    vp = ctypes.c_void_p
    a = dict(logits=0x10000, uniforms=0x10000, temperature=0x10000, out=0x10000, B=4, V=1024, dtype=1, kernel=0)
    if which in ("logits", "uniforms", "temperature", "out"):
        a[which] = 0
    elif which == "V":
        a["V"] = 0
    elif which == "dtype":
        a["dtype"] = 9
    elif which == "B0":
        a["B"] = 0
    elif which == "kernel1":  # 1 names no kernel
        a["kernel"] = 1
    opts = _native.Options(0, a["kernel"])
    rc = lib.spec_sample(vp(a["logits"]) if a["logits"] else None, vp(a["uniforms"]) if a["uniforms"] else None,
                         vp(a["temperature"]) if a["temperature"] else None, vp(a["out"]) if a["out"] else None,
                         a["B"], a["V"], a["dtype"], None, None, ctypes.byref(opts))
    assert rc == code


@pytest.mark.parametrize("over,code", [
    (dict(context=0), 1), (dict(lens=0), 1), (dict(num=0), 1), (dict(toks=0), 1), (dict(min_n=0), 1),
    (dict(max_n=65), 1), (dict(min_n=3, max_n=2), 1), (dict(gmax=17), 1), (dict(stride=0), 1), (dict(B=-1), 1),
    (dict(context=0x10002), 1), (dict(B=0), 0),
])
def test_ngram_argument_checks(lib, over, code):
    a = dict(context=0x10000, stride=64, lens=0x10000, B=4, min_n=1, max_n=4, gmax=4, toks=0x10000, num=0x10000)
    a.update(over)
    vp = ctypes.c_void_p
    rc = lib.spec_ngram_propose(vp(a["context"]) if a["context"] else None, a["stride"],
                                vp(a["lens"]) if a["lens"] else None, a["B"], a["min_n"], a["max_n"], a["gmax"],
                                vp(a["toks"]) if a["toks"] else None, vp(a["num"]) if a["num"] else None, None)
    assert rc == code


@pytest.mark.parametrize("over,code", [
    (dict(target=0), 1), (dict(parent=0), 1), (dict(tokens=0), 1), (dict(num_nodes=0), 1),
    (dict(uniforms=0), 1), (dict(temperature=0), 1), (dict(out_tokens=0), 1), (dict(out_num=0), 1),
    (dict(out_path=0x10002), 1), (dict(N=0), 1), (dict(N=257), 1), (dict(V=0), 1), (dict(B=-1), 1),
    (dict(dtype=5), 2), (dict(target=0x10001), 1), (dict(kernel=2), 1), (dict(cluster=17), 1), (dict(B=0), 0),
])
def test_tree_host_argument_checks(lib, over, code):
    # Never dereferenced: every case fails validation (or is B = 0) before a launch.
    fake = 0x10000
    a = dict(target=fake, parent=fake, tokens=fake, num_nodes=fake, uniforms=fake, temperature=fake,
             out_tokens=fake, out_num=fake, out_path=None, B=4, N=16, V=1024, dtype=1, kernel=0, cluster=0)
    a.update(over)
    vp = ctypes.c_void_p
    opts = _native.Options(a["cluster"], a["kernel"])
    rc = lib.spec_tree_verify(vp(a["target"]), vp(a["parent"]), vp(a["tokens"]), vp(a["num_nodes"]),
                              vp(a["uniforms"]), vp(a["temperature"]), vp(a["out_tokens"]), vp(a["out_num"]),
                              vp(a["out_path"]) if a["out_path"] else None, a["B"], a["N"], a["V"], a["dtype"],
                              None, None, ctypes.byref(opts))
    assert rc == code
