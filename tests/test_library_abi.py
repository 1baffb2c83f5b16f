"""The C library builds, loads without a GPU, exports every function that
include/avsg.h declares, agrees with the binding's struct layouts, and rejects
bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "avsg.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(avsg_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_step_interface():
    names = declared_functions()
    for n in ["avsg_create", "avsg_step", "avsg_destroy", "avsg_get_stats", "avsg_read_state"]:
        assert n in names
    assert len(names) >= 15


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_function():
    from decode_serving_gb300 import avsg
    assert set(declared_functions()) == set(avsg.SIGNATURES)
    for name in declared_functions():
        assert callable(getattr(avsg, name)), name


def test_struct_layouts_match_the_header(tmp_path):
    from decode_serving_gb300 import avsg
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "avsg.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(avsg_config),"
        " offsetof(avsg_config, num_entries), offsetof(avsg_config, softmax_scale),"
        " sizeof(avsg_stats), sizeof(avsg_info), sizeof(avsg_kernel_times)); return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(avsg.avsg_config), avsg.avsg_config.num_entries.offset,
            avsg.avsg_config.softmax_scale.offset, ctypes.sizeof(avsg.avsg_stats),
            ctypes.sizeof(avsg.avsg_info), ctypes.sizeof(avsg.avsg_kernel_times)]
    assert got == want


def _cfg(**kw):
    from decode_serving_gb300.session import make_config
    base = dict(requests=2, kv_heads=2, q_per_kv=4, num_entries=1024, head_dim=128, v_dim=128,
                buffer_slots=256, max_select=64)
    base.update(kw)
    return make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(requests=0), -1),
    (dict(head_dim=100), -1),
    (dict(num_entries=0), -1),
    (dict(max_tokens_per_step=9), -1),
    (dict(kv_shared=True, v_dim=64), -1),
    (dict(max_select=300), -2),                       # k larger than the buffer
    (dict(max_tokens_per_step=3, max_select=100), -2),
    # a step's miss set (2 * 8 * 2048 cells, rounded up) exceeds match's shared memory
    (dict(max_tokens_per_step=8, max_select=2048, buffer_slots=16384, num_entries=1 << 20), -2),
    (dict(q_per_kv=3), -7),                           # no attention kernel for G=3
    (dict(head_dim=96, v_dim=96), -7),
])
def test_create_rejects_bad_configs_on_the_host(lib, kw, code):
    from decode_serving_gb300 import avsg
    cfg = _cfg(**kw)
    h = ctypes.c_void_p()
    dummy = ctypes.create_string_buffer(16)
    rc = lib.avsg_create(ctypes.byref(cfg), ctypes.addressof(dummy), ctypes.addressof(dummy),
                         ctypes.byref(h))
    assert rc == code, avsg.avsg_strerror(rc)
    assert h.value is None


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.avsg_create(None, None, None, ctypes.byref(h)) == -1
    assert lib.avsg_step(None, 0, 1, 1, None, None, None, None, None, None) == -1
    assert lib.avsg_get_stats(None, None) == -1
    assert lib.avsg_destroy(None) == 0


def test_strerror(lib):
    from decode_serving_gb300 import avsg
    assert avsg.avsg_strerror(0) == "ok"
    for code in range(-8, 0):
        assert avsg.avsg_strerror(code) not in ("", "unknown error")
    assert avsg.avsg_strerror(-99) == "unknown error"
