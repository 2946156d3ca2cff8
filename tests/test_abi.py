"""CPU-side checks of the C ABI: the library builds, loads, exports every symbol the
header declares, and validates arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gptq.h")


@pytest.fixture(scope="module")
def clib():
    from post_weight_quantization_04_gb300 import build as b
    import post_weight_quantization_04_gb300 as g
    b.build()
    return g.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:int|int64_t|size_t|void|unsigned long long|const char\*)\s+(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declarations_match_binding():
    import post_weight_quantization_04_gb300 as g
    assert _declared() == sorted(g.EXPORTS)


def test_library_exports_every_declared_symbol(clib):
    for name in _declared():
        assert hasattr(clib, name), name


def test_host_only_helpers(clib):
    import post_weight_quantization_04_gb300 as g
    assert clib.gptq_packed_words_per_row(4096, 4) == 512
    assert clib.gptq_packed_words_per_row(4096, 3) == 384
    assert clib.gptq_packed_words_per_row(5, 3) == 1
    assert clib.gptq_prepare_workspace_bytes(4096, 0) >= 2 * 4096 * 4096 * 4
    assert clib.gptq_quantize_workspace_bytes(4096, 4096, g.qconfig(4, 128, True)) >= 4096 * 4096 * 4
    assert clib.gptq_status_string(3).decode().startswith("Hessian not positive")


def test_argument_validation_happens_before_any_launch(clib):
    import post_weight_quantization_04_gb300 as g
    p = ctypes.c_void_p(16)
    s = ctypes.c_void_p(0)
    # unsupported bit width / group size: rejected on the host
    assert clib.gptq_quantize(p, 4, 4, p, None, None, g.qconfig(5, 0, True), p, p, p, None, None, None, None,
                              p, 1 << 20, s) == 2
    assert clib.gptq_quantize(p, 4, 4, p, None, None, g.qconfig(4, 96, True), p, p, p, None, None, None, None,
                              p, 1 << 20, s) == 2
    assert clib.rtn_quantize(p, 4, 4, None, g.qconfig(1, 0, True), p, p, p, None, None, s) == 2
    assert clib.gptq_pack(p, 4, 4, 8, 1, p, s) == 2
    # empty inputs are a no-op
    assert clib.gptq_quantize(p, 0, 4, p, None, None, g.qconfig(4, 0, True), p, p, p, None, None, None, None,
                              p, 0, s) == 0
    assert clib.rtn_quantize(p, 4, 0, None, g.qconfig(4, 0, True), p, p, p, None, None, s) == 0
    # bad sizes / workspace
    assert clib.gptq_prepare(p, None, 0, 0.01, 0, p, p, p, p, 1 << 30, s) == 1
    assert clib.gptq_prepare(p, None, 8, 0.01, 1, p, p, p, p, 1 << 30, s) == 1   # act_order needs diag
    assert clib.gptq_prepare(p, None, 8, 0.01, 0, p, p, p, p, 16, s) == 6        # workspace too small
    assert clib.gptq_quantize(p, 4, 4, p, None, None, g.qconfig(4, 0, True), p, p, p, None, None, None, None,
                              p, 16, s) == 6
    h = ctypes.c_void_p()
    assert clib.gptq_hessian_create(0, ctypes.byref(h)) == 1


def test_status_mode_switch(clib):
    assert clib.gptq_set_status_mode(2) == 1          # INVALID_ARG
    prev = clib.gptq_status_mode()
    assert clib.gptq_set_status_mode(1) == 0
    assert clib.gptq_status_mode() == 1
    assert clib.gptq_set_status_mode(prev) == 0
