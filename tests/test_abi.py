"""libhe C ABI on the CPU: the library loads, exports every declared symbol, its
struct layouts match the header, and argument errors are reported without a GPU."""
import ctypes
import re
import subprocess
from pathlib import Path

import pytest

import decode_opt_step_gb300 as he
from decode_opt_step_gb300 import build as he_build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    he_build.build()
    return he.load_library()


def _declared_functions():
    names = []
    for h in sorted((ROOT / "include").glob("*.h")):
        text = h.read_text()
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(he_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_functions()
    assert "he_generate" in declared and "he_op_linear" in declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(declared) == set(he._SIGNATURES), "binding signatures out of sync with headers"
    out = subprocess.run(["nm", "-D", "--defined-only", str(he._LIB_PATH)], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (he_\w+)$", out, re.M))
    assert set(declared) <= exported


def test_struct_layouts_match_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "he.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(he_config),"
        " sizeof(he_layer_weights), sizeof(he_weights), sizeof(he_allocator), sizeof(he_stats),"
        " offsetof(he_stats, kclass_ms), offsetof(he_layer_weights, lora_b));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", str(ROOT / "include"), str(src), "-o", str(exe)], check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                       check=True).stdout.split()))
    want = [ctypes.sizeof(he.HeConfig), ctypes.sizeof(he.HeLayerWeights),
            ctypes.sizeof(he.HeWeights), ctypes.sizeof(he.HeAllocator), ctypes.sizeof(he.HeStats),
            he.HeStats.kclass_ms.offset, he.HeLayerWeights.lora_b.offset]
    assert got == want


def test_argument_errors_without_gpu(lib):
    out = ctypes.c_void_p(123)
    assert lib.he_create(None, None, None, 0, ctypes.byref(out)) == he.HE_ERR_ARG
    assert out.value is None
    assert b"NULL" in lib.he_last_error()
    cfg = he.HeConfig(2, 100, 3, 64, 10, 8, 2, 0, 1e-5, 1, 4, 8, 16.0, 0)
    w = he.HeWeights()
    assert lib.he_create(ctypes.byref(cfg), ctypes.byref(w), None, 0,
                         ctypes.byref(out)) == he.HE_ERR_ARG  # 100 % 3 != 0
    assert lib.he_destroy(None) == he.HE_OK
    assert lib.he_fuse_lora(None, None) == he.HE_ERR_ARG
    assert lib.he_unfuse_lora(None, None) == he.HE_ERR_ARG
    assert lib.he_generate(None, None, 1, 1, 1, None, None, None) == he.HE_ERR_ARG
    assert lib.he_release_workspace(None, None) == he.HE_ERR_ARG
    assert lib.he_retake_workspace(None, None) == he.HE_ERR_ARG
    assert lib.he_check(None, None) == he.HE_ERR_ARG
    assert lib.he_get_stats(None, None) == he.HE_ERR_ARG
    assert lib.he_op_linear(1, None, 8, None, 0, None, 1, 1, 8, 1, None, None) == he.HE_ERR_ARG
    assert lib.he_op_tile_weight(None, None, 128, 64, None) == he.HE_ERR_ARG
    assert lib.he_op_head_greedy(1, None, 64, None, 1, 128, 64, None, None, None,
                                 None) == he.HE_ERR_ARG
    assert lib.he_op_linear_fp8(None, 128, None, None, None, 1, 128, 128, 0, None,
                                None) == he.HE_ERR_ARG
    assert lib.he_op_attn_prefill(1, None, None, None, None, 1, 1, 1, 64, 8, 0, None,
                                  None) == he.HE_ERR_ARG
    dummy = 4096  # never dereferenced: the size checks fail first
    assert lib.he_op_attn_prefill(1, dummy, dummy, dummy, dummy, 1, 9, 1, 64, 8, 0, None,
                                  None) == he.HE_ERR_ARG  # Lp > max_seq
    assert lib.he_op_attn_prefill(1, dummy, dummy, dummy, dummy, 1, 4, 1, 64, 8, 2, None,
                                  None) == he.HE_ERR_ARG  # unknown flag
    assert lib.he_op_attn_prefill(1, dummy, dummy, dummy, dummy, 1, 4, 1, 96, 8, 0, None,
                                  None) == he.HE_ERR_UNSUPPORTED
    assert lib.he_set_weight_format(None, 1) == he.HE_ERR_ARG
    assert lib.he_read_fused_fp8(None, 0, 0, None, 0, None, None) == he.HE_ERR_ARG
    assert b"sm_103a" in lib.he_version()


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="libhe.so not found"):
        he.load_library(tmp_path / "libhe.so")
