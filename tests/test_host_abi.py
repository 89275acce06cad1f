"""Host-side checks of the C-ABI library (no GPU needed): it builds, loads, exports every
function include/lora.h declares, and rejects bad shapes before touching the device."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ags():
    import __graft_entry__

    __graft_entry__.build()
    import adapter_gemm_segment_gb300 as m

    return m


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(lora_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lora_pool_create", "lora_pool_load_slot", "lora_segment", "lora_linear_fwd"):
        assert required in names


def test_library_exports_every_declared_symbol(ags):
    lib = ctypes.CDLL(ags.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(ags.EXPORTED) <= set(declared_functions())


def test_pool_bytes_formula(ags):
    # table (16 B per slot, 256-aligned) + A slab + B slab, each 256-aligned
    S, R, h_in, h_out = 100, 8, 4096, 4096
    want = 1792 + S * R * h_in * 2 + S * h_out * R * 2
    assert ags.lora_pool_bytes(h_in, h_out, R, S, torch.float16) == want
    assert ags.lora_pool_bytes(256, 256, 8, 4, torch.float32) == 256 + 4 * 8 * 256 * 4 * 2


@pytest.mark.parametrize("shape", [(0, 256, 8, 4), (256, 256, 0, 4), (256, 256, 8, 0), (256, 256, 300, 4),
                                   (256, 256, 8, 5000), (250, 256, 8, 4), (256, 256, 12, 4)])
def test_bad_pool_shapes_rejected(ags, shape):
    with pytest.raises(ags.LoraError) as e:
        ags.lora_pool_bytes(*shape, torch.float16)
    assert e.value.code == ags.LORA_EINVAL
    assert ags.lora_last_error()


def test_segment_workspace_sizes(ags):
    assert ags.lora_segment_workspace_bytes(0, 4) > 0
    a = ags.lora_segment_workspace_bytes(64, 100)
    b = ags.lora_segment_workspace_bytes(16384, 100)
    assert b - a >= 2 * 4 * (16384 - 64)
    with pytest.raises(ags.LoraError):
        ags.lora_segment_workspace_bytes(-1, 4)
    with pytest.raises(ags.LoraError):
        ags.lora_segment_workspace_bytes(4, 0)


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "adapter_gemm_segment_gb300")
    pat = re.compile(r"^\s*(from\s+oracle|import\s+oracle)|lora_oracle", re.M)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                assert not pat.search(open(os.path.join(dirpath, f)).read()), f"{f} imports the oracle"
