"""The C-ABI library loads without a GPU and exports every entry point that
include/exl3.h declares; the host-only size functions follow the layout."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "exl3.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t)\s+(exl3_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return ctypes.CDLL(os.path.join(ROOT, "trellis_quantized_moe_gb300", "_lib",
                                    "libexl3_gb300.so"))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_sizes(lib):
    import trellis_quantized_moe_gb300 as X
    assert X.exl3_abi_version() == 1
    assert X.exl3_moe_workspace_bytes(1, 8, 192, 5120, 1536, 512) > 0
    assert X.exl3_moe_workspace_bytes(1, 8, 192, 5000, 1536, 512) == 0   # not a multiple of 128
    assert X.exl3_moe_workspace_bytes(1, 8, 2000, 5120, 1536, 512) == 0  # too many experts
    a = X.exl3_moe_workspace_bytes(64, 8, 288, 4096, 1408, 512)
    b = X.exl3_moe_workspace_bytes(128, 8, 288, 4096, 1408, 512)
    assert a % 256 == 0 and b > a
    assert X.exl3_route_pack_max_tiles(16, 2, 8, 3) == 32 // 3 + 8
    assert X.exl3_linear_workspace_bytes(5, 640, 384) > 5 * 640 * 2
