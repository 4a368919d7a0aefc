"""The numeric constants written into the CUDA sources as literals are the
correctly rounded float32 values of their definitions, and the codebook
constants of both kernels are the ones the oracle documents (read from the
sources as text; no GPU)."""
import math
import os
import re

import numpy as np

from oracle import exl3_oracle as O

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "trellis_quantized_moe_gb300", "csrc")


def _src(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def _float_literal(text, name):
    m = re.search(r"constexpr\s+float\s+" + name + r"\s*=\s*([0-9.eE+-]+)f\s*;", text)
    assert m, name
    return np.float32(float(m.group(1)))


def test_float_literals_are_correctly_rounded():
    common = _src("common.cuh")
    assert _float_literal(common, "kInvSqrt128") == np.float32(1.0 / math.sqrt(128.0))
    assert _float_literal(common, "kInvSqrtMul1") == np.float32(1.0 / math.sqrt(21845.0))
    assert _float_literal(common, "kSqrtMul1") == np.float32(math.sqrt(21845.0))


def test_codebook_constants_match_the_oracle():
    gemm = _src("expert_gemm.cuh")
    tc = _src("expert_tc.cuh")
    common = _src("common.cuh")
    for text in (gemm, tc):
        assert f"0x{O.A_MUL1:08X}u" in text
        assert f"0x{O.A_MCG:08X}u" in text
        assert f"{O.A_3INST}u" in text
    assert f"{O.B_3INST}u" in gemm and f"{O.B_3INST}u" in tc
    # the mask and exponent flip both kernels apply (held in registers)
    assert f"0x{O.HALF_MASK:08X}u" in common and f"0x{O.HALF_XOR:08X}u" in common
