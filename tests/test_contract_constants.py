"""Constants of the numerical contract, checked against the mathematics."""

import os
import re
import struct
from decimal import Decimal, getcontext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CONTRACT = os.path.join(ROOT, "bitwise_aligned_causal_gb300", "csrc", "kb_contract.cuh")


def test_score_scale_is_log2e_over_sqrt128_rounded_to_fp32():
    getcontext().prec = 60
    exact = (Decimal(1) / Decimal(2).ln()) / Decimal(128).sqrt()
    want = struct.unpack("<I", struct.pack("<f", float(exact)))[0]
    # the double nearest `exact` rounds to the same fp32 as `exact` itself here:
    # check that `exact` is not within double precision of an fp32 halfway point
    f = struct.unpack("<f", struct.pack("<I", want))[0]
    up = struct.unpack("<f", struct.pack("<I", want + 1))[0]
    dn = struct.unpack("<f", struct.pack("<I", want - 1))[0]
    assert abs(Decimal(f) - exact) < abs(Decimal(up) - exact)
    assert abs(Decimal(f) - exact) < abs(Decimal(dn) - exact)
    text = open(CONTRACT).read()
    m = re.search(r"kScoreScaleLog2Bits\s*=\s*(0x[0-9A-Fa-f]+)u", text)
    assert m, "scale constant not found in kb_contract.cuh"
    assert int(m.group(1), 16) == want == 0x3E0293EE


def test_tile_constants():
    text = open(CONTRACT).read()
    for name, val in (("kHeadDim", 128), ("kTileKeys", 128), ("kTileRows", 128), ("kGroup", 4)):
        m = re.search(rf"constexpr int {name}\s*=\s*(\d+);", text)
        assert m and int(m.group(1)) == val
