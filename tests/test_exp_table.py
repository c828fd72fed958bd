"""The route kernel's gate arithmetic rests on constants in
combine_moe_plan_gb300/csrc/exp_table.inc (written by gen_exp_table.py):
the committed file must be exactly what the generator writes, and the values
must have the accuracy the kernel's error bound assumes.  Host only."""
import os
import re
import subprocess
import sys

import pytest

mpmath = pytest.importorskip("mpmath")

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "combine_moe_plan_gb300", "csrc")
INC = os.path.join(CSRC, "exp_table.inc")


def _hexf(tok: str) -> float:
    tok = tok.rstrip("f")
    return 0.0 if tok in ("0.0", "-0.0") else float.fromhex(tok)


def test_committed_table_is_the_generators_output():
    out = subprocess.run([sys.executable, os.path.join(CSRC, "gen_exp_table.py")], capture_output=True, text=True,
                         check=True).stdout
    assert out == open(INC).read()


def test_table_and_ln2_split_accuracy():
    import numpy as np
    mpmath.mp.dps = 60
    src = open(INC).read()
    entries = re.findall(r"\{(\S+), (\S+)\},  // m = (-?\d+)", src)
    assert len(entries) == 361 and int(entries[0][2]) == -180 and int(entries[-1][2]) == 180
    worst = mpmath.mpf(0)
    for hi, lo, m in entries:
        h, l_ = _hexf(hi), _hexf(lo)
        assert float(np.float32(h)) == h and float(np.float32(l_)) == l_  # both are fp32 values
        assert abs(l_) <= abs(h) * 2.0 ** -24                             # a normalised pair
        e = mpmath.exp(mpmath.mpf(int(m)) / 512)
        worst = max(worst, abs(mpmath.mpf(h) + mpmath.mpf(l_) - e) / e)
    assert worst < mpmath.mpf(2) ** -49  # the kernel's bound takes 2^-49.1
    a, b, c = (_hexf(re.search(rf"{n} = (\S+);", src).group(1)) for n in ("kLn2A", "kLn2B", "kLn2C"))
    assert (a * 2 ** 16).is_integer() and 2 ** 15 <= a * 2 ** 16 < 2 ** 16  # 16 significant bits
    assert abs(mpmath.mpf(a) + b + c - mpmath.log(2)) < mpmath.mpf(2) ** -64
    inv = _hexf(re.search(r"kInvLn2 = (\S+);", src).group(1))
    assert abs(inv - 1 / float(mpmath.log(2))) < 2 ** -23


def test_reduction_range_stays_inside_the_table():
    """|r| <= ln2/2 plus the reduction's slack after n = rint(d / ln2) with
    the fp32 1/ln2; m = rint(512 r) must stay within [-180, 180]."""
    import math
    slack = 64 * 2 ** -23  # |d| <= 64 times the relative error of kInvLn2 and the product
    assert round(512 * (math.log(2) / 2 * (1 + slack) + 2 ** -18)) <= 178
