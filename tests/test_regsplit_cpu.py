"""Register budgets of the kernels' setmaxnreg splits, checked on the CPU.

Each kernel launches with one CTA per SM, so ptxas gives every thread the largest register
count that fits the 65536-register file, rounded down to a multiple of 8.  One warpgroup
then raises its count with setmaxnreg.inc and every other warp lowers it with
setmaxnreg.dec.  An increase waits until the decreases have released enough registers, so
a split whose total exceeds the launch's registers would never proceed.  This test reads the
thread counts and the two register counts from the kernel sources and checks:

- the total fits the launch;
- both counts are multiples of 8 within setmaxnreg's range of 24 to 256;
- the raised count is at least, and the lowered count at most, the launch count.
"""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(__file__), "..", "sparse_mla_attention_fwd_gb300", "csrc")
REGISTER_FILE = 65536


def constant(text, name):
    m = re.search(r"constexpr\s+int\s+" + name + r"\s*=\s*(\d+)\s*;", text)
    assert m, f"{name} not found"
    return int(m.group(1))


def launch_registers(threads):
    return (REGISTER_FILE // threads) // 8 * 8


@pytest.mark.parametrize("source, threads, raised, lowered", [
    ("sparse_mla_fwd.cu", "kThreads", "kSoftmaxRegs", "kOtherRegs"),
    ("sparse_mla_bwd.cuh", "kBwdThreads", "kBwdMathRegs", "kBwdOtherRegs"),
])
def test_setmaxnreg_split_fits_the_launch(source, threads, raised, lowered):
    text = open(os.path.join(CSRC, source)).read()
    n, hi, lo = constant(text, threads), constant(text, raised), constant(text, lowered)
    assert n % 128 == 0 and 128 < n <= 1024
    launch = launch_registers(n)
    for r in (hi, lo):
        assert r % 8 == 0 and 24 <= r <= 256
    assert lo <= launch <= hi
    # one warpgroup (128 threads) raised, the rest lowered
    assert 128 * hi + (n - 128) * lo <= n * launch
    # each count is used in exactly one setmaxnreg of the source
    assert text.count(f"reg_alloc<{raised}>") == 1
    assert text.count(f"reg_dealloc<{lowered}>") == 1


def test_launch_register_rule():
    # 512 threads get 128 registers each; 768 get 85, rounded down to 80
    assert launch_registers(512) == 128
    assert launch_registers(768) == 80
