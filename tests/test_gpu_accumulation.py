"""What the FP8 tensor-core accumulator keeps on this GPU (a hardware property, measured with
the kernels' own MMA helpers and the PV operand layout they use).

The FP8 Hopper forward adds each KV tile's PV to an fp32 O ("two-level accumulation")
because the Hopper FP8 accumulator keeps too few bits, which made O shrink at long key
lengths.  ``tcgen05_accumulation_probe.cu`` presets the TMEM accumulator to L and adds 128
products through four accumulating kind::f8f6f4 MMAs: the sums come out as fp32 arithmetic
gives them, so that failure mode does not exist on tcgen05.  The kernels keep the two-level
fold because the method specifies it; this test records why it is not needed for accuracy.
"""
import os
import subprocess

import pytest

from fp8_attention_forward_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("acc") / "acc_probe")
    cmd = [build.nvcc(), *build.ARCH, "-O2", "-std=c++17", "-I", os.path.join(build.ROOT, "include"),
           "-I", build.CSRC, "-o", exe, os.path.join(HERE, "tcgen05_accumulation_probe.cu"), "-lcuda"]
    subprocess.run(cmd, check=True, capture_output=True, timeout=600)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    res = {}
    for line in out.strip().splitlines():
        name, L, add, lo, hi, once, st = line.split("|")
        res[(name, float(L))] = dict(add=float(add), lo=float(lo), hi=float(hi), once=float(once), status=int(st))
    return res


def test_every_element_agrees_and_no_wait_timed_out(probe):
    for key, r in probe.items():
        assert r["status"] == 0 and r["lo"] == r["hi"], key


def test_small_products_survive_on_large_accumulators(probe):
    """128 x (1 * 2^-9) = 0.25 added onto L = 0 .. 2^16 is exact: 24 significant bits, where an
    accumulator with Hopper's FP8 precision loses the addends well before L = 2^16."""
    for L in (0.0, 16.0, 256.0, 4096.0, 65536.0):
        r = probe[("128 x (1 * 2^-9) onto L", L)]
        assert r["hi"] == L + 0.25, (L, r)
    for L in (0.0, 4096.0, 65536.0):
        r = probe[("128 x (1 * 0.5) onto L", L)]
        assert r["hi"] == L + 64.0, (L, r)


def test_mixed_magnitudes_inside_one_mma(probe):
    """256 * 1 plus 127 products of 2^-9 in one accumulation chain: exact in fp32."""
    r = probe[("256*1 + 127 x (1 * 2^-9), one MMA set", 0.0)]
    assert r["hi"] == 256.0 + 127.0 / 512.0, r
