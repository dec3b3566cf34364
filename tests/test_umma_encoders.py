"""CPU: the tcgen05 descriptor encoders of the GEMM (csrc/mx_umma.h), compiled
with the host C++ compiler and checked field by field against values worked out
by hand from the PTX ISA's descriptor tables (shared-memory matrix descriptor;
instruction descriptor of the block-scaled kinds). A wrong shift, a field in
the wrong place or a missing fixed bit changes one of these numbers."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mxfp8_block_scaled_rmsnorm_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "mx_umma.h"
using namespace mx::umma;
int main() {
    std::printf("%llx\n", (unsigned long long)smem_desc(0x400, 16, 1024, kSwizzle128B));
    std::printf("%llx\n", (unsigned long long)kmajor_sw128_desc(0x1C400));
    std::printf("%llx\n", (unsigned long long)scale_tile_desc(0x30200));
    std::printf("%x\n", idesc_mxf8(128, 256, 0, 0));
    std::printf("%x\n", idesc_mxf8(128, 256, 3, 1));
    std::printf("%x\n", idesc_mxf8(128, 128, 2, 2));
    std::printf("%x\n", tmem_addr(0x20, 96, 160));
    return 0;
}
"""


@pytest.fixture(scope="module")
def values(tmp_path_factory):
    d = tmp_path_factory.mktemp("umma")
    src, exe = d / "enc.cpp", d / "enc"
    src.write_text(PROGRAM)
    subprocess.run(["g++", "-std=c++17", "-O1", "-I" + CSRC, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    return [int(v, 16) for v in out.split()]


def fields64(d):
    return {"start": d & 0x3FFF, "lbo": (d >> 16) & 0x3FFF, "sbo": (d >> 32) & 0x3FFF,
            "fixed": (d >> 46) & 7, "base": (d >> 49) & 7, "lbo_mode": (d >> 52) & 1,
            "swizzle": (d >> 61) & 7, "reserved": ((d >> 14) & 3) | (((d >> 30) & 3) << 2)
            | (((d >> 53) & 0xFF) << 4)}


def test_shared_memory_descriptor(values):
    # start 0x400 >> 4, leading offset 16 >> 4, stride offset 1024 >> 4, the
    # fixed 0b001 at bit 46, 128-byte swizzle (2) at bit 61
    assert values[0] == 0x4000_4040_0001_0040
    f = fields64(values[0])
    assert f == {"start": 0x40, "lbo": 1, "sbo": 64, "fixed": 1, "base": 0, "lbo_mode": 0,
                 "swizzle": 2, "reserved": 0}
    # an operand tile of the GEMM: 8-row groups 1024 bytes apart, 128-byte swizzle
    assert values[1] == 0x4000_4040_0001_1C40
    # a scale tile: no swizzle, 8-row core matrices 128 bytes apart
    assert values[2] == 0x0000_4008_0000_3020
    assert fields64(values[2])["swizzle"] == 0 and fields64(values[2])["sbo"] == 8


def test_instruction_descriptor(values):
    # M = 128 (8 at bit 24), N = 256 (32 at bit 17), UE8M0 scales (bit 23),
    # E4M3 operands (formats 0), both K-major, no negation, dense
    assert values[3] == 0x08C0_0000
    # scale-factor ids: A at bits 29-30, B at bits 4-5
    assert values[4] == 0x68C0_0010
    assert (values[4] >> 29) & 3 == 3 and (values[4] >> 4) & 3 == 1
    assert values[5] == 0x48A0_0020
    assert (values[5] >> 17) & 0x3F == 128 >> 3 and (values[5] >> 24) & 0x1F == 128 >> 4


def test_tensor_memory_address(values):
    # lane in the high half-word, column in the low one
    assert values[6] == (96 << 16) + 0x20 + 160
