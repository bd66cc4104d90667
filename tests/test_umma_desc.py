"""The tcgen05 operand descriptors (umma_desc.h), checked field by field on the CPU.

The header's two encoders are compiled here with the host C++ compiler and their outputs
decoded with the bit positions of the public PTX ISA tables ("Matrix Descriptors" for
tcgen05: the shared-memory matrix descriptor and the instruction descriptor of kind::f16),
written out again below independently of the header.  One test per field, plus the bits that
must stay zero.  No GPU is needed.
"""

from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER_DIR = ROOT / "paged_kv_cache_244_gb300" / "csrc"

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include "umma_desc.h"
int main(int argc, char** argv) {
  if (argc == 5 && argv[1][0] == 's') {
    unsigned long long d = pa::umma_smem_desc(strtoul(argv[2], 0, 0), strtoul(argv[3], 0, 0),
                                              strtoul(argv[4], 0, 0));
    printf("%llu\n", d);
  } else if (argc == 6 && argv[1][0] == 'i') {
    unsigned d = pa::umma_idesc_bf16(atoi(argv[2]), atoi(argv[3]), atoi(argv[4]) != 0,
                                     atoi(argv[5]) != 0);
    printf("%u\n", d);
  } else {
    return 2;
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def encoder(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("umma")
    src = d / "enc.cpp"
    src.write_text(PROGRAM)
    exe = d / "enc"
    subprocess.run([cxx, "-std=c++17", "-O1", f"-I{HEADER_DIR}", str(src), "-o", str(exe)], check=True)

    def smem(addr, lbo, sbo):
        return int(subprocess.run([str(exe), "s", str(addr), str(lbo), str(sbo)], check=True,
                                  capture_output=True, text=True).stdout)

    def idesc(m, n, a_mn, b_mn):
        return int(subprocess.run([str(exe), "i", str(m), str(n), str(int(a_mn)), str(int(b_mn))],
                                  check=True, capture_output=True, text=True).stdout)

    return smem, idesc


def field(x, lo, hi):
    """Bits lo .. hi - 1 of x."""
    return (x >> lo) & ((1 << (hi - lo)) - 1)


# ---- shared-memory matrix descriptor -------------------------------------------------------

SMEM_CASES = [(0x0, 16, 1024), (0x400, 2048, 1024), (0x12340, 16, 1024), (0x3FFF0, 0x3FFF0, 0x3FFF0),
              (0x1C400 + 96, 16, 1024)]


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_start_address(encoder, addr, lbo, sbo):
    smem, _ = encoder
    assert field(smem(addr, lbo, sbo), 0, 14) == addr >> 4


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_leading_byte_offset(encoder, addr, lbo, sbo):
    smem, _ = encoder
    assert field(smem(addr, lbo, sbo), 16, 30) == lbo >> 4


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_stride_byte_offset(encoder, addr, lbo, sbo):
    smem, _ = encoder
    assert field(smem(addr, lbo, sbo), 32, 46) == sbo >> 4


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_version_is_one(encoder, addr, lbo, sbo):
    smem, _ = encoder
    assert field(smem(addr, lbo, sbo), 46, 48) == 1


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_base_offset_and_lbo_mode_zero(encoder, addr, lbo, sbo):
    smem, _ = encoder
    d = smem(addr, lbo, sbo)
    assert field(d, 49, 52) == 0      # swizzle pattern anchored at a 1024-byte boundary
    assert field(d, 52, 53) == 0      # leading offset is a relative byte offset


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_swizzle_is_128_byte(encoder, addr, lbo, sbo):
    smem, _ = encoder
    assert field(smem(addr, lbo, sbo), 61, 64) == 2


@pytest.mark.parametrize("addr,lbo,sbo", SMEM_CASES)
def test_smem_desc_reserved_bits_zero(encoder, addr, lbo, sbo):
    smem, _ = encoder
    d = smem(addr, lbo, sbo)
    for lo, hi in ((14, 16), (30, 32), (48, 49), (53, 61)):
        assert field(d, lo, hi) == 0, (lo, hi)


# ---- instruction descriptor, kind::f16 with bf16 operands ----------------------------------

IDESC_CASES = [(128, 32, False, False), (128, 128, False, True), (128, 16, False, False),
               (64, 256, True, False), (128, 256, True, True), (64, 8, False, False)]


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_sparsity_and_saturate_zero(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    assert field(idesc(m, n, a_mn, b_mn), 0, 4) == 0


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_accumulator_f32(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    assert field(idesc(m, n, a_mn, b_mn), 4, 6) == 1


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_a_and_b_bf16(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    d = idesc(m, n, a_mn, b_mn)
    assert field(d, 7, 10) == 1 and field(d, 10, 13) == 1   # same type on both sides


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_no_negation(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    assert field(idesc(m, n, a_mn, b_mn), 13, 15) == 0


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_major_bits(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    d = idesc(m, n, a_mn, b_mn)
    assert field(d, 15, 16) == int(a_mn) and field(d, 16, 17) == int(b_mn)


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_n_dimension(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    assert field(idesc(m, n, a_mn, b_mn), 17, 23) == n >> 3


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_m_dimension(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    assert field(idesc(m, n, a_mn, b_mn), 24, 29) == m >> 4


@pytest.mark.parametrize("m,n,a_mn,b_mn", IDESC_CASES)
def test_idesc_reserved_and_shift_zero(encoder, m, n, a_mn, b_mn):
    _, idesc = encoder
    d = idesc(m, n, a_mn, b_mn)
    assert field(d, 6, 7) == 0 and field(d, 23, 24) == 0 and field(d, 29, 32) == 0


def test_idesc_prefill_words(encoder):
    """The two words the prefill kernel issues, assembled by hand from the table: S = Q K^T
    (M 128, N 32, both K-major) and O += P V (M 128, N 128, V with N contiguous)."""
    _, idesc = encoder
    s_word = (1 << 4) | (1 << 7) | (1 << 10) | ((32 >> 3) << 17) | ((128 >> 4) << 24)
    pv_word = (1 << 4) | (1 << 7) | (1 << 10) | (1 << 16) | ((128 >> 3) << 17) | ((128 >> 4) << 24)
    assert idesc(128, 32, False, False) == s_word == 0x08080490
    assert idesc(128, 128, False, True) == pv_word == 0x08210490
