"""Bit layouts of the tcgen05 operand and instruction descriptors (CPU).

The library's encoders (csrc/kvc_tc.cuh) are compiled as host code with nvcc
and their outputs compared with fields assembled here from the PTX ISA's
tables: the shared-memory matrix descriptor (start address, leading and
stride byte offsets in 16-byte units, version 1 at bit 46, swizzle mode at
bits 61..63) and the kind::f16 instruction descriptor (f32 accumulator,
A/B type, major-ness, N >> 3 at bit 17, M >> 4 at bit 24).  A field moved by
one bit, a missing >> 4, or M and N exchanged fails here before any kernel
runs on a GPU.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "paged_kv_cache_kvc_gb300", "csrc", "kvc_tc.cuh")

SMEM_CASES = [(0x0, 16, 1024, 2), (0x1F0, 16, 1024, 2), (0x12340, 16384, 1024, 2), (0x30000, 8192, 1024, 2),
              (0x4000, 0, 512, 4), (0x8000, 2048, 256, 6), (0x10, 4096, 128, 0)]
ADVANCE_OFFSETS = [32, 96, 2048, 16384 + 96, 14336]
IDESC_CASES = [(128, 32, True, False, False), (128, 64, True, True, True), (128, 128, True, False, True),
               (64, 256, False, False, False), (128, 16, True, True, False), (256, 8, False, False, True)]

PROGRAM = r"""
#include <cstdio>
#include "%s"
int main() {
%s
  return 0;
}
"""


def _field(value, lsb, width):
    assert 0 <= value < (1 << width), (value, width)
    return value << lsb


def _smem_expected(addr, lbo, sbo, swizzle):
    return (_field((addr >> 4) & 0x3FFF, 0, 14) | _field((lbo >> 4) & 0x3FFF, 16, 14) |
            _field((sbo >> 4) & 0x3FFF, 32, 14) | _field(1, 46, 2) | _field(swizzle, 61, 3))


def _idesc_expected(M, N, bf16, a_mn, b_mn):
    t = 1 if bf16 else 0
    return (_field(1, 4, 2) | _field(t, 7, 3) | _field(t, 10, 3) | _field(int(a_mn), 15, 1) |
            _field(int(b_mn), 16, 1) | _field(N >> 3, 17, 6) | _field(M >> 4, 24, 5))


@pytest.fixture(scope="module")
def encoded():
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = shutil.which("nvcc")
    if not nvcc:
        pytest.skip("nvcc not available")
    lines = []
    for (a, l, s, z) in SMEM_CASES:
        lines.append(f'  printf("%llx\\n", (unsigned long long)kvc::tc_smem_desc({a}u, {l}u, {s}u, {z}u));')
    for (m, n, bf, am, bm) in IDESC_CASES:
        lines.append(f'  printf("%x\\n", kvc::tc_idesc_f16({m}, {n}, {str(bf).lower()}, {str(am).lower()}, '
                     f'{str(bm).lower()}));')
    for r in range(16):
        for c in range(8):
            lines.append(f'  printf("%u\\n", kvc::sw128({r}u, {c}u));')
    for (a, l, s_, z) in SMEM_CASES:
        for off in ADVANCE_OFFSETS:
            lines.append(f'  printf("%d\\n", (int)(kvc::tc_desc_advance(kvc::tc_smem_desc({a}u, {l}u, {s_}u, {z}u), '
                         f'{off}u) == kvc::tc_smem_desc({a + off}u, {l}u, {s_}u, {z}u)));')
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "enc.cu")
        with open(src, "w") as f:
            f.write(PROGRAM % (HEADER, "\n".join(lines)))
        exe = os.path.join(d, "enc")
        subprocess.check_call([nvcc, "-std=c++17", "-o", exe, src], cwd=d)
        out = subprocess.check_output([exe], text=True).split()
    return out


def test_shared_memory_descriptor_fields(encoded):
    for i, case in enumerate(SMEM_CASES):
        assert int(encoded[i], 16) == _smem_expected(*case), case


def test_instruction_descriptor_fields(encoded):
    off = len(SMEM_CASES)
    for i, case in enumerate(IDESC_CASES):
        assert int(encoded[off + i], 16) == _idesc_expected(*case), case


def test_128_byte_swizzle_chunk_placement(encoded):
    """Chunk c of row r sits at chunk c ^ (r mod 8) of the row: every row holds
    each chunk once, and a column of 8 rows spreads one chunk over 8 places."""
    off = len(SMEM_CASES) + len(IDESC_CASES)
    vals = [int(x) for x in encoded[off:]]
    for r in range(16):
        row = vals[r * 8:(r + 1) * 8]
        assert sorted(row) == [r * 128 + 16 * c for c in range(8)]
        for c in range(8):
            assert row[c] == r * 128 + 16 * (c ^ (r % 8))


def test_descriptor_advance_moves_only_the_start_address(encoded):
    """Stepping a descriptor along K (32 bytes inside a 128-byte band) or along rows (2 KiB
    per 16 rows) equals encoding the moved address: nothing carries out of the start field."""
    off = len(SMEM_CASES) + len(IDESC_CASES) + 16 * 8
    assert all(int(x) == 1 for x in encoded[off:off + len(SMEM_CASES) * len(ADVANCE_OFFSETS)])
