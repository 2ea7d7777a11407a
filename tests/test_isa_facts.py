"""Facts about the sm_103a instruction set that the GEMM design rests on.

The tensor-core GEMM computes its exact integer block sums with
tcgen05.mma kind::f16 on small integers, not with an int8 MMA, because the
PTX assembler rejects tcgen05.mma kind::i8 for sm_103a while it accepts it
for sm_100a.  These tests keep that on record by compiling a one-instruction
kernel for both targets (CPU only: nvcc cross-compiles without a GPU).  A
control kernel with kind::f16 must assemble for sm_103a, so a failure of the
first test cannot come from a broken toolchain.
"""
import os
import shutil
import subprocess

import pytest

NVCC = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc"
                                if os.path.exists("/usr/local/cuda/bin/nvcc") else None)

pytestmark = pytest.mark.skipif(NVCC is None, reason="nvcc not found")

_MMA_SRC = r"""
#include <cstdint>
__global__ void one_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}\n"
                 :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(0u));
}
"""


def _compile(tmp_path, kind, arch):
    src = tmp_path / f"mma_{kind}_{arch}.cu"
    src.write_text(_MMA_SRC.replace("KIND", kind))
    r = subprocess.run([NVCC, "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", str(src),
                        "-o", str(tmp_path / f"mma_{kind}_{arch}.o")],
                       capture_output=True, text=True, timeout=300)
    return r.returncode, r.stdout + r.stderr


def test_int8_mma_is_rejected_on_sm_103a(tmp_path):
    rc, out = _compile(tmp_path, "i8", "103a")
    assert rc != 0
    assert "kind::i8" in out and "not supported" in out and "sm_103a" in out, out


def test_int8_mma_assembles_on_sm_100a(tmp_path):
    rc, out = _compile(tmp_path, "i8", "100a")
    assert rc == 0, out


def test_f16_mma_assembles_on_sm_103a(tmp_path):
    rc, out = _compile(tmp_path, "f16", "103a")
    assert rc == 0, out
