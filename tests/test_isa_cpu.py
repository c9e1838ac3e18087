"""What the sm_103a compiler accepts: the evidence behind the integer contraction's
design.  tcgen05 has an 8-bit integer MMA kind on sm_100a but not on sm_103a
(GB300), so the exact integer latent score runs as kind::f16 MMAs on int8 codes
converted to fp16.  Only the compiler's verdict is read (its exit status and its
message); nothing it writes is inspected."""
import os
import shutil
import subprocess

import pytest

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

SRC = r'''
#include <cstdint>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::KIND [%0], %1, %2, %3, p;\n}\n"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
'''


def _compile(tmp_path, kind, arch):
    if not (os.path.exists(NVCC) or shutil.which("nvcc")):
        pytest.skip("nvcc not available")
    src = tmp_path / f"mma_{kind}_{arch}.cu"
    src.write_text(SRC.replace("KIND", kind))
    r = subprocess.run([NVCC if os.path.exists(NVCC) else "nvcc", "-gencode", f"arch=compute_{arch},code=sm_{arch}",
                        "-c", str(src), "-o", str(tmp_path / f"mma_{kind}_{arch}.o")],
                       capture_output=True, text=True)
    return r.returncode, r.stdout + r.stderr


def test_kind_i8_is_rejected_for_sm103a(tmp_path):
    rc, msg = _compile(tmp_path, "i8", "103a")
    assert rc != 0
    assert "kind::i8" in msg and "not supported" in msg and "sm_103a" in msg, msg


def test_kind_i8_is_accepted_for_sm100a(tmp_path):
    rc, msg = _compile(tmp_path, "i8", "100a")
    assert rc == 0, msg


def test_kind_f16_is_accepted_for_sm103a(tmp_path):
    rc, msg = _compile(tmp_path, "f16", "103a")
    assert rc == 0, msg
