"""Peak microbenchmarks for the rooflines of this library (sm_103a only).

Builds each probe in this directory with nvcc into a temporary directory and
runs it; every probe prints its own result.  Usage:

    python -m int8_head_kv_gb300.peaks [probe ...]

Probes: tcgen05_mma_rate (sustained kind::f16 MMA rate by N and A operand),
dsmem_exchange_rate (sustained 2-CTA st.async exchange), hbm_read_rate (HBM
read-only bandwidth), mma_sync_rate (warp-level s8 and f16 MMA rates).
"""
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
PROBES = ["tcgen05_mma_rate", "dsmem_exchange_rate", "hbm_read_rate", "mma_sync_rate"]


def main(argv):
    names = argv or PROBES
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    with tempfile.TemporaryDirectory() as tmp:
        for name in names:
            exe = os.path.join(tmp, name)
            subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                                   os.path.join(HERE, name + ".cu"), "-o", exe])
            print(f"== {name}", flush=True)
            subprocess.check_call([exe], timeout=300)


if __name__ == "__main__":
    main(sys.argv[1:])
