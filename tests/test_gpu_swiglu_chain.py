"""Exhaustive error bounds of the SwiGLU fast path (the packed fp32 chain the
fused kernels certify with rounding intervals): compiles
tests/probes/swiglu_chain.cu against the kernels' own numerics header and
runs it on every bf16 g.  The parity tests compare outputs with the oracle;
this proves the certification margins for all inputs, not only the sampled
ones."""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "block_scaled_mlp_gb300", "csrc")


def test_fast_path_bounds_every_bf16_g():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "swiglu_chain")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-I", CSRC,
                        os.path.join(HERE, "probes", "swiglu_chain.cu"), "-o", exe], check=True,
                       capture_output=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    out = r.stdout
    assert r.returncode == 0, out + r.stderr
    t_ulp = float(re.search(r"t max ulp ([0-9.]+)", out).group(1))
    silu = re.search(r"silu: (\d+) certified, (\d+) wrong", out)
    dg = re.search(r"dg: (\d+) g on the fast path, max needed/margin ([0-9.]+), (\d+) with needed >= margin, "
                   r"(\d+) sign errors", out)
    print(out)
    assert t_ulp < 2.6, out
    assert int(silu.group(1)) > 30000 and int(silu.group(2)) == 0, out
    assert int(dg.group(1)) > 30000 and float(dg.group(2)) < 0.5 and int(dg.group(3)) == 0, out
    assert int(dg.group(4)) == 0, out
