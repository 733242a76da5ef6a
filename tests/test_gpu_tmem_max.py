"""The row maxima the attention kernel takes from the TMEM loads themselves
(sm_103a `tcgen05.ld.red ... .max.f32`: the load returns, with the 32 scores of
a key block, their largest value).  A check build of the kernel
(SAGEATTN_CHECK_TMEM_MAX) also forms every unmasked tile's maximum from the
loaded scores and sets a device error bit if the two differ, then continues
with the software value.  This test compiles that build, links it with the
library's other objects and runs all three modes over several shapes in a
child process (the binding loads one library per process); a mismatch
surfaces as an error status."""
import os
import subprocess
import sys

import pytest

from sage_attention_forward_gb300 import build as lib_build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[2]); sys.path.insert(0, sys.argv[2] + "/tests")
import torch
import sage_attention_forward_gb300 as sa
sa._LIB_PATH = sys.argv[1]
from workloads import make_inputs, small_case, to_device
for (B, H, S, kw) in [(1, 2, 1000, {}), (2, 3, 1536, {}), (1, 2, 4000, dict(outlier_frac=0.05, outlier_gain=8.0)),
                      (1, 4, 3000, dict(k_channel_offset_std=2.0))]:
    g = to_device(make_inputs(small_case(B, H, S, 90 + S, **kw)), "cuda")
    sa.attn_fwd_bf16(g.q, g.k, g.v)
    sa.sage_attention(g.q, g.k, g.v)
    sa.sage_attention(g.q, g.k, g.v, pv="bf16")
    torch.cuda.synchronize()
    sa.attn_get_device_status()
print("tmem maxima agree")
'''


def test_tmem_load_maxima_match_the_loaded_scores(cuda_dev):
    lib_build.build()
    out = os.path.join(lib_build.OUT_DIR, "check")          # in-tree, next to the library
    os.makedirs(out, exist_ok=True)
    obj = os.path.join(out, "attn_fwd_check.o")
    so = os.path.join(out, "libsageattn_check.so")
    cmd = [lib_build.nvcc()] + lib_build._flags(["-DSAGEATTN_CHECK_TMEM_MAX"]) + [
        "-c", os.path.join(lib_build.CSRC, "attn_fwd.cu"), "-o", str(obj)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    others = [os.path.join(lib_build.OUT_DIR, f) for f in ("api.o", "sage_prepare.o")]
    r = subprocess.run([lib_build.nvcc()] + lib_build.ARCH + ["-shared", "-o", str(so), str(obj)] + others + ["-lcudart"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([sys.executable, "-c", CHILD, str(so), ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "tmem maxima agree" in r.stdout, (r.stdout[-1000:], r.stderr[-3000:])
