"""Concurrent first calls from several host threads.

The library keeps a few things per CUDA context that its first call fills in: the
kernels' shared-memory attributes, the device's SM count, the device check and the
tensor-map encoder.  This runs, in a fresh process whose library has made no call yet,
eight host threads that start together and each make their first calls (the BF16
forward, the one-call Sage op and its 16-bit P V mode) on a stream of their own;
ctypes drops the interpreter lock for the duration of a call, so the C side runs
concurrently.  Every output must equal, bit for bit, the same call made afterwards
from one thread.
"""
import os
import subprocess
import sys

import pytest

SCRIPT = r"""
import sys, threading
import torch
sys.path.insert(0, sys.argv[1])
import sage_attention_forward_gb300 as sa
from workloads import make_inputs, small_case

dev = torch.device("cuda:0")
inp = make_inputs(small_case(1, 3, 700, 4242))
q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
torch.cuda.synchronize()
sa.lib()                      # the shared object only: no library call has run yet
N = 8
calls = [lambda s: sa.attn_fwd_bf16(q, k, v, stream=s),
         lambda s: sa.sage_attention(q, k, v, stream=s),
         lambda s: sa.sage_attention(q, k, v, pv="bf16", stream=s)]
outs, errs = [None] * N, []
start = threading.Barrier(N)

def work(t):
    try:
        s = torch.cuda.Stream(dev)
        start.wait()
        with torch.cuda.stream(s):
            o = calls[t % 3](s)
        s.synchronize()
        outs[t] = o
    except Exception as e:   # reported below
        errs.append(f"thread {t}: {e!r}")

threads = [threading.Thread(target=work, args=(t,)) for t in range(N)]
for th in threads:
    th.start()
for th in threads:
    th.join()
assert not errs, errs
sa.attn_get_device_status()
ref = [c(torch.cuda.current_stream(dev)) for c in calls]
torch.cuda.synchronize()
for t in range(N):
    assert torch.equal(outs[t], ref[t % 3]), f"thread {t} differs"
print("threads ok")
"""


@pytest.mark.gpu
def test_concurrent_first_calls_from_host_threads(cuda_dev, tmp_path):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "threads.py"
    script.write_text(SCRIPT)
    r = subprocess.run([sys.executable, str(script), root], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
