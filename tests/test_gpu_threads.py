"""Concurrent host threads: four threads, each on its own CUDA stream, make the process's
first library calls at the same time -- dense FFN (one persistent launch) and grouped
experts on the two-CTA schedule -- so the per-device launch caches (tensor-map encoder,
cluster occupancy, shared-memory opt-in) are filled concurrently.  Every thread's
outputs must equal, bit for bit, the same calls made afterwards from one thread.  The
calls run in a fresh Python process so that the caches start empty."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading, torch
sys.path.insert(0, ROOT)
import situ_glu_activation_gb300 as situ
from situ_glu_activation_gb300 import workloads as wl

dev = torch.device("cuda:0")
torch.cuda.set_device(dev)
M, I, R = 512, 384, 1000
x, wgu, wd = wl.ffn_inputs(M, I, R, seed=3, device=dev)
T, k, E = 600, 2, 2            # 1200 routes over 2 experts: the two-CTA grouped schedule
gx = wl.normal((T, M), 1.0, seed=4, device=dev)
gwgu, gwd = wl.expert_weights(E, M, I, seed=5, device=dev)
g = torch.Generator().manual_seed(6)
ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32).to(dev)
torch.cuda.synchronize()

N = 4
outs = [None] * N
errors = []
barrier = threading.Barrier(N)

def work(i):
    try:
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            barrier.wait()
            y = situ.situ_ffn_forward(x, wgu, wd)
            off, tix = situ.situ_moe_build_index(ids, E)
            gy = situ.situ_moe_grouped_forward(gx, off, tix, gwgu, gwd, k)
        s.synchronize()
        outs[i] = (y, gy)
    except Exception as e:  # reported below
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(N)]
for t in threads:
    t.start()
for t in threads:
    t.join()
if errors:
    print("ERROR", errors)
    sys.exit(1)
y_ref = situ.situ_ffn_forward(x, wgu, wd)
off, tix = situ.situ_moe_build_index(ids, E)
gy_ref = situ.situ_moe_grouped_forward(gx, off, tix, gwgu, gwd, k)
torch.cuda.synchronize()
for i, (y, gy) in enumerate(outs):
    if not torch.equal(y.view(torch.int16), y_ref.view(torch.int16)):
        print("MISMATCH dense", i)
        sys.exit(1)
    if not torch.equal(gy.view(torch.int16), gy_ref.view(torch.int16)):
        print("MISMATCH grouped", i)
        sys.exit(1)
st = situ.device_status(clear=True)
print("OK", st)
sys.exit(0 if st == 0 else 1)
"""


def test_concurrent_first_calls(cuda_dev):
    code = SCRIPT.replace("ROOT", repr(ROOT))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-2000:])
    assert "OK 0" in r.stdout
