"""Concurrent first use from several host threads.

The library sets up each kernel once per device on first use (shared-memory
attributes, occupancy queries, the device error word's address, the
tensor-map encoder). Host threads that make their first calls at the same
time, each on its own stream with its own workspace, must all succeed and
produce the same bytes as the same calls made one at a time afterwards.

The threads run in a fresh interpreter, so that no set-up has happened yet
when they start; the weights are quantized by the oracle on the CPU for the
same reason. The calls cover the CTA-pair GEMM behind the cooperative
dynamic quantizer, the decode kernel behind the one-cluster quantizer, the
fused decode kernel, and the re-quantizing epilogue.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys, threading
import numpy as np
import torch
sys.path.insert(0, ROOT)
sys.path.insert(0, ROOT + "/tests")
import oracle
from helpers import bf16_bits, sf_rowmajor_to_mma
import nvfp4_block_scaled_28_b300 as nv
from nvfp4_block_scaled_28_b300 import workloads

oracle.build()
nv.load_library()
N_, K_ = 1024, 2048
w = workloads.make_w(N_, K_, seed=3)
wb = bf16_bits(w)
gw = oracle.global_scale(wb)
wq, ws = oracle.quantize(wb, gw)
Wq = torch.from_numpy(wq).cuda()
Ws = torch.from_numpy(sf_rowmajor_to_mma(ws)).cuda()
g_w = torch.tensor([np.float32(gw)], dtype=torch.float32, device="cuda")
bias = workloads.make_bias(N_, seed=4).cuda()

# (M, mode, requant): pair GEMM + cooperative quantizer, decode kernel +
# one-cluster quantizer, fused decode, decode kernel + the small quantizer,
# pair GEMM with the re-quantizing epilogue
JOBS = [(2048, 0, False), (64, 0, False), (4, 1, False), (16, 0, False), (256, 0, True)] * 2
xs = [workloads.make_x("outlier", M, K_, seed=10 + i).cuda() for i, (M, _, _) in enumerate(JOBS)]
torch.cuda.synchronize()

def call(i):
    M, mode, requant = JOBS[i]
    ws_t = torch.empty(nv.linear_workspace_bytes(M, N_, K_, mode), dtype=torch.uint8,
                       device="cuda")
    if requant:
        Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(xs[i], Wq, Ws, g_w, bias=bias,
                                                              workspace=ws_t)
        return [Y.view(torch.int16), g_y.view(torch.int32), Yq, Ys]
    return [nv.nvfp4_linear(xs[i], Wq, Ws, g_w, mode=mode, workspace=ws_t).view(torch.int16)]

start = threading.Barrier(len(JOBS))
got, errors = [None] * len(JOBS), []

def worker(i):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            start.wait()
            out = call(i)
        s.synchronize()
        got[i] = out
    except Exception as e:  # reported by the parent
        errors.append("job %d: %r" % (i, e))

threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(JOBS))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
torch.cuda.synchronize()
assert nv.nvfp4_device_error() == 0
for i in range(len(JOBS)):
    ref = call(i)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(got[i], ref)), "job %d differs" % i
print("threads ok")
"""


def test_concurrent_first_calls_from_host_threads():
    env = dict(os.environ)
    code = "ROOT = %r\n" % ROOT + _CHILD
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
