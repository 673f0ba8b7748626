"""Several host threads making the library's first launches at the same time.

The library keeps kernel attributes, resident CTA-pair counts and SM counts per device,
set up by whichever call comes first.  A fresh child process (so that nothing is set up
yet) starts four threads behind a barrier; each makes its own calls on its own stream —
the projection engine on CTA pairs, the top-K cache, the fused forward — and the results
must equal those of the same calls made one after another afterwards.  ctypes releases the
interpreter lock during each call, so the threads really are inside the library together.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import threading
import torch
import sparse_teacher_kl_gb300 as kd
from synth import Workload, make_dense_teacher_logits, make_inputs

dev = torch.device("cuda:0")
torch.cuda.init()

def job(i, stream):
    """One thread's calls on `stream`: returns the outputs to compare."""
    g = torch.Generator(device=dev).manual_seed(100 + i)
    out = {}
    with torch.cuda.stream(stream):
        A = torch.randn((512, 320), generator=g, device=dev).to(torch.bfloat16)
        B = torch.randn((768, 320), generator=g, device=dev).to(torch.bfloat16)
        C, _ = kd.gemm_bf16(A, B, 512, 768, 320)
        X = make_dense_teacher_logits(700, 9000, seed=7 + i, device=dev)
        ids, vals = kd.topk_cache(X, 100)
        w = Workload("thr", 1, 384, 256, 4096, 16, 128, "zipf", 0.9, 2000 + i)
        H, W, tid, tlog, mask = make_inputs(w, dev)
        loss, lse, ws = kd.fused_kl_forward(H, W, tid, tlog, mask, chunk=128)
        stream.synchronize()
        out.update(C=C, ids=ids, vals=vals, loss=loss, lse=lse)
        assert kd.device_error(ws) == (0, 0)
    return out

streams = [torch.cuda.Stream(dev) for _ in range(4)]
barrier = threading.Barrier(4)
results, errors = [None] * 4, []

def run(i):
    try:
        barrier.wait()
        results[i] = job(i, streams[i])
    except Exception as e:  # reported below
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(4)]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
torch.cuda.synchronize()
for i in range(4):
    ref = job(i, torch.cuda.current_stream(dev))
    for k, v in ref.items():
        assert torch.equal(results[i][k], v), (i, k)
print("threads ok")
'''


def test_first_launches_from_four_threads(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "threads ok" in r.stdout
