"""The checked build (KD_DEBUG, libkdkl_debug.so): kernels check the indices they compute
and report one out of range through the workspace error word instead of using it.

Runs, in a child process that loads the checked library, the cases that stress those
indices most: top-K rows where every element becomes a candidate (ascending values),
rows of one value (ties everywhere), both warp-per-row buffer sizes and the block kernel
for K > 256, warps of several rows whose speculative starts miss (their first 4096 values
far above the rest), the fused teacher projection, and a fused fwd + bwd.  Every result
must match the oracle and every error word must stay clean.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import numpy as np
import torch

import oracle
import sparse_teacher_kl_gb300 as kd
from synth import WORKLOADS, Workload, bf16_bits, make_dense_teacher_logits, make_inputs

assert kd._abi.LIB_PATH.endswith("libkdkl_debug.so"), kd._abi.LIB_PATH
dev = torch.device("cuda:0")
stream = torch.cuda.current_stream().cuda_stream


def device_error(ws):
    st, detail = kd.device_error(ws)
    assert st == 0, f"device error {st}, detail {detail:#x}"


def topk_case(X, K):
    N, V = X.shape
    Xd = X.to(dev)
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = kd.workspace(kd._abi.kd_topk_cache_workspace(N, V, K), dev)
    dropped = torch.empty((N,), dtype=torch.float32, device=dev)
    st = kd._abi.kd_topk_cache(Xd.data_ptr(), N, V, V, K, ids.data_ptr(), vals.data_ptr(), None, dropped.data_ptr(),
                               ws.data_ptr(), ws.numel(), stream)
    assert st == 0
    device_error(ws)
    rid, rval = oracle.topk_cache(bf16_bits(X), K)
    assert np.array_equal(ids.cpu().numpy(), rid), (N, V, K)
    assert np.array_equal(vals.cpu().numpy().view(np.uint32), rval.view(np.uint32)), (N, V, K)


g = torch.Generator().manual_seed(11)
for (N, V, K) in [(300, 20000, 100), (64, 9000, 200), (8, 40000, 1024)]:
    X = make_dense_teacher_logits(N, V, seed=N + V + K)
    X[0] = torch.linspace(-4, 4, V)       # ascending: every element is a candidate
    X[1] = 0.75                           # one value everywhere
    X[2, ::3] = -0.0
    topk_case(X.to(torch.bfloat16), K)

# several rows per warp with scales jumping between rows, rows of few values, and rows whose
# first 4096 values sit far above the rest: speculative starts that miss, and the selection
# of such a row a second time from its exact bound
N, V = 5000, 12000  # rows 16-byte aligned (ld = V)
X = torch.randn((N, V), generator=g) * 10.0 ** (torch.rand((N, 1), generator=g) * 4 - 2)
X[1::5] = torch.randint(-2, 3, (len(range(1, N, 5)), V), generator=g).float()
X[0::3, :4096] += 6.0 * X[0::3].std(dim=1, keepdim=True)
topk_case(X.to(torch.bfloat16), 100)

# teacher projection + top-K with exact small-integer logits
N, dt, V, K = 300, 64, 3000, 50
Ht = torch.randint(-2, 3, (N, dt), generator=g).to(torch.bfloat16)
Wt = torch.randint(-2, 3, (V, dt), generator=g).to(torch.bfloat16)
ws = kd.workspace(kd._abi.kd_teacher_topk_workspace(N, dt, V, K, 128), dev)
ids, vals = kd.teacher_topk(Ht.to(dev), Wt.to(dev), K, chunk=128, ws=ws)
device_error(ws)
logits = oracle.teacher_logits_bf16(bf16_bits(Ht), bf16_bits(Wt))
rid, rval = oracle.topk_cache(logits, K)
assert np.array_equal(ids.cpu().numpy(), rid)
assert np.array_equal(vals.cpu().numpy(), rval)

# fused fwd + bwd on the tiny workload
w = WORKLOADS["tiny"]
H, W, tid, tlog, mask = make_inputs(w)
Hd, Wd, idd, tld = H.to(dev), W.to(dev), tid.to(dev), tlog.to(dev)
ws = kd.workspace(kd._abi.kd_fused_kl_workspace(w.N, w.d, w.V, w.K, w.chunk), dev)
loss, lse, _ = kd.fused_kl_forward(Hd, Wd, idd, tld, None, chunk=w.chunk, ws=ws)
gH, gW = kd.fused_kl_backward(Hd, Wd, idd, tld, None, lse, torch.ones(1, device=dev), chunk=w.chunk, ws=ws,
                              grad_H_fp32=True)
device_error(ws)
ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), tid.numpy(), tlog.numpy(), None)
assert abs(loss.item() - ref.loss) <= 1e-3 * abs(ref.loss)
for got, want in ((gH.cpu().numpy(), ref.grad_H), (gW.cpu().numpy(), ref.grad_W)):
    assert np.max(np.abs(got - want)) <= 2e-2 * np.max(np.abs(want))
print("checked build ok")
'''


def test_checked_build_parity_and_clean_error_word(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library(debug=True)
    env = dict(os.environ, KD_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked build ok" in r.stdout
