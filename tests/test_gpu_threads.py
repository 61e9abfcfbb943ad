"""Concurrent calls from several host threads, each on a stream of its own (needs a GB300).

The library keeps per-device and per-stream state on the host (tensor-map cache,
stream-K workspaces and counters, dequantisation buffers) behind locks.  Four
threads run a mix of every kernel form at once, each on its own stream, many
times over; with exact inputs every result must equal, bit for bit, the one a
single-threaded call gives.
"""
import threading

import numpy as np
import pytest
import torch

from gpu_helpers import DEV, device_status, run
from tensor_core_gemm_02_gb300 import binding, workloads
from tensor_core_gemm_02_gb300.workloads import OUT_BF16, OUT_F32

pytestmark = pytest.mark.gpu


def _fp4(seed, M, N, K):
    rng = np.random.default_rng(seed)
    A = torch.from_numpy((rng.integers(-4, 5, (M, K)) / 4).astype(np.float32)).to(torch.bfloat16)
    Bq = torch.from_numpy(rng.integers(0, 256, (N, K // 2)).astype(np.uint8))
    Bs = torch.from_numpy(rng.integers(125, 130, (K // 32, N)).astype(np.uint8))
    C = torch.from_numpy((rng.integers(-4, 5, (M, N)) / 4).astype(np.float32))
    return workloads.Problem(f"fp4_{M}x{N}x{K}", A, Bq, C, alpha=0.5, beta=1.0, out=OUT_F32, Bs=Bs)


def _problems():
    q = dict(values="quarter")
    acc = workloads.random_problem(57, 16, 2048, 1024, dtype="bf16", with_c=True, alpha=-0.5, **q)
    return [
        # skinny stream-K (split tiles, last-arriver reduction)
        workloads.random_problem(51, 16, 4096, 2048, dtype="bf16", with_c=True, alpha=0.5, **q),
        # tile kernel, ragged
        workloads.random_problem(52, 300, 520, 264, dtype="f16", with_c=True, alpha=2.0,
                                 beta=0.5, out=OUT_BF16, **q),
        # gathered rows
        workloads.random_problem(53, 600, 2048, 512, dtype="bf16", with_c=True, alpha=0.5,
                                 gather_rows=333, **q),
        # scattered rows
        workloads.random_problem(54, 200, 300, 264, dtype="bf16", with_c=True, alpha=0.5,
                                 scatter_rows=700, **q),
        # FP4 weights (skinny form with converter warps)
        _fp4(55, 16, 2048, 1024),
        # dense 256 x 512 pair form
        workloads.random_problem(56, 1024, 2048, 2048, dtype="bf16", **q),
        # accumulate into float32 D (atomic adds; exact, so the order does not matter)
        workloads.Problem("acc", acc.A, acc.B, None, alpha=acc.alpha, beta=0.0, out=OUT_F32,
                          D0=acc.C, accumulate=True),
    ]


def test_threads_on_own_streams_match_single_threaded():
    problems = _problems()
    want = [run(p).cpu() for p in problems]
    torch.cuda.synchronize()
    failures = []

    def worker(tid):
        try:
            s = torch.cuda.Stream(device=DEV)
            with torch.cuda.stream(s):
                for it in range(8):
                    outs = [run(p, stream=s) for p in problems]
                    s.synchronize()
                    for k, (got, ref) in enumerate(zip(outs, want)):
                        if not torch.equal(got.cpu(), ref):
                            failures.append((tid, it, problems[k].name))
        except Exception as e:  # noqa: BLE001 -- reported below
            failures.append((tid, -1, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads)
    assert not failures, failures[:5]
    assert device_status() == binding.GEMM_OK
