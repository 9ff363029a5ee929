"""Several states driven from different host threads at once.

Each thread creates its own state and steps it on its own CUDA stream.  The
child process starts with no kernel configured, so the threads race on the
library's process-wide launch settings (the shared-memory limits raised once
per device, the cooperative stage's resident-CTA count).  Every state must
produce the same bits as the same state stepped alone afterwards.
"""

import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    import torch
    from powersgd_rank_gradient_gb300 import PowerSGDState

    SHAPES = [(1030, 700), (700,), (512, 2048), (64, 3, 7, 7)]
    N = 1030 * 700 + 700 + 512 * 2048 + 64 * 3 * 7 * 7
    CASES = [(1, 2), (4, 2), (8, 5), (16, 3), (32, 1), (4, 8)]   # (rank, replicas)
    STEPS = 3

    def run(rank, world, seed, results, key, barrier=None):
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            st = PowerSGDState(SHAPES, world, matrix_approximation_rank=rank, start_powerSGD_iter=0,
                               min_compression_rate=1.0, random_seed=seed, device="cuda:0")
            gen = torch.Generator(device="cpu").manual_seed(seed)
            host = [[torch.randn(N, generator=gen).mul_(1e-3) for _ in range(world)] for _ in range(STEPS)]
            outs = []
            if barrier is not None:
                barrier.wait()
            for k in range(STEPS):
                grads = [h.to("cuda:0", non_blocking=False) for h in host[k]]
                outs.append(st.step(grads, stream=stream).clone())
            stream.synchronize()
            results[key] = [o.cpu() for o in outs]
            st.close()

    threaded, alone = {}, {}
    bar = threading.Barrier(len(CASES), timeout=120)
    ths = [threading.Thread(target=run, args=(r, w, 11 + i, threaded, i, bar)) for i, (r, w) in enumerate(CASES)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert len(threaded) == len(CASES), "a thread failed"
    for i, (r, w) in enumerate(CASES):
        run(r, w, 11 + i, alone, i)
        for k in range(STEPS):
            if not torch.equal(threaded[i][k], alone[i][k]):
                raise SystemExit(f"rank {r} W {w} step {k}: threaded output differs")
    print("threads ok")
""")


def test_states_on_concurrent_threads_match_sequential():
    p = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    assert "threads ok" in p.stdout
