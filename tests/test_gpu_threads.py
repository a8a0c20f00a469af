"""Calls from several host threads at once, each on its own stream, in a fresh process so
that the library's one-time set-up (error word, kernel attributes, tensor-map encoder,
SM count) is raced too: every thread's result equals the serial call's, bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
import numpy as np, torch
sys.path.insert(0, ROOT)
from paged_kv_cache_293_gb300 import _build, workloads
_build.build()
from paged_kv_cache_293_gb300 import pagedkv as P

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=dev)
g = workloads.build("threads_gqa", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=16, context_lens=[5, 700, 1500, 4000, 33, 260], seed=71,
                    device=dev)
m = workloads.build("threads_mha", dtype="f16", num_q_heads=8, num_kv_heads=8, head_dim=64,
                    block_size=32, context_lens=[1, 90, 2100, 640], seed=72, device=dev)
c = workloads.build("threads_cascade", dtype="bf16", num_q_heads=32, num_kv_heads=8,
                    head_dim=128, block_size=16, context_lens=[200, 300, 129, 900], seed=73,
                    device=dev, shared_prefix_blocks=8)
torch.cuda.synchronize()


def decode(w, psize, out):
    nb = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, w.max_context_len,
                                      psize)
    ws = P.workspace_tensor(nb, dev) if nb else None
    P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, i32(w.block_tables),
                                 i32(w.context_lens), w.scale, out, w.max_context_len, psize, ws)
    return ws


def cascade(w, out):
    nb = P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 32, w.max_context_len, 128, 0)
    ws = P.workspace_tensor(nb, dev)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, i32(w.block_tables),
                                         i32(w.context_lens), w.scale, out, w.max_context_len,
                                         128, ws)
    return ws


jobs = [("gqa", lambda o: decode(g, 0, o), g), ("gqa_split", lambda o: decode(g, 512, o), g),
        ("mha", lambda o: decode(m, 0, o), m), ("mha_split", lambda o: decode(m, 256, o), m),
        ("cascade", lambda o: cascade(c, o), c)]
N = 3 * len(jobs)
results, keep, errors = [None] * N, [None] * N, []
start = threading.Barrier(N, timeout=120)


def run(i):
    name, fn, w = jobs[i % len(jobs)]
    try:
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                             dtype=torch.float32, device=dev)
        start.wait()
        with torch.cuda.stream(s):
            keep[i] = fn(out)
        s.synchronize()
        results[i] = out
    except Exception as e:  # reported below
        errors.append("%s: %r" % (name, e))


threads = [threading.Thread(target=run, args=(i,)) for i in range(N)]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
for i in range(N):
    name, fn, w = jobs[i % len(jobs)]
    ref = torch.full_like(results[i], float("nan"))
    fn(ref)
    torch.cuda.synchronize()
    assert torch.equal(results[i], ref), name
assert P.pkv_get_device_error() == 0
print("ok", N)
"""


def test_concurrent_first_calls_from_threads():
    proc = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD],
                          capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert proc.returncode == 0, proc.stdout[-2000:] + proc.stderr[-4000:]
    assert proc.stdout.strip().endswith("ok 15")
