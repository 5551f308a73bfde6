"""First use of the library from several host threads at once: a fresh process
starts eight threads that call four entry points concurrently, each on its own
stream, so the per-device set-up (device check, error word, shared-memory
opt-ins, SM count) runs under contention; every result must match the oracle."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import oracle, workloads as W
    from chunked_prefill_gqa_gb300 import build
    build.build()
    import chunked_prefill_gqa_gb300 as cp
    torch.cuda.set_device(0)
    inp = W.edge(100, 77, seed=3)
    ref = oracle.prefill(inp)
    kv = W.to_bf16(inp)
    ref16 = oracle.prefill_bf16kv(inp.q, kv.k, kv.v, inp.P)
    paths = ["attn_prefill", "attn_prefill_bf16x3", "attn_prefill_ffma", "attn_prefill_bf16kv"] * 2
    results, errors = {{}}, []
    barrier = threading.Barrier(len(paths))
    def run(i, path):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                q = torch.from_numpy(inp.q).cuda()
                if path == "attn_prefill_bf16kv":
                    k = torch.from_numpy(kv.k.view(np.int16)).cuda().view(torch.bfloat16)
                    v = torch.from_numpy(kv.v.view(np.int16)).cuda().view(torch.bfloat16)
                else:
                    k = torch.from_numpy(inp.k).cuda(); v = torch.from_numpy(inp.v).cuda()
                out = torch.full_like(q, float("nan"))
                s.synchronize()
                barrier.wait()
                getattr(cp, path)(q, k, v, out, inp.P, s)
                s.synchronize()
                results[i] = (path, out.cpu().numpy())
        except Exception as e:
            errors.append(repr(e))
    ts = [threading.Thread(target=run, args=(i, p)) for i, p in enumerate(paths)]
    [t.start() for t in ts]; [t.join() for t in ts]
    assert not errors, errors
    assert cp.attn_get_device_error() == 0
    for i, (path, got) in results.items():
        rep = oracle.check(got, ref16 if path == "attn_prefill_bf16kv" else ref)
        assert rep["n_bad"] == 0, (path, rep)
    print("OK", len(results))
""")


def test_concurrent_first_calls_from_host_threads():
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "OK 8" in r.stdout
