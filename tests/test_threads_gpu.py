"""Host threads calling the library at once. A fresh process starts four threads together.
Each thread has its own handle and stream, and runs its own pack three times from the first
call on, so the once-per-process and once-per-device set-up (SM count, kernel attributes,
the tensor-map entry point) is taken concurrently. Every result must equal, bit for bit,
the same packs run one after another afterwards."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import threading, sys
import numpy as np, torch
from packed_linear_attention_gb300 import gdn
from packed_linear_attention_gb300 import inputs as I

torch.cuda.set_device(0)
packs = [I.make_pack(lens, num_k_heads=2, num_v_heads=4, head_dim=128, io_dtype="bf16",
                     seed=70 + i, init_std=0.02,
                     ckpt_lists=[[64] if n >= 64 else [] for n in lens])
         for i, lens in enumerate([[300, 200], [128, 64, 77], [1024], [65, 1, 190]])]
bufs = [gdn.to_device(p) for p in packs]
torch.cuda.synchronize()
results, errors = [None] * 4, []
start = threading.Barrier(4)

def work(i):
    try:
        h = gdn.gdn_handle_create(0, 0)
        stream = torch.cuda.Stream()
        start.wait()
        outs = []
        for _ in range(3):
            gdn.prefill(h, bufs[i], stream)
            stream.synchronize()
            assert gdn.gdn_read_device_status(bufs[i].workspace) == 0
            outs.append([x.clone() for x in (bufs[i].o, bufs[i].ckpt, bufs[i].final)])
        results[i] = outs
        gdn.gdn_handle_destroy(h)
    except Exception as e:  # reported by the parent
        errors.append(f"thread {i}: {e!r}")

threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
for t in threads: t.start()
for t in threads: t.join()
if errors:
    print("\n".join(errors)); sys.exit(1)
h = gdn.gdn_handle_create(0, 0)
for i, b in enumerate(bufs):
    gdn.prefill(h, b)
    torch.cuda.synchronize()
    want = (b.o, b.ckpt, b.final)
    for r, outs in enumerate(results[i]):
        for got, ref in zip(outs, want):
            if not torch.equal(got, ref):
                print(f"pack {i} call {r}: differs from the sequential run"); sys.exit(1)
gdn.gdn_handle_destroy(h)
print("THREADS_OK")
"""


def test_threads_take_first_use_set_up_together():
    from packed_linear_attention_gb300 import build
    build.build()
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "THREADS_OK" in r.stdout, r.stdout + r.stderr
