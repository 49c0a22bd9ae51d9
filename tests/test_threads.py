"""First calls from two host threads at once, in a fresh process.

The library looks up per-device facts (SM count, the addresses of its device
words) on the first call that uses a device, and the no-allocation entry
point does the same for its table.  Two threads make their first calls at the
same moment -- one through kda_chunk_prefill, one through
kda_chunk_prefill_noalloc, on two streams -- and both results must equal, bit
for bit, the same calls made one after the other afterwards.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import kda_linear_attention_chunk_gb300 as kda
from kda_linear_attention_chunk_gb300 import synthetic as syn

w = syn.Workload("threads", [300, 1, 64, 129, 700], H=4, dk=128, dv=128, init_state=True, seed=31)
x = syn.draw(w)
dev = {k: (torch.from_numpy(v.view(np.int16)).view(torch.bfloat16) if v.dtype == np.uint16
           else torch.from_numpy(v)).cuda() for k, v in x.items()}
cu = torch.from_numpy(w.cu_seqlens()).cuda()
s0 = torch.from_numpy(syn.draw_initial_state(w)).cuda()
outs = [torch.empty((w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
fins = [torch.empty((w.N, w.H, w.dv, w.dk), dtype=torch.float32, device="cuda") for _ in range(4)]
streams = [torch.cuda.Stream(), torch.cuda.Stream()]
torch.cuda.synchronize()
args = lambda i: (dev["q"].data_ptr(), dev["k"].data_ptr(), dev["v"].data_ptr(), dev["g"].data_ptr(),
                  dev["beta"].data_ptr(), cu.data_ptr(), s0.data_ptr(), outs[i].data_ptr(),
                  fins[i].data_ptr(), w.N, w.T, w.H, w.dk, w.dv, int(streams[i % 2].cuda_stream))
gate = threading.Barrier(2)
status = [None, None]

def first(i):
    gate.wait()
    fn = kda.kda_chunk_prefill if i == 0 else kda.kda_chunk_prefill_noalloc
    status[i] = fn(*args(i))

kda.load()
th = [threading.Thread(target=first, args=(i,)) for i in range(2)]
for t in th: t.start()
for t in th: t.join()
torch.cuda.synchronize()
assert status == [kda.KDA_OK, kda.KDA_OK], status
assert kda.kda_chunk_prefill(*args(2)) == kda.KDA_OK
torch.cuda.synchronize()
assert kda.kda_chunk_prefill_noalloc(*args(3)) == kda.KDA_OK
torch.cuda.synchronize()
assert kda.device_error(reset=True) == 0
for a, b in ((0, 2), (1, 3), (0, 1)):
    assert torch.equal(outs[a], outs[b]) and torch.equal(fins[a], fins[b]), (a, b)
print("THREADS-OK")
"""


@pytest.mark.gpu
def test_first_calls_from_two_threads():
    res = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "THREADS-OK" in res.stdout, res.stdout + res.stderr
