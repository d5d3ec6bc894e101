"""Device-side failure detection, exercised without faulting the GPU.

Every wait inside the kernels is bounded.  With SINK_ATTN_DEBUG_WITHHOLD_COPIES=1
the TMA producers (prefill, tensor-core decode) issue no copies, so no barrier a
consumer waits on ever completes: each wait gives up after
SINK_ATTN_WAIT_LIMIT_MS, records a bit in the library's device error word and
the kernel returns.  The host then reads SINK_ATTN_ERR_TIMEOUT from
sink_attn_get_device_error().  The single-token chunk kernel has no such wait
(each warp waits only for its own asynchronous copies), so it still reports
nothing.  Nothing traps, faults or hangs; a fresh process afterwards computes
correct results.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, {root!r})
import gqa_attention_head_sink_gb300 as sa
from gqa_attention_head_sink_gb300 import workloads
sa.load()
# 4 new tokens x group 8 = 32 rows per kv head: the tensor-core decode kernel
d = workloads.make_decode([100, 40], num_q_heads=16, num_kv_heads=2, seed=1, num_splits=2, q_len=4, device="cuda")
sa.sink_attn_decode_multi(d.q, d.k_pages, d.v_pages, d.page_table, d.seqlens_t, d.sinks, d.scale, num_splits=2)
st_decode = sa.sink_attn_get_device_error()
p = workloads.make_prefill([200], num_q_heads=4, num_kv_heads=2, seed=2, device="cuda")
sa.sink_attn_prefill(p.q, p.k, p.v, p.sinks, p.cu_seqlens, p.scale, max_seqlen=200)
st_prefill = sa.sink_attn_get_device_error()
st_clear = sa.sink_attn_get_device_error()   # the word is cleared once read
e = workloads.make_decode([100, 40], num_q_heads=16, num_kv_heads=2, seed=3, num_splits=2, device="cuda")
sa.sink_attn_decode(e.q, e.k_pages, e.v_pages, e.page_table, e.seqlens_t, e.sinks, e.scale, num_splits=2)
st_chunk = sa.sink_attn_get_device_error()
torch.cuda.synchronize()
print("STATUS", st_decode, st_prefill, st_clear, st_chunk)
"""


def _run_child(env_extra):
    from gqa_attention_head_sink_gb300 import build
    build.build()
    env = dict(os.environ)
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [l for l in r.stdout.splitlines() if l.startswith("STATUS")][-1]
    return [int(x) for x in line.split()[1:]]


@pytest.mark.gpu
def test_withheld_copies_time_out_and_are_reported():
    st = _run_child({"SINK_ATTN_DEBUG_WITHHOLD_COPIES": "1", "SINK_ATTN_WAIT_LIMIT_MS": "50"})
    assert st == [4, 4, 0, 0]  # SINK_ATTN_ERR_TIMEOUT for each waiting kernel, cleared; none for the chunk kernel


@pytest.mark.gpu
def test_normal_process_reports_no_timeout():
    st = _run_child({"SINK_ATTN_WAIT_LIMIT_MS": "50"})
    assert st == [0, 0, 0, 0]
