"""The NCCL branches of the multi-rank code on one GPU, in a one-rank NCCL process group (no
second GPU is needed and no kernel waits on another rank): bench.py's timing reduction and
barrier, and the data-parallel step-result exchange (dp_allreduce_step_result), whose device
tensors take the NCCL all-gather. With one rank the exchange must return the rank's own result
combined by grpo_combine_step_results, and the timing reduction its own figures."""
import os
import socket
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys, json
sys.path.insert(0, os.environ["GRPO_ROOT"])
import torch
import torch.distributed as dist
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
import bench
from rl_post_token_gb300 import step as S, _lib
# the world size passed as 2 makes both helpers take their collective branches on this group
bench.barrier(2, dev)
el, units = bench.reduce_timing(2.5, 77.0, 2, dev)
res = dict(loss_sum=1.5, n_valid=3, n_clipped=1, n_nonfinite=0, n_tokens=4, status=0, kernel_flags=2)
got = S.dp_allreduce_step_result(res, divisor=6)
want = S.combine_step_results([res], 6)
dist.destroy_process_group()
print("RESULT " + json.dumps({"el": el, "units": units, "got": got, "want": want}), flush=True)
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_nccl_one_rank_exchange(grpo_lib, tmp_path):
    assert torch.cuda.is_available()
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()), RANK="0", WORLD_SIZE="1",
               LOCAL_RANK="0", GRPO_ROOT=ROOT, NCCL_NVLS_ENABLE="0")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True, timeout=300,
                       cwd=str(tmp_path))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    import json
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")]
    assert lines, r.stdout[-2000:] + r.stderr[-2000:]
    out = json.loads(lines[-1][len("RESULT "):])
    assert out["el"] == 2.5 and out["units"] == 77.0
    assert out["got"] == out["want"]
    assert out["got"]["loss"] == 1.5 / 6 and out["got"]["n_valid"] == 3 and out["got"]["kernel_flags"] == 2
