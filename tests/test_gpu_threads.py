"""Concurrent callers: several host threads, each on its own stream with its own outputs,
call every row-pass instance, the row pass over host logits and both LM-head backward paths
at once, each followed by its step finish, starting from empty launch caches (a fresh
process). Each result equals the same call made alone, bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_concurrent_host_threads_same_bits(grpo_lib):
    r = subprocess.run([sys.executable, "-m", "tests._threads_child"], cwd=ROOT, capture_output=True,
                       text=True, timeout=900)
    out = r.stdout + r.stderr
    assert r.returncode == 0 and "THREADS_OK" in r.stdout, out[-3000:]
    assert int(r.stdout.split("THREADS_OK")[1].split()[0]) > 0
