"""Register and spill budget of the product kernels, from the ptxas report the build records
(no GPU needed). The cluster row pass runs 17 warps per SM, so a thread has at most 96
registers; a spill in one of the instances the dispatcher selects by default costs that
instance a large share of its bandwidth, so none is allowed."""
import os
import re

import pytest

from rl_post_token_gb300 import build as B


def _report(src):
    path = B.ptxas_report(src)
    if not os.path.exists(path):
        pytest.skip("library not built here")
    # ptxas prints, per entry function, "Compiling entry function NAME", then "Function
    # properties for F" blocks (for NAME and for any non-inlined callee F), each followed by
    # its stack/spill line, then NAME's register count
    kernels = {}
    entry = prop = None
    for line in open(path):
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            entry = prop = m.group(1)
            continue
        m = re.search(r"Function properties for (\S+)", line)
        if m:
            prop = m.group(1)
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and entry and prop == entry:
            kernels.setdefault(entry, {})["spill"] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m and entry:
            kernels.setdefault(entry, {})["regs"] = int(m.group(1))
    return kernels


def _cluster(T, C, NCW, VPT, MINB, ENT, TERMS):
    t = {"bf16": "13__nv_bfloat16", "f32": "f"}[T]
    return f"_ZN4grpo18row_cluster_kernelI{t}Li{C}ELi{NCW}ELi{VPT}ELi{MINB}ELb{ENT}ELi{TERMS}EEEvNS_7RowArgsEii"


# (dtype, cluster, consumer warps, vectors per thread, CTAs per SM, entropy, terms) as
# dispatched for vocabularies that fit one CTA per SM (bf16: 2-CTA cluster; f32: 4-CTA)
DEFAULT_ROW_PASS = [
    # bf16, 2-CTA cluster: no terms, KL, weights, KL + weights, entropy, entropy + weights
    ("bf16", 2, 16, 4, 1, 0, 0), ("bf16", 2, 16, 4, 1, 0, 1), ("bf16", 2, 16, 4, 1, 0, 2),
    ("bf16", 2, 16, 4, 1, 0, 3), ("bf16", 2, 16, 4, 1, 1, 1), ("bf16", 2, 16, 4, 1, 1, 3),
    # bf16, 4-CTA cluster (rows too long for two CTAs)
    ("bf16", 4, 16, 4, 1, 0, 0), ("bf16", 4, 16, 4, 1, 0, 1), ("bf16", 4, 16, 4, 1, 0, 2),
    ("bf16", 4, 16, 4, 1, 0, 3), ("bf16", 4, 16, 4, 1, 1, 1), ("bf16", 4, 16, 4, 1, 1, 3),
    # float32, 4-CTA cluster
    ("f32", 4, 16, 4, 1, 0, 0), ("f32", 4, 16, 4, 1, 0, 1), ("f32", 4, 16, 4, 1, 0, 2),
    ("f32", 4, 16, 4, 1, 0, 3), ("f32", 4, 16, 4, 1, 1, 1), ("f32", 4, 16, 4, 1, 1, 3)]


def test_row_pass_default_instances_do_not_spill(grpo_lib):
    k = _report("grpo_rowpass.cu")
    for inst in DEFAULT_ROW_PASS:
        name = _cluster(*inst)
        assert name in k, (inst, "not compiled")
        assert k[name]["spill"] == 0, (inst, k[name])
        assert k[name]["regs"] <= 96, (inst, k[name])


# the forward-only streaming instances (dtype, cluster, consumer warps, vectors per thread)
FORWARD_ONLY = [("bf16", 2, 16, 4), ("bf16", 4, 16, 4), ("f32", 4, 16, 4)]


def test_forward_only_instances_do_not_spill(grpo_lib):
    k = _report("grpo_rowpass.cu")
    for T, C, NCW, VPT in FORWARD_ONLY:
        t = {"bf16": "13__nv_bfloat16", "f32": "f"}[T]
        name = f"_ZN4grpo14row_fwd_kernelI{t}Li{C}ELi{NCW}ELi{VPT}EEEvNS_7RowArgsEii"
        assert name in k, (T, "not compiled")
        assert k[name]["spill"] == 0, (T, k[name])
        assert k[name]["regs"] <= 96, (T, k[name])


def test_lmhead_and_step_kernels_do_not_spill(grpo_lib):
    for src, pat in (("grpo_lmhead.cu", r"gemm_kernel|reduce_kernel|partition_kernel|gather_kernel"),
                     ("grpo_step.cu", r"finish_kernel|adv_")):
        k = _report(src)
        hits = [n for n in k if re.search(pat, n)]
        assert hits, (src, "no kernel found")
        for n in hits:
            assert k[n]["spill"] == 0, (n, k[n])


def test_lmhead_gemm_instances_do_not_spill(grpo_lib):
    # every instance of the LM-head GEMM template (CTA group 1 and 2; partials, dlogits and
    # float32 epilogues with their operand layouts) and the per-token reduce: no spill and no
    # stack frame (a local array indexed at run time would live in local memory)
    k = _report("grpo_lmhead.cu")
    gemm = [n for n in k if "lmhead11gemm_kernel" in n]
    assert len(gemm) == 10, sorted(gemm)
    for name in gemm + [n for n in k if "lmhead13reduce_kernel" in n]:
        assert k[name]["spill"] == 0, (name, k[name])
        assert k[name]["regs"] <= 255, (name, k[name])
    stack = re.findall(r"Compiling entry function '(\S*gemm_kernel\S*)'.*?\n\s+(\d+) bytes stack frame",
                       open(B.ptxas_report("grpo_lmhead.cu")).read(), flags=re.S)
    assert stack and all(int(b) == 0 for _, b in stack), stack
