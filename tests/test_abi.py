"""The C-ABI library loads without a GPU and exports every entry point the header declares."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        names += re.findall(r"GRPO_API\s+[\w\s\*]*?\b(grpo_\w+)\s*\(", text)
    return names


def test_header_declares_entry_points():
    names = _declared()
    for n in ("grpo_plan_microbatches", "grpo_group_advantage", "grpo_logprob_loss_fwd_bwd",
              "grpo_finish_step"):
        assert n in names


def test_library_exports_every_declared_symbol(grpo_lib):
    missing = [n for n in _declared() if not hasattr(grpo_lib, n)]
    assert missing == []


def test_status_strings_and_version(grpo_lib):
    grpo_lib.grpo_status_string.restype = ctypes.c_char_p
    assert grpo_lib.grpo_status_string(0) == b"ok"
    assert b"N" in grpo_lib.grpo_status_string(-8)
    assert grpo_lib.grpo_version() >= 100


def test_struct_sizes_match_header(grpo_lib):
    from rl_post_token_gb300 import _lib
    assert ctypes.sizeof(_lib.grpo_step_result) == 64
    assert _lib.ACC_BYTES == 128


def test_binding_constants_match_header():
    # every integer constant the binding names after a header #define has the header's value
    from rl_post_token_gb300 import _lib
    text = open(os.path.join(ROOT, "include", "grpo.h")).read()
    defs = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define GRPO_(\w+)\s+\(?(-?\d+)\)?", text)}
    named = [k for k in defs if isinstance(getattr(_lib, k, None), int)]
    for k in named:
        assert getattr(_lib, k) == defs[k], k
    for k in ("OK", "STEP_SKIPPED_NONFINITE", "ERR_UNSUPPORTED", "DTYPE_BF16", "AGG_SEQ_MEAN_TOKEN_MEAN",
              "KL_K1", "KL_K3"):
        assert k in named, k


def test_header_is_plain_c_and_a_c_client_links(grpo_lib, tmp_path):
    # the boundary is a C ABI: the plain-C client compiles as C11 against grpo.h (with warnings
    # as errors) and links against the library; running it needs a GPU (its own GPU test)
    import shutil
    import subprocess
    import pytest
    gcc = shutil.which("gcc")
    cuda = next((c for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda")
                 if c and os.path.exists(os.path.join(c, "include", "cuda_runtime_api.h"))), None)
    if not gcc or not cuda:
        pytest.skip("gcc or the CUDA headers not found")
    pkg = os.path.join(ROOT, "rl_post_token_gb300")
    cmd = [gcc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror", f"-I{ROOT}/include", f"-I{cuda}/include",
           os.path.join(ROOT, "tests", "c_abi", "loss_step.c"), "-o", str(tmp_path / "loss_step"), f"-L{pkg}",
           "-lgrpo", f"-L{cuda}/lib64", "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
