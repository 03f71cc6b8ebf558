"""Argument checks of the C ABI, on the CPU: every call below is invalid (or empty) and is
answered by the host-side checks before any device memory or CUDA call is touched, so no GPU
is needed. The pointers are placeholders that are never dereferenced. On a machine with a GPU
the module is skipped: its GPU tests run real calls."""
import ctypes as C
import math

import pytest

from rl_post_token_gb300 import _lib

P = 0x100000  # a 256-byte-aligned placeholder address


@pytest.fixture(scope="module", autouse=True)
def _no_gpu(grpo_lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-side argument checks are exercised without a GPU")
    return grpo_lib


def _row(dtype=_lib.DTYPE_BF16, T=8, V=16, ld=16, logits=P, target=P, adv=P, mask=P, dl=None, ld_out=0,
         loss=P, acc=P, terms=None):
    t = C.byref(terms) if terms is not None else None
    return _lib.lib().grpo_logprob_loss_fwd_bwd_ex(logits, dtype, T, V, ld, None, target, None, adv, mask,
                                                   C.c_float(0.2), C.c_float(1.0), dl, ld_out, loss, None, t,
                                                   acc, None)


@pytest.mark.parametrize("kw, code", [
    (dict(dtype=7), _lib.ERR_UNSUPPORTED),
    (dict(T=-1), _lib.ERR_INVALID),
    (dict(V=0), _lib.ERR_INVALID),
    (dict(ld=15), _lib.ERR_INVALID),
    (dict(acc=None), _lib.ERR_INVALID),
    (dict(dl=P, ld_out=15), _lib.ERR_INVALID),
    (dict(logits=None), _lib.ERR_INVALID),
    (dict(target=None), _lib.ERR_INVALID),
    (dict(adv=None), _lib.ERR_INVALID),
    (dict(mask=None), _lib.ERR_INVALID),
    (dict(loss=None), _lib.ERR_INVALID),
    (dict(V=2 ** 31, ld=2 ** 31), _lib.ERR_INVALID),
    (dict(T=2 ** 31), _lib.ERR_INVALID),
    (dict(T=0), _lib.OK),  # nothing to do: nothing launched
    (dict(T=0, logits=None, target=None, adv=None, mask=None, loss=None), _lib.OK),
])
def test_row_pass_argument_checks(kw, code):
    assert _row(**kw) == code


@pytest.mark.parametrize("terms", [
    dict(kl_kind=5),
    dict(kl_kind=-1),
    dict(kl_kind=_lib.KL_K1),  # a KL term without reference log-probs
    dict(kl_kind=_lib.KL_K3, ref_logp=P, kl_coef=math.nan),
    dict(ent_coef=math.inf),
    dict(ent_coef=-math.inf),
])
def test_row_pass_term_checks(terms):
    tm = _lib.grpo_loss_terms(terms.get("kl_kind", 0), terms.get("kl_coef", 0.0), terms.get("ref_logp"),
                              terms.get("ent_coef", 0.0), None, None)
    assert _row(terms=tm) == _lib.ERR_INVALID
    # the same terms are rejected even for an empty call
    assert _row(T=0, terms=tm) == _lib.ERR_INVALID


def _host(T=8, V=16, ld=16, logits=P, staging=P, block_rows=4, acc=P, dl=None, ld_out=0):
    return _lib.lib().grpo_logprob_loss_fwd_bwd_host(logits, _lib.DTYPE_BF16, T, V, ld, None, P, None, P, P,
                                                     C.c_float(0.2), C.c_float(1.0), dl, ld_out, P, None, None,
                                                     acc, staging, block_rows, None, None)


@pytest.mark.parametrize("kw, code", [
    (dict(staging=P + 8), _lib.ERR_INVALID),  # the staging buffer must be 16-byte aligned
    (dict(staging=None), _lib.ERR_INVALID),
    (dict(logits=None), _lib.ERR_INVALID),
    (dict(block_rows=0), _lib.ERR_INVALID),
    (dict(acc=None), _lib.ERR_INVALID),
    (dict(ld=8), _lib.ERR_INVALID),
    (dict(dl=P, ld_out=8), _lib.ERR_INVALID),
    (dict(T=0), _lib.OK),
])
def test_host_entry_argument_checks(kw, code):
    assert _host(**kw) == code


def _lm(T=256, V=1024, H=128, h=P, W=P, ws=P, ws_bytes=1 << 30, acc=P, target=P, flags=0, d_h=P, dW=P):
    return _lib.lib().grpo_lmhead_loss_fwd_bwd(h, W, T, V, H, target, None, P, P, C.c_float(0.2),
                                               C.c_float(1.0), d_h, dW, flags, P, None, acc, ws, ws_bytes, None)


@pytest.mark.parametrize("kw, code", [
    (dict(H=100), _lib.ERR_INVALID),  # H a multiple of 64
    (dict(flags=4), _lib.ERR_INVALID),  # unknown flag bits
    (dict(H=32), _lib.ERR_INVALID),
    (dict(V=0), _lib.ERR_INVALID),
    (dict(T=-1), _lib.ERR_INVALID),
    (dict(acc=None), _lib.ERR_INVALID),
    (dict(h=P + 8), _lib.ERR_INVALID),  # TMA sources 16-byte aligned
    (dict(W=P + 8), _lib.ERR_INVALID),
    (dict(ws=P + 16), _lib.ERR_INVALID),  # the workspace (GEMM scratch included) 256-byte aligned
    (dict(ws=None), _lib.ERR_INVALID),
    (dict(d_h=P + 4), _lib.ERR_INVALID),  # the float32 outputs' rows are written 16 bytes at a time
    (dict(dW=P + 8), _lib.ERR_INVALID),
    (dict(target=None), _lib.ERR_INVALID),
    (dict(T=2 ** 30), _lib.ERR_INVALID),
    (dict(T=0), _lib.OK),
])
def test_lmhead_argument_checks(kw, code):
    assert _lm(**kw) == code


def test_lmhead_workspace_too_small_is_capacity():
    # one byte short of the documented workspace
    need = _lib.grpo_lmhead_workspace_size(256, 1024, 128)
    assert _lm(ws_bytes=need - 1) == _lib.ERR_CAPACITY


def test_lmhead_workspace_sizes():
    up = lambda x: (x + 255) // 256 * 256
    for T, V, H, chunk_tiles in [(1, 1, 64, 1), (256, 1024, 128, 4), (300, 40000, 512, 53),
                                 (16384, 151936, 2048, 66), (8, 256 * 66, 64, 66), (8, 256 * 67, 64, 34)]:
        plain = _lib.grpo_lmhead_workspace_size(T, V, H)
        nct = (V + 255) // 256
        # partials (two float arrays per tile and token), three per-token floats, two bf16
        # dlogits chunk buffers (the tiles split into ceil(tiles / 66) chunks of equal width),
        # then the entropy's third partial per tile and token and two per-token floats, then
        # the backward's token partition (an int32 per token), its live count and the compact
        # bf16 hidden states [T, H]
        n_chunks = -(-nct // 66)
        assert -(-nct // n_chunks) == chunk_tiles
        base = 2 * up(4 * nct * T) + 3 * up(4 * T)
        assert plain == (base + 2 * up(2 * T * 256 * chunk_tiles) + up(4 * nct * T) + 2 * up(4 * T)
                         + up(4 * T) + 256 + up(2 * T * H))
    for bad in [(0, 8, 64), (8, 0, 64), (8, 8, 0), (-1, 8, 64)]:
        assert _lib.grpo_lmhead_workspace_size(*bad) == 0
    assert _lib.lib().grpo_lmhead_forward_noalloc_max_scratch() == 16 << 20
