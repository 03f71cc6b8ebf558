"""ctypes binding of ``libgrpo.so`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does nothing but turn
Python/torch arguments into pointers and sizes, call the library, and turn a negative status
into ``GrpoError``. All computation happens in the library. If the library has not been
built, every call raises instead of falling back to anything.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgrpo.so")

OK = 0
STEP_SKIPPED_NONFINITE = 1
ERR_INVALID = -1
ERR_DIVISIBILITY = -2
ERR_ROLLOUT_COUNT = -3
ERR_TOKEN_BUDGET = -4
ERR_INCOMPATIBLE = -5
ERR_CAPACITY = -6
ERR_CUDA = -7
ERR_N_MISMATCH = -8
ERR_KERNEL = -9
ERR_UNSUPPORTED = -10
DTYPE_F32 = 0
DTYPE_BF16 = 1
AGG_TOKEN_MEAN = 0
AGG_SEQ_MEAN_TOKEN_SUM = 1
AGG_SEQ_MEAN_TOKEN_MEAN = 2
# GRPO_KL_*: the KL estimator of the regulariser term
KL_NONE = 0
KL_K1 = 1
KL_K3 = 2
ACC_BYTES = 128

_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)


class GrpoError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib().grpo_status_string(code).decode() if _LIB is not None else str(code)
        super().__init__(f"{where}: {msg} (status {code})")
        self.code = code


class grpo_plan_cfg(C.Structure):
    _fields_ = [("batch", C.c_int32), ("mini", C.c_int32), ("micro", C.c_int32),
                ("group_size", C.c_int32), ("dynamic", C.c_int32), ("workload", C.c_int32),
                ("max_token_len", C.c_int64), ("min_bins", C.c_int32), ("bin_multiple", C.c_int32),
                ("balance_ends", C.c_int32), ("compaction", C.c_int32), ("n_gpus", C.c_int32),
                ("logprob_batch", C.c_int32), ("sequence_packing", C.c_int32),
                ("interleaved_pipeline", C.c_int32), ("use_rollout_logprobs", C.c_int32)]


class grpo_plan(C.Structure):
    _fields_ = [("cap_rows", C.c_int32), ("cap_chunks", C.c_int32), ("cap_steps", C.c_int32),
                ("n_rows", C.c_int32), ("n_chunks", C.c_int32), ("n_steps", C.c_int32),
                ("n_micro", C.c_int32), ("q", C.c_int32), ("n_pad_rows", C.c_int32),
                ("needs_old_logp_cache", C.c_int32),
                ("row_src", _i32p), ("row_pad", _i32p), ("row_gpu", _i32p), ("row_rollout", _i32p),
                ("inv_perm", _i32p), ("chunk_row_off", _i32p), ("step_chunk_off", _i32p),
                ("step_in_row_off", _i32p), ("chunk_tokens", _i64p), ("step_valid_tokens", _i64p),
                ("step_valid_rows", _i32p)]


class grpo_window(C.Structure):
    _fields_ = [("n_micro", C.c_int32), ("pos", C.c_int32), ("remaining_drop", C.c_int32),
                ("reserved0", C.c_int32), ("denom", C.c_int64), ("loss_x_denom", C.c_double),
                ("steps", C.c_int64), ("skipped_windows", C.c_int64), ("dropped_chunks", C.c_int64),
                ("batch_loss_x_denom", C.c_double), ("batch_denom", C.c_int64)]


class grpo_loss_terms(C.Structure):
    _fields_ = [("kl_kind", C.c_int32), ("kl_coef", C.c_float), ("ref_logp", C.c_void_p),
                ("ent_coef", C.c_float), ("entropy_tok", C.c_void_p), ("w_tok", C.c_void_p)]


class grpo_step_result(C.Structure):
    _fields_ = [("loss", C.c_double), ("loss_sum", C.c_double), ("clipfrac", C.c_double),
                ("n_valid", C.c_int64), ("n_clipped", C.c_int64), ("n_nonfinite", C.c_int64),
                ("n_tokens", C.c_int64), ("status", C.c_int32), ("kernel_flags", C.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


_PLAN_CFG_FIELDS = [f for f, _ in grpo_plan_cfg._fields_]
_LIB: Optional[C.CDLL] = None


def _lib() -> C.CDLL:
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run `python -m rl_post_token_gb300.build` "
                           "(the library has no fallback path)")
    lib = C.CDLL(LIB_PATH)
    vp = C.c_void_p
    lib.grpo_plan_microbatches.argtypes = [C.POINTER(grpo_plan_cfg), C.c_int32, C.c_int32, _i32p,
                                           _i32p, _i32p, C.POINTER(grpo_plan)]
    lib.grpo_plan_token_index.argtypes = [C.POINTER(grpo_plan), C.c_int32, _i64p, _i64p, C.c_int64,
                                          _i64p]
    lib.grpo_group_advantage.argtypes = [vp, C.c_int32, C.c_int32, C.c_float, C.c_int32, vp, vp, vp,
                                         C.c_int32, vp, vp]
    lib.grpo_logprob_loss_fwd_bwd.argtypes = [vp, C.c_int32, C.c_int64, C.c_int64, C.c_int64, vp, vp,
                                              vp, vp, vp, C.c_float, C.c_float, vp, C.c_int64, vp, vp,
                                              vp, vp]
    lib.grpo_logprob_loss_fwd_bwd_ex.argtypes = [vp, C.c_int32, C.c_int64, C.c_int64, C.c_int64, vp, vp,
                                                 vp, vp, vp, C.c_float, C.c_float, vp, C.c_int64, vp, vp,
                                                 C.POINTER(grpo_loss_terms), vp, vp]
    lib.grpo_logprob_loss_fwd_bwd_ex.restype = C.c_int
    lib.grpo_logprob_loss_fwd_bwd_host.argtypes = [vp, C.c_int32, C.c_int64, C.c_int64, C.c_int64, vp, vp,
                                                   vp, vp, vp, C.c_float, C.c_float, vp, C.c_int64, vp, vp,
                                                   C.POINTER(grpo_loss_terms), vp, vp, C.c_int64, vp, vp]
    lib.grpo_logprob_loss_fwd_bwd_host.restype = C.c_int
    lib.grpo_finish_step.argtypes = [vp, vp, C.c_int64, C.c_int64, C.c_int32, C.POINTER(vp), _i64p,
                                     _i32p, C.c_int32, C.POINTER(grpo_step_result), vp]
    lib.grpo_finish_step_ex.argtypes = [vp, vp, C.c_int64, vp, C.c_int64, C.c_int64, C.c_int32, C.POINTER(vp),
                                        _i64p, _i32p, C.c_int32, C.POINTER(grpo_step_result), vp]
    lib.grpo_finish_step_ex.restype = C.c_int
    lib.grpo_plan_token_weights.argtypes = [C.POINTER(grpo_plan), C.c_int32, _i64p, _i32p, C.c_int32, _i64p,
                                            C.POINTER(C.c_float), C.POINTER(C.c_float)]
    lib.grpo_plan_token_weights.restype = C.c_int
    lib.grpo_combine_step_results.argtypes = [C.POINTER(grpo_step_result), C.c_int32, C.c_int64,
                                              C.POINTER(grpo_step_result)]
    lib.grpo_combine_step_results.restype = C.c_int
    lib.grpo_lmhead_workspace_size.argtypes = [C.c_int64, C.c_int64, C.c_int64]
    lib.grpo_lmhead_workspace_size.restype = C.c_size_t
    lib.grpo_lmhead_loss_fwd_bwd.argtypes = [vp, vp, C.c_int64, C.c_int64, C.c_int64, vp, vp, vp, vp, C.c_float,
                                             C.c_float, vp, vp, C.c_uint32, vp, vp, vp, vp, C.c_size_t, vp]
    lib.grpo_lmhead_loss_fwd_bwd.restype = C.c_int
    lib.grpo_lmhead_loss_fwd_bwd_ex.argtypes = [vp, vp, C.c_int64, C.c_int64, C.c_int64, vp, vp, vp, vp,
                                                C.c_float, C.c_float, vp, vp, C.c_uint32, vp, vp,
                                                C.POINTER(grpo_loss_terms), vp, vp, C.c_size_t, vp]
    lib.grpo_lmhead_loss_fwd_bwd_ex.restype = C.c_int
    lib.grpo_lmhead_forward_noalloc.argtypes = [vp, vp, C.c_int64, C.c_int64, C.c_int64, vp, vp, vp, vp,
                                                C.c_float, C.c_float, vp, vp, vp, vp]
    lib.grpo_lmhead_forward_noalloc.restype = C.c_int
    lib.grpo_lmhead_forward_noalloc_max_scratch.argtypes = []
    lib.grpo_lmhead_forward_noalloc_max_scratch.restype = C.c_size_t
    lib.grpo_window_init.argtypes = [C.POINTER(grpo_window), C.c_int32]
    lib.grpo_window_chunk.argtypes = [C.POINTER(grpo_window), C.c_int32, C.c_double, C.c_int64,
                                      C.POINTER(C.c_int32), C.POINTER(C.c_double)]
    lib.grpo_window_rollup.argtypes = [C.POINTER(grpo_window), C.POINTER(C.c_double), _i64p, _i64p]
    for f in ("grpo_window_init", "grpo_window_chunk", "grpo_window_rollup"):
        getattr(lib, f).restype = C.c_int
    lib.grpo_status_string.argtypes = [C.c_int]
    lib.grpo_status_string.restype = C.c_char_p
    lib.grpo_version.argtypes = []
    lib.grpo_selftest_wait_timeout.argtypes = [vp, vp]
    for f in ("grpo_plan_microbatches", "grpo_plan_token_index", "grpo_group_advantage",
              "grpo_logprob_loss_fwd_bwd", "grpo_finish_step", "grpo_version", "grpo_selftest_wait_timeout"):
        getattr(lib, f).restype = C.c_int
    _LIB = lib
    return lib


def lib() -> C.CDLL:
    """The loaded library (raises if it is not built)."""
    return _lib()


def _ptr(t) -> Optional[int]:
    """Device/host address of a torch tensor (None -> NULL)."""
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _np_i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p32(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_i32p)


# ---- planner (host) ------------------------------------------------------------------------

def grpo_plan_microbatches(cfg: dict, row_len, row_valid, seg_counts=None,
                           n_rollouts: Optional[int] = None) -> dict:
    """Plan one collected batch; returns the plan as a dict of scalars and numpy arrays."""
    L = _lib()
    c = grpo_plan_cfg()
    for k, v in cfg.items():
        if k not in _PLAN_CFG_FIELDS:
            raise KeyError(f"unknown planner field {k}")
        setattr(c, k, int(v))
    if "bin_multiple" not in cfg:
        c.bin_multiple = 1
    if "n_gpus" not in cfg:
        c.n_gpus = 1
    if "logprob_batch" not in cfg:
        c.logprob_batch = 1
    rl = _np_i32(row_len)
    rv = _np_i32(row_valid)
    sc = None if seg_counts is None else _np_i32(seg_counts)
    n_in = rl.shape[0]
    if n_rollouts is None:
        n_rollouts = sc.shape[0] if sc is not None else n_in
    p = grpo_plan()
    rc = L.grpo_plan_microbatches(C.byref(c), n_rollouts, n_in, _p32(rl), _p32(rv), _p32(sc), C.byref(p))
    if rc not in (OK, ERR_CAPACITY):
        raise GrpoError(rc, "grpo_plan_microbatches")
    nr, nc, ns = max(p.n_rows, 1), max(p.n_chunks, 1), max(p.n_steps, 1)
    arr = {
        "row_src": np.zeros(nr, np.int32), "row_pad": np.zeros(nr, np.int32),
        "row_gpu": np.zeros(nr, np.int32), "row_rollout": np.zeros(nr, np.int32),
        "inv_perm": np.zeros(max(n_in, 1), np.int32), "chunk_row_off": np.zeros(nc + 1, np.int32),
        "step_chunk_off": np.zeros(ns + 1, np.int32), "step_in_row_off": np.zeros(ns + 1, np.int32),
        "chunk_tokens": np.zeros(nc, np.int64), "step_valid_tokens": np.zeros(ns, np.int64),
        "step_valid_rows": np.zeros(ns, np.int32),
    }
    p = grpo_plan()
    p.cap_rows, p.cap_chunks, p.cap_steps = nr, nc, ns
    for k, a in arr.items():
        setattr(p, k, a.ctypes.data_as(_i64p if a.dtype == np.int64 else _i32p))
    rc = L.grpo_plan_microbatches(C.byref(c), n_rollouts, n_in, _p32(rl), _p32(rv), _p32(sc), C.byref(p))
    if rc != OK:
        raise GrpoError(rc, "grpo_plan_microbatches")
    out = {k: getattr(p, k) for k in ("n_rows", "n_chunks", "n_steps", "n_micro", "q", "n_pad_rows",
                                      "needs_old_logp_cache")}
    lens = {"row_src": p.n_rows, "row_pad": p.n_rows, "row_gpu": p.n_rows, "row_rollout": p.n_rows,
            "inv_perm": n_in, "chunk_row_off": p.n_chunks + 1, "step_chunk_off": p.n_steps + 1,
            "step_in_row_off": p.n_steps + 1, "chunk_tokens": p.n_chunks,
            "step_valid_tokens": p.n_steps, "step_valid_rows": p.n_steps}
    for k, a in arr.items():
        out[k] = a[:lens[k]].copy()
    return out


def grpo_plan_token_index(plan: dict, row_len) -> np.ndarray:
    """Exec-order token -> input-order token index (negative -1-i for padding rows)."""
    L = _lib()
    rl = np.asarray(row_len, np.int64)
    off = np.zeros(rl.shape[0] + 1, np.int64)
    np.cumsum(rl, out=off[1:])
    p = grpo_plan()
    p.n_rows = int(plan["n_rows"])
    rs = _np_i32(plan["row_src"])
    rp = _np_i32(plan["row_pad"])
    p.row_src, p.row_pad = _p32(rs), _p32(rp)
    n = C.c_int64(0)
    rc = L.grpo_plan_token_index(C.byref(p), rl.shape[0], off.ctypes.data_as(_i64p), None, 0, C.byref(n))
    if rc not in (OK, ERR_CAPACITY):
        raise GrpoError(rc, "grpo_plan_token_index")
    out = np.zeros(max(n.value, 1), np.int64)
    rc = L.grpo_plan_token_index(C.byref(p), rl.shape[0], off.ctypes.data_as(_i64p),
                                 out.ctypes.data_as(_i64p), out.shape[0], C.byref(n))
    if rc != OK:
        raise GrpoError(rc, "grpo_plan_token_index")
    return out[:n.value]


def grpo_plan_token_weights(plan: dict, row_len, row_valid, agg: int, want_w: bool = True,
                            want_scale: bool = False):
    """(step_divisor int64 [n_steps], w_tok float32 [tokens] or None) of an aggregation mode;
    with want_scale a third item, step_grad_scale float32 [n_steps] (1/max(D_s, 1))."""
    rl = np.asarray(row_len, np.int64)
    off = np.zeros(rl.shape[0] + 1, np.int64)
    np.cumsum(rl, out=off[1:])
    rv = _np_i32(row_valid)
    p = grpo_plan()
    p.n_steps = int(plan["n_steps"])
    so = _np_i32(plan["step_in_row_off"])
    p.step_in_row_off = _p32(so)
    div = np.zeros(max(p.n_steps, 1), np.int64)
    w = np.zeros(max(int(off[-1]), 1), np.float32) if want_w else None
    sc = np.zeros(max(p.n_steps, 1), np.float32) if want_scale else None
    fp = C.POINTER(C.c_float)
    rc = _lib().grpo_plan_token_weights(C.byref(p), rl.shape[0], off.ctypes.data_as(_i64p), _p32(rv), int(agg),
                                        div.ctypes.data_as(_i64p), None if w is None else w.ctypes.data_as(fp),
                                        None if sc is None else sc.ctypes.data_as(fp))
    if rc != OK:
        raise GrpoError(rc, "grpo_plan_token_weights")
    out = (div[:p.n_steps], None if w is None else w[:int(off[-1])])
    return out + (sc[:p.n_steps],) if want_scale else out


def grpo_combine_step_results(per_rank, divisor: int) -> dict:
    """One step's result (dict) from the per-rank results (dicts with the grpo_step_result
    fields; the list order is the rank order and the summation order)."""
    n = len(per_rank)
    arr = (grpo_step_result * max(n, 1))()
    for k, r in enumerate(per_rank):
        for name, ctype in grpo_step_result._fields_:
            v = r.get(name, 0)
            setattr(arr[k], name, float(v) if ctype is C.c_double else int(v))
    out = grpo_step_result()
    rc = _lib().grpo_combine_step_results(arr, n, int(divisor), C.byref(out))
    if rc != OK:
        raise GrpoError(rc, "grpo_combine_step_results")
    return out.as_dict()


# ---- device entry points ---------------------------------------------------------------------

def grpo_group_advantage(rewards, group_size: int, eps: float, unbiased_std: bool, adv_out,
                         row_rollout=None, row_tok_off=None, adv_tok=None, stream=None) -> None:
    """rewards/adv_out float32 device tensors; optional token broadcast into adv_tok."""
    n_rows = 0 if row_tok_off is None else row_tok_off.numel() - 1
    rc = _lib().grpo_group_advantage(_ptr(rewards), rewards.numel(), int(group_size), float(eps),
                                     int(bool(unbiased_std)), _ptr(adv_out), _ptr(row_rollout),
                                     _ptr(row_tok_off), n_rows, _ptr(adv_tok), _stream(stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_group_advantage")


def grpo_logprob_loss_fwd_bwd(logits, target, old_logp, adv_tok, mask, clip_eps: float,
                              grad_scale: float, dlogits, loss_tok, logp_tok, acc, tok_src=None,
                              V: Optional[int] = None, stream=None, terms: Optional[dict] = None) -> None:
    """logits [T, ld] (float32 or bfloat16) on the device; see grpo.h for the rest.

    ``terms`` (optional) = dict(kl_kind=0|1|2, kl_coef=..., ref_logp=tensor, ent_coef=...,
    entropy_tok=tensor, w_tok=tensor) selects grpo_logprob_loss_fwd_bwd_ex."""
    import torch

    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D tensor with unit inner stride")
    dt = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}[logits.dtype]
    T, ld = logits.shape[0], logits.stride(0) if logits.shape[0] > 1 else logits.shape[1]
    V = logits.shape[1] if V is None else V
    ld_out = 0
    if dlogits is not None:
        if dlogits.dtype != logits.dtype or dlogits.dim() != 2 or dlogits.stride(1) != 1:
            raise ValueError("dlogits must match logits' dtype, 2-D, unit inner stride")
        if dlogits.shape[0] != T:
            raise ValueError("dlogits must have the same row count as logits")
        ld_out = dlogits.stride(0) if T > 1 else dlogits.shape[1]
    if terms is None:
        rc = _lib().grpo_logprob_loss_fwd_bwd(_ptr(logits), dt, T, V, ld, _ptr(tok_src), _ptr(target),
                                              _ptr(old_logp), _ptr(adv_tok), _ptr(mask), float(clip_eps),
                                              float(grad_scale), _ptr(dlogits), ld_out, _ptr(loss_tok),
                                              _ptr(logp_tok), _ptr(acc), _stream(stream))
    else:
        tm = grpo_loss_terms(int(terms.get("kl_kind", 0)), float(terms.get("kl_coef", 0.0)),
                             _ptr(terms.get("ref_logp")), float(terms.get("ent_coef", 0.0)),
                             _ptr(terms.get("entropy_tok")), _ptr(terms.get("w_tok")))
        rc = _lib().grpo_logprob_loss_fwd_bwd_ex(_ptr(logits), dt, T, V, ld, _ptr(tok_src), _ptr(target),
                                                 _ptr(old_logp), _ptr(adv_tok), _ptr(mask), float(clip_eps),
                                                 float(grad_scale), _ptr(dlogits), ld_out, _ptr(loss_tok),
                                                 _ptr(logp_tok), C.byref(tm), _ptr(acc), _stream(stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_logprob_loss_fwd_bwd")


def grpo_logprob_loss_fwd_bwd_host(logits_host, target, old_logp, adv_tok, mask, clip_eps: float,
                                   grad_scale: float, dlogits, loss_tok, logp_tok, acc, staging,
                                   block_rows: int, tok_src=None, V: Optional[int] = None, stream=None,
                                   copy_stream=None, terms: Optional[dict] = None) -> None:
    """logits_host [T, ld] (float32 or bfloat16) in host memory (pinned for the link's full
    rate), streamed through ``staging`` (a device uint8 tensor of at least
    2 * block_rows * ld * element-size bytes) in blocks of ``block_rows``; the rest as
    grpo_logprob_loss_fwd_bwd. See grpo.h."""
    import torch

    if logits_host.device.type != "cpu" or logits_host.dim() != 2 or logits_host.stride(1) != 1:
        raise ValueError("logits_host must be a 2-D host tensor with unit inner stride")
    dt = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}[logits_host.dtype]
    T = logits_host.shape[0]
    ld = logits_host.stride(0) if T > 1 else logits_host.shape[1]
    V = logits_host.shape[1] if V is None else V
    need = 2 * min(int(block_rows), max(T, 1)) * ld * logits_host.element_size()
    if staging.device.type != "cuda" or staging.numel() * staging.element_size() < need:
        raise ValueError(f"staging must be a device buffer of at least {need} bytes")
    ld_out = 0
    if dlogits is not None:
        if dlogits.dtype != logits_host.dtype or dlogits.dim() != 2 or dlogits.stride(1) != 1 or dlogits.shape[0] != T:
            raise ValueError("dlogits must match logits' dtype and rows, 2-D, unit inner stride")
        ld_out = dlogits.stride(0) if T > 1 else dlogits.shape[1]
    terms = terms or {}
    tm = grpo_loss_terms(int(terms.get("kl_kind", 0)), float(terms.get("kl_coef", 0.0)),
                         _ptr(terms.get("ref_logp")), float(terms.get("ent_coef", 0.0)),
                         _ptr(terms.get("entropy_tok")), _ptr(terms.get("w_tok")))
    st = _stream(stream)
    rc = _lib().grpo_logprob_loss_fwd_bwd_host(logits_host.data_ptr(), dt, T, V, ld, _ptr(tok_src), _ptr(target),
                                               _ptr(old_logp), _ptr(adv_tok), _ptr(mask), float(clip_eps),
                                               float(grad_scale), _ptr(dlogits), ld_out, _ptr(loss_tok),
                                               _ptr(logp_tok), C.byref(tm), _ptr(acc), _ptr(staging),
                                               int(block_rows), st, st if copy_stream is None else _stream(copy_stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_logprob_loss_fwd_bwd_host")


def _grad_arrays(grad_bufs):
    import torch

    nb = len(grad_bufs)
    bufs = (C.c_void_p * max(nb, 1))(*[g.data_ptr() for g in grad_bufs])
    numels = (C.c_int64 * max(nb, 1))(*[g.numel() for g in grad_bufs])
    dts = (C.c_int32 * max(nb, 1))(*[{torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}[g.dtype]
                                      for g in grad_bufs])
    return nb, bufs, numels, dts


def _finish_rc(rc: int, res, sync: bool, where: str):
    if rc < 0 and not sync:
        raise GrpoError(rc, where)
    if rc < 0 and rc not in (ERR_N_MISMATCH, ERR_KERNEL):
        raise GrpoError(rc, where)
    return res.as_dict() if sync else None


def grpo_finish_step(acc, loss_tok, n_tok: Optional[int] = None, expected_N: int = -1,
                     deferred: bool = False, grad_bufs: Sequence = (), sync: bool = True,
                     stream=None):
    """Close the step. With sync=True returns the result dict (the call waits on the stream);
    with sync=False returns None and the result stays on the device in acc."""
    n_tok = loss_tok.numel() if n_tok is None else n_tok
    nb, bufs, numels, dts = _grad_arrays(grad_bufs)
    res = grpo_step_result()
    rc = _lib().grpo_finish_step(_ptr(acc), _ptr(loss_tok), int(n_tok), int(expected_N), int(bool(deferred)),
                                 bufs, numels, dts, nb, C.byref(res) if sync else None, _stream(stream))
    return _finish_rc(rc, res, sync, "grpo_finish_step")


def grpo_finish_step_ex(acc, loss_tok, w_tok=None, divisor: int = -1, n_tok: Optional[int] = None,
                        expected_N: int = -1, deferred: bool = False, grad_bufs: Sequence = (),
                        sync: bool = True, stream=None):
    """grpo_finish_step with per-token weights (device float, or None) and a divisor (-1 = N)."""
    n_tok = loss_tok.numel() if n_tok is None else n_tok
    nb, bufs, numels, dts = _grad_arrays(grad_bufs)
    res = grpo_step_result()
    rc = _lib().grpo_finish_step_ex(_ptr(acc), _ptr(loss_tok), int(n_tok), _ptr(w_tok), int(divisor),
                                    int(expected_N), int(bool(deferred)), bufs, numels, dts, nb,
                                    C.byref(res) if sync else None, _stream(stream))
    return _finish_rc(rc, res, sync, "grpo_finish_step_ex")


def grpo_lmhead_workspace_size(T: int, V: int, H: int) -> int:
    return int(_lib().grpo_lmhead_workspace_size(T, V, H))


LMHEAD_DW_ACCUMULATE = 1
LMHEAD_SKIP_MASKED = 2


def grpo_lmhead_loss_fwd_bwd(h, W, target, old_logp, adv_tok, mask, clip_eps: float, grad_scale: float,
                             d_h, dW, loss_tok, logp_tok, acc, workspace, stream=None,
                             dw_accumulate: bool = False, terms: Optional[dict] = None,
                             skip_masked: bool = False) -> None:
    """h [T, H] and W [V, H] bf16 device tensors; d_h / dW float32 or None; dw_accumulate adds
    this call's dW to the buffer instead of overwriting it; skip_masked runs the forward GEMM
    over the mask=1 tokens only; ``terms`` (as for grpo_logprob_loss_fwd_bwd) selects
    grpo_lmhead_loss_fwd_bwd_ex; see grpo.h."""
    T, H = h.shape
    V = W.shape[0]
    flags = (LMHEAD_DW_ACCUMULATE if dw_accumulate else 0) | (LMHEAD_SKIP_MASKED if skip_masked else 0)
    if terms is not None:
        tm = grpo_loss_terms(int(terms.get("kl_kind", 0)), float(terms.get("kl_coef", 0.0)),
                             _ptr(terms.get("ref_logp")), float(terms.get("ent_coef", 0.0)),
                             _ptr(terms.get("entropy_tok")), _ptr(terms.get("w_tok")))
        rc = _lib().grpo_lmhead_loss_fwd_bwd_ex(_ptr(h), _ptr(W), T, V, H, _ptr(target), _ptr(old_logp),
                                                _ptr(adv_tok), _ptr(mask), float(clip_eps), float(grad_scale),
                                                _ptr(d_h), _ptr(dW), flags, _ptr(loss_tok), _ptr(logp_tok),
                                                C.byref(tm), _ptr(acc), _ptr(workspace),
                                                workspace.numel() * workspace.element_size(), _stream(stream))
        if rc != OK:
            raise GrpoError(rc, "grpo_lmhead_loss_fwd_bwd_ex")
        return
    rc = _lib().grpo_lmhead_loss_fwd_bwd(_ptr(h), _ptr(W), T, V, H, _ptr(target), _ptr(old_logp),
                                         _ptr(adv_tok), _ptr(mask), float(clip_eps), float(grad_scale),
                                         _ptr(d_h), _ptr(dW), flags,
                                         _ptr(loss_tok), _ptr(logp_tok), _ptr(acc),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_lmhead_loss_fwd_bwd")


def grpo_lmhead_forward_noalloc(h, W, target, old_logp, adv_tok, mask, clip_eps: float,
                                grad_scale: float, loss_tok, logp_tok, acc, stream=None) -> None:
    """Forward-only LM-head loss with the library's own fixed scratch (no allocation)."""
    T, H = h.shape
    V = W.shape[0]
    rc = _lib().grpo_lmhead_forward_noalloc(_ptr(h), _ptr(W), T, V, H, _ptr(target), _ptr(old_logp),
                                            _ptr(adv_tok), _ptr(mask), float(clip_eps), float(grad_scale),
                                            _ptr(loss_tok), _ptr(logp_tok), _ptr(acc), _stream(stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_lmhead_forward_noalloc")


def grpo_lmhead_forward_noalloc_max_scratch() -> int:
    return int(_lib().grpo_lmhead_forward_noalloc_max_scratch())


class Window:
    """The host accumulation window (grpo_window_* entry points)."""

    def __init__(self, n_micro: int):
        self._w = grpo_window()
        rc = _lib().grpo_window_init(C.byref(self._w), int(n_micro))
        if rc != OK:
            raise GrpoError(rc, "grpo_window_init")

    def grpo_window_chunk(self, finite: bool, loss: float, denom: int):
        act, scale = C.c_int32(0), C.c_double(0.0)
        rc = _lib().grpo_window_chunk(C.byref(self._w), int(bool(finite)), float(loss), int(denom),
                                      C.byref(act), C.byref(scale))
        if rc != OK:
            raise GrpoError(rc, "grpo_window_chunk")
        return act.value, scale.value

    def grpo_window_rollup(self):
        loss, denom, steps = C.c_double(0.0), C.c_int64(0), C.c_int64(0)
        rc = _lib().grpo_window_rollup(C.byref(self._w), C.byref(loss), C.byref(denom), C.byref(steps))
        if rc != OK:
            raise GrpoError(rc, "grpo_window_rollup")
        return loss.value, denom.value, steps.value

    @property
    def state(self) -> dict:
        return {k: getattr(self._w, k) for k, _ in grpo_window._fields_}


def new_step_acc(device="cuda"):
    """A zeroed device-resident grpo_step_acc (caller-owned, 128 bytes)."""
    import torch
    return torch.zeros(ACC_BYTES, dtype=torch.uint8, device=device)


def read_step_result(acc) -> dict:
    """Decode acc->result after an asynchronous grpo_finish_step (copies 64 bytes to host)."""
    raw = acc[64:128].cpu().numpy().tobytes()
    return grpo_step_result.from_buffer_copy(raw).as_dict()


def grpo_version() -> int:
    return _lib().grpo_version()


def grpo_selftest_wait_timeout(acc, stream=None) -> None:
    """One bounded wait that nothing completes: sets acc's wait-timeout flag after about a
    second (see grpo.h); the next grpo_finish_step on acc reports ERR_KERNEL."""
    rc = _lib().grpo_selftest_wait_timeout(_ptr(acc), _stream(stream))
    if rc != OK:
        raise GrpoError(rc, "grpo_selftest_wait_timeout")
