"""fp64 CPU oracle of the speculative-decoding verify/commit step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU baseline and
``--impl reference`` arm) import this package.  It wraps ``spec_oracle.c`` through
ctypes and numpy; it imports nothing from the CUDA package and the CUDA package
imports nothing from it.

Functions whose results no pin fixes are marked "parity unpinned" in their docstring.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libspecoracle.so")
_lock = threading.Lock()
_lib = None

BF16, F32 = 0, 1

# near-tie flag bits (see spec_oracle.c)
FL_THRESH, FL_GUMBEL, FL_DEGENERATE, FL_ILLCOND = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into libspecoracle.so (gcc, fp64, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, U64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_rand_word.argtypes = [U64, U64, I32, I32, I32, I32]
        lib.oracle_rand_word.restype = ctypes.c_uint32
        lib.oracle_u01.argtypes = [ctypes.c_uint32]
        lib.oracle_u01.restype = D
        lib.oracle_gumbel.argtypes = [ctypes.c_uint32]
        lib.oracle_gumbel.restype = D
        lib.oracle_row_logprobs.argtypes = [P, I32, D, P]
        lib.oracle_accept_prob.argtypes = [D, D]
        lib.oracle_accept_prob.restype = D
        lib.oracle_residual_weights.argtypes = [P, P, I32, P]
        lib.oracle_gumbel_sample.argtypes = [P, I32, U64, U64, I32, I32, I32]
        lib.oracle_gumbel_sample.restype = I32
        lib.oracle_verify_sample.argtypes = [P, P, I32, I32, I32, I32, I64, P, P, P, U64, U64,
                                             P, P, P, P, P, P, P, P, I32]
        lib.oracle_verify_sample.restype = I32
        lib.oracle_verify_greedy.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, P, P, I32]
        lib.oracle_verify_greedy.restype = I32
        lib.oracle_verify_sample_early_exit.argtypes = lib.oracle_verify_sample.argtypes
        lib.oracle_verify_sample_early_exit.restype = I32
        lib.oracle_verify_greedy_early_exit.argtypes = lib.oracle_verify_greedy.argtypes
        lib.oracle_verify_greedy_early_exit.restype = I32
        lib.oracle_schedule_verify_len.argtypes = [P, P, I32, I32, P, I32, I32, I32, P, P, P]
        lib.oracle_schedule_verify_len.restype = I32
        lib.oracle_schedule_threshold.argtypes = [P, P, I32, I32, ctypes.c_float, P]
        lib.oracle_schedule_threshold.restype = I32
        lib.oracle_schedule_verify_len_stale.argtypes = [P, P, P, I32, I32, P, I32, I32, I32, P, P, P]
        lib.oracle_schedule_verify_len_stale.restype = I32
        lib.oracle_markov_draft.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, I32, P, U64, U64, I32, P, P, P,
                                            P, I32]
        lib.oracle_markov_draft.restype = I32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- RNG
def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 of one counter (4 x uint32) under key (2 x uint32)."""
    lib = _load()
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib.oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def rand_word(seed: int, step: int, b: int, row: int, purpose: int, v: int) -> int:
    return int(_load().oracle_rand_word(seed, step, b, row, purpose, v))


def u01(w: int) -> float:
    return float(_load().oracle_u01(w))


def gumbel(w: int) -> float:
    return float(_load().oracle_gumbel(w))


# ------------------------------------------------------------------ method steps
def row_logprobs(x, T: float) -> np.ndarray:
    """log softmax(x / T) of one row in fp64."""
    lib = _load()
    xx = _c(x, np.float64)
    out = np.empty_like(xx)
    lib.oracle_row_logprobs(_ptr(xx), xx.size, float(T), _ptr(out))
    return out


def accept_prob(P: float, Q: float) -> float:
    return float(_load().oracle_accept_prob(float(P), float(Q)))


def residual_weights(p, q) -> np.ndarray:
    lib = _load()
    pp, qq = _c(p, np.float64), _c(q, np.float64)
    out = np.empty_like(pp)
    lib.oracle_residual_weights(_ptr(pp), _ptr(qq), pp.size, _ptr(out))
    return out


def gumbel_sample(w, seed: int, step: int, b: int = 0, row: int = 0, purpose: int = 1) -> int:
    lib = _load()
    ww = _c(w, np.float64)
    return int(lib.oracle_gumbel_sample(_ptr(ww), ww.size, seed, step, b, row, purpose))


# ------------------------------------------------------------------------ verify
def _logit_array(a):
    """Return (contiguous array, dtype code).  bf16 logits are given as uint16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    return np.ascontiguousarray(a, dtype=np.float32), F32


def verify_sample(target, draft, draft_tokens, num_draft, temperature, seed: int, step: int,
                  nthreads: int = 1, early_exit: bool = False) -> dict:
    """Sampling verify of a padded batch.

    target [B, K+1, V] and draft [B, K, V] as float32 or bf16 bit patterns (uint16);
    draft_tokens [B, K] int32; num_draft [B] int32 or None; temperature [B] float32.
    early_exit: read rows in position order and stop at the first rejection (status 4
    only for rows read; p and q stay -1 past the first rejected position).
    Near-tie outputs: flags [B] (bits FL_*), flag_pos [B] (first scanned position whose
    acceptance test is a threshold near-tie, -1 if none) and gap [B] (top-2 gap of the
    Gumbel draw).
    """
    lib = _load()
    t, dt = _logit_array(target)
    d, dd = _logit_array(draft)
    assert dt == dd
    B, K1, V = t.shape
    K = K1 - 1
    assert d.shape == (B, K, V)
    x = _c(draft_tokens, np.int32).reshape(B, K)
    nd = None if num_draft is None else _c(num_draft, np.int32)
    T = _c(temperature, np.float32)
    out = dict(tokens=np.full((B, K + 1), -1, np.int32), accepted=np.zeros(B, np.int32),
               p=np.full((B, K), -1.0), q=np.full((B, K), -1.0), status=np.zeros(B, np.int32),
               flags=np.zeros(B, np.int32), flag_pos=np.full(B, -1, np.int32), gap=np.zeros(B))
    fn = lib.oracle_verify_sample_early_exit if early_exit else lib.oracle_verify_sample
    rc = fn(_ptr(t), _ptr(d), dt, B, K, V, V, _ptr(x), _ptr(nd), _ptr(T),
                                  seed & (2**64 - 1), step & (2**64 - 1),
                                  _ptr(out["tokens"]), _ptr(out["accepted"]), _ptr(out["p"]),
                                  _ptr(out["q"]), _ptr(out["status"]), _ptr(out["flags"]),
                                  _ptr(out["flag_pos"]), _ptr(out["gap"]), nthreads)
    assert rc == 0
    return out


def verify_greedy(target, draft_tokens, num_draft, nthreads: int = 1, early_exit: bool = False) -> dict:
    """Greedy verify of a padded batch; early_exit as in verify_sample."""
    lib = _load()
    t, dt = _logit_array(target)
    B, K1, V = t.shape
    K = K1 - 1
    x = _c(draft_tokens, np.int32).reshape(B, K)
    nd = None if num_draft is None else _c(num_draft, np.int32)
    out = dict(tokens=np.full((B, K + 1), -1, np.int32), accepted=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    fn = lib.oracle_verify_greedy_early_exit if early_exit else lib.oracle_verify_greedy
    rc = fn(_ptr(t), dt, B, K, V, V, _ptr(x), _ptr(nd), _ptr(out["tokens"]),
                                  _ptr(out["accepted"]), _ptr(out["status"]), nthreads)
    assert rc == 0
    return out


def schedule_verify_len(conf, max_len, step_time_us, budget: int, min_len: int) -> dict | None:
    """Confidence-scheduled verify lengths; None for invalid arguments."""
    lib = _load()
    c = _c(conf, np.float32)
    B, K = c.shape
    ml = None if max_len is None else _c(max_len, np.int32)
    tau = _c(step_time_us, np.float32)
    out_len = np.zeros(B, np.int32)
    info = np.zeros(3)
    flags = np.zeros(1, np.int32)
    rc = lib.oracle_schedule_verify_len(_ptr(c), _ptr(ml), B, K, _ptr(tau), tau.size, budget, min_len,
                                        _ptr(out_len), _ptr(info), _ptr(flags))
    if rc != 0:
        return None
    return dict(len=out_len, n=int(info[0]), expected_tokens=float(info[1]),
                tokens_per_us=float(info[2]), flags=int(flags[0]))


def schedule_threshold(conf, max_len, threshold: float) -> np.ndarray | None:
    """Static threshold truncation: L_b = the first position whose confidence is
    below the threshold (NaN counts as below), else maxlen_b; None if invalid."""
    lib = _load()
    c = _c(conf, np.float32)
    B, K = c.shape
    ml = None if max_len is None else _c(max_len, np.int32)
    out = np.zeros(B, np.int32)
    if lib.oracle_schedule_threshold(_ptr(c), _ptr(ml), B, K, float(threshold), _ptr(out)) != 0:
        return None
    return out


def schedule_verify_len_stale(conf_stale, conf, max_len, step_time_us, budget: int, min_len: int) -> dict | None:
    """Two-step-stale batch sizing: the total n* from conf_stale, the slots by conf."""
    lib = _load()
    cs = _c(conf_stale, np.float32)
    c = _c(conf, np.float32)
    B, K = c.shape
    assert cs.shape == c.shape
    ml = None if max_len is None else _c(max_len, np.int32)
    tau = _c(step_time_us, np.float32)
    out_len = np.zeros(B, np.int32)
    info = np.zeros(3)
    flags = np.zeros(1, np.int32)
    rc = lib.oracle_schedule_verify_len_stale(_ptr(cs), _ptr(c), _ptr(ml), B, K, _ptr(tau), tau.size, budget,
                                              min_len, _ptr(out_len), _ptr(info), _ptr(flags))
    if rc != 0:
        return None
    return dict(len=out_len, n=int(info[0]), expected_tokens=float(info[1]),
                tokens_per_us=float(info[2]), flags=int(flags[0]))


# ------------------------------------------------------------------ Markov-head drafting
def markov_draft(base, anchor, emb, proj, temperature, seed: int, step: int, topk: int = 0,
                 nthreads: int = 1, want_logits: bool = True) -> dict:
    """Semi-autoregressive drafting of one block with a rank-r Markov head.

    base [B, K, V] float32 or bf16 bit patterns (uint16): the backbone's logits;
    anchor [B] int32: the token before the block; emb, proj [V, r] in base's dtype;
    temperature [B] float32 (0: greedy) or None (all greedy); topk = 0: the whole
    vocabulary, else only the topk largest base logits are corrected and drawn from.
    Returns tokens [B, K], logits [B, K, V] (the corrected z, -inf outside the
    candidates), status [B] and tie [B] (first position decided within the near-tie
    band, K if none).
    """
    lib = _load()
    u, du = _logit_array(base)
    e, de = _logit_array(emb)
    pr, dp = _logit_array(proj)
    assert du == de == dp
    B, K, V = u.shape
    r = e.shape[1]
    assert e.shape == (V, r) and pr.shape == (V, r)
    a = _c(anchor, np.int32)
    T = None if temperature is None else _c(temperature, np.float32)
    out = dict(tokens=np.full((B, K), -1, np.int32),
               logits=np.zeros((B, K, V)) if want_logits else None,
               status=np.zeros(B, np.int32), tie=np.zeros(B, np.int32))
    rc = lib.oracle_markov_draft(_ptr(u), du, B, K, V, V, _ptr(a), _ptr(e), _ptr(pr), r, _ptr(T),
                                 seed & (2**64 - 1), step & (2**64 - 1), topk, _ptr(out["tokens"]),
                                 _ptr(out["logits"]), _ptr(out["status"]), _ptr(out["tie"]), nthreads)
    assert rc == 0
    return out
