"""ctypes binding of libspecverify.so (include/spec_verify.h).

Argument marshalling only: every step of the verify path runs in the library's
CUDA kernels.  Functions named like the C entry points take torch CUDA tensors,
check shapes / dtypes / devices, pass raw pointers and the current stream, and
raise SpecError on a non-zero return code.  The library must be built
(``__graft_entry__.build()`` or ``_build.build()``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import _build

SPEC_OK, SPEC_EINVAL, SPEC_ECUDA, SPEC_EUNSUPPORTED, SPEC_EWORKSPACE = 0, 1, 2, 3, 4
SPEC_ESCRATCH = 5
SPEC_BF16, SPEC_F32 = 0, 1
STATUS_OK, STATUS_BAD_TOKEN, STATUS_BAD_K, STATUS_BAD_TEMPERATURE, STATUS_NONFINITE = 0, 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


class SpecError(RuntimeError):
    def __init__(self, fn: str, rc: int, lib=None):
        msg = f"{fn} failed: {rc}"
        if lib is not None:
            msg += f" ({lib.spec_error_string(rc).decode()})"
            if rc == SPEC_ECUDA:
                msg += f", cudaError {lib.spec_last_cuda_error()}"
        super().__init__(msg)
        self.rc = rc


def lib_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load libspecverify.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build() (needs nvcc)")
        lib = ctypes.CDLL(p)
        P, I32, I64, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
        lib.spec_verify_workspace_size.argtypes = [I32, I32, I32, I32]
        lib.spec_verify_workspace_size.restype = SZ
        lib.spec_verify_greedy.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, P, P, P, SZ, P]
        lib.spec_verify_greedy.restype = I32
        lib.spec_verify_sample.argtypes = [P, P, I32, I32, I32, I32, I64, P, P, P, U64, U64, P, P, P, P, P,
                                           P, SZ, P]
        lib.spec_verify_sample.restype = I32
        lib.spec_verify_greedy_flat.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, P, P, P, SZ, P]
        lib.spec_verify_greedy_flat.restype = I32
        lib.spec_verify_sample_flat.argtypes = [P, P, I32, I32, I32, I32, I64, P, P, P, U64, U64, P, P, P, P, P,
                                                P, SZ, P]
        lib.spec_verify_sample_flat.restype = I32
        lib.spec_verify_sample_early_exit.argtypes = [P, P, I32, I32, I32, I32, I64, P, P, P, U64, U64, P, P, P,
                                                      P, P, P]
        lib.spec_verify_sample_early_exit.restype = I32
        lib.spec_verify_greedy_early_exit.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, P, P, P]
        lib.spec_verify_greedy_early_exit.restype = I32
        lib.spec_markov_draft.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, I32, P, U64, U64, P, P, P, P]
        lib.spec_markov_draft.restype = I32
        lib.spec_markov_topk_workspace_size.argtypes = [I32, I32, I32, I32]
        lib.spec_markov_topk_workspace_size.restype = SZ
        lib.spec_markov_draft_topk.argtypes = [P, I32, I32, I32, I32, I64, P, P, P, I32, P, U64, U64, I32, P, P, P,
                                               P, SZ, P]
        lib.spec_markov_draft_topk.restype = I32
        lib.spec_verify_sample_noalloc.argtypes = [P, P, I32, I32, I32, I32, I64, P, P, P, U64, U64, P, P, P,
                                                   P, P, P]
        lib.spec_verify_sample_noalloc.restype = I32
        lib.spec_schedule_verify_len.argtypes = [P, P, I32, I32, P, I32, I32, I32, P, P, P]
        lib.spec_schedule_verify_len.restype = I32
        lib.spec_schedule_verify_len_stale.argtypes = [P, P, P, I32, I32, P, I32, I32, I32, P, P, P]
        lib.spec_schedule_verify_len_stale.restype = I32
        lib.spec_schedule_threshold.argtypes = [P, P, I32, I32, ctypes.c_float, P, P]
        lib.spec_schedule_threshold.restype = I32
        lib.spec_error_string.argtypes = [I32]
        lib.spec_error_string.restype = ctypes.c_char_p
        lib.spec_last_cuda_error.argtypes = []
        lib.spec_last_cuda_error.restype = I32
        lib.spec_profile_enable.argtypes = [I32]
        lib.spec_profile_enable.restype = I32
        lib.spec_profile_read.argtypes = [P, I32]
        lib.spec_profile_read.restype = I32
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/spec_verify.h declares."""
    hdr = os.path.join(_build.INCLUDE, "spec_verify.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


# ------------------------------------------------------------------ marshalling
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    """The stream to launch on: the given one (it must belong to `device`), else the
    current stream of `device`, the device that holds the call's tensors."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _call(lib, name: str, device, *args):
    """Call entry point `name` with `device` current: the library launches on the
    current device and looks its per-device state (SM count, scratch) up there."""
    with torch.cuda.device(device):
        rc = getattr(lib, name)(*args)
    if rc != SPEC_OK:
        raise SpecError(name, rc, lib)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need(t, name, dtype=None, shape=None, device=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _logits_layout(t: torch.Tensor, rows_per_req: int):
    """(B, V, ld_row) of a [B, rows, V] logits tensor whose last dim is contiguous."""
    if t.dim() != 3 or t.shape[1] != rows_per_req:
        raise ValueError(f"logits must be [B, {rows_per_req}, V], got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    B, R, V = t.shape
    ld = t.stride(1) if R > 1 else (t.stride(0) if B > 1 else V)
    if V > 1 and t.stride(2) != 1:
        raise ValueError("logits must have V contiguous")
    if ld < V or (R > 1 and B > 1 and t.stride(0) != R * ld) or (R == 1 and B > 1 and t.stride(0) != ld):
        raise ValueError("logit rows must be evenly strided: row (b, i) at (b * rows + i) * ld_row")
    return B, V, ld


def spec_verify_workspace_size(B: int, Kmax: int, V: int, dtype: int) -> int:
    return int(load().spec_verify_workspace_size(B, Kmax, V, dtype))


def spec_verify_greedy(target, draft_tokens, num_draft, out_tokens, out_accepted, out_status, workspace,
                       stream=None) -> None:
    lib = load()
    K1 = target.shape[1]
    Kmax = K1 - 1
    B, V, ld = _logits_layout(target, K1)
    dev = target.device
    _need(draft_tokens, "draft_tokens", torch.int32, (B, Kmax), dev)
    if num_draft is not None:
        _need(num_draft, "num_draft", torch.int32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K1), dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    _call(lib, "spec_verify_greedy", dev, _ptr(target), _dtype_code(target), B, Kmax, V, ld, _ptr(draft_tokens),
                                _ptr(num_draft), _ptr(out_tokens), _ptr(out_accepted), _ptr(out_status),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))


def spec_verify_sample(target, draft, draft_tokens, num_draft, temperature, seed: int, step: int, out_tokens,
                       out_accepted, out_p, out_q, out_status, workspace, stream=None) -> None:
    lib = load()
    K1 = target.shape[1]
    Kmax = K1 - 1
    B, V, ld = _logits_layout(target, K1)
    dev = target.device
    if draft.dtype != target.dtype:
        raise TypeError("target and draft logits must share a dtype")
    if Kmax > 0:
        Bd, Vd, ldd = _logits_layout(draft, Kmax)
        if (Bd, Vd, ldd) != (B, V, ld):
            raise ValueError("draft logits must be [B, Kmax, V] with the target's row stride")
    if draft.device != dev:
        raise ValueError("draft logits must be on the target's device")
    _need(draft_tokens, "draft_tokens", torch.int32, (B, Kmax), dev)
    if num_draft is not None:
        _need(num_draft, "num_draft", torch.int32, (B,), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K1), dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    if out_p is not None:
        _need(out_p, "out_p", torch.float32, (B, Kmax), dev)
    if out_q is not None:
        _need(out_q, "out_q", torch.float32, (B, Kmax), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    _call(lib, "spec_verify_sample", dev, _ptr(target), _ptr(draft), _dtype_code(target), B, Kmax, V, ld,
                                _ptr(draft_tokens), _ptr(num_draft), _ptr(temperature),
                                int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out_tokens),
                                _ptr(out_accepted), _ptr(out_p), _ptr(out_q), _ptr(out_status),
                                _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))


def spec_verify_sample_early_exit(target, draft, draft_tokens, num_draft, temperature, seed: int, step: int,
                                  out_tokens, out_accepted, out_p, out_q, out_status, stream=None) -> None:
    """spec_verify_sample that reads rows in position order and stops at the first
    rejection (no workspace); tensors as for spec_verify_sample."""
    lib = load()
    K1 = target.shape[1]
    Kmax = K1 - 1
    B, V, ld = _logits_layout(target, K1)
    dev = target.device
    if draft.dtype != target.dtype:
        raise TypeError("target and draft logits must share a dtype")
    if Kmax > 0:
        Bd, Vd, ldd = _logits_layout(draft, Kmax)
        if (Bd, Vd, ldd) != (B, V, ld):
            raise ValueError("draft logits must be [B, Kmax, V] with the target's row stride")
    _need(draft_tokens, "draft_tokens", torch.int32, (B, Kmax), dev)
    if num_draft is not None:
        _need(num_draft, "num_draft", torch.int32, (B,), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K1), dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    for t, n in ((out_p, "out_p"), (out_q, "out_q")):
        if t is not None:
            _need(t, n, torch.float32, (B, Kmax), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _call(lib, "spec_verify_sample_early_exit", dev, _ptr(target), _ptr(draft), _dtype_code(target), B, Kmax, V, ld,
                                           _ptr(draft_tokens), _ptr(num_draft), _ptr(temperature),
                                           int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out_tokens),
                                           _ptr(out_accepted), _ptr(out_p), _ptr(out_q), _ptr(out_status),
                                           _stream_handle(stream, dev))


def spec_verify_greedy_early_exit(target, draft_tokens, num_draft, out_tokens, out_accepted, out_status,
                                  stream=None) -> None:
    lib = load()
    K1 = target.shape[1]
    Kmax = K1 - 1
    B, V, ld = _logits_layout(target, K1)
    dev = target.device
    _need(draft_tokens, "draft_tokens", torch.int32, (B, Kmax), dev)
    if num_draft is not None:
        _need(num_draft, "num_draft", torch.int32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K1), dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _call(lib, "spec_verify_greedy_early_exit", dev, _ptr(target), _dtype_code(target), B, Kmax, V, ld, _ptr(draft_tokens),
                                           _ptr(num_draft), _ptr(out_tokens), _ptr(out_accepted),
                                           _ptr(out_status), _stream_handle(stream, dev))


def spec_markov_draft(base, anchor, emb, proj, temperature, seed: int, step: int, out_tokens, out_logits,
                      out_status, stream=None) -> None:
    """Markov-head drafting of one block.  base [B, K, V] (or a [B, K, ld] view with
    unit stride over V), emb / proj [V, r] contiguous in base's dtype, anchor [B]
    int32, temperature [B] float32 or None; outputs tokens [B, K] int32, logits
    [B, K, V] float32, status [B] int32."""
    lib = load()
    B, K = base.shape[0], base.shape[1]
    _, V, ld = _logits_layout(base, K) if K > 0 else (B, base.shape[2], base.shape[2])
    dev = base.device
    if emb.dtype != base.dtype or proj.dtype != base.dtype:
        raise TypeError("the factors must have the base logits' dtype")
    if emb.dim() != 2 or emb.shape[0] != V or proj.shape != emb.shape or not emb.is_contiguous() \
            or not proj.is_contiguous():
        raise ValueError("emb and proj must be contiguous [V, r]")
    _need(anchor, "anchor", torch.int32, (B,), dev)
    if temperature is not None:
        _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K), dev)
    _need(out_logits, "out_logits", torch.float32, (B, K, V), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _call(lib, "spec_markov_draft", dev, _ptr(base), _dtype_code(base), B, K, V, ld, _ptr(anchor), _ptr(emb), _ptr(proj),
                               emb.shape[1], _ptr(temperature), int(seed) & (2**64 - 1), int(step) & (2**64 - 1),
                               _ptr(out_tokens), _ptr(out_logits), _ptr(out_status), _stream_handle(stream, dev))


def spec_markov_topk_workspace_size(B: int, K: int, V: int, topk: int) -> int:
    return int(load().spec_markov_topk_workspace_size(B, K, V, topk))


def spec_markov_draft_topk(base, anchor, emb, proj, temperature, seed: int, step: int, topk: int, out_tokens,
                           out_logits, out_status, ws, stream=None) -> None:
    """Top-K Markov-head drafting of one block: as spec_markov_draft, with only the
    topk largest backbone logits of each position corrected and drawn from.
    out_logits may be None; ws is a uint8 device tensor of at least
    spec_markov_topk_workspace_size(B, K, V, topk) bytes."""
    lib = load()
    B, K = base.shape[0], base.shape[1]
    _, V, ld = _logits_layout(base, K) if K > 0 else (B, base.shape[2], base.shape[2])
    dev = base.device
    if emb.dtype != base.dtype or proj.dtype != base.dtype:
        raise TypeError("the factors must have the base logits' dtype")
    if emb.dim() != 2 or emb.shape[0] != V or proj.shape != emb.shape or not emb.is_contiguous() \
            or not proj.is_contiguous():
        raise ValueError("emb and proj must be contiguous [V, r]")
    _need(anchor, "anchor", torch.int32, (B,), dev)
    if temperature is not None:
        _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K), dev)
    if out_logits is not None:
        _need(out_logits, "out_logits", torch.float32, (B, K, V), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    if ws is not None and ws.device != dev:
        raise ValueError("the workspace must be on the logits' device")
    _call(lib, "spec_markov_draft_topk", dev, _ptr(base), _dtype_code(base), B, K, V, ld, _ptr(anchor), _ptr(emb),
          _ptr(proj), emb.shape[1], _ptr(temperature), int(seed) & (2**64 - 1), int(step) & (2**64 - 1), int(topk),
          _ptr(out_tokens), _ptr(out_logits), _ptr(out_status), _ptr(ws), 0 if ws is None else ws.numel(),
          _stream_handle(stream, dev))


def spec_verify_sample_noalloc(target, draft, draft_tokens, num_draft, temperature, seed: int, step: int,
                               out_tokens, out_accepted, out_p, out_q, out_status, stream=None) -> None:
    """spec_verify_sample on the library's fixed per-device scratch (no workspace).
    Calls on one device must not overlap; sizes beyond the scratch raise SpecError
    with rc SPEC_ESCRATCH."""
    lib = load()
    K1 = target.shape[1]
    Kmax = K1 - 1
    B, V, ld = _logits_layout(target, K1)
    dev = target.device
    if draft.dtype != target.dtype or draft.device != dev:
        raise TypeError("target and draft logits must share a dtype and a device")
    if Kmax > 0 and _logits_layout(draft, Kmax) != (B, V, ld):
        raise ValueError("draft logits must be [B, Kmax, V] with the target's row stride")
    _need(draft_tokens, "draft_tokens", torch.int32, (B, Kmax), dev)
    if num_draft is not None:
        _need(num_draft, "num_draft", torch.int32, (B,), dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, (B, K1), dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    for t, n in ((out_p, "out_p"), (out_q, "out_q")):
        if t is not None:
            _need(t, n, torch.float32, (B, Kmax), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _call(lib, "spec_verify_sample_noalloc", dev, _ptr(target), _ptr(draft), _dtype_code(target), B, Kmax, V, ld,
                                        _ptr(draft_tokens), _ptr(num_draft), _ptr(temperature),
                                        int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out_tokens),
                                        _ptr(out_accepted), _ptr(out_p), _ptr(out_q), _ptr(out_status),
                                        _stream_handle(stream, dev))


def _flat_rows(t: torch.Tensor, name: str):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be [rows, V] with V contiguous")
    return t.shape[1], t.stride(0)


def spec_verify_greedy_flat(target, cu_draft, draft_tokens, out_tokens, out_accepted, out_status, workspace,
                            Kmax: int, stream=None) -> None:
    """Flattened layout: target [sum_b (k_b + 1), V]; cu_draft [B + 1] int32 offsets of the
    draft positions; draft_tokens [sum_b k_b] int32; out_tokens [sum_b (k_b + 1)]."""
    lib = load()
    dev = target.device
    V, ld = _flat_rows(target, "target")
    B = cu_draft.numel() - 1
    _need(cu_draft, "cu_draft", torch.int32, None, dev)
    _need(draft_tokens, "draft_tokens", torch.int32, None, dev)
    _need(out_tokens, "out_tokens", torch.int32, None, dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    _call(lib, "spec_verify_greedy_flat", dev, _ptr(target), _dtype_code(target), B, int(Kmax), V, ld, _ptr(cu_draft),
                                     _ptr(draft_tokens), _ptr(out_tokens), _ptr(out_accepted), _ptr(out_status),
                                     _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))


def spec_verify_sample_flat(target, draft, cu_draft, draft_tokens, temperature, seed: int, step: int, out_tokens,
                            out_accepted, out_p, out_q, out_status, workspace, Kmax: int, stream=None) -> None:
    """Flattened layout; draft [sum_b k_b, V]; out_p / out_q [sum_b k_b] or None."""
    lib = load()
    dev = target.device
    V, ld = _flat_rows(target, "target")
    Vd, ldd = _flat_rows(draft, "draft")
    if Vd != V or ldd != ld or draft.dtype != target.dtype:
        raise ValueError("draft must match target in V, row stride and dtype")
    B = cu_draft.numel() - 1
    _need(cu_draft, "cu_draft", torch.int32, None, dev)
    _need(draft_tokens, "draft_tokens", torch.int32, None, dev)
    _need(temperature, "temperature", torch.float32, (B,), dev)
    _need(out_tokens, "out_tokens", torch.int32, None, dev)
    _need(out_accepted, "out_accepted", torch.int32, (B,), dev)
    _need(out_status, "out_status", torch.int32, (B,), dev)
    for t, n in ((out_p, "out_p"), (out_q, "out_q")):
        if t is not None:
            _need(t, n, torch.float32, None, dev)
    _need(workspace, "workspace", torch.uint8, None, dev)
    _call(lib, "spec_verify_sample_flat", dev, _ptr(target), _ptr(draft), _dtype_code(target), B, int(Kmax), V, ld,
                                     _ptr(cu_draft), _ptr(draft_tokens), _ptr(temperature),
                                     int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _ptr(out_tokens),
                                     _ptr(out_accepted), _ptr(out_p), _ptr(out_q), _ptr(out_status),
                                     _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))


def spec_schedule_verify_len(conf, max_len, step_time_us, budget: int, min_len: int, out_len, out_info=None,
                             stream=None) -> None:
    lib = load()
    if conf.dim() != 2:
        raise ValueError("conf must be [B, Kmax]")
    B, Kmax = conf.shape
    dev = conf.device
    _need(conf, "conf", torch.float32, None, dev)
    if max_len is not None:
        _need(max_len, "max_len", torch.int32, (B,), dev)
    _need(step_time_us, "step_time_us", torch.float32, None, dev)
    _need(out_len, "out_len", torch.int32, (B,), dev)
    if out_info is not None:
        _need(out_info, "out_info", torch.float64, (3,), dev)
    _call(lib, "spec_schedule_verify_len", dev, _ptr(conf), _ptr(max_len), B, Kmax, _ptr(step_time_us),
                                      step_time_us.numel(), int(budget), int(min_len), _ptr(out_len),
                                      _ptr(out_info), _stream_handle(stream, dev))


def spec_schedule_verify_len_stale(conf_stale, conf, max_len, step_time_us, budget: int, min_len: int, out_len,
                                   out_info=None, stream=None) -> None:
    lib = load()
    if conf.dim() != 2 or conf_stale.shape != conf.shape:
        raise ValueError("conf and conf_stale must both be [B, Kmax]")
    B, Kmax = conf.shape
    dev = conf.device
    _need(conf, "conf", torch.float32, None, dev)
    _need(conf_stale, "conf_stale", torch.float32, None, dev)
    if max_len is not None:
        _need(max_len, "max_len", torch.int32, (B,), dev)
    _need(step_time_us, "step_time_us", torch.float32, None, dev)
    _need(out_len, "out_len", torch.int32, (B,), dev)
    if out_info is not None:
        _need(out_info, "out_info", torch.float64, (3,), dev)
    _call(lib, "spec_schedule_verify_len_stale", dev, _ptr(conf_stale), _ptr(conf), _ptr(max_len), B, Kmax,
                                            _ptr(step_time_us), step_time_us.numel(), int(budget), int(min_len),
                                            _ptr(out_len), _ptr(out_info), _stream_handle(stream, dev))


def spec_schedule_threshold(conf, max_len, threshold: float, out_len, stream=None) -> None:
    lib = load()
    if conf.dim() != 2:
        raise ValueError("conf must be [B, Kmax]")
    B, Kmax = conf.shape
    dev = conf.device
    _need(conf, "conf", torch.float32, None, dev)
    if max_len is not None:
        _need(max_len, "max_len", torch.int32, (B,), dev)
    _need(out_len, "out_len", torch.int32, (B,), dev)
    _call(lib, "spec_schedule_threshold", dev, _ptr(conf), _ptr(max_len), B, Kmax, float(threshold), _ptr(out_len),
                                     _stream_handle(stream, dev))


def profile_enable(on: bool) -> None:
    load().spec_profile_enable(1 if on else 0)


def profile_read(n: int = 4) -> list[float]:
    buf = (ctypes.c_float * n)()
    k = load().spec_profile_read(buf, n)
    if k < 0:
        raise SpecError("spec_profile_read", -k, load())
    return [float(buf[i]) for i in range(k)]
