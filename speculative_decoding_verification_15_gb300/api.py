"""Convenience layer over the C ABI: allocates outputs and a cached workspace.

Every call goes through the C entry points in ``binding``; this module only
manages tensors.  Shapes follow the C ABI: target logits [B, K+1, V], draft logits
[B, K, V] (bfloat16 or float32), draft tokens [B, K] int32.
"""
from __future__ import annotations

import threading

import torch

from . import binding

_ws_lock = threading.Lock()
_ws_cache: dict[int, torch.Tensor] = {}


def workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """A cached uint8 workspace of at least nbytes on device (grown on demand).

    It is zero-filled when allocated: the verify calls need a zeroed workspace
    before its first use and leave it ready for the next call."""
    idx = torch.device(device).index
    if idx is None:
        idx = torch.cuda.current_device()
    with _ws_lock:
        ws = _ws_cache.get(idx)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 1), dtype=torch.uint8, device=torch.device("cuda", idx))
            _ws_cache[idx] = ws
        return ws


def _as_i32(t, device):
    return None if t is None else t.to(device=device, dtype=torch.int32).contiguous()


def verify_sample(target, draft, draft_tokens, temperature, seed: int, step: int, num_draft=None,
                  stream=None, want_probs: bool = True) -> dict:
    dev = target.device
    B, K1, V = target.shape
    K = K1 - 1
    x = _as_i32(draft_tokens, dev)
    nd = _as_i32(num_draft, dev)
    T = temperature.to(device=dev, dtype=torch.float32).contiguous()
    out = dict(tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev),
               p=torch.empty((B, K), dtype=torch.float32, device=dev) if want_probs else None,
               q=torch.empty((B, K), dtype=torch.float32, device=dev) if want_probs else None)
    ws = workspace(dev, binding.spec_verify_workspace_size(B, K, V, binding._dtype_code(target)))
    binding.spec_verify_sample(target, draft, x, nd, T, seed, step, out["tokens"], out["accepted"], out["p"],
                               out["q"], out["status"], ws, stream)
    return out


def verify_greedy(target, draft_tokens, num_draft=None, stream=None) -> dict:
    dev = target.device
    B, K1, V = target.shape
    x = _as_i32(draft_tokens, dev)
    nd = _as_i32(num_draft, dev)
    out = dict(tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = workspace(dev, binding.spec_verify_workspace_size(B, K1 - 1, V, binding._dtype_code(target)))
    binding.spec_verify_greedy(target, x, nd, out["tokens"], out["accepted"], out["status"], ws, stream)
    return out


def schedule_verify_len(conf, step_time_us, budget: int, min_len: int, max_len=None, stream=None):
    dev = conf.device
    B = conf.shape[0]
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    info = torch.empty(3, dtype=torch.float64, device=dev)
    binding.spec_schedule_verify_len(conf.to(torch.float32).contiguous(), _as_i32(max_len, dev),
                                     step_time_us.to(device=dev, dtype=torch.float32).contiguous(), budget,
                                     min_len, out_len, info, stream)
    return out_len, info


def verify_sample_early_exit(target, draft, draft_tokens, temperature, seed: int, step: int, num_draft=None,
                             stream=None) -> dict:
    """Sampling verify that stops reading at each request's first rejection."""
    dev = target.device
    B, K1, V = target.shape
    K = K1 - 1
    out = dict(tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               p=torch.empty((B, K), dtype=torch.float32, device=dev),
               q=torch.empty((B, K), dtype=torch.float32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    binding.spec_verify_sample_early_exit(target, draft, _as_i32(draft_tokens, dev), _as_i32(num_draft, dev),
                                          temperature.to(device=dev, dtype=torch.float32).contiguous(), seed, step,
                                          out["tokens"], out["accepted"], out["p"], out["q"], out["status"],
                                          stream)
    return out


def verify_greedy_early_exit(target, draft_tokens, num_draft=None, stream=None) -> dict:
    """Greedy verify that stops reading at each request's first mismatch."""
    dev = target.device
    B, K1, V = target.shape
    out = dict(tokens=torch.empty((B, K1), dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    binding.spec_verify_greedy_early_exit(target, _as_i32(draft_tokens, dev), _as_i32(num_draft, dev),
                                          out["tokens"], out["accepted"], out["status"], stream)
    return out


def markov_draft(base, anchor, emb, proj, temperature=None, seed: int = 0, step: int = 0, stream=None) -> dict:
    """Markov-head drafting of one block: tokens [B, K], corrected logits [B, K, V]
    (float32) and status [B]."""
    dev = base.device
    B, K, V = base.shape
    out = dict(tokens=torch.empty((B, K), dtype=torch.int32, device=dev),
               logits=torch.empty((B, K, V), dtype=torch.float32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    T = None if temperature is None else temperature.to(device=dev, dtype=torch.float32).contiguous()
    binding.spec_markov_draft(base, _as_i32(anchor, dev), emb, proj, T, seed, step, out["tokens"], out["logits"],
                              out["status"], stream)
    return out


def markov_draft_topk(base, anchor, emb, proj, topk: int, temperature=None, seed: int = 0, step: int = 0,
                      want_logits: bool = True, stream=None) -> dict:
    """Top-K Markov-head drafting of one block: tokens [B, K], corrected logits
    [B, K, V] (float32, -inf outside each position's topk candidates; None unless
    want_logits) and status [B]."""
    dev = base.device
    B, K, V = base.shape
    out = dict(tokens=torch.empty((B, K), dtype=torch.int32, device=dev),
               logits=torch.empty((B, K, V), dtype=torch.float32, device=dev) if want_logits else None,
               status=torch.empty(B, dtype=torch.int32, device=dev))
    T = None if temperature is None else temperature.to(device=dev, dtype=torch.float32).contiguous()
    ws = torch.empty(max(binding.spec_markov_topk_workspace_size(B, K, V, topk), 16), dtype=torch.uint8, device=dev)
    binding.spec_markov_draft_topk(base, _as_i32(anchor, dev), emb, proj, T, seed, step, topk, out["tokens"],
                                   out["logits"], out["status"], ws, stream)
    return out


def verify_sample_flat(target, draft, cu_draft, draft_tokens, temperature, seed: int, step: int, Kmax: int,
                       stream=None) -> dict:
    """Flattened ragged layout (no padding rows): target [sum_b (k_b + 1), V], draft
    [sum_b k_b, V], cu_draft [B + 1] offsets of the draft positions, draft_tokens
    [sum_b k_b]; Kmax bounds every k_b.  Outputs are flattened the same way."""
    dev = target.device
    cu = _as_i32(cu_draft, dev)
    B = cu.numel() - 1
    n_tok = target.shape[0]
    out = dict(tokens=torch.empty(n_tok, dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               p=torch.empty(draft.shape[0], dtype=torch.float32, device=dev),
               q=torch.empty(draft.shape[0], dtype=torch.float32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = workspace(dev, binding.spec_verify_workspace_size(B, Kmax, target.shape[1], binding._dtype_code(target)))
    binding.spec_verify_sample_flat(target, draft, cu, _as_i32(draft_tokens, dev),
                                    temperature.to(device=dev, dtype=torch.float32).contiguous(), seed, step,
                                    out["tokens"], out["accepted"], out["p"], out["q"], out["status"], ws, Kmax,
                                    stream)
    return out


def verify_greedy_flat(target, cu_draft, draft_tokens, Kmax: int, stream=None) -> dict:
    """Greedy verify in the flattened ragged layout (see verify_sample_flat)."""
    dev = target.device
    cu = _as_i32(cu_draft, dev)
    B = cu.numel() - 1
    out = dict(tokens=torch.empty(target.shape[0], dtype=torch.int32, device=dev),
               accepted=torch.empty(B, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    ws = workspace(dev, binding.spec_verify_workspace_size(B, Kmax, target.shape[1], binding._dtype_code(target)))
    binding.spec_verify_greedy_flat(target, cu, _as_i32(draft_tokens, dev), out["tokens"], out["accepted"],
                                    out["status"], ws, Kmax, stream)
    return out


def schedule_verify_len_stale(conf_stale, conf, step_time_us, budget: int, min_len: int, max_len=None,
                              stream=None):
    dev = conf.device
    B = conf.shape[0]
    out_len = torch.empty(B, dtype=torch.int32, device=dev)
    info = torch.empty(3, dtype=torch.float64, device=dev)
    binding.spec_schedule_verify_len_stale(conf_stale.to(device=dev, dtype=torch.float32).contiguous(),
                                           conf.to(torch.float32).contiguous(), _as_i32(max_len, dev),
                                           step_time_us.to(device=dev, dtype=torch.float32).contiguous(), budget,
                                           min_len, out_len, info, stream)
    return out_len, info


def schedule_threshold(conf, threshold: float, max_len=None, stream=None):
    dev = conf.device
    out_len = torch.empty(conf.shape[0], dtype=torch.int32, device=dev)
    binding.spec_schedule_threshold(conf.to(torch.float32).contiguous(), _as_i32(max_len, dev), threshold,
                                    out_len, stream)
    return out_len


def verify_sample_host(target_h, draft_h, tokens_h, temperature_h, seed: int, step: int, num_draft_h=None,
                       device=None, dev_buffers: dict | None = None) -> dict:
    """End-to-end call from host (ideally pinned) tensors: copy in, verify, copy the
    emitted tokens, accepted counts and statuses back.  Returns host tensors."""
    device = torch.device(device or "cuda")
    bufs = dev_buffers if dev_buffers is not None else {}

    def dev_copy(name, t):
        if t is None:
            return None
        d = bufs.get(name)
        if d is None or d.shape != t.shape or d.dtype != t.dtype:
            d = torch.empty(t.shape, dtype=t.dtype, device=device)
            bufs[name] = d
        d.copy_(t, non_blocking=True)
        return d

    t = dev_copy("target", target_h)
    d = dev_copy("draft", draft_h)
    x = dev_copy("tokens", tokens_h)
    T = dev_copy("temperature", temperature_h)
    nd = dev_copy("num_draft", num_draft_h)
    out = verify_sample(t, d, x, T, seed, step, num_draft=nd, want_probs=False)
    host = {k: v.to("cpu", non_blocking=True) for k, v in out.items() if v is not None}
    torch.cuda.current_stream().synchronize()
    return host
