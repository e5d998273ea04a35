"""Seeded synthetic inputs for the verify/commit step and the verify-length scheduler.

Shared by the tests (both the CUDA path and the oracle are fed from here) and by
bench.py.  Every generator draws on the CPU by default; with ``device`` given, the
same recipe draws with that device's generator (other numbers from the same data
seed), which is how bench.py makes its large batches quickly.  This module holds none of the verify method's arithmetic: it only draws
logits, drafts, temperatures and confidences with ``torch.Generator`` on the CPU.
Draft tokens are drawn the way a drafter would propose them (a categorical draw
from softmax(draft / T) with torch's own sampler, or the draft's argmax when T = 0);
that draw precedes the verify step and is not part of it.

Workloads (sizes and distributions follow the pages' setting: Qwen3-sized vocab
151,936, block 7, temperatures 1.0 / 0, batch 64-512):

  tiny     B=1,   K=4,  V=1024,   fp32  t ~ N(0,3^2), d = t + N(0,1), T = 1.0
  small    B=8,   K=8,  V=32000,  bf16  t ~ N(0,3^2) + Zipf, d = t + N(0, s_b^2),
                                        s_b from {0.25, 0.5, 1, 2}, T = 0.8
  main     B=64,  K=7,  V=151936, bf16  t ~ N(0,4^2) + Zipf, d = t + N(0,1),
                                        T_b ~ U[0.6, 1.0]
  ragged   B=256, Kmax=16, V=129280, bf16  confidences Beta(4,1.5) * 0.95^i,
                                        step time 12 + 0.02 n us, budget 1024,
                                        logits as "small" at this V
  stress   B=512, K=4,  V=151936, fp32  even b greedy (T=0), odd b T=1.0, with
                                        adversarial requests (q == p, q off p's
                                        top-50, exact bf16 ties at the argmax)

Zipf prior: -1.1 * ln(v + 1) added to the target logit of token v.
Data seed of step s of workload w: 1000 * w + s (w = 1..5 in the order above).
"""
from __future__ import annotations

import math

import numpy as np
import torch

WORKLOADS = {"tiny": 1, "small": 2, "main": 3, "ragged": 4, "stress": 5}

ZIPF_S = 1.1


def _gen(seed: int, device=None) -> torch.Generator:
    g = torch.Generator(device=device) if device is not None else torch.Generator()
    g.manual_seed(int(seed))
    return g


def zipf_prior(V: int, device=None) -> torch.Tensor:
    return -ZIPF_S * torch.log(torch.arange(V, dtype=torch.float64, device=device) + 1.0)


def _round(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return x.to(dtype)


def _draw_drafts(d_rows: torch.Tensor, T: float, g: torch.Generator) -> torch.Tensor:
    """Propose one token per draft row: categorical from softmax(d / T), or argmax if T == 0."""
    d = d_rows.to(torch.float64)
    if T == 0.0:
        return torch.argmax(d, dim=-1).to(torch.int32)
    probs = torch.softmax(d / T, dim=-1)
    return torch.multinomial(probs, 1, generator=g).squeeze(-1).to(torch.int32)


def make_batch(B: int, K: int, V: int, dtype: torch.dtype, seed: int, *, t_sigma: float = 3.0,
               zipf: bool = False, noise_sigmas=(1.0,), temperature=(1.0, 1.0), greedy_mask=None,
               num_draft=None, unused_fill: float | None = None, device=None) -> dict:
    """Draw one padded verify batch (on the CPU, or with device's generator there).

    temperature: (lo, hi) for T_b ~ U[lo, hi] (lo == hi: constant).
    noise_sigmas: per-request draft noise sigma drawn uniformly from this tuple.
    greedy_mask: optional bool [B]; greedy requests get T = 0 and drafts = argmax(d).
    num_draft: optional int [B] (ragged k_b); rows beyond it are filled with
    ``unused_fill`` (default NaN) so that reading them is detectable.
    """
    g = _gen(seed, device)
    prior = zipf_prior(V, device) if zipf else None
    target = torch.empty((B, K + 1, V), dtype=dtype, device=device)
    draft = torch.empty((B, K, V), dtype=dtype, device=device)
    tokens = torch.zeros((B, K), dtype=torch.int32, device=device)
    lo, hi = temperature
    temps = (lo + (hi - lo) * torch.rand(B, generator=g, dtype=torch.float64, device=device)).to(torch.float32)
    sig_idx = torch.randint(0, len(noise_sigmas), (B,), generator=g, device=device).tolist()
    if greedy_mask is not None:
        temps = torch.where(torch.as_tensor(greedy_mask, device=device), torch.zeros_like(temps), temps)
    temps_h = temps.tolist()
    fill = float("nan") if unused_fill is None else unused_fill
    for b in range(B):
        kb = K if num_draft is None else int(num_draft[b])
        t = t_sigma * torch.randn((K + 1, V), generator=g, dtype=torch.float64, device=device)
        if prior is not None:
            t = t + prior
        d = t[:K] + noise_sigmas[int(sig_idx[b])] * torch.randn((K, V), generator=g, dtype=torch.float64,
                                                                device=device)
        tb = _round(t, dtype)
        db = _round(d, dtype)
        T = float(temps_h[b])
        if kb > 0:
            tokens[b, :kb] = _draw_drafts(db[:kb], T, g)
        if kb < K:
            tb[kb + 1:] = fill
            db[kb:] = fill
        target[b] = tb
        draft[b] = db
    return dict(target=target, draft=draft, draft_tokens=tokens,
                num_draft=None if num_draft is None else torch.as_tensor(num_draft, dtype=torch.int32, device=device),
                temperature=temps, B=B, K=K, V=V, dtype=dtype)


def tiny(step: int = 0, device=None) -> dict:
    b = make_batch(1, 4, 1024, torch.float32, 1000 * 1 + step, t_sigma=3.0, noise_sigmas=(1.0,),
                   temperature=(1.0, 1.0), device=device)
    b.update(seed=1, step=step, name="tiny")
    return b


def small(step: int = 0, V: int = 32000, device=None) -> dict:
    b = make_batch(8, 8, V, torch.bfloat16, 1000 * 2 + step, t_sigma=3.0, zipf=True,
                   noise_sigmas=(0.25, 0.5, 1.0, 2.0), temperature=(0.8, 0.8), device=device)
    b.update(seed=2, step=step, name="small")
    return b


def main(step: int = 0, B: int = 64, device=None) -> dict:
    b = make_batch(B, 7, 151936, torch.bfloat16, 1000 * 3 + step, t_sigma=4.0, zipf=True,
                   noise_sigmas=(1.0,), temperature=(0.6, 1.0), device=device)
    b.update(seed=3, step=step, name="main")
    return b


def ragged_schedule_inputs(step: int = 0, B: int = 256, Kmax: int = 16) -> dict:
    """Confidences Beta(4, 1.5) * 0.95^i, step-time table 12 + 0.02 n us (n = 0..1024)."""
    g = _gen(1000 * 4 + step)
    # Beta(4, 1.5) as X / (X + Y) with X ~ Gamma(4), Y ~ Gamma(1.5), drawn with the seeded generator
    x = _gamma(4.0, (B, Kmax), g)
    y = _gamma(1.5, (B, Kmax), g)
    beta = x / (x + y)
    decay = 0.95 ** torch.arange(Kmax, dtype=torch.float64)
    conf = (beta * decay).to(torch.float32)
    n = torch.arange(1025, dtype=torch.float64)
    tau = (12.0 + 0.02 * n).to(torch.float32)
    return dict(conf=conf, step_time_us=tau, budget=1024, min_len=1, B=B, Kmax=Kmax)


def _gamma(shape: float, size, g: torch.Generator) -> torch.Tensor:
    """Gamma(shape, 1) by Marsaglia-Tsang squeeze, vectorised, from the seeded generator."""
    out = torch.empty(size, dtype=torch.float64).view(-1)
    n = out.numel()
    boost = shape < 1.0
    a = shape + 1.0 if boost else shape
    dd = a - 1.0 / 3.0
    cc = 1.0 / math.sqrt(9.0 * dd)
    filled = 0
    while filled < n:
        m = 2 * (n - filled) + 16
        z = torch.randn(m, generator=g, dtype=torch.float64)
        u = torch.rand(m, generator=g, dtype=torch.float64)
        v = (1.0 + cc * z) ** 3
        ok = (v > 0) & (torch.log(u.clamp_min(1e-300)) < 0.5 * z * z + dd - dd * v + dd * torch.log(v.clamp_min(1e-300)))
        acc = (dd * v)[ok]
        take = min(acc.numel(), n - filled)
        out[filled:filled + take] = acc[:take]
        filled += take
    if boost:
        u = torch.rand(n, generator=g, dtype=torch.float64)
        out = out * u ** (1.0 / shape)
    return out.view(size)


def ragged(step: int = 0, num_draft=None, V: int = 129280, B: int = 256, Kmax: int = 16, device=None) -> dict:
    """Verify inputs of the ragged workload: 'small'-style logits at V, k_b = num_draft."""
    if num_draft is None:
        num_draft = [Kmax] * B
    b = make_batch(B, Kmax, V, torch.bfloat16, 1000 * 4 + 500 + step, t_sigma=3.0, zipf=True,
                   noise_sigmas=(0.25, 0.5, 1.0, 2.0), temperature=(0.8, 0.8), num_draft=num_draft, device=device)
    b.update(seed=4, step=step, name="ragged")
    return b


def stress(step: int = 0, B: int = 512, V: int = 151936, n_adv: int = 8, device=None) -> dict:
    """Half greedy (even b), half sampling at T = 1 (odd b), fp32, with adversarial requests.

    Adversarial sets (n_adv each, drawn from the first requests of each parity):
      odd b  3, 7, ...: draft logits bitwise equal to the target's (q == p);
      odd b  1, 5, ...: draft = target - 1e4 on the target's 50 largest entries, so
                        the proposals fall outside p's top-50;
      even b 0, 2, ...: a row where two entries share the exact (bf16-valued) max and
                        the draft proposes the higher of the two indices.
    Draft logits of greedy requests are never read; they are filled with NaN.
    """
    K = 4
    g = _gen(1000 * 5 + step, device)
    prior = zipf_prior(V, device)
    target = torch.empty((B, K + 1, V), dtype=torch.float32, device=device)
    draft = torch.empty((B, K, V), dtype=torch.float32, device=device)
    tokens = torch.zeros((B, K), dtype=torch.int32, device=device)
    temps = torch.where(torch.arange(B, device=device) % 2 == 0, 0.0, 1.0).to(torch.float32)
    temps_h = temps.tolist()
    kinds = ["plain"] * B
    odd = [b for b in range(B) if b % 2 == 1]
    even = [b for b in range(B) if b % 2 == 0]
    for b in odd[0:2 * n_adv:2]:
        kinds[b] = "top50_off"
    for b in odd[1:2 * n_adv:2]:
        kinds[b] = "q_eq_p"
    for b in even[:n_adv]:
        kinds[b] = "tie"
    for b in range(B):
        t = 4.0 * torch.randn((K + 1, V), generator=g, dtype=torch.float64, device=device) + prior
        if kinds[b] == "tie":
            t = t.to(torch.bfloat16).to(torch.float64)  # bf16-valued entries
            for i in range(K + 1):
                top2 = torch.topk(t[i], 2).indices
                lo_i, hi_i = sorted(int(v) for v in top2)
                t[i, hi_i] = t[i, lo_i]
        tb = t.to(torch.float32)
        if temps_h[b] == 0.0:
            db = torch.full((K, V), float("nan"), dtype=torch.float32, device=device)
            if kinds[b] == "tie":
                for i in range(K):
                    mx = tb[i].max()
                    idx = torch.nonzero(tb[i] == mx).flatten()
                    tokens[b, i] = int(idx.max())
            else:
                d = t[:K] + 0.5 * torch.randn((K, V), generator=g, dtype=torch.float64, device=device)
                tokens[b] = torch.argmax(d, dim=-1).to(torch.int32)
        else:
            if kinds[b] == "q_eq_p":
                db = tb[:K].clone()
            else:
                d = t[:K] + 1.0 * torch.randn((K, V), generator=g, dtype=torch.float64, device=device)
                if kinds[b] == "top50_off":
                    for i in range(K):
                        top = torch.topk(t[i], 50).indices
                        d[i, top] = d[i, top] - 1e4
                db = d.to(torch.float32)
            tokens[b] = _draw_drafts(db, float(temps_h[b]), g)
        target[b] = tb
        draft[b] = db
    return dict(target=target, draft=draft, draft_tokens=tokens, num_draft=None, temperature=temps,
                B=B, K=K, V=V, dtype=torch.float32, seed=5, step=step, name="stress", kinds=kinds)


def markov(step: int = 0, B: int = 64, K: int = 7, V: int = 151936, r: int = 256,
           dtype: torch.dtype = torch.bfloat16, greedy_every: int = 0) -> dict:
    """Inputs of one Markov-head drafting block: backbone logits U ~ N(0, 3^2) + Zipf,
    factors emb ~ N(0, 0.5^2) and proj ~ N(0, 0.1^2) ([V, r]; the bias of a token
    then has standard deviation ~0.8), anchors uniform over the vocabulary,
    T_b ~ U[0.6, 1.0] (every greedy_every-th request greedy if greedy_every > 0).
    Random weights: no trained head is used."""
    g = _gen(1000 * 6 + step)
    prior = zipf_prior(V)
    base = _round(3.0 * torch.randn((B, K, V), generator=g, dtype=torch.float64) + prior, dtype)
    emb = _round(0.5 * torch.randn((V, r), generator=g, dtype=torch.float64), dtype)
    proj = _round(0.1 * torch.randn((V, r), generator=g, dtype=torch.float64), dtype)
    anchor = torch.randint(0, V, (B,), generator=g, dtype=torch.int64).to(torch.int32)
    temps = (0.6 + 0.4 * torch.rand(B, generator=g, dtype=torch.float64)).to(torch.float32)
    if greedy_every > 0:
        temps[::greedy_every] = 0.0
    return dict(base=base, emb=emb, proj=proj, anchor=anchor, temperature=temps, B=B, K=K, V=V, r=r,
                dtype=dtype, seed=6, step=step, name="markov")


def as_oracle_array(x: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy for the oracle (bf16 as uint16 bit patterns)."""
    x = x.contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()
