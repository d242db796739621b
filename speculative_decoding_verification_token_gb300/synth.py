"""Seeded synthetic inputs for the verify / draft / schedule workloads.

This module only draws random inputs with the shapes and value distributions of the five
workloads; it holds none of the method's arithmetic (no softmax, no sampling, no verification).
Both the CUDA path and the CPU oracle are fed from it.

Workloads (logits are row-major, one row per (request, position)):

* ``token_small``  -- 4 requests, 4 drafted positions + 1 bonus, V = 1024, fp32; target logits
  N(0, 2^2), draft = target + N(0, 0.5^2).
* ``token_large``  -- 64 requests, 5 drafted positions, V = 151936, bf16; target N(0, 3^2) plus a
  Zipf(1.1) log-prior -1.1 * ln(v + 1) over token ids; draft = target + N(0, 1).
* ``block_large``  -- 128 requests, 7 drafted positions, V = 129280, bf16; target as above; draft =
  target + N(0, sigma_r^2) with sigma_r ~ U[0.3, 1.5] per request.
* ``markov``       -- 256 requests, block length 16, V = 151936; backbone logits N(0, 2^2) bf16;
  U [V, 256] and W [256, V] bf16 N(0, 0.02^2); anchors uniform over the vocabulary; confidence
  scores N(0, 1); per-position STS temperatures U[0.8, 1.2].
* ``lmhead``       -- 64 requests, 5 drafted positions, V = 151936, hidden size 2560; bf16 hidden
  rows and output projection whose products give the ``token_large`` logit recipe.
* ``scheduled``    -- 512 requests x 16 positions; conditional acceptance c[i, k] = Beta(8, 2) draw
  times 0.97^(k-1); engine curve SPS(B) = 1 / (2 ms + B * 0.4 us) for B <= 8192; logits for all 17
  target and 16 draft rows per request as in ``token_large`` with V = 129280.

Draft tokens are not drawn here: they are sampled from q by the method itself (the CUDA sampler on
the product path, the oracle's sampler in tests).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class TokenWorkload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: torch.dtype
    target_std: float
    zipf: float            # exponent of the log-prior over token ids (0 = none)
    draft_noise: float     # std of the draft perturbation (ignored if noise_range is set)
    noise_range: tuple | None  # per-request std range (block workload)
    seed: int              # Philox seed of the method's uniforms
    gen_seed: int          # seed of the input generator


TOKEN_SMALL = TokenWorkload("token_small", 4, 4, 1024, torch.float32, 2.0, 0.0, 0.5, None, 0, 1001)
TOKEN_LARGE = TokenWorkload("token_large", 64, 5, 151936, torch.bfloat16, 3.0, 1.1, 1.0, None, 1,
                            1002)
BLOCK_LARGE = TokenWorkload("block_large", 128, 7, 129280, torch.bfloat16, 3.0, 1.1, 1.0,
                            (0.3, 1.5), 2, 1003)
SCHEDULED_VERIFY = TokenWorkload("scheduled", 512, 16, 129280, torch.bfloat16, 3.0, 1.1, 1.0,
                                 None, 4, 1005)


def scaled(w: TokenWorkload, **kw) -> TokenWorkload:
    """The same recipe at other sizes (for tests that the oracle must finish in seconds)."""
    return replace(w, **kw)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def token_inputs(w: TokenWorkload, device="cpu", draft_len=None):
    """Logits and row layout of a verify workload.

    Request r owns target rows r*(gamma+1) .. r*(gamma+1)+gamma and draft rows r*gamma ..
    r*gamma+gamma-1 (``draft_len`` may shorten a request: its rows stay where they are, the
    verifier reads only the first draft_len[r] + 1 target and draft_len[r] draft rows).
    """
    B, G, V = w.B, w.gamma, w.V
    g = _gen(device, w.gen_seed)
    n_t, n_d = B * (G + 1), B * G
    target = torch.randn((n_t, V), generator=g, device=device, dtype=torch.float32)
    target.mul_(w.target_std)
    if w.zipf:
        prior = -w.zipf * torch.log(torch.arange(V, device=device, dtype=torch.float32) + 1.0)
        target.add_(prior)
    # draft rows follow the target rows of the same request and position
    t_view = target.view(B, G + 1, V)[:, :G, :].reshape(n_d, V)
    noise = torch.randn((n_d, V), generator=g, device=device, dtype=torch.float32)
    if w.noise_range is not None:
        lo, hi = w.noise_range
        sig = lo + (hi - lo) * torch.rand((B, 1), generator=g, device=device)
        noise.view(B, G, V).mul_(sig.view(B, 1, 1))
    else:
        noise.mul_(w.draft_noise)
    draft = t_view + noise
    target = target.to(w.dtype)
    draft = draft.to(w.dtype)
    if draft_len is None:
        draft_len = torch.full((B,), G, dtype=torch.int32)
    draft_len = torch.as_tensor(draft_len, dtype=torch.int32).to(device)
    return {
        "target": target,
        "draft": draft,
        "V": V,
        "ld": V,
        "target_row0": (torch.arange(B, dtype=torch.int64) * (G + 1)).to(device),
        "draft_row0": (torch.arange(B, dtype=torch.int64) * G).to(device),
        "draft_len": draft_len,
        "max_draft_len": G,
        "B": B,
        "seed": w.seed,
    }


def ragged_lengths(B, gamma_max, seed):
    """Per-request drafted lengths uniform over 0..gamma_max (ragged batches in tests)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, gamma_max + 1, size=B).astype(np.int32)


@dataclass(frozen=True)
class MarkovWorkload:
    name: str
    B: int
    K: int
    V: int
    R: int
    backbone_std: float
    weight_std: float
    seed: int
    gen_seed: int


# The drafting workload: backbone ~ N(0, 2^2), U and W ~ N(0, 0.02^2) (bias std 0.0064).
MARKOV = MarkovWorkload("markov", 256, 16, 151936, 256, 2.0, 0.02, 3, 1004)
# Parity case: several M-blocks and vocabulary tiles with ragged tails (B % 128 != 0,
# V % 64 != 0); U, W ~ N(0, 0.25^2) give the bias U[x] . W unit scale, so the contraction moves
# z by many bf16 ulps and an error in it cannot hide below the backbone's rounding.
MARKOV_SMALL = MarkovWorkload("markov_small", 200, 3, 1000, 256, 2.0, 0.25, 5, 1006)


def markov_inputs(w: MarkovWorkload, device="cpu"):
    g = _gen(device, w.gen_seed)
    B, K, V, R = w.B, w.K, w.V, w.R
    backbone = (torch.randn((B, K, V), generator=g, device=device) * w.backbone_std)
    U = torch.randn((V, R), generator=g, device=device) * w.weight_std
    W = torch.randn((R, V), generator=g, device=device) * w.weight_std
    anchor = torch.randint(0, V, (B,), generator=g, device=device, dtype=torch.int64)
    scores = torch.randn((B, K), generator=g, device=device)
    T = 0.8 + 0.4 * torch.rand((K,), generator=g, device=device)
    return {
        "backbone": backbone.to(torch.bfloat16),
        "U": U.to(torch.bfloat16),
        "W": W.to(torch.bfloat16),
        "Wt": W.t().contiguous().to(torch.bfloat16),
        "anchor": anchor.to(torch.int32),
        "scores": scores.float(),
        "T": T.float(),
        "B": B, "K": K, "V": V, "R": R,
        "seed": w.seed,
    }


@dataclass(frozen=True)
class LmHeadWorkload:
    name: str
    B: int
    gamma: int
    V: int
    H: int
    target_std: float      # std of the target logits h . W[v] (before the prior)
    zipf: float            # exponent of the log-prior over token ids, carried by hidden column 0
    draft_noise: float     # std of the draft logits' deviation from the target's
    seed: int
    gen_seed: int


# Verification from hidden states: 64 requests, 5 drafted positions, V = 151936, hidden size 2560
# (a Qwen3-4B-sized target), bf16.  Logits h . W[v] ~ N(0, 3^2) plus the Zipf(1.1) prior, draft
# logits = target + N(0, 1): the token_large logit recipe, produced through an output projection.
LMHEAD = LmHeadWorkload("lmhead", 64, 5, 151936, 2560, 3.0, 1.1, 1.0, 6, 1007)
# Parity case: several slot blocks and vocabulary tiles with ragged tails (V % 256 != 0), and an
# odd number of 64-wide k-blocks.
LMHEAD_SMALL = LmHeadWorkload("lmhead_small", 24, 5, 4099, 320, 3.0, 1.1, 1.0, 7, 1008)


def lmhead_inputs(w: LmHeadWorkload, device="cpu", draft_len=None):
    """Hidden rows and the output projection of a verify-from-hidden-states workload.

    Target hidden rows h ~ N(0, 1) and W ~ N(0, (target_std / sqrt(H - 1))^2) make h . W[v] ~
    N(0, target_std^2); hidden column 0 is the constant 1 and W[v][0] = -zipf ln(v + 1), so every
    logit carries the prior.  Draft row j of a request is its target row j plus
    N(0, (draft_noise / target_std)^2) in columns 1.., so draft logits = target + N(0,
    draft_noise^2).  Row layout as in token_inputs: request r owns target rows r (gamma + 1) + j and
    draft rows r gamma + j.
    """
    B, G, V, H = w.B, w.gamma, w.V, w.H
    g = _gen(device, w.gen_seed)
    n_t, n_d = B * (G + 1), B * G
    target = torch.randn((n_t, H), generator=g, device=device, dtype=torch.float32)
    W = torch.randn((V, H), generator=g, device=device, dtype=torch.float32)
    W.mul_(w.target_std / math.sqrt(H - 1))
    target[:, 0] = 1.0
    W[:, 0] = -w.zipf * torch.log(torch.arange(V, device=device, dtype=torch.float32) + 1.0)
    t_view = target.view(B, G + 1, H)[:, :G, :].reshape(n_d, H)
    noise = torch.randn((n_d, H), generator=g, device=device, dtype=torch.float32)
    noise.mul_(w.draft_noise / w.target_std)
    noise[:, 0] = 0.0
    draft = t_view + noise
    if draft_len is None:
        draft_len = torch.full((B,), G, dtype=torch.int32)
    draft_len = torch.as_tensor(draft_len, dtype=torch.int32).to(device)
    return {
        "target_hidden": target.to(torch.bfloat16),
        "draft_hidden": draft.to(torch.bfloat16),
        "W": W.to(torch.bfloat16),
        "V": V,
        "H": H,
        "target_row0": (torch.arange(B, dtype=torch.int64) * (G + 1)).to(device),
        "draft_row0": (torch.arange(B, dtype=torch.int64) * G).to(device),
        "draft_len": draft_len,
        "max_draft_len": G,
        "B": B,
        "seed": w.seed,
    }


@dataclass(frozen=True)
class ScheduleWorkload:
    name: str
    N: int
    K: int
    B_max: int
    fixed_ms: float
    per_row_us: float
    decay: float
    beta_a: float
    beta_b: float
    gen_seed: int


SCHEDULE = ScheduleWorkload("scheduled", 512, 16, 8192, 2.0, 0.4, 0.97, 8.0, 2.0, 1005)


def schedule_inputs(w: ScheduleWorkload, max_len=None):
    """Conditional acceptance probabilities [N, K] (float32) and the engine curve SPS[0..B_max]."""
    rng = np.random.default_rng(w.gen_seed)
    c = rng.beta(w.beta_a, w.beta_b, size=(w.N, w.K))
    c = c * (w.decay ** np.arange(w.K))[None, :]
    Bs = np.arange(w.B_max + 1, dtype=np.float64)
    sps = 1.0 / (w.fixed_ms * 1e-3 + Bs * w.per_row_us * 1e-6)
    if max_len is None:
        max_len = np.full(w.N, w.K, dtype=np.int32)
    return {
        "cond_accept": c.astype(np.float32),
        "max_len": np.asarray(max_len, dtype=np.int32),
        "sps": sps,
        "N": w.N, "K": w.K, "B_max": w.B_max,
    }


def bytes_of_rows(n_rows, V, dtype):
    return int(n_rows) * int(V) * torch.empty((), dtype=dtype).element_size()


def nearest_multiple(x, m):
    return int(math.ceil(x / m) * m)
