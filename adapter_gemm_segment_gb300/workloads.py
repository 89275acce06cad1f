"""Seeded synthetic inputs for the multi-LoRA segmented linear.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the layer's arithmetic; both the CUDA path (tests, bench)
and the CPU oracle receive the tensors it returns.

Shapes and distributions follow the workloads of the multi-LoRA serving pages
("LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排", blog.lonae.com: a 7B base
with hidden size 4096, rank-8/alpha-16 adapters, up to 100 adapters, batch 1-64
at decode; 512-token prefill chunks from the fair-scheduling page):

* W_base ~ N(0, 0.02), A ~ U(-1/sqrt(h_in), +1/sqrt(h_in)), B ~ N(0, 0.01),
  x ~ N(0, 1); everything is drawn in float64 with numpy's PCG64 and rounded
  once (round-to-nearest-even) to the workload dtype.
* Adapter choice: a finite Zipf law p(k) ~ k^-1.1, k = 1..S, mapped to slot
  k-1 (slot 0 is the hottest); "10 % base-only" means an independent
  Bernoulli(0.1) per token that sets idx = -1.
* Draw order inside one case is fixed: idx, W, A, B, x.

Every case is a plain dict of CPU tensors (see ``LinearCase``).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass
class AdapterSet:
    """Adapters at their true rank, as an adapter file would hold them."""

    A: List[torch.Tensor]  # slot s: [rank_s, h_in]
    B: List[torch.Tensor]  # slot s: [h_out, rank_s]
    ranks: List[int]
    alphas: List[float]
    r_max: int

    @property
    def n_slots(self) -> int:
        return len(self.ranks)


@dataclasses.dataclass
class LinearCase:
    """One LoRA-augmented linear over one batch."""

    name: str
    x: torch.Tensor  # [n, h_in]
    W: torch.Tensor  # [h_out, h_in]
    adapters: AdapterSet
    idx: torch.Tensor  # int32 [n]; -1 = base only

    @property
    def n(self) -> int:
        return int(self.x.shape[0])

    @property
    def h_in(self) -> int:
        return int(self.x.shape[1])

    @property
    def h_out(self) -> int:
        return int(self.W.shape[0])

    @property
    def dtype(self) -> torch.dtype:
        return self.x.dtype


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(key))


def _round(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(dtype)


def zipf_probs(n_slots: int, s: float = 1.1) -> np.ndarray:
    k = np.arange(1, n_slots + 1, dtype=np.float64)
    p = k ** (-s)
    return p / p.sum()


def draw_zipf_idx(rng: np.random.Generator, n: int, n_slots: int, p_base: float = 0.0,
                  s: float = 1.1) -> np.ndarray:
    """Zipf slot per token; with probability p_base the token is base-only (-1)."""
    base = rng.random(n) < p_base if p_base > 0 else np.zeros(n, dtype=bool)
    cdf = np.cumsum(zipf_probs(n_slots, s))
    u = rng.random(n)
    slot = np.minimum(np.searchsorted(cdf, u, side="right"), n_slots - 1)
    return np.where(base, -1, slot).astype(np.int32)


def draw_uniform_idx(rng: np.random.Generator, n: int, n_slots: int, with_base: bool = True) -> np.ndarray:
    lo = -1 if with_base else 0
    return rng.integers(lo, n_slots, size=n).astype(np.int32)


def draw_weight(rng: np.random.Generator, h_out: int, h_in: int, dtype: torch.dtype,
                std: float = 0.02) -> torch.Tensor:
    return _round(rng.standard_normal((h_out, h_in)) * std, dtype)


def draw_adapters(rng: np.random.Generator, h_in: int, h_out: int, ranks: Sequence[int],
                  alphas: Sequence[float], dtype: torch.dtype, r_max: Optional[int] = None) -> AdapterSet:
    """A ~ U(+-1/sqrt(h_in)) [r, h_in] for every slot, then B ~ N(0, 0.01) [h_out, r]."""
    bound = 1.0 / np.sqrt(h_in)
    A = [_round(rng.uniform(-bound, bound, size=(r, h_in)), dtype) for r in ranks]
    B = [_round(rng.standard_normal((h_out, r)) * 0.01, dtype) for r in ranks]
    return AdapterSet(A=A, B=B, ranks=list(ranks), alphas=[float(a) for a in alphas],
                      r_max=int(r_max if r_max is not None else max(ranks)))


def draw_x(rng: np.random.Generator, n: int, h_in: int, dtype: torch.dtype) -> torch.Tensor:
    return _round(rng.standard_normal((n, h_in)), dtype)


# ----------------------------------------------------------------------------------------
# The five workloads
# ----------------------------------------------------------------------------------------

def tiny(seed: int = 0) -> LinearCase:
    """16 tokens, 256 -> 256 fp32, 4 adapters rank 8 alpha 16, idx uniform over {-1..3}."""
    rng = _rng(seed)
    idx = draw_uniform_idx(rng, 16, 4)
    W = draw_weight(rng, 256, 256, torch.float32)
    ad = draw_adapters(rng, 256, 256, [8] * 4, [16.0] * 4, torch.float32)
    x = draw_x(rng, 16, 256, torch.float32)
    return LinearCase("tiny", x, W, ad, torch.from_numpy(idx))


def decode_q_proj(seed: int = 1, n: int = 64, layer: int = 0, h: int = 4096, n_slots: int = 100,
                  dtype: torch.dtype = torch.float16) -> LinearCase:
    """Decode q_proj of a 7B-shaped model: n tokens, h x h, 100 adapters rank 8 alpha 16,
    idx Zipf(1.1) with 10 % base-only. ``layer`` selects an independent copy (the bench
    cycles through copies the way a model cycles through layers)."""
    rng = _rng(seed, layer)
    idx = draw_zipf_idx(rng, n, n_slots, p_base=0.1)
    W = draw_weight(rng, h, h, dtype)
    ad = draw_adapters(rng, h, h, [8] * n_slots, [16.0] * n_slots, dtype)
    x = draw_x(rng, n, h, dtype)
    return LinearCase(f"decode_q_proj_n{n}_l{layer}", x, W, ad, torch.from_numpy(idx))


MIXED_RANKS = (8, 8, 16, 16, 64, 64)


def mixed_rank(n: int, seed: int = 2, h: int = 4096, layer: int = 0,
               dtype: torch.dtype = torch.float16) -> LinearCase:
    """6 adapters of ranks {8,8,16,16,64,64} padded to 64, alpha = 2r; idx uniform over
    {-1, 0..5}; one independent draw per batch size n."""
    rng = _rng(seed, n, layer)
    idx = draw_uniform_idx(rng, n, len(MIXED_RANKS))
    W = draw_weight(rng, h, h, dtype)
    ad = draw_adapters(rng, h, h, MIXED_RANKS, [2.0 * r for r in MIXED_RANKS], dtype, r_max=64)
    x = draw_x(rng, n, h, dtype)
    return LinearCase(f"mixed_rank_n{n}", x, W, ad, torch.from_numpy(idx))


def prefill(seed: int = 3, n_req: int = 32, chunk: int = 512, h: int = 4096, n_slots: int = 100,
            dtype: torch.dtype = torch.bfloat16) -> List[LinearCase]:
    """32 requests x 512 tokens; one Zipf(1.1) adapter per request (no base-only tokens);
    q_proj and v_proj (h -> h each) share x and the token->slot map, each with its own
    base weight and its own pool of 100 rank-16 alpha-32 adapters."""
    rng = _rng(seed)
    req_slot = draw_zipf_idx(rng, n_req, n_slots)
    idx = np.repeat(req_slot, chunk).astype(np.int32)
    cases = []
    Ws, ads = [], []
    for _proj in ("q_proj", "v_proj"):
        Ws.append(draw_weight(rng, h, h, dtype))
        ads.append(draw_adapters(rng, h, h, [16] * n_slots, [32.0] * n_slots, dtype))
    x = draw_x(rng, n_req * chunk, h, dtype)
    for name, W, ad in zip(("q_proj", "v_proj"), Ws, ads):
        cases.append(LinearCase(f"prefill_{name}", x, W, ad, torch.from_numpy(idx)))
    return cases


LAYER_PROJS = (  # name, h_in, h_out; x shared by q/k/v and by gate/up
    ("q_proj", 4096, 4096), ("k_proj", 4096, 4096), ("v_proj", 4096, 4096),
    ("o_proj", 4096, 4096), ("gate_proj", 4096, 11008), ("up_proj", 4096, 11008),
    ("down_proj", 11008, 4096),
)


def full_layer(layer: int, seed: int = 4, n: int = 256, n_slots: int = 100, r: int = 16,
               alpha: float = 32.0, dtype: torch.dtype = torch.bfloat16,
               projs: Optional[Sequence[str]] = None) -> List[LinearCase]:
    """One decoder layer of a 7B-shaped model at decode: 256 tokens, LoRA rank 16 on all
    seven projections, 100 adapters each, Zipf(1.1) idx shared by the whole batch.
    Inputs: x_attn feeds q/k/v, x_o feeds o, x_mlp feeds gate/up, x_down feeds down."""
    rng = _rng(seed)
    idx = draw_zipf_idx(rng, n, n_slots)  # one routing for every layer of the batch
    lrng = _rng(seed, 1000 + layer)
    xs = {"attn": draw_x(lrng, n, 4096, dtype), "o": draw_x(lrng, n, 4096, dtype),
          "mlp": draw_x(lrng, n, 4096, dtype), "down": draw_x(lrng, n, 11008, dtype)}
    feed = {"q_proj": "attn", "k_proj": "attn", "v_proj": "attn", "o_proj": "o",
            "gate_proj": "mlp", "up_proj": "mlp", "down_proj": "down"}
    cases = []
    for name, h_in, h_out in LAYER_PROJS:
        prng = _rng(seed, 1000 + layer, LAYER_PROJS.index((name, h_in, h_out)))
        W = draw_weight(prng, h_out, h_in, dtype)
        ad = draw_adapters(prng, h_in, h_out, [r] * n_slots, [alpha] * n_slots, dtype)
        if projs is None or name in projs:
            cases.append(LinearCase(f"layer{layer}_{name}", xs[feed[name]], W, ad, torch.from_numpy(idx)))
    return cases


def random_case(seed: int, n: int, h_in: int, h_out: int, ranks: Sequence[int],
                alphas: Optional[Sequence[float]] = None, r_max: Optional[int] = None,
                dtype: torch.dtype = torch.float16, p_base: float = 0.1,
                idx: Optional[np.ndarray] = None) -> LinearCase:
    """General small case for edge tests (ragged sizes, many slots, custom idx)."""
    rng = _rng(seed, n, h_in, h_out)
    S = len(ranks)
    if idx is None:
        idx = draw_zipf_idx(rng, n, S, p_base=p_base) if S > 0 else np.full(n, -1, np.int32)
    W = draw_weight(rng, h_out, h_in, dtype)
    if alphas is None:
        alphas = [2.0 * r for r in ranks]
    ad = draw_adapters(rng, h_in, h_out, ranks, alphas, dtype, r_max=r_max)
    x = draw_x(rng, n, h_in, dtype)
    return LinearCase(f"random_s{seed}_n{n}_{h_in}x{h_out}", x, W, ad,
                      torch.from_numpy(np.asarray(idx, dtype=np.int32)))


def random_group(seed: int, n: int, h_in: int, h_outs: Sequence[int], ranks: Sequence[int],
                 r_max: Optional[int] = None, dtype: torch.dtype = torch.float16, p_base: float = 0.1,
                 slice_ranks: Optional[Sequence[Sequence[int]]] = None) -> List[LinearCase]:
    """Projections that share x and idx (q, k, v of one attention block): one case per slice,
    all holding the same x and idx tensors, each with its own W and adapters (slot s of every
    slice is mounted; ``slice_ranks[q]`` overrides the ranks of slice q).  Draw order: idx, x,
    then W, A, B of every slice in turn."""
    rng = _rng(seed, n, h_in, *h_outs)
    S = len(ranks)
    idx = torch.from_numpy(np.asarray(draw_zipf_idx(rng, n, S, p_base=p_base), dtype=np.int32))
    x = draw_x(rng, n, h_in, dtype)
    cases = []
    for q, h_out in enumerate(h_outs):
        rq = list(ranks if slice_ranks is None else slice_ranks[q])
        W = draw_weight(rng, h_out, h_in, dtype)
        ad = draw_adapters(rng, h_in, h_out, rq, [2.0 * r for r in rq], dtype, r_max=r_max)
        cases.append(LinearCase(f"group_s{seed}_n{n}_{h_in}_slice{q}", x, W, ad, idx))
    return cases
