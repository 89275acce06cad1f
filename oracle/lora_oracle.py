"""CPU oracle for the multi-LoRA segmented linear -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the CPU-baseline leg of the benchmark may
import this module.  The product path (the CUDA library and its Python binding)
never calls it and never falls back to it.

What it computes, in float64, straight from the definitions:

* ``pad_pool``: the HBM adapter pool.  Every adapter is stored at the common rank
  r_max; rows of A and columns of B beyond the adapter's own rank are exactly zero.
  ("LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排", blog.lonae.com, section on
  tensor concatenation: zero-pad the low-rank adapters to the high rank before they
  are concatenated, accepting some wasted work for correct shapes.)  The per-slot
  scale is alpha / r with r the adapter's *true* rank (the LoRA convention for the
  alpha/r factor; dividing by r_max would make padding change the result).

* ``segments``: the adapter-level bucketing of a mixed batch.  Tokens are put into
  buckets by adapter slot with a stable counting sort (ties keep token order); the
  key -1 (base only) is the smallest key.  Each non-empty bucket, in ascending key
  order, is one segment.  (Same page, section on two-level bucketing -- request
  level, then adapter level; "Multi-LoRA 在线服务隔离" (ai.codenodex.com), section
  "请求身份决定适配器，而非客户端参数": one dispatch may mix adapters as long as the
  index map stays per request.)

* ``lora_linear``: y[t] = x[t] W^T + (alpha_s / r_s) (x[t] A_s^T) B_s^T with s = idx[t],
  and no LoRA term when idx[t] = -1 (the routing default ``base_only`` of the
  xpshop.cn article 492 case study, section 三).  The adapter execution unit of the
  blog.lonae.com page adds the low-rank product to the base hidden state; the exact
  formula is the LoRA definition.

* Errors: an idx outside [-1, n_slots) or one that names a slot with no adapter
  loaded is an explicit error and produces no output -- there is no fallback to the
  base model or to another adapter (ai.codenodex.com page, section
  "请求身份决定适配器，而非客户端参数": default deny, a missing mapping is an error).

* ``lora_linear_group``: projections sharing x and idx, side by side (see its docstring).

* ``within_tolerance``: the elementwise float bar |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.

Arithmetic: float64 throughout; the base term and the per-token shrink/expand products use
numpy's matmul (a library primitive) with no blocking or reordering of its own.

Pins (tests/test_oracle_pins.py): brute force in pure-Python loops on tiny inputs (full
batches and ``rows=`` subsets in any order), numpy's stable argsort for the segment order,
the merged-weight identity, zero-pad invariance, permutation equivariance, the unit-vector
selector closed form, the rank-1 outer product, hand-computed pairs on both sides of the
tolerance bound, and a hand-worked golden example in tests/golden/.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import numpy as np

# status codes shared in meaning (not in code) with the C library's lora_status
OK = 0
EIDX = -6


class OracleError(Exception):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


def _f64(t) -> np.ndarray:
    """Exact upcast of an already-rounded tensor/array to float64."""
    if hasattr(t, "detach"):
        t = t.detach().to("cpu")
        import torch  # local: only needed to upcast 16-bit torch tensors exactly

        return t.to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


@dataclasses.dataclass
class OraclePool:
    A: np.ndarray  # [S, r_max, h_in] float64, zero-padded rows
    B: np.ndarray  # [S, h_out, r_max] float64, zero-padded columns
    scale: np.ndarray  # [S] alpha / true rank
    loaded: np.ndarray  # [S] bool

    @property
    def n_slots(self) -> int:
        return int(self.A.shape[0])


def pad_pool(A_list: Sequence, B_list: Sequence, ranks: Sequence[int], alphas: Sequence[float],
             r_max: int, h_in: int, h_out: int, n_slots: Optional[int] = None,
             slots: Optional[Sequence[int]] = None) -> OraclePool:
    """Build the zero-padded pool.  Adapter i goes to slot ``slots[i]`` (default i)."""
    S = n_slots if n_slots is not None else len(ranks)
    slots = list(range(len(ranks))) if slots is None else list(slots)
    A = np.zeros((S, r_max, h_in))
    B = np.zeros((S, h_out, r_max))
    scale = np.zeros(S)
    loaded = np.zeros(S, dtype=bool)
    for a, b, r, alpha, s in zip(A_list, B_list, ranks, alphas, slots):
        if not (1 <= r <= r_max):
            raise OracleError(-4, f"rank {r} outside [1, {r_max}]")
        a = _f64(a)
        b = _f64(b)
        assert a.shape == (r, h_in) and b.shape == (h_out, r)
        A[s, :r, :] = a
        B[s, :, :r] = b
        scale[s] = float(alpha) / float(r)
        loaded[s] = True
    return OraclePool(A, B, scale, loaded)


def validate_idx(idx: np.ndarray, pool_or_nslots) -> None:
    """Default deny: every idx must be -1 or name a loaded slot."""
    if isinstance(pool_or_nslots, OraclePool):
        S, loaded = pool_or_nslots.n_slots, pool_or_nslots.loaded
    else:
        S, loaded = int(pool_or_nslots), None
    for t, k in enumerate(idx.tolist()):
        if k < -1 or k >= S:
            raise OracleError(EIDX, f"token {t}: idx {k} outside [-1, {S})")
        if k >= 0 and loaded is not None and not loaded[k]:
            raise OracleError(EIDX, f"token {t}: slot {k} has no adapter loaded")


def segments(idx, pool_or_nslots) -> Tuple[np.ndarray, np.ndarray, np.ndarray, int]:
    """Stable counting sort of token positions by key idx (-1 first).

    Returns (perm, seg_start, seg_slot, nseg): perm[j] is the original position of
    the j-th token in sorted order; segment i covers sorted positions
    seg_start[i] .. seg_start[i+1]-1, all with key seg_slot[i] (which may be -1 for
    the base-only run); seg_start has nseg+1 entries, seg_start[nseg] = n.
    """
    idx = np.asarray(idx, dtype=np.int64)
    validate_idx(idx, pool_or_nslots)
    S = pool_or_nslots.n_slots if isinstance(pool_or_nslots, OraclePool) else int(pool_or_nslots)
    n = idx.shape[0]
    # 1. histogram over the S+1 keys -1..S-1 (key k lives in bucket k+1)
    count = [0] * (S + 1)
    for k in idx.tolist():
        count[k + 1] += 1
    # 2. exclusive prefix sum -> first sorted position of every key
    start = [0] * (S + 1)
    acc = 0
    for b in range(S + 1):
        start[b] = acc
        acc += count[b]
    # 3. stable placement: visit tokens in their original order
    perm = np.empty(n, dtype=np.int32)
    nxt = list(start)
    for t, k in enumerate(idx.tolist()):
        perm[nxt[k + 1]] = t
        nxt[k + 1] += 1
    # 4. maximal runs of equal key, ascending key order; empty keys give no segment
    seg_start, seg_slot = [], []
    for b in range(S + 1):
        if count[b] > 0:
            seg_start.append(start[b])
            seg_slot.append(b - 1)
    seg_start.append(n)
    return (perm, np.asarray(seg_start, dtype=np.int32), np.asarray(seg_slot, dtype=np.int32),
            len(seg_slot))


def lora_linear(x, W, pool: OraclePool, idx, rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """y[t] = x[t] W^T + scale_s (x[t] A_s^T) B_s^T for s = idx[t] >= 0, in float64.

    ``rows`` restricts the evaluation to a subset of tokens (the result has one row
    per requested token, in the order given); validation still covers the whole batch
    because an invalid token anywhere makes the whole call fail.
    """
    idx = np.asarray(idx, dtype=np.int64)
    validate_idx(idx, pool)
    rows = np.arange(idx.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    W64 = _f64(W)
    if hasattr(x, "index_select"):
        import torch

        xs = _f64(x.index_select(0, torch.from_numpy(rows)))
    else:
        xs = _f64(x)[rows]
    y = xs @ W64.T  # base linear (nn.Linear layout: W is [h_out, h_in])
    for i, t in enumerate(rows.tolist()):
        s = int(idx[t])
        if s < 0:
            continue
        u = pool.A[s] @ xs[i]  # shrink: [r_max]
        y[i] += pool.scale[s] * (pool.B[s] @ u)  # expand: [h_out]
    return y


def lora_linear_group(x, Ws: Sequence, pools: Sequence[OraclePool], idx,
                      rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Several projections that read the same x with the same token-to-adapter map (q, k
    and v of one attention block): slice q is ``lora_linear`` of W_q with pool q, and the
    result puts the slices side by side, slice 0's columns first.

    One adapter identity covers all of its target modules (the registry entry of the
    ai.codenodex.com page, section "适配器先进入可信注册表", lists target modules q_proj
    and v_proj), so an idx must be valid in every pool of the group.
    """
    return np.concatenate([lora_linear(x, W, p, idx, rows=rows) for W, p in zip(Ws, pools)], axis=1)


def lora_linear_case(case, rows=None) -> np.ndarray:
    """Convenience: run ``lora_linear`` on a ``workloads.LinearCase``."""
    ad = case.adapters
    pool = pad_pool(ad.A, ad.B, ad.ranks, ad.alphas, ad.r_max, case.h_in, case.h_out)
    return lora_linear(case.x, case.W, pool, case.idx.numpy(), rows=rows)


def pool_of_case(case) -> OraclePool:
    ad = case.adapters
    return pad_pool(ad.A, ad.B, ad.ranks, ad.alphas, ad.r_max, case.h_in, case.h_out)


def within_tolerance(y, y_ref, atol: float = 1e-2, rtol: float = 1e-2) -> np.ndarray:
    """Elementwise |y - y_ref| <= atol + rtol |y_ref| (the stated float bar)."""
    y = _f64(y)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    return np.abs(y - y_ref) <= atol + rtol * np.abs(y_ref)
