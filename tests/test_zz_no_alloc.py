"""The workspace-free linear forward (lora_linear_fwd_static_ws).

It serves callers that cannot hand the library any device memory of their own -- a plugin
inside another engine that only receives its inputs and outputs, or code enqueueing work
during CUDA graph capture, where cudaMalloc is not allowed.  Its scratch is a fixed device
array inside the library.  This file runs last (pytest collects files in name order), so a
run that stops at the first failure has executed every other test before it.

Each case is called twice in a row through the C ABI, and both results must agree with the
regular entry point (caller workspace) within the same tolerance the parity tests use.
"""
import numpy as np
import pytest
import torch

from adapter_gemm_segment_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    ("decode fp16 n=64", lambda: wl.random_case(31, 64, 1024, 512, [8, 8, 8, 8], r_max=8, dtype=torch.float16)),
    ("mixed rank n=7", lambda: wl.random_case(32, 7, 512, 256, [8, 16, 64], r_max=64, dtype=torch.float16)),
    ("long batch bf16 n=300", lambda: wl.random_case(33, 300, 512, 384, [16, 16], r_max=16, dtype=torch.bfloat16)),
    ("fp32 n=16", lambda: wl.tiny()),
]


def _close(a: torch.Tensor, b: torch.Tensor) -> bool:
    a64, b64 = a.double().cpu().numpy(), b.double().cpu().numpy()
    return bool(np.all(np.abs(a64 - b64) <= 1e-2 + 1e-2 * np.abs(b64)))


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_matches_caller_workspace(lib, name, make):
    case = make()
    ad = case.adapters
    pool = lib.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, case.dtype, "cuda")
    for s in range(ad.n_slots):
        pool.load_slot(s, ad.A[s].cuda(), ad.B[s].cuda(), ad.alphas[s])
    seg = pool.segment(case.idx.cuda())
    W, x = case.W.cuda(), case.x.cuda()
    y_ref = pool.linear(W, x, seg).clone()
    outs = []
    for _ in range(2):  # two calls in a row share (and overwrite) the library's scratch array
        y = torch.full((case.n, case.h_out), float("nan"), dtype=case.dtype, device="cuda")
        lib.lora_linear_fwd_static_ws(pool.handle, W, x, y, seg)
        outs.append(y)
    torch.cuda.synchronize()
    for y in outs:
        assert _close(y, y_ref), f"{name}: static-workspace result differs from the caller-workspace result"


def test_static_workspace_refuses_oversized_batches(lib):
    # 4 MiB hold 1 Mi floats: 16384 tokens x r_max 128 (one part above 256 tokens) do not fit
    pool = lib.LoraPool(64, 64, 128, 2, torch.bfloat16, "cuda")
    seg = pool.segment(torch.full((16384,), -1, dtype=torch.int32, device="cuda"))
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(16384, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(16384, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.LoraError) as e:
        lib.lora_linear_fwd_static_ws(pool.handle, W, x, y, seg)
    assert e.value.code == lib.LORA_ENOSPACE
