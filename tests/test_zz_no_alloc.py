"""The workspace-free linear forward (lora_linear_fwd_static_ws).

It serves callers that cannot hand the library any device memory of their own -- an operator
plugin inside another engine that only receives its inputs and outputs while the engine owns
every allocation, or a host held to a fixed device-memory budget.  Its scratch (the shrink
output) is a fixed device array inside the library.  This file runs last (pytest collects
files in name order), so a run that stops at the first failure has executed every other test
before it; it also passes when run alone in a fresh process.

Each case is called twice in a row through the C ABI.  Both results must equal the regular
entry point's (caller workspace) bit for bit: the kernels and their inputs are the same, only
the address of the scratch differs.
"""
import pytest
import torch

from adapter_gemm_segment_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    ("decode fp16 n=64", lambda: wl.random_case(31, 64, 1024, 512, [8, 8, 8, 8], r_max=8, dtype=torch.float16)),
    # h_in 4096 at 64 tokens: the decode shrink writes 4 K-parts (64 x 8 x 4 floats of scratch)
    ("decode fp16 n=64 h_in=4096, 4 shrink parts",
     lambda: wl.random_case(34, 64, 4096, 256, [8, 8, 8], r_max=8, dtype=torch.float16)),
    ("mixed rank n=7", lambda: wl.random_case(32, 7, 512, 256, [8, 16, 64], r_max=64, dtype=torch.float16)),
    ("long batch bf16 n=300", lambda: wl.random_case(33, 300, 512, 384, [16, 16], r_max=16, dtype=torch.bfloat16)),
    ("fp32 n=16", lambda: wl.tiny()),
]


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
    for k, y in enumerate(outs):
        assert torch.equal(y, y_ref), f"{name}: call {k + 1} differs from the caller-workspace result"


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
