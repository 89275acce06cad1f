"""Failure paths on the GPU, exercised without a fault: a bounded pipeline wait that runs out.

Every pipeline wait of the tensor-core kernels gives up after a time limit, records
LORA_ETIMEOUT in the status word and skips the output (no trap, no endless spin).  The test
runs that same wait (lora_wait_selftest) on a barrier that nothing completes, with a 2 ms
limit, and checks the status, the untouched output, and that the context stays usable.
"""
import pytest
import torch

from adapter_gemm_segment_gb300 import workloads as wl
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(4096, dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    lib.lora_wait_selftest(status, out, arrive=False, limit_ns=2_000_000)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == lib.LORA_ETIMEOUT
    assert int(torch.count_nonzero(out).item()) == 0, "the output of a wait that gave up was written"
    ms = e0.elapsed_time(e1)
    assert 1.5 <= ms <= 100.0, f"the wait gave up after {ms:.3f} ms, not after about its 2 ms limit"


def test_completed_wait_writes_output_and_context_stays_usable(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(5000, dtype=torch.float32, device="cuda")
    lib.lora_wait_selftest(status, out, arrive=False, limit_ns=1_000_000)  # runs out first
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.lora_wait_selftest(status2, out, arrive=True, limit_ns=1_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) == lib.LORA_ETIMEOUT and int(status2.item()) == 0
    assert bool((out == 1.0).all())
    # a LoRA linear still runs correctly on the same context afterwards
    case = wl.random_case(70, 40, 512, 256, [8, 16], r_max=16, dtype=torch.float16)
    ad = case.adapters
    pool = lib.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, case.dtype, "cuda")
    for s in range(ad.n_slots):
        pool.load_slot(s, ad.A[s].cuda(), ad.B[s].cuda(), ad.alphas[s])
    seg = pool.segment(case.idx.cuda())
    y = pool.linear(case.W.cuda(), case.x.cuda(), seg).cpu()
    assert O.within_tolerance(y, O.lora_linear_case(case)).all()


def test_selftest_argument_errors(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(8, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.LoraError) as e:
        lib.lora_wait_selftest(status, out, arrive=False, limit_ns=10**9)  # above the 0.1 s cap
    assert e.value.code == lib.LORA_EINVAL
    assert int(status.item()) == 0
