"""The adapter loader: background mounts on a copy stream and draining remounts.

A remount of a slot waits for every release fence recorded on it since its last mount, so
linears still queued on the compute stream keep reading the old adapter; a compute stream
that acquires a slot sees its new adapter.  Checked through the C ABI against the float64
oracle, with W = 0 so that y is the LoRA term alone (a stale or torn adapter cannot hide in
the base term).
"""
import numpy as np
import pytest
import torch

from adapter_gemm_segment_gb300 import workloads as wl
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu

H, R, S = 4096, 8, 4


def _adapters(seed):
    ad = wl.draw_adapters(np.random.default_rng(seed), H, H, [8, 8, 4, 8], [16.0, 16.0, 8.0, 16.0],
                          torch.float16, r_max=R)
    return [a.contiguous().pin_memory() for a in ad.A], [b.contiguous().pin_memory() for b in ad.B], ad


def _lora_only_ref(x, ad_list, idx):
    """Oracle of the LoRA term (W = 0) for slot s holding ad_list[s] = (A, B, rank, alpha)."""
    pool = O.pad_pool([a[0] for a in ad_list], [a[1] for a in ad_list], [a[2] for a in ad_list],
                      [a[3] for a in ad_list], R, H, H)
    return O.lora_linear(x, np.zeros((H, H)), pool, idx)


def _close(y, ref):
    y64 = y.double().cpu().numpy()
    return bool(np.all(np.abs(y64 - ref) <= 1e-2 * np.abs(ref).max() + 1e-2 * np.abs(ref)))


def test_draining_remount_under_load(lib):
    dev = torch.device("cuda")
    compute, copy = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    pool = lib.LoraPool(H, H, R, S, torch.float16, dev)
    loader = lib.LoraLoader([pool], copy)
    XA, XB, X = _adapters(1)
    YA, YB, Y = _adapters(2)
    rng = np.random.default_rng(3)
    idx = torch.from_numpy(np.where(rng.random(64) < 0.7, 0, rng.integers(1, S, 64)).astype(np.int32))
    x = wl.draw_x(rng, 64, H, torch.float16)
    W = torch.zeros(H, H, dtype=torch.float16, device=dev)
    n_lin = 24
    ys1 = [torch.empty(64, H, dtype=torch.float16, device=dev) for _ in range(n_lin)]
    ys2 = [torch.empty(64, H, dtype=torch.float16, device=dev) for _ in range(n_lin)]
    loader.mount(list(range(S)), [XA], [XB], X.alphas)
    with torch.cuda.stream(compute):
        xd, idd = x.to(dev, non_blocking=True), idx.to(dev, non_blocking=True)
        ws = pool.linear_workspace(64, dev)
        loader.acquire(list(range(S)), compute)
        # hold the compute stream for a few ms so that the whole first batch is still queued when
        # the remount below reaches the (idle) copy stream: only the drain keeps it from landing
        torch.cuda._sleep(20_000_000)
        seg = pool.segment(idd, stream=compute)
        for y in ys1:  # a long batch on slot 0 (and the others), still running when the remount is enqueued
            pool.linear(W, xd, seg, y=y, ws=ws, stream=compute)
        loader.release(list(range(S)), compute)
        # slot 0 gets adapter Y on the copy stream: it must drain the batch above first
        loader.mount([0], [[YA[0]]], [[YB[0]]], [Y.alphas[0]])
        loader.acquire([0], compute)
        seg2 = pool.segment(idd, ws=torch.zeros_like(seg._ws), stream=compute)
        ws2 = pool.linear_workspace(64, dev)
        for y in ys2:
            pool.linear(W, xd, seg2, y=y, ws=ws2, stream=compute)
        loader.release([0], compute)
    torch.cuda.synchronize()
    ref_x = _lora_only_ref(x, [(X.A[s], X.B[s], X.ranks[s], X.alphas[s]) for s in range(S)], idx.numpy())
    mixed = [(Y.A[0], Y.B[0], Y.ranks[0], Y.alphas[0])] + [(X.A[s], X.B[s], X.ranks[s], X.alphas[s])
                                                           for s in range(1, S)]
    ref_y = _lora_only_ref(x, mixed, idx.numpy())
    assert not _close(ys1[0], ref_y), "the two adapters must be told apart by the check"
    for k, y in enumerate(ys1):
        assert torch.equal(y, ys1[0]), f"linear {k} of the first batch saw a different adapter"
    assert _close(ys1[0], ref_x), "the first batch does not match the old adapter"
    for k, y in enumerate(ys2):
        assert torch.equal(y, ys2[0]), f"linear {k} of the second batch differs"
    assert _close(ys2[0], ref_y), "the second batch does not match the remounted adapter"
    st = loader.stats()
    assert st["mounts"] == S + 1 and st["drained_fences"] == 1
    loader.close()


def test_background_mount_into_a_free_slot(lib):
    """Double buffering: the next adapter lands in a free slot on the copy stream while linears
    on the other slots run; after acquire, a batch naming it is exact against the oracle."""
    dev = torch.device("cuda")
    compute, copy = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    pool = lib.LoraPool(H, H, R, S, torch.float16, dev)
    loader = lib.LoraLoader([pool], copy)
    XA, XB, X = _adapters(4)
    loader.mount([0, 1, 2], [XA[:3]], [XB[:3]], X.alphas[:3])
    rng = np.random.default_rng(5)
    idx1 = torch.from_numpy(rng.integers(-1, 3, 64).astype(np.int32))
    idx2 = torch.from_numpy(rng.integers(-1, 4, 64).astype(np.int32))
    x = wl.draw_x(rng, 64, H, torch.float16)
    W = torch.zeros(H, H, dtype=torch.float16, device=dev)
    with torch.cuda.stream(compute):
        xd = x.to(dev, non_blocking=True)
        loader.acquire([0, 1, 2], compute)
        seg = pool.segment(idx1.to(dev, non_blocking=True), stream=compute)
        ws = pool.linear_workspace(64, dev)
        y1 = [pool.linear(W, xd, seg, ws=ws, stream=compute) for _ in range(12)]
        loader.release([0, 1, 2], compute)
        loader.mount([3], [[XA[3]]], [[XB[3]]], [X.alphas[3]])  # in the background, slot 3 was free
        loader.acquire([3], compute)
        seg2 = pool.segment(idx2.to(dev, non_blocking=True), stream=compute)
        y2 = pool.linear(W, xd, seg2, ws=ws, stream=compute)
    torch.cuda.synchronize()
    all4 = [(X.A[s], X.B[s], X.ranks[s], X.alphas[s]) for s in range(S)]
    assert _close(y1[-1], _lora_only_ref(x, all4, idx1.numpy()))
    assert _close(y2, _lora_only_ref(x, all4, idx2.numpy()))
    assert loader.stats()["drained_fences"] == 0
    loader.close()


def test_loader_errors(lib):
    dev = torch.device("cuda")
    copy = torch.cuda.Stream(dev)
    pool = lib.LoraPool(256, 256, 8, 4, torch.float16, dev)
    loader = lib.LoraLoader([pool], copy)
    A = torch.zeros(8, 256, dtype=torch.float16).pin_memory()
    B = torch.zeros(256, 8, dtype=torch.float16).pin_memory()
    A16 = torch.zeros(16, 256, dtype=torch.float16).pin_memory()
    B16 = torch.zeros(256, 16, dtype=torch.float16).pin_memory()
    cases = [([4], [[A]], [[B]], lib.LORA_ESLOT), ([1, 1], [[A, A]], [[B, B]], lib.LORA_EBUSY),
             ([2], [[A16]], [[B16]], lib.LORA_ERANK)]
    for slots, As, Bs, code in cases:
        with pytest.raises(lib.LoraError) as e:
            loader.mount(slots, As, Bs, [16.0] * len(slots))
        assert e.value.code == code
    assert loader.stats()["mounts"] == 0
    with pytest.raises(ValueError):
        loader.mount([0], [[A.cuda()]], [[B.cuda()]], [16.0])  # device tensors are not the host tier
    other = lib.LoraPool(256, 256, 8, 5, torch.float16, dev)
    with pytest.raises(lib.LoraError):
        lib.LoraLoader([pool, other], copy)  # different slot counts
    loader.close()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_one_mount_call_across_pools_is_byte_exact(lib, dtype):
    """One lora_loader_mount over pools of different shapes (one kernel for every pool and slot
    of the call for 16-bit pools; the pools' own mounts for float32) leaves every pool's bytes
    identical to lora_pool_load_slot into a fresh pool: zero padding, ranks that are not
    multiples of 8, slot table."""
    dev = torch.device("cuda")
    copy = torch.cuda.Stream(dev)
    shapes = [(4096, 4096), (4096, 1024), (1024, 4096)]
    r_max, S = 16, 6
    slots, ranks = [4, 0, 5], [16, 5, 8]
    rng = np.random.default_rng(9)
    pools = [lib.LoraPool(hi, ho, r_max, S, dtype, dev) for hi, ho in shapes]
    refs = [lib.LoraPool(hi, ho, r_max, S, dtype, dev) for hi, ho in shapes]
    loader = lib.LoraLoader(pools, copy)
    As, Bs = [], []
    for (hi, ho), ref in zip(shapes, refs):
        ad = wl.draw_adapters(rng, hi, ho, ranks, [2.0 * r for r in ranks], dtype, r_max=r_max)
        As.append([a.contiguous().pin_memory() for a in ad.A])
        Bs.append([b.contiguous().pin_memory() for b in ad.B])
        for sl, a, b, al in zip(slots, ad.A, ad.B, ad.alphas):
            ref.load_slot(sl, a.to(dev), b.to(dev), al)
    loader.mount(slots, As, Bs, [2.0 * r for r in ranks])
    torch.cuda.synchronize()
    for p, (pool, ref) in enumerate(zip(pools, refs)):
        assert torch.equal(pool.mem, ref.mem), f"pool {p} differs from per-slot mounts"
    loader.close()
