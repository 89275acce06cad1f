"""GPU parity of the CUDA path (through the C ABI) against the float64 CPU oracle.

Bars: segment outputs bit-exact; floats elementwise |y - y_ref| <= 1e-2 + 1e-2 |y_ref|.
Because that bar is loose next to the LoRA term at the workloads' scales, every config is
also run with W = 0 (y is then the LoRA term alone, compared against a bar scaled by the
largest |y_ref|), and a negative control (outputs compared with the oracle of a shuffled
idx) must fail.
"""
import numpy as np
import pytest
import torch

from adapter_gemm_segment_gb300 import workloads as wl
from oracle import lora_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"


# ------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------

def make_pool(ags, case, n_slots=None, load=True):
    ad = case.adapters
    S = n_slots or ad.n_slots
    pool = ags.LoraPool(case.h_in, case.h_out, ad.r_max, S, case.dtype, DEV)
    if load:
        for s in range(ad.n_slots):
            pool.load_slot(s, ad.A[s].to(DEV), ad.B[s].to(DEV), ad.alphas[s])
    return pool


class Guarded:
    """A device buffer between two guard zones of canary bytes (the stand-in for a memory
    checker): a kernel writing past either end of the buffer it was given changes a canary.
    The interior starts as canary bytes too (or NaN for outputs), so results cannot depend
    on the library finding zeros in its workspaces."""

    ZONE = 4096
    CANARY = 0xA5

    def __init__(self, nbytes, what):
        self.nbytes, self.what = int(nbytes), what
        pad = (self.nbytes + 255) // 256 * 256
        self.full = torch.full((2 * self.ZONE + pad,), self.CANARY, dtype=torch.uint8, device=DEV)
        self.bytes = self.full[self.ZONE:self.ZONE + self.nbytes]

    @classmethod
    def tensor(cls, shape, dtype, what):
        es = torch.empty(0, dtype=dtype).element_size()
        g = cls(int(np.prod(shape)) * es, what)
        g.t = g.bytes.view(dtype).view(*shape)
        g.t.fill_(float("nan"))
        return g

    def check(self):
        z = self.ZONE
        front, back = self.full[:z], self.full[z + self.nbytes:]
        assert bool((front == self.CANARY).all()), f"{self.what}: write before the start of the buffer"
        assert bool((back == self.CANARY).all()), f"{self.what}: write past the end of the buffer"


def run(ags, case, variant=0, W=None, idx=None, pool=None):
    pool = pool or make_pool(ags, case)
    idx = case.idx if idx is None else idx
    n = int(idx.numel())
    seg_g = Guarded(ags.lora_segment_workspace_bytes(n, pool.n_slots), "segment workspace")
    seg = pool.segment(idx.to(DEV), ws=seg_g.bytes)
    lin_g = Guarded(ags.lora_linear_workspace_bytes(pool.handle, n), "linear workspace")
    y_g = Guarded.tensor((n, case.h_out), case.dtype, "y")
    Wd = (case.W if W is None else W).to(DEV)
    y = pool.linear(Wd, case.x.to(DEV), seg, variant=variant, y=y_g.t, ws=lin_g.bytes)
    torch.cuda.synchronize()
    for g in (seg_g, lin_g, y_g):
        g.check()
    return y.cpu(), pool, seg


def assert_parity(y, y_ref, what=""):
    ok = O.within_tolerance(y, y_ref)
    bad = np.count_nonzero(~ok)
    if bad:
        y64 = y.double().numpy()
        i = np.unravel_index(np.argmax(np.abs(y64 - y_ref)), y_ref.shape)
        pytest.fail(f"{what}: {bad}/{ok.size} elements outside tolerance; worst at {i}: got {y64[i]}, want {y_ref[i]}")


def assert_lora_only_parity(y, y_ref, what=""):
    y64 = y.double().numpy()
    bound = 1e-2 * np.abs(y_ref).max() + 1e-2 * np.abs(y_ref)
    bad = np.count_nonzero(np.abs(y64 - y_ref) > bound)
    assert bad == 0, f"{what}: {bad} elements of the LoRA-only output outside tolerance"


def seg_arrays(ags, seg):
    return {k: v.cpu().numpy() for k, v in ags.segment_arrays(seg).items()}


def check_segments(ags, seg, idx, S, ranks):
    """ranks[s]: the true rank mounted in slot s (it travels with the shrink work items)."""
    got = seg_arrays(ags, seg)
    perm, ss, sl, nseg = O.segments(np.asarray(idx), S)
    assert int(got["status"][0]) == 0
    assert int(got["nseg"][0]) == nseg
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["seg_start"][:nseg + 1], ss)
    assert np.array_equal(got["seg_slot"][:nseg], sl)
    assert np.array_equal(got["idx"], np.asarray(idx))
    # shrink work items: every adapter segment cut into runs of up to 4 sorted tokens,
    # {slot, count, tokens, padded with the run's first token}; derived from the segments
    want = []
    for i in range(nseg):
        if sl[i] < 0:
            continue
        for j0 in range(ss[i], ss[i + 1], 4):
            toks = [int(t) for t in perm[j0:min(j0 + 4, ss[i + 1])]]
            want.append([int(sl[i]), len(toks)] + toks + [toks[0]] * (4 - len(toks)) + [int(ranks[sl[i]])])
    assert int(got["nseg"][1]) == len(want)
    items = got["items"].reshape(-1, 8)[:len(want), :7]
    assert np.array_equal(items, np.array(want, dtype=np.int32).reshape(-1, 7))


# ------------------------------------------------------------------------------------------
# pool
# ------------------------------------------------------------------------------------------

def test_pool_load_is_exact_zero_pad(lib):
    case = wl.random_case(1, 8, 64, 48, [3, 8, 1], r_max=16, dtype=torch.float16)
    pool = make_pool(lib, case, n_slots=5)
    torch.cuda.synchronize()
    S, R = 5, 16
    mem = pool.mem
    table = mem[:S * 16].view(torch.int32).view(S, 4).cpu().numpy()
    scale = mem[:S * 16].view(torch.float32).view(S, 4)[:, 2].cpu().numpy()
    ad = case.adapters
    ref = O.pad_pool(ad.A, ad.B, ad.ranks, ad.alphas, R, 64, 48, n_slots=S)
    assert table[:, 0].tolist() == [3, 8, 1, 0, 0]
    assert table[:, 1].tolist() == [1, 1, 1, 0, 0]
    assert np.array_equal(scale, ref.scale.astype(np.float32))
    a_off = 256
    A = mem[a_off:a_off + S * R * 64 * 2].view(torch.float16).view(S, R, 64).cpu().double().numpy()
    b_off = a_off + S * R * 64 * 2
    b_off = (b_off + 255) // 256 * 256
    B = mem[b_off:b_off + S * 48 * R * 2].view(torch.float16).view(S, 48, R).cpu().double().numpy()
    assert np.array_equal(A, ref.A) and np.array_equal(B, ref.B)


def test_pool_load_from_pinned_host_is_identical(lib):
    # the mounting kernel reads pinned host memory directly (no staging copy): same bytes
    case = wl.random_case(5, 24, 256, 192, [8, 3, 16], r_max=16, dtype=torch.bfloat16)
    ad = case.adapters
    pool_d = make_pool(lib, case)
    pool_h = lib.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, case.dtype, DEV)
    hA = [a.contiguous().pin_memory() for a in ad.A]
    hB = [b.contiguous().pin_memory() for b in ad.B]
    for s in range(ad.n_slots):
        pool_h.load_slot(s, hA[s], hB[s], ad.alphas[s])
    torch.cuda.synchronize()
    assert torch.equal(pool_h.mem, pool_d.mem)
    y, _, _ = run(lib, case, 1, pool=pool_h)
    assert_parity(y, O.lora_linear_case(case), "linear over a pool mounted from host")
    with pytest.raises(ValueError):
        pool_h.load_slot(0, ad.A[0], ad.B[0], ad.alphas[0])  # pageable host memory is refused


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_pool_batched_mount_is_identical(lib, dtype):
    # one call for every slot (ranks 1..16, some not multiples of 8), from device and from
    # pinned host memory, byte-identical to one lora_pool_load_slot per slot
    ranks = [8, 3, 16, 1, 9, 16, 5]
    case = wl.random_case(6, 8, 264, 136, ranks, r_max=16, dtype=dtype)
    ad = case.adapters
    ref = make_pool(lib, case)
    slots = list(range(ad.n_slots))[::-1]
    for src in ("device", "host"):
        pool = lib.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, case.dtype, DEV)
        As = [ad.A[s].contiguous() for s in slots]
        Bs = [ad.B[s].contiguous() for s in slots]
        As = [a.to(DEV) if src == "device" else a.pin_memory() for a in As]
        Bs = [b.to(DEV) if src == "device" else b.pin_memory() for b in Bs]
        pool.load_slots(slots, As, Bs, [ad.alphas[s] for s in slots])
        torch.cuda.synchronize()
        assert torch.equal(pool.mem, ref.mem), src
    with pytest.raises(lib.LoraError) as e:  # a slot named twice: nothing is mounted
        pool2 = lib.LoraPool(case.h_in, case.h_out, ad.r_max, ad.n_slots, case.dtype, DEV)
        pool2.load_slots([0, 0], [ad.A[0].to(DEV)] * 2, [ad.B[0].to(DEV)] * 2, [1.0, 1.0])
    assert e.value.code == lib.LORA_EBUSY
    pool2.load_slots([0], [ad.A[0].to(DEV)], [ad.B[0].to(DEV)], [1.0])  # slot 0 is still free


def test_pool_mount_errors(lib):
    case = wl.random_case(2, 4, 64, 64, [8, 8], r_max=8, dtype=torch.float16)
    pool = make_pool(lib, case)
    A, B = case.adapters.A[0].to(DEV), case.adapters.B[0].to(DEV)
    with pytest.raises(lib.LoraError) as e:
        pool.load_slot(0, A, B, 16.0)
    assert e.value.code == lib.LORA_EBUSY
    with pytest.raises(lib.LoraError) as e:
        pool.load_slot(2, A, B, 16.0)
    assert e.value.code == lib.LORA_ESLOT
    big = torch.zeros(9, 64, dtype=torch.float16, device=DEV)
    with pytest.raises(lib.LoraError) as e:
        lib.lora_pool_load_slot(pool.handle, 1, big, torch.zeros(64, 9, dtype=torch.float16, device=DEV), 9, 1.0)
    assert e.value.code == lib.LORA_ERANK
    pool.unload_slot(0)
    pool.load_slot(0, A, B, 16.0)  # unmount, then mount again


# ------------------------------------------------------------------------------------------
# segments
# ------------------------------------------------------------------------------------------

SEG_CASES = {
    "all_base": (np.full(37, -1), 4),
    "one_slot": (np.full(50, 2), 4),
    "single_token": (np.array([3]), 4),
    "every_slot": (np.arange(100)[::-1].copy(), 100),
    "zipf_decode_64": (wl.draw_zipf_idx(np.random.default_rng(1), 64, 100, 0.1), 100),
    "uniform_1500": (np.random.default_rng(2).integers(-1, 7, 1500), 7),
    "prefill_16384": (np.repeat(wl.draw_zipf_idx(np.random.default_rng(3), 32, 100), 512), 100),
    "max_slots": (np.random.default_rng(4).integers(-1, 2048, 5000), 2048),
    "long_run_3000": (np.concatenate([np.full(3000, 5), np.full(10, -1), np.full(1030, 1)]), 8),
}


@pytest.mark.parametrize("name", list(SEG_CASES))
def test_segments_bitexact(lib, name):
    idx, S = SEG_CASES[name]
    idx = np.asarray(idx, np.int32)
    pool = lib.LoraPool(64, 64, 8, S, torch.float16, DEV)
    A = torch.zeros(8, 64, dtype=torch.float16, device=DEV)
    B = torch.zeros(64, 8, dtype=torch.float16, device=DEV)
    for s in sorted(set(idx.tolist()) - {-1}):
        pool.load_slot(s, A, B, 8.0)
    seg = pool.segment(torch.from_numpy(idx).to(DEV))
    torch.cuda.synchronize()
    check_segments(lib, seg, idx, S, [8] * S)


def test_segments_empty_batch(lib):
    pool = lib.LoraPool(64, 64, 8, 4, torch.float16, DEV)
    seg = pool.segment(torch.zeros(0, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = seg_arrays(lib, seg)
    assert int(got["nseg"][0]) == 0 and int(got["seg_start"][0]) == 0 and int(got["status"][0]) == 0
    y = pool.linear(torch.zeros(64, 64, dtype=torch.float16, device=DEV),
                    torch.zeros(0, 64, dtype=torch.float16, device=DEV), seg)
    assert y.shape == (0, 64)


@pytest.mark.parametrize("bad", ["out_of_range", "below_minus_one", "unmounted"])
@pytest.mark.parametrize("n", [16, 300])
def test_invalid_idx_is_an_error_and_y_untouched(lib, bad, n):
    case = wl.random_case(3, n, 128, 128, [8, 8, 8], r_max=8, dtype=torch.float16)
    pool = make_pool(lib, case, n_slots=4)  # slot 3 stays empty
    idx = case.idx.clone()
    idx[n // 2] = {"out_of_range": 4, "below_minus_one": -2, "unmounted": 3}[bad]
    seg = pool.segment(idx.to(DEV))
    assert lib.lora_segment_status(seg) == lib.LORA_EIDX
    y = torch.full((n, 128), 7.0, dtype=torch.float16, device=DEV)
    for variant in (1, 2, 3):
        pool.linear(case.W.to(DEV), case.x.to(DEV), seg, variant=variant, y=y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()), "y was written although the batch names an invalid slot"


# ------------------------------------------------------------------------------------------
# linear: small cases, all variants
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [1, 2, 3])
def test_tiny_fp32(lib, variant):
    case = wl.tiny()
    y, pool, seg = run(lib, case, variant)
    torch.cuda.synchronize()
    check_segments(lib, seg, case.idx.numpy(), 4, case.adapters.ranks)
    assert_parity(y, O.lora_linear_case(case), f"tiny variant {variant}")
    y0, _, _ = run(lib, case, variant, W=torch.zeros_like(case.W))
    pool0 = O.pool_of_case(case)
    assert_lora_only_parity(y0, O.lora_linear(case.x, torch.zeros_like(case.W), pool0, case.idx.numpy()))


SMALL = [
    # (seed, n, h_in, h_out, ranks, r_max, dtype)
    (10, 16, 256, 256, [8, 8, 8], 8, torch.float16),
    (11, 1, 128, 256, [8], 8, torch.float16),
    (12, 17, 200, 136, [8, 16], 16, torch.bfloat16),
    (13, 64, 512, 384, [8, 8, 16, 64, 64, 16], 64, torch.float16),
    (14, 255, 136, 264, [16, 8, 4, 1], 16, torch.bfloat16),
    (15, 256, 256, 128, [8] * 10, 8, torch.float16),
    (16, 257, 256, 520, [16, 16, 16], 16, torch.bfloat16),
    (17, 300, 512, 256, [16, 3, 16], 16, torch.bfloat16),
    (18, 700, 136, 392, [8, 8], 8, torch.float16),
    (19, 129, 4104, 64, [8, 8], 8, torch.bfloat16),
    # two K chunks per decode stage: whole stages, and a split whose last stage is half past h_in
    (20, 64, 1024, 256, [8, 8], 8, torch.bfloat16),
    (21, 40, 704, 136, [8, 16, 16], 16, torch.float16),
    # r_max 64 at 100 tokens: the segmented shrink (4-token items), ragged K (4104 features)
    (22, 100, 4104, 64, [64, 8, 16, 64, 1], 64, torch.bfloat16),
    # the limits of the pool: the largest rank (256) and the most slots (2048)
    (23, 40, 512, 264, [256, 100, 8, 33], 256, torch.float16),
    (24, 100, 64, 72, [8] * 2048, 8, torch.float16),
]


@pytest.mark.parametrize("variant", [3, 1, 2])
@pytest.mark.parametrize("spec", SMALL, ids=[f"n{s[1]}_{s[2]}x{s[3]}_R{s[5]}" for s in SMALL])
def test_small_cases(lib, spec, variant):
    seed, n, h_in, h_out, ranks, r_max, dtype = spec
    case = wl.random_case(seed, n, h_in, h_out, ranks, r_max=r_max, dtype=dtype, p_base=0.15)
    y, pool, seg = run(lib, case, variant)
    check_segments(lib, seg, case.idx.numpy(), len(ranks), ranks)
    assert_parity(y, O.lora_linear_case(case), f"{case.name} variant {variant}")
    y0, _, _ = run(lib, case, variant, W=torch.zeros_like(case.W), pool=pool)
    assert_lora_only_parity(y0, O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case),
                                              case.idx.numpy()), f"{case.name} W=0 variant {variant}")


def test_l2_prefetch_hint_does_not_change_results(lib):
    case = wl.decode_q_proj(n=32, h=1024)
    pool = make_pool(lib, case)
    seg = pool.segment(case.idx.to(DEV))
    W, x = case.W.to(DEV), case.x.to(DEV)
    ws = pool.linear_workspace(case.n)
    W_next = torch.randn(1024, 1024, device=DEV).half()
    y0 = torch.empty(case.n, case.h_out, dtype=case.dtype, device=DEV)
    y1 = torch.empty_like(y0)
    lib.lora_linear_fwd(pool.handle, W, x, y0, seg, ws, 1)
    lib.lora_linear_fwd_ex(pool.handle, W, x, y1, seg, ws, 1, prefetch=W_next)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert_parity(y1.cpu(), O.lora_linear_case(case), "prefetch hint")


def test_repeated_calls_are_bit_identical(lib):
    case = wl.decode_q_proj(n=48, h=1024)
    pool = make_pool(lib, case)
    seg = pool.segment(case.idx.to(DEV))
    W, x = case.W.to(DEV), case.x.to(DEV)
    ys = [pool.linear(W, x, seg, variant=1).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_variant_policy_follows_the_measured_sweep(lib):
    """LORA_VARIANT_AUTO against the fused-vs-separate sweep on GB300 (4096 x 4096 fp16):
    r_max 8 with 100 adapters fused up to 128 tokens, separate at 192 and 256; r_max 64 on 6
    adapters fused up to 96 tokens, separate at 128 and 256."""
    dec = lib.LoraPool(4096, 4096, 8, 100, torch.float16, DEV)  # empty slots count at r_max 8
    mix = make_pool(lib, wl.mixed_rank(8))  # ranks {8, 8, 16, 16, 64, 64} mounted, as in the sweep
    F, S = lib.LORA_VARIANT_FUSED, lib.LORA_VARIANT_SEPARATE
    for n, want in ((1, F), (8, F), (64, F), (96, F), (128, F), (192, S), (256, S)):
        assert lib.lora_linear_policy(dec.handle, n) == want, f"r_max 8, {n} tokens"
    for n, want in ((1, F), (64, F), (96, F), (128, S), (256, S)):
        assert lib.lora_linear_policy(mix.handle, n) == want, f"r_max 64, {n} tokens"
    assert lib.lora_linear_policy(dec.handle, 4096) == F  # prefill batches are fused


@pytest.mark.parametrize("n", [1, 8])
def test_fused_decode_repeated_over_one_segment_table(lib, n):
    """Fused decode linears over one segment table on one stream hand x over from the shrink
    to the GEMM through two words of the segment workspace, which every such linear leaves at
    zero: a chain of them, and a chain after a rebuilt segment table, stays exact."""
    case = wl.decode_q_proj(n=n, h=4096)
    pool = make_pool(lib, case)
    W, x = case.W.to(DEV), case.x.to(DEV)
    ref = O.lora_linear_case(case)
    seg = pool.segment(case.idx.to(DEV))
    y = pool.linear(W, x, seg, variant=1)
    ys = [pool.linear(W, x, seg, variant=1) for _ in range(6)]
    seg2 = pool.segment(case.idx.to(DEV))
    ys += [pool.linear(W, x, seg2, variant=1) for _ in range(3)]
    torch.cuda.synchronize()
    assert_parity(y.cpu(), ref, "fused decode")
    for k, yk in enumerate(ys):
        assert torch.equal(yk, y), f"linear {k} of the chain differs"
    for sg in (seg, seg2):
        words = lib.segment_arrays(sg)["nseg"].cpu().tolist()
        assert words[2:] == [0, 0], f"hand-off words left at {words[2:]}"


@pytest.mark.parametrize("n,h_out", [(1, 4096), (16, 4096), (48, 10240)])
def test_fused_decode_with_the_shrink_kernel(lib, n, h_out):
    """A fused decode linear is two launches: the shrink kernel, then the GEMM with the LoRA
    expand in its epilogue."""
    case = wl.random_case(72, n, 256, h_out, [8, 16, 8], r_max=16, dtype=torch.bfloat16)
    pool = make_pool(lib, case)
    seg = pool.segment(case.idx.to(DEV))
    torch.cuda.synchronize()
    c0 = lib.lora_kernel_launch_count()
    y = pool.linear(case.W.to(DEV), case.x.to(DEV), seg, variant=1)
    assert lib.lora_kernel_launch_count() - c0 == 2
    torch.cuda.synchronize()
    assert_parity(y.cpu(), O.lora_linear_case(case), "fused decode after the shrink kernel")
    y0 = pool.linear(torch.zeros_like(case.W).to(DEV), case.x.to(DEV), seg, variant=1).cpu()
    assert_lora_only_parity(y0, O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case),
                                              case.idx.numpy()), "fused decode after the shrink kernel, W=0")


@pytest.mark.parametrize("n", [16, 48])
def test_chained_fused_decode_hands_x_over_from_the_shrink(lib, n):
    """Fused decode GEMMs after the per-token shrink start streaming their weight while the
    previous linear finishes and read x once the shrink has published a value unique to the
    pair (the x-ready word of the segments).  A chain of linears over one set of segments,
    each fed the previous output: every output against the oracle run on the GPU's own input,
    the hand-off words cleared after the chain, and a graph replay of the chain (the same
    values again) bit-identical to the eager run, twice."""
    h, L = 512, 6
    case = wl.random_case(73, n, h, h, [8, 16, 8, 4], r_max=16, dtype=torch.float16)
    pool = make_pool(lib, case)
    seg = pool.segment(case.idx.to(DEV))
    rng = np.random.default_rng(74)
    Ws = [torch.from_numpy(rng.standard_normal((h, h)) * 0.05).to(torch.float16).to(DEV) for _ in range(L)]
    ys = [torch.empty(n, h, dtype=torch.float16, device=DEV) for _ in range(L)]
    ws = torch.empty(lib.lora_linear_workspace_bytes(pool.handle, n), dtype=torch.uint8, device=DEV)
    x0 = case.x.to(DEV)

    def chain():
        x = x0
        for i in range(L):
            pool.linear(Ws[i], x, seg, variant=1, y=ys[i], ws=ws)
            x = ys[i]

    chain()
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    ref_pool = O.pool_of_case(case)
    for i in range(L):
        xin = x0 if i == 0 else eager[i - 1]
        y_ref = O.lora_linear(xin.cpu(), Ws[i].cpu(), ref_pool, case.idx.numpy())
        assert_parity(eager[i].cpu(), y_ref, f"chained linear {i}")
    words = seg_arrays(lib, seg)["nseg"]
    assert words[2:].tolist() == [0, 0]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            chain()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i in range(L):
            assert torch.equal(ys[i], eager[i]), f"graph replay of chained linear {i}"
        assert seg_arrays(lib, seg)["nseg"][2:].tolist() == [0, 0]


# ------------------------------------------------------------------------------------------
# the five workloads
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [1, 2])
def test_decode_q_proj_full(lib, variant):
    case = wl.decode_q_proj()
    y, pool, seg = run(lib, case, variant)
    check_segments(lib, seg, case.idx.numpy(), 100, case.adapters.ranks)
    y_ref = O.lora_linear_case(case)
    assert_parity(y, y_ref, f"decode q_proj variant {variant}")
    y0, _, _ = run(lib, case, variant, W=torch.zeros_like(case.W), pool=pool)
    y0_ref = O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case), case.idx.numpy())
    assert_lora_only_parity(y0, y0_ref, "decode q_proj W=0")
    # negative control: the LoRA-only output must not match the oracle of a shuffled routing
    idx_sh = case.idx.numpy()[np.random.default_rng(0).permutation(case.n)]
    y0_wrong = O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case), idx_sh)
    bound = 1e-2 * np.abs(y0_wrong).max() + 1e-2 * np.abs(y0_wrong)
    assert np.count_nonzero(np.abs(y0.double().numpy() - y0_wrong) > bound) > 0


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
def test_mixed_rank_sweep(lib, n):
    case = wl.mixed_rank(n)
    for variant in (1, 2):
        y, pool, seg = run(lib, case, variant)
        assert_parity(y, O.lora_linear_case(case), f"mixed rank n={n} variant {variant}")
        y0, _, _ = run(lib, case, variant, W=torch.zeros_like(case.W), pool=pool)
        y0_ref = O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case), case.idx.numpy())
        assert_lora_only_parity(y0, y0_ref, f"mixed rank n={n} W=0 variant {variant}")


def test_prefill_full_sampled(lib):
    cases = wl.prefill()
    rows = np.sort(np.random.default_rng(7).choice(16384, 192, replace=False))
    rows = np.unique(np.concatenate([rows, [0, 127, 128, 511, 512, 16383]]))
    for case in cases:
        for variant in (1, 2):
            y, pool, seg = run(lib, case, variant)
            if variant == 1:
                check_segments(lib, seg, case.idx.numpy(), 100, case.adapters.ranks)
            assert_parity(y[rows], O.lora_linear_case(case, rows=rows), f"{case.name} variant {variant}")
        y0, _, _ = run(lib, case, 1, W=torch.zeros_like(case.W), pool=pool)
        y0_ref = O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case), case.idx.numpy(), rows=rows)
        assert_lora_only_parity(y0[rows], y0_ref, f"{case.name} W=0")


def test_full_layer_sampled(lib):
    cases = wl.full_layer(layer=0)
    rows = np.array([0, 1, 63, 64, 100, 200, 254, 255])
    for case in cases:
        y, pool, seg = run(lib, case, 0)
        assert_parity(y[rows], O.lora_linear_case(case, rows=rows), case.name)


# ------------------------------------------------------------------------------------------
# the full-size configurations through the exact calls the benchmark times
# ------------------------------------------------------------------------------------------

LAYER_GROUPS = (("q_proj", "k_proj", "v_proj"), ("o_proj",), ("gate_proj", "up_proj"), ("down_proj",))


def _negative_control(y0, cases, pools_ref, rows=None, seed=5):
    """The LoRA-only output against the oracle of a shuffled routing must fail somewhere."""
    idx = cases[0].idx.numpy()
    shuffled = np.random.default_rng(seed).permutation(idx)
    if np.array_equal(shuffled, idx):
        return
    wrong = O.lora_linear_group(cases[0].x, [torch.zeros_like(c.W) for c in cases], pools_ref, shuffled, rows=rows)
    assert not O.within_tolerance(y0, wrong).all(), "a shuffled routing passes the LoRA-only check"


@pytest.mark.parametrize("variant", [0, 1, 2])
def test_full_layer_grouped_every_row(lib, variant):
    """The 7B-shaped layer (256 tokens bf16, rank 16, 100 adapters, Zipf) as the benchmark runs
    it: q|k|v, o, gate|up and down as four grouped calls (the 256-row-tile GEMM with its token
    split for q|k|v and gate|up under the policy).  Every row of every call against the oracle,
    a LoRA-only run (W = 0) of each, and a negative control."""
    cases = {c.name.split("_", 1)[1]: c for c in wl.full_layer(layer=0)}
    for names in LAYER_GROUPS:
        group = [cases[nm] for nm in names]
        pools_ref = [O.pool_of_case(c) for c in group]
        y, pools, _ = run_group(lib, group, variant)
        ref = O.lora_linear_group(group[0].x, [c.W for c in group], pools_ref, group[0].idx.numpy())
        assert_parity(y, ref, f"{'|'.join(names)} variant {variant}")
        y0, _, _ = run_group(lib, group, variant, pools=pools, zero_w=True)
        ref0 = O.lora_linear_group(group[0].x, [torch.zeros_like(c.W) for c in group], pools_ref,
                                   group[0].idx.numpy())
        assert_lora_only_parity(y0, ref0, f"{'|'.join(names)} W=0 variant {variant}")
        _negative_control(y0, group, pools_ref)
        del pools


def _prefill_rows():
    """One whole 128-token tile of every 512-token request (a different tile position per
    request), the first and last token of every request, and a seeded sample."""
    rows = [np.arange(512 * i + 128 * (i % 4), 512 * i + 128 * (i % 4) + 128) for i in range(32)]
    rows.append(np.concatenate([[512 * i, 512 * i + 511] for i in range(32)]))
    rows.append(np.random.default_rng(8).choice(16384, 256, replace=False))
    return np.unique(np.concatenate(rows))


@pytest.mark.parametrize("variant", [0, 2])
def test_prefill_grouped_tiles(lib, variant):
    """Prefill (32 x 512 tokens bf16) as the benchmark runs it: q_proj and v_proj as one grouped
    call (the grouped tensor-core shrink and the 8192-wide prefill GEMM under the policy)."""
    group = wl.prefill()
    rows = _prefill_rows()
    pools_ref = [O.pool_of_case(c) for c in group]
    y, pools, seg = run_group(lib, group, variant)
    check_segments(lib, seg, group[0].idx.numpy(), 100, group[0].adapters.ranks)
    ref = O.lora_linear_group(group[0].x, [c.W for c in group], pools_ref, group[0].idx.numpy(), rows=rows)
    assert_parity(y[rows], ref, f"prefill q|v variant {variant}")
    y0, _, _ = run_group(lib, group, variant, pools=pools, zero_w=True)
    ref0 = O.lora_linear_group(group[0].x, [torch.zeros_like(c.W) for c in group], pools_ref,
                               group[0].idx.numpy(), rows=rows)
    assert_lora_only_parity(y0[rows], ref0, f"prefill q|v W=0 variant {variant}")
    _negative_control(y0[rows], group, pools_ref, rows=rows)


# (seed, r_max, true ranks, run length, dtype): adapters in runs of `run length` tokens, every
# seventh token base-only, so a 128-token tile holds the number of adapters noted
PREFILL_BLOCK_CASES = [
    (70, 8, [8] * 10, 16, torch.bfloat16),          # 8 per tile: the largest block at r_max 8
    (71, 8, [8, 3] * 6, 13, torch.float16),         # 10-11 per tile: the epilogue's SIMT expand
    (72, 16, [16, 5, 16, 9], 40, torch.bfloat16),   # 3-5 per tile (4 fit a block at r_max 16)
    (73, 32, [32, 17, 32], 64, torch.float16),      # 2-3 per tile at r_max 32
    (74, 64, [64, 33], 128, torch.bfloat16),        # one per tile
    (75, 64, [64, 33, 50], 100, torch.float16),     # 1 or 2 per tile (SIMT when 2)
]


@pytest.mark.parametrize("seed,r_max,ranks,run_len,dtype", PREFILL_BLOCK_CASES)
def test_prefill_lora_block_on_the_tensor_core(lib, seed, r_max, ranks, run_len, dtype):
    """The prefill GEMM adds the LoRA term of a tile as one more tensor-core K block when the
    tile's adapters fit it (count x r_max <= 64), else in its epilogue: tiles of both kinds
    in one call, with base-only tokens, a ragged last token tile and a ragged column tile.
    Every element against the oracle, and the LoRA term alone (W = 0)."""
    n, S = 5 * 128 + 37, len(ranks)
    idx = (np.arange(n) // run_len) % S
    idx[::7] = -1
    case = wl.random_case(seed, n, 256, 320, ranks, r_max=r_max, dtype=dtype, idx=idx)
    y, pool, _ = run(lib, case, 1)
    assert_parity(y, O.lora_linear_case(case), f"prefill LoRA block r_max {r_max} runs of {run_len}")
    y0, _, _ = run(lib, case, 1, W=torch.zeros_like(case.W), pool=pool)
    y0_ref = O.lora_linear(case.x, torch.zeros_like(case.W), O.pool_of_case(case), case.idx.numpy())
    assert_lora_only_parity(y0, y0_ref, f"prefill LoRA block r_max {r_max} W=0")


# ------------------------------------------------------------------------------------------
# segments shared by pools whose slots hold different ranks
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [1, 2])
def test_segments_shared_with_a_pool_of_larger_ranks(lib, variant):
    """The shrink work items carry the ranks of the pool the segments were built on; a pool
    that holds the same slots at larger ranks (r_max 64, 64 tokens: the segmented shrink)
    must still apply every row of its own adapters."""
    small = wl.random_case(50, 64, 4096, 256, [8, 8, 16], r_max=64, dtype=torch.float16)
    big = wl.random_case(51, 64, 4096, 256, [64, 40, 64], r_max=64, dtype=torch.float16,
                         idx=small.idx.numpy())
    pool_small, pool_big = make_pool(lib, small), make_pool(lib, big)
    seg = pool_small.segment(small.idx.to(DEV))
    y = pool_big.linear(big.W.to(DEV), big.x.to(DEV), seg, variant=variant).cpu()
    assert_parity(y, O.lora_linear_case(big), f"shared segments variant {variant}")
    y0 = pool_big.linear(torch.zeros_like(big.W).to(DEV), big.x.to(DEV), seg, variant=variant).cpu()
    assert_lora_only_parity(y0, O.lora_linear(big.x, torch.zeros_like(big.W), O.pool_of_case(big),
                                              big.idx.numpy()), f"shared segments W=0 variant {variant}")


# ------------------------------------------------------------------------------------------
# grouped projections: slices sharing x and segments, one concatenated weight
# ------------------------------------------------------------------------------------------

def group_pools(ags, cases):
    return [make_pool(ags, c) for c in cases]


def run_group(ags, cases, variant=0, pools=None, zero_w=False, ws=None):
    pools = pools or group_pools(ags, cases)
    x, idx = cases[0].x.to(DEV), cases[0].idx.to(DEV)
    n = cases[0].n
    seg_g = Guarded(ags.lora_segment_workspace_bytes(n, pools[0].n_slots), "segment workspace")
    seg = pools[0].segment(idx, ws=seg_g.bytes)
    W = torch.cat([c.W for c in cases], 0).to(DEV)
    if zero_w:
        W.zero_()
    y_g = Guarded.tensor((n, W.shape[0]), cases[0].dtype, "y")
    handles = [p.handle for p in pools]
    guards = [seg_g, y_g]
    if ws is None:
        ws_g = Guarded(ags.lora_linear_group_workspace_bytes(handles, n), "group workspace")
        ws = ws_g.bytes
        guards.append(ws_g)
    ags.lora_linear_fwd_group(handles, W, x, y_g.t, seg, ws, variant)
    torch.cuda.synchronize()
    for g in guards:
        g.check()
    return y_g.t.cpu(), pools, seg


def group_ref(cases, zero_w=False):
    Ws = [torch.zeros_like(c.W) if zero_w else c.W for c in cases]
    return O.lora_linear_group(cases[0].x, Ws, [O.pool_of_case(c) for c in cases], cases[0].idx.numpy())


GROUPS = [
    # (seed, n, h_in, slice h_out, ranks, r_max, dtype)
    (40, 16, 256, [256, 128, 128], [8, 8, 8], 8, torch.float16),  # q, k, v with narrower k/v
    (41, 64, 1024, [512, 512, 512], [8, 16, 8, 16], 16, torch.bfloat16),
    (42, 1, 512, [256, 256], [8], 8, torch.float16),
    (43, 100, 4104, [384, 128], [16, 8, 16, 16, 4], 16, torch.bfloat16),  # ragged K
    (44, 256, 512, [176, 304], [16, 8, 16], 16, torch.bfloat16),  # slice edges inside tiles
    (45, 64, 4096, [512, 256], [64, 8, 64], 64, torch.float16),  # segmented shrink, 2 slices
    (46, 300, 512, [256, 128, 128], [16, 16], 16, torch.bfloat16),  # prefill path
    (47, 700, 256, [272, 528], [8, 8, 8], 8, torch.float16),  # prefill, slice edge inside a tile
    (48, 130, 256, [128, 128, 128, 128], [8, 8], 8, torch.float16),  # four slices
    # prefill tensor-core shrink over every slice: slices x r_max = 256 (one slot per pass),
    # an odd number of 8-row blocks (r_max 8, three slices), many slots per tile (several
    # passes), and slices x r_max above 256 (one shrink launch per slice)
    (49, 300, 256, [128, 128, 128, 128], [64, 8, 64], 64, torch.bfloat16),
    (50, 500, 256, [256, 128, 128], [8, 4, 8, 8, 1], 8, torch.float16),
    (51, 300, 256, [128, 128, 128], [16] * 20, 16, torch.bfloat16),
    (52, 300, 256, [128, 256, 128], [128, 96], 128, torch.float16),
    # the 256-row-tile GEMM just above its switch (65 tokens: N = 80), a ragged last tile
    # (528 rows) and 5 K blocks
    (53, 65, 320, [256, 272], [8, 16, 16], 16, torch.bfloat16),
    # the 256-row-tile GEMM with a single K block, and with 80 tiles (20480 rows)
    (54, 100, 64, [128, 256], [8, 8], 8, torch.float16),
    (55, 80, 128, [10240, 10240], [8, 8], 8, torch.bfloat16),
]


@pytest.mark.parametrize("variant", [0, 1, 2])
@pytest.mark.parametrize("spec", GROUPS, ids=[f"n{s[1]}_{s[2]}x{'+'.join(map(str, s[3]))}" for s in GROUPS])
def test_group_parity(lib, spec, variant):
    seed, n, h_in, h_outs, ranks, r_max, dtype = spec
    cases = wl.random_group(seed, n, h_in, h_outs, ranks, r_max=r_max, dtype=dtype, p_base=0.15)
    y, pools, _ = run_group(lib, cases, variant)
    assert_parity(y, group_ref(cases), f"group {seed} variant {variant}")
    y0, _, _ = run_group(lib, cases, variant, pools=pools, zero_w=True)
    assert_lora_only_parity(y0, group_ref(cases, zero_w=True), f"group {seed} W=0 variant {variant}")
    # negative control: every LoRA token moved to another adapter must not pass
    idx = cases[0].idx.numpy()
    if (idx >= 0).any():
        S = len(ranks)
        moved = np.where(idx >= 0, (idx + 1) % S if S > 1 else -1, idx).astype(np.int32)
        wrong = O.lora_linear_group(cases[0].x, [torch.zeros_like(c.W) for c in cases],
                                    [O.pool_of_case(c) for c in cases], moved)
        assert not O.within_tolerance(y0, wrong).all()


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("n", [1, 8, 16, 64, 300])
def test_group_of_one_is_the_single_linear(lib, n, variant):
    case = wl.random_case(60, n, 512, 384, [8, 16, 8], r_max=16, dtype=torch.bfloat16)
    y1, pools, seg = run_group(lib, [case], variant)
    y = pools[0].linear(case.W.to(DEV), case.x.to(DEV), seg, variant=variant).cpu()
    assert torch.equal(y1, y)


def test_group_slices_with_different_ranks(lib):
    cases = wl.random_group(61, 64, 4096, [256, 256], [8, 8, 8], r_max=64, dtype=torch.float16,
                            slice_ranks=[[8, 8, 8], [64, 33, 64]])
    for variant in (1, 2):
        y0, _, _ = run_group(lib, cases, variant, zero_w=True)
        assert_lora_only_parity(y0, group_ref(cases, zero_w=True), f"mixed slice ranks variant {variant}")


def test_group_errors(lib):
    cases = wl.random_group(62, 16, 256, [128, 128], [8, 8], dtype=torch.float16)
    pools = group_pools(lib, cases)
    handles = [p.handle for p in pools]
    x, W = cases[0].x.to(DEV), torch.cat([c.W for c in cases], 0).to(DEV)
    y = torch.zeros(16, 256, dtype=torch.float16, device=DEV)
    seg = pools[0].segment(cases[0].idx.to(DEV))
    ws = lib._device_bytes(lib.lora_linear_group_workspace_bytes(handles, 16), DEV)

    def code(fn):
        with pytest.raises(lib.LoraError) as e:
            fn()
        return e.value.code

    assert code(lambda: lib.lora_linear_fwd_group([], W, x, y, seg, ws)) == lib.LORA_EINVAL
    assert code(lambda: lib.lora_linear_fwd_group(handles * 3, W, x, y, seg, ws)) == lib.LORA_EINVAL  # 6 > 4
    assert code(lambda: lib.lora_linear_fwd_group(handles, W, x, y, seg, ws, 3)) == lib.LORA_EUNSUP
    small_ws = lib._device_bytes(256, DEV)
    assert code(lambda: lib.lora_linear_fwd_group(handles, W, x, y, seg, small_ws)) == lib.LORA_ENOSPACE
    other = lib.LoraPool(512, 128, 8, 2, torch.float16, DEV)  # different h_in
    assert code(lambda: lib.lora_linear_fwd_group([handles[0], other.handle], W, x, y, seg, ws)) == lib.LORA_EINVAL
    ragged = lib.LoraPool(256, 136, 8, 2, torch.float16, DEV)  # h_out not a multiple of 16
    for s in range(2):
        ragged.load_slot(s, cases[0].adapters.A[s].to(DEV), torch.zeros(136, 8, dtype=torch.float16, device=DEV), 16.0)
    assert code(lambda: lib.lora_linear_group_workspace_bytes([handles[0], ragged.handle], 16)) == lib.LORA_EINVAL
    partial = lib.LoraPool(256, 128, 8, 2, torch.float16, DEV)  # slot 1 not mounted
    partial.load_slot(0, cases[1].adapters.A[0].to(DEV), cases[1].adapters.B[0].to(DEV), 16.0)
    assert code(lambda: lib.lora_linear_fwd_group([handles[0], partial.handle], W, x, y, seg, ws)) == lib.LORA_EINVAL
    f32 = lib.LoraPool(256, 128, 8, 2, torch.float32, DEV)
    assert code(lambda: lib.lora_linear_group_workspace_bytes([f32.handle], 16)) == lib.LORA_EUNSUP
    assert torch.count_nonzero(y) == 0  # nothing ran
    assert lib.lora_linear_group_policy(handles, 64) == lib.LORA_VARIANT_SEPARATE
    assert lib.lora_linear_group_policy(handles, 4096) == lib.LORA_VARIANT_FUSED
    for n in (1, 64, 256, 4096):  # a group of one follows the single-linear policy
        assert lib.lora_linear_group_policy(handles[:1], n) == lib.lora_linear_policy(handles[0], n)


@pytest.mark.parametrize("n", [16, 300])
def test_group_invalid_idx_leaves_y_untouched(lib, n):
    cases = wl.random_group(63, n, 256, [128, 256], [8, 8], dtype=torch.bfloat16)
    pools = group_pools(lib, cases)
    idx = cases[0].idx.clone()
    idx[n // 2] = 7  # no such slot
    seg = pools[0].segment(idx.to(DEV))
    handles = [p.handle for p in pools]
    W = torch.cat([c.W for c in cases], 0).to(DEV)
    y = torch.full((n, 384), 3.0, dtype=torch.bfloat16, device=DEV)
    ws = lib._device_bytes(lib.lora_linear_group_workspace_bytes(handles, n), DEV)
    for variant in (1, 2):
        lib.lora_linear_fwd_group(handles, W, cases[0].x.to(DEV), y, seg, ws, variant)
        torch.cuda.synchronize()
        assert lib.lora_segment_status(seg) == lib.LORA_EIDX
        assert torch.all(y == 3.0)


# ------------------------------------------------------------------------------------------
# host-tier adapter cache: pinned host adapters, LRU eviction of slots the batch does not use
# ------------------------------------------------------------------------------------------

def lru_model(n_slots, batches):
    """Independent model of the replacement rule: hits keep their slot; a miss takes the lowest
    free slot, else the least recently used slot not named by the batch (ties: lowest slot)."""
    slot_of, last, owner, clock, out = {}, [0] * n_slots, [None] * n_slots, 0, []
    for ids in batches:
        clock += 1
        need = sorted({i for i in ids if i >= 0})
        for i in need:
            if i in slot_of:
                last[slot_of[i]] = clock
        for i in need:
            if i in slot_of:
                continue
            free = [s for s in range(n_slots) if owner[s] is None]
            if free:
                s = free[0]
            else:
                cand = [s for s in range(n_slots) if last[s] != clock]
                s = min(cand, key=lambda k: (last[k], k))
                del slot_of[owner[s]]
            owner[s], slot_of[i], last[s] = i, s, clock
        out.append([slot_of[i] if i >= 0 else -1 for i in ids])
    return out


def test_cache_lru_mapping_and_parity(lib):
    n_ad, S, n = 10, 4, 24
    h_in, shapes, R = 256, [(256, 128), (256, 384)], 16  # two projections share the cache
    rng = np.random.default_rng(70)
    ranks = [int(r) for r in rng.choice([4, 8, 16], n_ad)]
    host, oracle_ad = {}, {}
    pools = [lib.LoraPool(hi, ho, R, S, torch.bfloat16, DEV) for hi, ho in shapes]
    cache = lib.LoraCache(pools)
    for a in range(n_ad):
        As, Bs = [], []
        for hi, ho in shapes:
            As.append(torch.from_numpy(rng.uniform(-0.06, 0.06, (ranks[a], hi))).to(torch.bfloat16).pin_memory())
            Bs.append(torch.from_numpy(rng.standard_normal((ho, ranks[a])) * 0.01).to(torch.bfloat16).pin_memory())
        cache.register(100 + a, As, Bs, [2.0 * ranks[a]] * len(shapes))
        oracle_ad[100 + a] = (As, Bs)
    Ws = [torch.from_numpy(rng.standard_normal((ho, hi)) * 0.02).to(torch.bfloat16) for hi, ho in shapes]
    batches = []
    for b in range(6):  # each batch names at most S adapters
        names = rng.choice(n_ad, size=int(rng.integers(1, S + 1)), replace=False) + 100
        batches.append([int(rng.choice(names)) if rng.random() > 0.2 else -1 for _ in range(n)])
    want_slots = lru_model(S, batches)
    evictions = 0
    for b, ids in enumerate(batches):
        idx, mounts = cache.map(ids)
        assert idx.tolist() == want_slots[b], f"batch {b}"
        x = torch.from_numpy(rng.standard_normal((n, h_in))).to(torch.bfloat16)
        seg = pools[0].segment(idx.to(DEV))
        for q, (pool, W) in enumerate(zip(pools, Ws)):
            y = pool.linear(W.to(DEV), x.to(DEV), seg, variant=0).cpu()
            # the oracle sees the adapters by identity, not by slot
            used = sorted({i for i in ids if i >= 0})
            op = O.pad_pool([oracle_ad[i][0][q] for i in used], [oracle_ad[i][1][q] for i in used],
                            [ranks[i - 100] for i in used], [2.0 * ranks[i - 100] for i in used], R, h_in,
                            shapes[q][1])
            local = np.array([used.index(i) if i >= 0 else -1 for i in ids], np.int32)
            assert_parity(y, O.lora_linear(x, W, op, local), f"cache batch {b} projection {q}")
            y0 = pool.linear(torch.zeros_like(W).to(DEV), x.to(DEV), seg, variant=0).cpu()
            assert_lora_only_parity(y0, O.lora_linear(x, torch.zeros_like(W), op, local), f"cache W=0 {b}/{q}")
    st = cache.stats()
    assert st["hits"] + st["misses"] == sum(len({i for i in ids if i >= 0}) for ids in batches)
    assert st["evictions"] > 0 and st["evictions"] == st["misses"] - min(S, st["misses"])
    cache.close()


def test_cache_errors(lib):
    S = 2
    pools = [lib.LoraPool(128, 128, 8, S, torch.float16, DEV)]
    cache = lib.LoraCache(pools)
    A = torch.zeros(8, 128, dtype=torch.float16).pin_memory()
    B = torch.zeros(128, 8, dtype=torch.float16).pin_memory()
    for i in range(3):
        cache.register(i, [A], [B], [16.0])

    def code(fn):
        with pytest.raises(lib.LoraError) as e:
            fn()
        return e.value.code

    assert code(lambda: cache.register(1, [A], [B], [16.0])) == lib.LORA_EBUSY
    big = torch.zeros(16, 128, dtype=torch.float16).pin_memory()
    assert code(lambda: cache.register(7, [big], [torch.zeros(128, 16, dtype=torch.float16).pin_memory()],
                                       [1.0])) == lib.LORA_ERANK
    assert code(lambda: cache.map([0, 5])) == lib.LORA_EIDX  # unknown adapter: nothing mounted
    assert cache.slot_of(0) == -1 and cache.stats() == {"hits": 0, "misses": 0, "evictions": 0}
    assert code(lambda: cache.map([0, 1, 2])) == lib.LORA_ENOSPACE  # three adapters, two slots
    idx, mounts = cache.map([0, -1, 1, 0])
    assert idx.tolist() == [0, -1, 1, 0] and mounts == 2
    idx, mounts = cache.map([2, 1])  # 0 is least recently used and not named: evicted
    assert idx.tolist() == [0, 1] and mounts == 1 and cache.slot_of(0) == -1
    cache.unregister(2)
    assert cache.slot_of(1) == 1 and code(lambda: cache.slot_of(2)) == lib.LORA_EIDX
    busy = lib.LoraPool(128, 128, 8, S, torch.float16, DEV)
    busy.load_slot(0, A.to(DEV), B.to(DEV), 16.0)
    assert code(lambda: lib.LoraCache([busy])) == lib.LORA_EBUSY
    other = lib.LoraPool(128, 128, 8, S + 1, torch.float16, DEV)
    fresh = lib.LoraPool(128, 128, 8, S, torch.float16, DEV)
    assert code(lambda: lib.LoraCache([fresh, other])) == lib.LORA_EINVAL  # slot counts differ
    cache.close()


# ------------------------------------------------------------------------------------------
# B tiles staged at true ranks: a graph captured with low ranks, replayed after remounting
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", [1, 0])
def test_graph_replay_after_remount_at_larger_ranks(lib, variant):
    """The decode GEMM sizes its staging of B tiles from the ranks mounted when it is
    launched; a CUDA graph keeps that launch.  After slots are remounted at r_max the replay
    must still be exact (tiles that no longer fit take the late path)."""
    n, h, R = 64, 4096, 64
    low = wl.random_case(80, n, h, 512, [8, 8, 16, 16, 8, 8], r_max=R, dtype=torch.float16, p_base=0.0)
    high = wl.random_case(81, n, h, 512, [64, 64, 64, 64, 64, 64], r_max=R, dtype=torch.float16,
                          idx=low.idx.numpy())
    pool = make_pool(lib, low)
    seg = pool.segment(low.idx.to(DEV))
    W, x = low.W.to(DEV), low.x.to(DEV)
    y = torch.empty(n, 512, dtype=torch.float16, device=DEV)
    ws = pool.linear_workspace(n)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        lib.lora_linear_fwd(pool.handle, W, x, y, seg, ws, variant)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        lib.lora_linear_fwd(pool.handle, W, x, y, seg, ws, variant)
    g.replay()
    torch.cuda.synchronize()
    assert_parity(y.cpu(), O.lora_linear_case(low), "graph, low ranks")
    for s in range(6):  # same slots, now at r_max (on the capture stream, ordered before the replay)
        pool.unload_slot(s, stream=st)
        pool.load_slot(s, high.adapters.A[s].to(DEV), high.adapters.B[s].to(DEV), high.adapters.alphas[s], stream=st)
    with torch.cuda.stream(st):
        g.replay()
    torch.cuda.synchronize()
    want = O.lora_linear(low.x, low.W, O.pool_of_case(high), low.idx.numpy())
    assert_parity(y.cpu(), want, "graph replayed after remounting at r_max")
    y0 = torch.empty_like(y)
    lib.lora_linear_fwd(pool.handle, torch.zeros_like(W), x, y0, seg, ws, variant)
    torch.cuda.synchronize()
    assert_lora_only_parity(y0.cpu(), O.lora_linear(low.x, torch.zeros_like(low.W), O.pool_of_case(high),
                                                    low.idx.numpy()), "remounted, W=0")
