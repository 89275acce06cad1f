// Grouped tensor-core shrink for long batches (prefill): s[t, :] = (alpha_s/r_s) x[t] A_s^T.
//
// One CTA per 128-token tile in original token order.  The CTA first finds the distinct adapter
// slots its tokens name (the adapter-level bucket of "LLM 多 LoRA 推理服务工程 2026：从热插拔到
// 租户编排", blog.lonae.com, restricted to the tile), then runs a tcgen05 GEMM whose N operand is
// the concatenation of those slots' zero-padded A rows (gathered per K-block by one TMA box per
// slot from the pool's A slab) -- the pages' concatenated matmul, but only over the adapters the
// tile touches.  Each token keeps the r_max columns of its own slot.  A prefill tile usually
// holds one request and therefore one slot, so N = r_max and x is read once at HBM speed.
// Tiles touching more than 256 / r_max slots run several passes over K.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace lora {
namespace tc {

using namespace ptx;

constexpr int kShrBM = 128;
constexpr int kShrBK = 64;
constexpr int kShrMaxN = 256;
constexpr int kShrStages = 4;
constexpr int kShrThreads = 192;
constexpr uint32_t kShrXBytes = kShrBM * kShrBK * 2;
constexpr uint32_t kShrBBytes = kShrMaxN * kShrBK * 2;
constexpr uint32_t kShrStageBytes = kShrXBytes + kShrBBytes;
constexpr size_t kShrSmem = (size_t)kShrStages * kShrStageBytes + 1024 + 4096;

struct ShrinkArgs {
    PoolView pool;
    GroupView grp;  // slices sharing x and idx; slice q's output at s_out + q * grp.s_stride
    SegView seg;
    float* s_out;
    int n, kb_total, bf16;
};

// The N operand of a pass holds, for each of its slots and then each slice, that slice's
// r_max rows of the slot's A: a token's G * r_max accumulator columns are contiguous.
template <typename T>
__global__ void __launch_bounds__(kShrThreads, 1)
shrink_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA0,
                 const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2,
                 const __grid_constant__ CUtensorMap tmA3, const ShrinkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align(smem_raw, 1024);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kShrStages * kShrStageBytes);
    uint64_t* empty = full + kShrStages;
    uint64_t* acc_full = empty + kShrStages;  // [2]
    uint64_t* acc_empty = acc_full + 2;       // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] abort, [4..7] scan
    int* tok_slot = const_cast<int*>(flags) + 8;  // [128]
    int* fidx = tok_slot + kShrBM;                // [128]
    int* dloc = fidx + kShrBM;                    // [128]
    int* dlist = dloc + kShrBM;                   // [128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kShrBM;
    const int R = a.pool.R;

    pdl_wait();  // idx, status and x come from earlier kernels
    pdl_trigger();
    if (__ldcg(a.seg.status) != LORA_OK) return;

    // ---- the tile's distinct slots (threads 0..127, one token each) ----
    const int q = threadIdx.x;
    if (q < kShrBM) tok_slot[q] = (m0 + q < a.n) ? __ldcg(a.seg.idx + m0 + q) : -1;
    __syncthreads();
    bool is_first = false;
    if (q < kShrBM) {
        int f = -1;
        if (tok_slot[q] >= 0) {
            f = q;
            for (int q2 = 0; q2 < q; ++q2)
                if (tok_slot[q2] == tok_slot[q]) {
                    f = q2;
                    break;
                }
        }
        fidx[q] = f;
        is_first = f == q;
    }
    int* wsum = const_cast<int*>(flags) + 4;
    const unsigned bal = __ballot_sync(0xffffffffu, is_first);
    if (q < kShrBM && lane == 0) wsum[warp] = __popc(bal);
    __syncthreads();
    if (is_first) {
        int base = 0;
        for (int w = 0; w < warp; ++w) base += wsum[w];
        const int d = base + __popc(bal & ((1u << lane) - 1u));
        dloc[q] = d;
        dlist[d] = tok_slot[q];
    }
    const int D = wsum[0] + wsum[1] + wsum[2] + wsum[3];
    __syncthreads();
    if (q < kShrBM && !is_first) dloc[q] = fidx[q] >= 0 ? dloc[fidx[q]] : -1;
    if (D == 0) return;  // base-only tile: nothing to shrink

    const int G = a.grp.count;
    const int GR = G * R;            // accumulator columns per slot
    const int spp = kShrMaxN / GR;   // slots per pass
    const int passes = (D + spp - 1) / spp;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kShrStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        flags[0] = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmA0);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * kShrMaxN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nkb = a.kb_total;

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int p = 0; p < passes && !flags[0]; ++p) {
                const int d0 = p * spp, dn = min(spp, D - d0);
                const int rows = dn * GR, rows_pad = (rows + 15) / 16 * 16;
                const uint32_t bytes = kShrXBytes + rows_pad * kShrBK * 2;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % kShrStages;
                    if (it >= kShrStages && !mbar_wait(&empty[s], ((it / kShrStages) & 1) ^ 1, flags)) break;
                    mbar_arrive_expect_tx(&full[s], bytes);
                    uint8_t* st = smem + s * kShrStageBytes;
                    tma_load_2d(st, &tmX, &full[s], kb * kShrBK, m0);
                    for (int d = 0; d < dn; ++d)
                        for (int q = 0; q < G; ++q) {
                            const CUtensorMap* mA = q == 0 ? &tmA0 : q == 1 ? &tmA1 : q == 2 ? &tmA2 : &tmA3;
                            tma_load_2d(st + kShrXBytes + (d * G + q) * R * 128, mA, &full[s], kb * kShrBK,
                                        dlist[d0 + d] * R);
                        }
                    if (rows_pad > rows) {  // r_max = 8 and an odd row-block count: repeat the last block
                        const int q = G - 1;
                        const CUtensorMap* mA = q == 0 ? &tmA0 : q == 1 ? &tmA1 : q == 2 ? &tmA2 : &tmA3;
                        tma_load_2d(st + kShrXBytes + rows * 128, mA, &full[s], kb * kShrBK, dlist[d0 + dn - 1] * R);
                    }
                }
            }
            if (flags[0]) {
                report_timeout_status(a.seg.status);
                for (int i = max(0, it - kShrStages); i < it; ++i) {
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&full[i % kShrStages], (i / kShrStages) & 1) &&
                           globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int p = 0; p < passes && ok; ++p) {
                const int buf = p & 1;
                const int rows_pad = (min(spp, D - p * spp) * GR + 15) / 16 * 16;
                const uint32_t idesc = idesc_f16(kShrBM, rows_pad, a.bf16 != 0);
                if (!mbar_wait(&acc_empty[buf], ((p >> 1) & 1) ^ 1, flags)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % kShrStages;
                    if (!mbar_wait(&full[s], (it / kShrStages) & 1, flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xa = smem_u32(smem + s * kShrStageBytes);
                    const uint32_t ba = xa + kShrXBytes;
#pragma unroll
                    for (int k = 0; k < kShrBK / 16; ++k)
                        umma_f16(tmem + buf * kShrMaxN, sdesc_sw128(xa + k * 32), sdesc_sw128(ba + k * 32), idesc,
                                 (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[s]);
                }
                umma_commit(&acc_full[buf]);
            }
            if (!ok) report_timeout_status(a.seg.status);
        }
    } else {
        // ---- epilogue: thread <-> token row; keep the r_max columns of the token's own slot ----
        const int row = (warp & 3) * 32 + lane;
        const int t = m0 + row;
        const int slot = tok_slot[row];
        const int dl = dloc[row];
        float scale[kMaxGroup];  // alpha / r of the token's slot in every slice
#pragma unroll
        for (int q = 0; q < kMaxGroup; ++q)
            scale[q] = (slot >= 0 && q < G) ? group_slice(a.grp, q).table[slot].scale : 0.f;
        for (int p = 0; p < passes; ++p) {
            const int buf = p & 1;
            const bool got = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (p >> 1) & 1, flags));
            if (!got) break;
            tc_fence_after();
            const int d0 = p * spp, dn = min(spp, D - d0);
            const int rows_pad = (dn * GR + 15) / 16 * 16;
            const bool mine = slot >= 0 && dl >= d0 && dl < d0 + dn;
            const int col0 = (dl - d0) * GR;  // the token's G * r_max columns
            const uint32_t taddr = tmem + buf * kShrMaxN + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            for (int c0 = 0; c0 < rows_pad; c0 += 16) {
                uint32_t r[16];
                __syncwarp();
                tmem_ld16(taddr + c0, r);
                tmem_ld_wait();
                if (mine && c0 + 16 > col0 && c0 < col0 + GR) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int col = c0 + c - col0;
                        if (col >= 0 && col < GR) {
                            const int q = col / R, j = col - q * R;
                            float sc = scale[0];
#pragma unroll
                            for (int i = 1; i < kMaxGroup; ++i)
                                if (i == q) sc = scale[i];
                            a.s_out[q * a.grp.s_stride + (long long)t * R + j] = sc * __uint_as_float(r[c]);
                        }
                    }
                }
            }
            tc_fence_before();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * kShrMaxN);
}

template <typename T>
static int launch_shrink_tc_t(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                              cudaStream_t st) {
    const int n = sv.n;
    if (n == 0) return LORA_OK;
    if (grp.count < 1 || grp.count > kMaxGroup || grp.count * pv.R > kShrMaxN)
        return set_error(LORA_EINVAL, "internal: tensor-core shrink of %d slices of rank %d", grp.count, pv.R);
    const int bf16 = pv.dtype == LORA_BF16;
    CUtensorMap mX, mA[kMaxGroup];
    int rc = make_map(&mX, x, bf16, pv.h_in, n, kShrBM);
    if (rc) return rc;
    for (int q = 0; q < kMaxGroup; ++q) {  // unused maps repeat slice 0's
        rc = make_map(&mA[q], grp.A[q < grp.count ? q : 0], bf16, pv.h_in, (uint64_t)pv.S * pv.R, pv.R);
        if (rc) return rc;
    }
    ShrinkArgs a;
    a.pool = pv;
    a.grp = grp;
    a.seg = sv;
    a.s_out = s_out;
    a.n = n;
    a.kb_total = (pv.h_in + kShrBK - 1) / kShrBK;
    a.bf16 = bf16;
    static bool attr_set = false;
    if (!attr_set) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(shrink_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kShrSmem));
        attr_set = true;
    }
    void* args[] = {(void*)&mX, (void*)&mA[0], (void*)&mA[1], (void*)&mA[2], (void*)&mA[3], (void*)&a};
    LORA_CUDA_TRY(launch_pdl((const void*)shrink_tc_kernel<T>, dim3((n + kShrBM - 1) / kShrBM), dim3(kShrThreads),
                             kShrSmem, st, args));
    return LORA_OK;
}

}  // namespace tc

int shrink_tc_supported(const PoolView& pv) {
    return (pv.dtype == LORA_F16 || pv.dtype == LORA_BF16) && pv.h_in % 8 == 0 && pv.R % 8 == 0 &&
           pv.R <= tc::kShrMaxN;
}

int launch_shrink_tc(const PoolView& pv, const SegView& sv, const void* x, float* s_out, cudaStream_t st) {
    return launch_shrink_tc_group(pv, single_group(pv), sv, x, s_out, st);
}

int launch_shrink_tc_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                           cudaStream_t st) {
    if (pv.dtype == LORA_F16) return tc::launch_shrink_tc_t<__half>(pv, grp, sv, x, s_out, st);
    return tc::launch_shrink_tc_t<__nv_bfloat16>(pv, grp, sv, x, s_out, st);
}

int shrink_tc_group_supported(const PoolView& pv, int count) {
    return shrink_tc_supported(pv) && count >= 1 && count <= kMaxGroup && count * pv.R <= tc::kShrMaxN;
}

}  // namespace lora
