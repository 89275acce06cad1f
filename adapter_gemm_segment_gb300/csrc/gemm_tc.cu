// Tensor-core base GEMM of the LoRA-augmented linear on sm_103a (tcgen05 + TMEM + TMA),
// with the LoRA expand fused into the epilogue.
//
// The "fused kernel" design of the adapter execution unit ("LLM 多 LoRA 推理服务工程 2026：
// 从热插拔到租户编排", blog.lonae.com) computes the base linear and the A/B product in one
// launch; here the base product x W^T accumulates in tensor memory and the epilogue adds
// scale_s * s[t,:] B_s^T (s from the shrink kernel, scale folded in) before rounding y once.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 owns TMEM and issues tcgen05.mma
// from one thread, warps 2..5 drain the accumulator (warp w may only touch TMEM lanes
// 32*(w%4) .. 32*(w%4)+31).  A ring of shared-memory stages with full/empty mbarriers
// connects producer and MMA; tcgen05.commit releases stages and publishes accumulators.
//
// Decode (n <= 256 tokens): swap-AB.  The weight tile (128 output features) is the MMA M side
// and the tokens (padded to a multiple of 16) the N side, so the whole batch is one N tile and
// W streams through exactly once.  K is split over the CTAs of a thread-block cluster (up to 8)
// to fill the GPU: each CTA parks its float32 partial tile in shared memory, the partials are
// exchanged by shared-to-remote-shared bulk copies (DSMEM) so that each CTA of the cluster owns
// a slice of the tokens, and each CTA sums its slice in split order, adds the LoRA term and
// stores its tokens of y with a TMA store.  Behind the per-token shrink kernel the GEMM is
// released at the shrink's start and reads x once the shrink has published the pair's x-ready
// value (its weight stream overlaps the previous linear's tail).
//
// Prefill (n > 256): 128-token x 256-feature tiles, persistent CTAs over the tile list,
// double-buffered accumulators (2 x 256 TMEM columns) so the epilogue of one tile overlaps the
// main loop of the next.  A tile's LoRA term is one more tensor-core K block when its adapters
// fit one (below), and y leaves through shared memory and TMA stores.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace lora {
namespace tc {

using namespace ptx;

constexpr int BM = 128;       // MMA M
constexpr int BK = 64;        // K per stage (one 128-byte swizzle row of 16-bit elements)
constexpr int UMMA_K = 16;    // K per tcgen05.mma of kind::f16
constexpr int kThreads = 192;
constexpr int kPrefillBN = 256;
constexpr int kDecodeMaxN = 256;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kLsmMaxTokens = 32;
constexpr int kYChunk = 32;  // tokens per TMA store of the decode output
constexpr int kYBatch = 16;  // tokens whose partials one epilogue thread loads before adding them

struct DecodeArgs {
    PoolView pool;
    SegView seg;
    const float* s_in;
    void* y;
    int n, n_pad, kb_total, splits, kb_per_split, stages, tmem_cols, fuse, bf16;
    int nacc;     // independent TMEM accumulators the K-blocks rotate over (summed in the epilogue)
    int kc;       // 64-wide K chunks per pipeline stage (one TMA box per operand and stage)
    int s_parts;  // K-parts of the shrink output to sum
    int bpre_bytes;  // room for B tiles staged during the main loop
    int compact;     // stage each tile at its slot's true rank (else at r_max, no table read)
    int push;     // exchange partials by bulk copies (1) or remote loads (0)
    const char* prefetch;  // optional range streamed into L2 once this CTA's accumulator is complete
    size_t prefetch_bytes;
    unsigned long long* stamp;  // benchmark instrumentation (nullptr: off)
    // x-ready hand-off with the shrink kernel before this grid (nonzero: the value it publishes
    // in *xword once every earlier kernel is complete; xword[1] counts this grid's readers)
    int xready;
    int* xword;
};

struct PrefillArgs {
    PoolView pool;
    GroupView grp;  // output slices (one for a single linear); y row stride grp.ldy
    SegView seg;
    const float* s_in;
    void* y;
    int n, m_tiles, n_tiles, kb_total, stages, fuse, bf16;
    int lora_mma;  // one more pipeline block per tile: the LoRA expand on the tensor core
    unsigned long long* stamp;  // benchmark instrumentation (nullptr: off)
};

// Tile order of the persistent prefill kernel: output columns in groups of kPrefillNGroup
// tiles (4096 features), and inside a group every token tile before the next group.  A wave of
// CTAs then shares one group's weight (33.5 MB at 4096 inputs), which stays in L2 while the
// token tiles stream past; x is read once per group.  Odd groups walk the token tiles in
// reverse, so the first ones they need are the last the previous group read (still in L2).
// Measured on GB300 (q|v as one 8192-wide launch, 16384 tokens bf16): DRAM reads 377 MB in
// order, 367 MB snaking, same time; walking all 32 column tiles in every wave evicted the
// weight (1.74 GB of reads, 5 % slower), also with evict-last hints on the weight's loads.
constexpr int kPrefillNGroup = 16;

__device__ __forceinline__ void prefill_tile(int tile, int m_tiles, int n_tiles, int& m0, int& n0) {
    const int per_group = m_tiles * kPrefillNGroup;
    const int g = tile / per_group;
    const int gw = min(kPrefillNGroup, n_tiles - g * kPrefillNGroup);  // column tiles in this group
    const int r = tile - g * per_group;
    m0 = ((g & 1) ? (m_tiles - 1 - r / gw) : (r / gw)) * BM;
    n0 = (g * kPrefillNGroup + r % gw) * kPrefillBN;
}

// LoRA term of one (token, feature): sum_j s[t, j] * B_slot[o, j]; s already carries alpha/r.
template <typename T>
__device__ __forceinline__ float lora_term(const T* __restrict__ Brow, const float* __restrict__ srow, int R) {
    float acc = 0.f;
    for (int j = 0; j < R; j += 8) {
        float b[8];
        unpack8<T>(__ldg(reinterpret_cast<const uint4*>(Brow + j)), b);
        const float4 s0 = __ldcg(reinterpret_cast<const float4*>(srow + j));
        const float4 s1 = __ldcg(reinterpret_cast<const float4*>(srow + j + 4));
        acc = fmaf(b[0], s0.x, acc);
        acc = fmaf(b[1], s0.y, acc);
        acc = fmaf(b[2], s0.z, acc);
        acc = fmaf(b[3], s0.w, acc);
        acc = fmaf(b[4], s1.x, acc);
        acc = fmaf(b[5], s1.y, acc);
        acc = fmaf(b[6], s1.z, acc);
        acc = fmaf(b[7], s1.w, acc);
    }
    return acc;
}

// Two float32 values rounded to the 16-bit type, packed (low half first).
template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Eight float32 values rounded to the 16-bit type, as one 16-byte chunk.
template <typename T>
__device__ __forceinline__ uint4 pack8(const float4& lo, const float4& hi) {
    alignas(16) T v[8] = {from_f32<T>(lo.x), from_f32<T>(lo.y), from_f32<T>(lo.z), from_f32<T>(lo.w),
                          from_f32<T>(hi.x), from_f32<T>(hi.y), from_f32<T>(hi.z), from_f32<T>(hi.w)};
    return *reinterpret_cast<const uint4*>(v);
}

// dot(B row of one feature, s row of one token) over r_max, both in shared memory.  Lanes walk
// the 16-byte chunks of their rows in a staggered order so that a warp whose lanes read
// consecutive B rows (row pitch r_max*2 bytes) hits distinct banks for any r_max.
template <typename T>
__device__ __forceinline__ float lora_dot_smem(const uint4* __restrict__ br, const float* __restrict__ sr, int chunks,
                                               int lane) {
    float acc = 0.f;
    for (int jj = 0; jj < chunks; ++jj) {
        const int jc = (jj + lane) % chunks;
        float b[8];
        unpack8<T>(br[jc], b);
        const float4 s0 = reinterpret_cast<const float4*>(sr + jc * 8)[0];
        const float4 s1 = reinterpret_cast<const float4*>(sr + jc * 8)[1];
        acc = fmaf(b[0], s0.x, acc);
        acc = fmaf(b[1], s0.y, acc);
        acc = fmaf(b[2], s0.z, acc);
        acc = fmaf(b[3], s0.w, acc);
        acc = fmaf(b[4], s1.x, acc);
        acc = fmaf(b[5], s1.y, acc);
        acc = fmaf(b[6], s1.z, acc);
        acc = fmaf(b[7], s1.w, acc);
    }
    return acc;
}

// LoRA term of one feature (B row `row`) for up to 8 tokens q0..q0+7 at once, all operands in
// shared memory; every load of the batch is issued before it is used.  Tokens whose slot index
// (dloc - g0) is outside [0, Dg) get 0.
template <typename T>
__device__ __forceinline__ void lora_batch8(const T* __restrict__ Bg, const float* __restrict__ S_sm,
                                            const int* __restrict__ dloc_sm, int q0, int cnt, int g0, int Dg, int row,
                                            int R, int lane, float (&acc)[8]) {
    const int chunks = R / 8;
    int d[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        d[u] = q0 + u < cnt ? dloc_sm[q0 + u] - g0 : -1;
        if (d[u] >= Dg) d[u] = -1;
        acc[u] = 0.f;
    }
    if (Dg <= 0) return;  // nothing staged: do not touch the (empty) B region
    const uint4* B4 = reinterpret_cast<const uint4*>(Bg);
    for (int jj = 0; jj < chunks; ++jj) {
        const int jc = (jj + lane) % chunks;  // staggered: conflict-free rows for any r_max
        uint4 bv[8];
        float4 s0[8], s1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int du = d[u] < 0 ? 0 : d[u];
            bv[u] = B4[(size_t)(du * BM + row) * chunks + jc];
            const float4* sp = reinterpret_cast<const float4*>(S_sm + min(q0 + u, cnt - 1) * R + jc * 8);
            s0[u] = sp[0];
            s1[u] = sp[1];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float b[8];
            unpack8<T>(bv[u], b);
            float v = acc[u];
            v = fmaf(b[0], s0[u].x, v);
            v = fmaf(b[1], s0[u].y, v);
            v = fmaf(b[2], s0[u].z, v);
            v = fmaf(b[3], s0[u].w, v);
            v = fmaf(b[4], s1[u].x, v);
            v = fmaf(b[5], s1[u].y, v);
            v = fmaf(b[6], s1[u].z, v);
            v = fmaf(b[7], s1[u].w, v);
            acc[u] = d[u] >= 0 ? v : 0.f;
        }
    }
}

// The same for slots staged at their true rank: staged slot d's tile is pre_sm[1 + kMaxPre + d]
// chunk blocks of [128 rows][8 columns] (16 bytes per row), the first at uint4 offset
// pre_sm[1 + d]; a warp's 32 consecutive rows read 32 consecutive 16-byte words.  Columns past
// a slot's rank are zero in B and in s, so they are skipped; the loop runs over the largest
// chunk count among the eight tokens.
constexpr int kMaxPre = 32;

template <typename T>
__device__ __forceinline__ void lora_batch8_pre(const uint4* __restrict__ Bp4, const int* __restrict__ pre_sm,
                                                const float* __restrict__ S_sm, const int* __restrict__ dloc_sm,
                                                int q0, int cnt, int Dg, int row, int R, int lane, float (&acc)[8]) {
    int off[8], c[8];
    int cmax = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        int d = q0 + u < cnt ? dloc_sm[q0 + u] : -1;
        if (d >= Dg) d = -1;
        c[u] = d >= 0 ? pre_sm[1 + kMaxPre + d] : 0;
        off[u] = d >= 0 ? pre_sm[1 + d] + row : 0;
        cmax = max(cmax, c[u]);
        acc[u] = 0.f;
    }
    for (int jc = 0; jc < cmax; ++jc) {
        uint4 bv[8];
        float4 s0[8], s1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            bv[u] = jc < c[u] ? Bp4[off[u] + jc * BM] : make_uint4(0, 0, 0, 0);
            const float4* sp = reinterpret_cast<const float4*>(S_sm + min(q0 + u, cnt - 1) * R + jc * 8);
            s0[u] = sp[0];
            s1[u] = sp[1];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float b[8];
            unpack8<T>(bv[u], b);
            float v = acc[u];
            v = fmaf(b[0], s0[u].x, v);
            v = fmaf(b[1], s0[u].y, v);
            v = fmaf(b[2], s0[u].z, v);
            v = fmaf(b[3], s0[u].w, v);
            v = fmaf(b[4], s1[u].x, v);
            v = fmaf(b[5], s1[u].y, v);
            v = fmaf(b[6], s1[u].z, v);
            v = fmaf(b[7], s1[u].w, v);
            acc[u] = v;
        }
    }
}

// ============================================================================================
// decode: swap-AB + split-K over a thread-block cluster
// ============================================================================================
// The `splits` CTAs that share one 128-feature tile form a cluster (cluster dims 1 x splits);
// CTA r owns the reduction of tokens [r*per, r*per + per).
//  phase A (epilogue warps, overlapping the main loop): the slot ids of the owned tokens, their
//          distinct slots, and -- by bulk copies -- the B rows of those slots for this feature
//          tile and the owned tokens' shrink output; then the LoRA term of every owned
//          (token, feature) pair.
//  phase B: the float32 partial tile [n_pad tokens][128 features] is parked in the idle stages.
//  phase C: after a cluster barrier, each CTA bulk-copies the partial rows of the tokens another
//          CTA owns into that CTA's receive buffer (completion on the receiver's mbarrier); when
//          the buffers do not fit, owners read the partials remotely instead.
//  phase D: owners add the partials, the LoRA term and store y.  No global scratch.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
gemm_decode_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmYtail,
                   const __grid_constant__ CUtensorMap tmB, const DecodeArgs a) {
    stamp_start(a.stamp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align(smem_raw, 1024);
    const int stages = a.stages;
    const int kc = a.kc;
    const uint32_t w_bytes = BM * BK * 2 * kc;
    const uint32_t x_bytes = static_cast<uint32_t>(a.n_pad) * BK * 2 * kc;
    const uint32_t stage_bytes = w_bytes + x_bytes;
    const int R = a.pool.R;
    const int per = (a.n_pad + a.splits - 1) / a.splits;  // tokens reduced by each CTA
    const bool use_lsm = per <= kLsmMaxTokens;
    // dedicated region after the stages (layout mirrored by plan_decode)
    int* slot_sm = reinterpret_cast<int*>(smem + (size_t)stages * stage_bytes);  // [per]
    int* dloc_sm = slot_sm + per;                                               // [per]
    int* dlist = dloc_sm + per;                                                 // [per]
    int* fidx_sm = dlist + per;                                                 // [per]
    int* pre_sm = fidx_sm + per;  // [1 + 2 kMaxPre]: staged slots; their uint4 offsets; chunks per row
    float* S_sm = smem_align(reinterpret_cast<float*>(pre_sm + 1 + 2 * kMaxPre), 16);  // [s_parts][per][R]
    float* L_sm = S_sm + (size_t)a.s_parts * per * R;                            // [per][128] if use_lsm
    T* Bpre = smem_align(reinterpret_cast<T*>(L_sm + (use_lsm ? (size_t)per * BM : 0)), 128);  // bpre_bytes
    uint64_t* full = smem_align(reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(Bpre) + a.bpre_bytes), 8);
    uint64_t* empty = full + stages;
    uint64_t* tmem_full = empty + stages;
    uint64_t* lbar = tmem_full + 1;  // LoRA operands staged
    uint64_t* rbar = lbar + 1;       // partial rows received
    uint64_t* xbar = rbar + 1;       // x-ready: the producer has seen the shrink's signal
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // abort, go, D, status, wsum[4]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tile = blockIdx.x, split = blockIdx.y;
    // K range of this split in 64-wide blocks, walked in stages of kc blocks
    const int kb0 = split * a.kb_per_split;
    const int nkb = (min(a.kb_total, kb0 + a.kb_per_split) - kb0 + kc - 1) / kc;  // stages
    // Every feature tile reads the same x slice; starting each tile's walk over its K range at a
    // different stage keeps the concurrent reads of x spread over different lines.
    const int kb_rot = nkb > 0 ? m_tile % nkb : 0;
    const int n = a.n, h_out = a.pool.h_out;
    const int rank = static_cast<int>(cluster_ctarank());
    const int t0 = rank * per;
    const int cnt = max(0, min(n, t0 + per) - t0);
    const int rows_valid = min(BM, h_out - m_tile * BM);
    // stage area after the main loop: P [n_pad][128] | Rcv [splits][per][128] | late B tiles
    float* P = reinterpret_cast<float*>(smem);
    float* Rcv = P + (size_t)a.n_pad * BM;
    const bool push = a.push != 0;

    // stage i of this CTA's K walk: its W box and x box, counted on full[i % stages]
    auto issue_w = [&](int i) {  // expects the whole stage, loads its W box
        const int s = i % stages;
        const int kb = kb0 + ((i + kb_rot) % nkb) * kc;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        if (kc == 1)
            tma_load_2d_cta(smem + s * stage_bytes, &tmW, &full[s], kb * BK, m_tile * BM);
        else
            tma_load_3d_cta(smem + s * stage_bytes, &tmW, &full[s], 0, m_tile * BM, kb);
    };
    auto issue_x = [&](int i) {
        const int s = i % stages;
        const int kb = kb0 + ((i + kb_rot) % nkb) * kc;
        if (kc == 1)
            tma_load_2d_cta(smem + s * stage_bytes + w_bytes, &tmX, &full[s], kb * BK, 0);
        else
            tma_load_3d_cta(smem + s * stage_bytes + w_bytes, &tmX, &full[s], 0, 0, kb);
    };
    auto issue_stage = [&](int i) {
        issue_w(i);
        issue_x(i);
    };
    // The producer thread initialises the barriers and fills the ring right away, so the first
    // HBM round trip overlaps the TMEM allocation and the CTA-wide barrier below.  With the
    // x-ready hand-off the previous linear may still be running, so only the W boxes go out now
    // (a weight is never written by the kernels of the linear chain); the x boxes follow the
    // hand-off.
    const int pre = min(stages, nkb);
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tmem_full, 1);
        mbar_init(lbar, 1);
        mbar_init(rbar, 1);
        mbar_init(xbar, 1);
        for (int i = 0; i < 8; ++i) flags[i] = 0;
        fence_barrier_init();
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
        for (int i = 0; i < pre; ++i) {
            if (a.xready)
                issue_w(i);
            else
                issue_stage(i);
        }
        prefetch_tmap(&tmY);
        prefetch_tmap(&tmYtail);
        if (a.compact && a.fuse) prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    const int et = threadIdx.x - 64;  // 0..127 in the epilogue warps
    const int row = (warp & 3) * 32 + lane;
    const int o = m_tile * BM + row;
    const int chunks = R / 8;  // 16-byte chunks per B row
    const T* B = static_cast<const T*>(a.pool.B);

    if (warp == 0) {
        // Without a hand-off, W and x are complete when this grid starts if a shrink kernel
        // precedes it in the stream: it releases its dependents only after its own
        // grid-dependency wait, and only the shrink output (read by the epilogue warps) needs
        // this grid's wait.  With the x-ready hand-off the shrink released this grid at its
        // start, and x is read once the shrink has published the pair's value.
        if (lane == 0) {
            if (a.xready) {
                // The shrink kernel before this grid released it at its start and publishes the
                // value once every earlier kernel is complete: x may then be read (through TMA,
                // after a proxy fence); the weight boxes are already on their way.  The last CTA
                // to read the value clears the word for the next linear over these segments.
                const unsigned long long t0w = globaltimer();
                bool seen = true;
                while (ld_acquire_gpu(a.xword) != a.xready) {
                    if (globaltimer() - t0w > kWaitLimitNs) {
                        seen = false;
                        break;
                    }
                    __nanosleep(32);
                }
                if (seen) {
                    if (atomicAdd(a.xword + 1, 1) == (int)(gridDim.x * gridDim.y) - 1) {
                        atomicExch(a.xword, 0);
                        atomicExch(a.xword + 1, 0);
                    }
                } else {  // y is not written; x is still loaded, so that every copy completes
                    flags[0] = 1;
                    report_timeout_status(a.seg.status);
                }
                fence_proxy_async_global();
                mbar_arrive(xbar);  // the epilogue warps may read the segments
                for (int i = 0; i < pre; ++i) issue_x(i);
            }
            int issued = pre;  // stages 0 .. pre-1 went out before the CTA-wide barrier
            for (int i = pre; i < nkb; ++i) {
                const int s = i % stages;
                if (i >= stages && !mbar_wait(&empty[s], ((i / stages) & 1) ^ 1, flags)) break;
                issue_stage(i);
                ++issued;
            }
            if (flags[0]) {  // aborted: let copies already in flight land before the CTA exits
                report_timeout_status(a.seg.status);
                for (int i = max(0, issued - stages); i < issued; ++i) {
                    const unsigned long long tw = globaltimer();
                    while (!mbar_try_wait(&full[i % stages], (i / stages) & 1) && globaltimer() - tw < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // With only n_pad tokens on N an MMA is short, and a chain of MMAs into one
            // accumulator waits on each other; K-blocks therefore rotate over nacc accumulators.
            const uint32_t idesc = idesc_f16(BM, a.n_pad, a.bf16 != 0);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % stages;
                if (!mbar_wait(&full[s], (i / stages) & 1, flags)) {
                    report_timeout_status(a.seg.status);
                    break;
                }
                tc_fence_after();
                const uint32_t wa = smem_u32(smem + s * stage_bytes);
                const uint32_t xa = wa + w_bytes;
                const uint32_t acc = tmem + static_cast<uint32_t>((i % a.nacc) * a.n_pad);
                for (int c = 0; c < kc; ++c) {
                    const uint32_t wc = wa + c * BM * BK * 2, xc = xa + c * a.n_pad * BK * 2;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        umma_f16(acc, sdesc_sw128(wc + k * UMMA_K * 2), sdesc_sw128(xc + k * UMMA_K * 2), idesc,
                                 (i >= a.nacc || c > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(tmem_full);  // also on abort: fires once the issued MMAs have finished
        }
    } else {
        // ---- phase A (overlaps the main loop): stage this CTA's LoRA operands ----
        // s, idx and the status word come from earlier kernels.  With the x-ready hand-off every kernel before the shrink is complete once the producer
        // has seen its signal: the segments are read then, and only s waits for this grid's
        // dependency wait (below, after the B tiles are on their way).
        if (a.xready) {
            if (et == 0) mbar_wait(xbar, 0, flags);
        } else {
            pdl_wait();
        }
        if (et == 0) flags[3] = flags[0] ? LORA_ETIMEOUT : __ldcg(a.seg.status);
        named_bar_sync(1, 128);
        const bool lora = flags[3] == LORA_OK && a.fuse;
        // With the x-ready hand-off, this grid completes only after the shrink before it (as
        // every later kernel's dependency wait assumes): the LoRA path waits below, this one here.
        if (!lora && a.xready) pdl_wait();
        if (lora) {
            for (int q = et; q < cnt; q += 128) slot_sm[q] = __ldcg(a.seg.idx + t0 + q);
            named_bar_sync(1, 128);
            // distinct slots of this CTA's tokens: dloc_sm[q] = index of token q's slot in dlist
            for (int q = et; q < cnt; q += 128) {
                int first = -1;
                if (slot_sm[q] >= 0) {
                    first = q;
                    for (int q2 = 0; q2 < q; ++q2)
                        if (slot_sm[q2] == slot_sm[q]) {
                            first = q2;
                            break;
                        }
                }
                fidx_sm[q] = first;
            }
            int* wsum = const_cast<int*>(flags) + 4;
            int running = 0;
            for (int c0 = 0; c0 < cnt; c0 += 128) {  // block-wide exclusive scan of "first occurrence"
                const int q = c0 + et;
                named_bar_sync(1, 128);
                const bool is_first = q < cnt && fidx_sm[q] == q;
                const unsigned bal = __ballot_sync(0xffffffffu, is_first);
                if (lane == 0) wsum[et >> 5] = __popc(bal);
                named_bar_sync(1, 128);
                int base = running;
                for (int w = 0; w < (et >> 5); ++w) base += wsum[w];
                if (is_first) {
                    const int d = base + __popc(bal & ((1u << lane) - 1u));
                    dloc_sm[q] = d;
                    dlist[d] = slot_sm[q];
                }
                running += wsum[0] + wsum[1] + wsum[2] + wsum[3];
            }
            named_bar_sync(1, 128);
            for (int q = et; q < cnt; q += 128) {
                const int f = fidx_sm[q];
                if (f != q) dloc_sm[q] = f >= 0 ? dloc_sm[f] : -1;
            }
            // compact staging: the slots' true ranks in whole 8-column chunks (this pool's table
            // decides); otherwise every tile at r_max, without the dependent table read
            if (a.compact) {
                if (et < min(running, kMaxPre))
                    pre_sm[1 + kMaxPre + et] = (min(max(__ldg(&a.pool.table[dlist[et]].rank), 1), R) + 7) / 8;
                named_bar_sync(1, 128);
            }
            if (et == 0) {
                flags[2] = running;
                const uint32_t s_bytes = static_cast<uint32_t>(cnt * R * 4);
                if (a.compact) {
                    // the first distinct slots whose true-rank tiles fit in the room planned
                    int off = 0, ns = 0;
                    for (int d = 0; d < min(running, kMaxPre); ++d) {
                        const int c = pre_sm[1 + kMaxPre + d];
                        if ((off + BM * c) * 16 > a.bpre_bytes) break;
                        pre_sm[1 + d] = off;
                        off += BM * c;
                        ++ns;
                    }
                    pre_sm[0] = ns;
                    // bulk copies of the owned tokens' shrink parts (unless they come after this
                    // grid's dependency wait), then one TMA box per staged slot and 8-column
                    // chunk: [128 feature rows][8 columns] of B
                    const uint32_t sb = (cnt > 0 && !a.xready) ? a.s_parts * s_bytes : 0;
                    if (a.xready)
                        mbar_expect_tx(lbar, static_cast<uint32_t>(off) * 16);  // s: arrival below
                    else
                        mbar_arrive_expect_tx(lbar, sb + static_cast<uint32_t>(off) * 16);
                    if (sb)
                        for (int k = 0; k < a.s_parts; ++k)
                            bulk_g2s(S_sm + (size_t)k * per * R, a.s_in + ((size_t)k * n + t0) * R, s_bytes, lbar);
                    uint4* Bp4 = reinterpret_cast<uint4*>(Bpre);
                    for (int d = 0; d < ns; ++d)
                        for (int cc = 0; cc < pre_sm[1 + kMaxPre + d]; ++cc)
                            tma_load_3d_cta(Bp4 + pre_sm[1 + d] + cc * BM, &tmB, lbar, 0, cc,
                                            dlist[d] * h_out + m_tile * BM);
                } else {
                    // every tile at r_max ([128 rows][r_max], one contiguous bulk copy each)
                    const uint32_t b_bytes = static_cast<uint32_t>(rows_valid * R * 2);
                    const int ns = min(min(running, kMaxPre), a.bpre_bytes / (BM * R * 2));
                    pre_sm[0] = ns;
                    const uint32_t sb = (cnt > 0 && !a.xready) ? a.s_parts * s_bytes : 0;
                    if (a.xready)
                        mbar_expect_tx(lbar, ns * b_bytes);  // s: arrival below
                    else
                        mbar_arrive_expect_tx(lbar, sb + ns * b_bytes);
                    if (sb)
                        for (int k = 0; k < a.s_parts; ++k)
                            bulk_g2s(S_sm + (size_t)k * per * R, a.s_in + ((size_t)k * n + t0) * R, s_bytes, lbar);
                    for (int d = 0; d < ns; ++d)
                        bulk_g2s(Bpre + (size_t)d * BM * R, B + ((size_t)dlist[d] * h_out + m_tile * BM) * R, b_bytes,
                                 lbar);
                }
            }
            named_bar_sync(1, 128);
            if (a.xready) {  // the shrink output: after this grid's dependency wait
                pdl_wait();
                if (et == 0) {
                    const uint32_t s_bytes = static_cast<uint32_t>(cnt * R * 4);
                    mbar_arrive_expect_tx(lbar, cnt > 0 ? a.s_parts * s_bytes : 0);
                    if (cnt > 0)
                        for (int k = 0; k < a.s_parts; ++k)
                            bulk_g2s(S_sm + (size_t)k * per * R, a.s_in + ((size_t)k * n + t0) * R, s_bytes, lbar);
                }
            }
            const int Dg = pre_sm[0];
            const bool staged = mbar_wait(lbar, 0, flags);
            // sum the shrink's K-parts once (part 0 receives the total)
            for (int e = et; e < cnt * R; e += 128) {
                float v = S_sm[e];
                for (int k = 1; k < a.s_parts; ++k) v += S_sm[(size_t)k * per * R + e];
                S_sm[e] = v;
            }
            named_bar_sync(1, 128);
            // LoRA term of this thread's feature for every owned token whose slot is pre-staged
            if (use_lsm) {
                for (int q0 = 0; q0 < cnt; q0 += 8) {
                    float acc[8];
                    if (a.compact)
                        lora_batch8_pre<T>(reinterpret_cast<const uint4*>(Bpre), pre_sm, S_sm, dloc_sm, q0, cnt,
                                           staged ? Dg : 0, row, R, lane, acc);
                    else
                        lora_batch8<T>(Bpre, S_sm, dloc_sm, q0, cnt, 0, staged ? Dg : 0, row, R, lane, acc);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (q0 + u < cnt) L_sm[(q0 + u) * BM + row] = acc[u];
                }
            }
        } else if (use_lsm) {
            for (int q = 0; q < cnt; ++q) L_sm[q * BM + row] = 0.f;
        }
        // ---- phase B: park the partial tile in the idle stages ----
        const bool got = mbar_wait(tmem_full, 0, flags);
        tc_fence_after();
        if (et == 0 && got && a.prefetch && a.prefetch_bytes) {
            // This CTA's share of W has been consumed and HBM would idle through the epilogue:
            // stream this CTA's slice of the caller's prefetch range (typically the next
            // linear's weight) into L2 meanwhile.
            const size_t ncta = (size_t)gridDim.x * gridDim.y;
            const size_t cta = (size_t)blockIdx.y * gridDim.x + blockIdx.x;
            const size_t slice = ((a.prefetch_bytes + ncta - 1) / ncta + 15) & ~size_t(15);
            const size_t beg = cta * slice;
            const size_t cap = a.prefetch_bytes & ~size_t(15);
            const size_t end = cap < beg + slice ? cap : beg + slice;
            for (size_t off = beg; off < end; off += 65536)
                prefetch_l2_bulk(a.prefetch + off, static_cast<uint32_t>(end - off < 65536 ? end - off : 65536));
        }
        if (et == 0) {
            flags[1] = (got && !flags[0] && flags[3] == LORA_OK) ? 1 : 0;
            // receive buffer: one bulk copy of this CTA's token rows from every other CTA
            if (push && flags[1] && cnt > 0) mbar_arrive_expect_tx(rbar, (uint32_t)((a.splits - 1) * cnt * BM * 4));
        }
        named_bar_sync(1, 128);
        if (flags[1]) {
            const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
            const int used = min(a.nacc, nkb);  // accumulators that received K-blocks
            const int cols = min(a.n_pad, (n + 15) & ~15);
            // 64 columns per round: all TMEM loads of the round, one wait, then the stores
            // (one warp per scheduler runs this, so serial load-wait-store rounds are slow)
            for (int c0 = 0; c0 < cols; c0 += 64) {
                float v[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) v[c] = 0.f;
                for (int j = 0; j < used; ++j) {
                    uint32_t r[64];
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (c0 + 16 * q < cols)
                            tmem_ld16(taddr + static_cast<uint32_t>(j * a.n_pad + c0 + 16 * q),
                                      *reinterpret_cast<uint32_t(*)[16]>(&r[16 * q]));
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 64; ++c) v[c] += __uint_as_float(r[c]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (c0 + 16 * q < cols)
#pragma unroll
                        for (int c = 0; c < 16; ++c) P[(c0 + 16 * q + c) * BM + row] = v[16 * q + c];
            }
            fence_proxy_async_smem();  // the parked rows are read by bulk copies
        }
    }

    tc_fence_before();
    cluster_sync();  // every CTA of the cluster is past its main loop and has parked its partials

    // ---- phase C: send the partial rows of tokens owned by other CTAs ----
    if (push && threadIdx.x >= 64 && threadIdx.x < 64 + a.splits && flags[1]) {
        // one thread per peer, so the copies are issued side by side
        const int dst = threadIdx.x - 64;
        const int dt0 = dst * per;
        const int dcnt = max(0, min(n, dt0 + per) - dt0);
        if (dst != rank && dcnt > 0) {
            const int slot_idx = rank < dst ? rank : rank - 1;  // sender index in dst's buffer
            const uint32_t dst_addr =
                mapa_shared(smem_u32(Rcv + (size_t)slot_idx * per * BM), static_cast<uint32_t>(dst));
            const uint32_t dst_bar = mapa_shared(smem_u32(rbar), static_cast<uint32_t>(dst));
            bulk_s2cluster(dst_addr, P + (size_t)dt0 * BM, static_cast<uint32_t>(dcnt * BM * 4), dst_bar);
        }
    }

    // ---- phase D: late LoRA groups, reduction over the cluster, store ----
    // The closing cluster barrier keeps every CTA alive until the copies out of its parked rows
    // have landed.  With pushed partials, a CTA's incoming copies are complete once its receive
    // barrier fires, so its epilogue threads announce their arrival right then and only wait
    // at the very end: the barrier's latency overlaps the reduction and the y store.
    bool arrived = false;
    if (warp >= 2 && flags[1]) {
        float* own = P + (size_t)t0 * BM;  // this CTA's partials of its own tokens (LoRA added here)
        const int D = flags[2];
        const int Dpre = D > 0 ? pre_sm[0] : 0;     // slots staged during the main loop
        const int g_begin = use_lsm ? Dpre : 0;  // with L_sm the pre-staged group is already applied
        if (a.fuse && D > g_begin) {
            T* Blate = smem_align(reinterpret_cast<T*>(Rcv + (push ? (size_t)(a.splits - 1) * per * BM : 0)), 128) +
                       (size_t)2 * kYChunk * BM;  // after the two y buffers
            const size_t late_bytes = (size_t)stages * stage_bytes - (reinterpret_cast<uint8_t*>(Blate) - smem);
            const int dlate = max(1, static_cast<int>(late_bytes / ((size_t)BM * R * sizeof(T))));
            for (int g0 = g_begin; g0 < D;) {
                const bool pre = g0 == 0 && Dpre > 0;
                const int Dg = pre ? min(D, Dpre) : min(D - g0, dlate);
                const T* Bg = Blate;
                if (!pre) {
                    named_bar_sync(1, 128);
                    const int total = Dg * BM * chunks;
                    for (int e0 = et; e0 < total; e0 += 8 * 128) {
                        uint4 v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int e = e0 + u * 128;
                            v[u] = make_uint4(0, 0, 0, 0);
                            if (e < total) {
                                const int d = e / (BM * chunks);
                                const int rem = e - d * (BM * chunks);
                                const int oo = m_tile * BM + rem / chunks;
                                if (oo < h_out)
                                    v[u] = __ldg(reinterpret_cast<const uint4*>(
                                        B + ((size_t)dlist[g0 + d] * h_out + oo) * R + (rem % chunks) * 8));
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (e0 + u * 128 < total) reinterpret_cast<uint4*>(Blate)[e0 + u * 128] = v[u];
                    }
                    named_bar_sync(1, 128);
                }
                for (int q0 = 0; q0 < cnt; q0 += 8) {
                    float acc[8];
                    if (pre && a.compact)
                        lora_batch8_pre<T>(reinterpret_cast<const uint4*>(Bpre), pre_sm, S_sm, dloc_sm, q0, cnt, Dg,
                                           row, R, lane, acc);
                    else
                        lora_batch8<T>(pre ? Bpre : Bg, S_sm, dloc_sm, q0, cnt, g0, Dg, row, R, lane, acc);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (q0 + u < cnt) own[(q0 + u) * BM + row] += acc[u];
                }
                g0 += Dg;
            }
        }
        bool recv = true;
        if (push && cnt > 0 && a.splits > 1) recv = __all_sync(0xffffffffu, mbar_wait(rbar, 0, flags));
        if (push) {
            cluster_arrive();
            arrived = true;
        }
        // y is assembled in shared memory 32 tokens at a time (two buffers of [32][128], after
        // the receive buffer) and written with TMA stores; rows/columns outside y are clipped
        T* Ysm = smem_align(reinterpret_cast<T*>(Rcv + (push ? (size_t)(a.splits - 1) * per * BM : 0)), 128);
        // store boxes never cross into the next CTA's tokens: ychunk = min(32, per) rows, and the
        // last (per % ychunk)-row piece of a share goes through the tail map
        const int ychunk = min(kYChunk, per);
        for (int c0 = 0; c0 < cnt; c0 += ychunk) {
            T* Yb = Ysm + (size_t)((c0 / ychunk) & 1) * kYChunk * BM;
            named_bar_sync(1, 128);  // this buffer's previous TMA store has finished reading it
            if (recv) {
                for (int q0 = c0; q0 < min(cnt, c0 + ychunk); q0 += kYBatch) {  // kYBatch tokens, all loads first
                    float v[kYBatch];
#pragma unroll
                    for (int u = 0; u < kYBatch; ++u) {
                        const int q = min(q0 + u, cnt - 1);
                        v[u] = own[q * BM + row];
                        if (use_lsm) v[u] += L_sm[q * BM + row];
                    }
                    if (push && a.splits == 4) {
                        // the usual 4-way split: all three peers' partials loaded before any add
                        float r0[kYBatch], r1[kYBatch], r2[kYBatch];
#pragma unroll
                        for (int u = 0; u < kYBatch; ++u) {
                            const size_t q = (size_t)min(q0 + u, cnt - 1);
                            r0[u] = Rcv[q * BM + row];
                            r1[u] = Rcv[((size_t)per + q) * BM + row];
                            r2[u] = Rcv[((size_t)2 * per + q) * BM + row];
                        }
#pragma unroll
                        for (int u = 0; u < kYBatch; ++u) v[u] += (r0[u] + r1[u]) + r2[u];
                    } else if (push) {
#pragma unroll
                        for (int c = 0; c < 7; ++c) {
                            if (c < a.splits - 1) {
                                float r8[kYBatch];
#pragma unroll
                                for (int u = 0; u < kYBatch; ++u)
                                    r8[u] = Rcv[((size_t)c * per + min(q0 + u, cnt - 1)) * BM + row];
#pragma unroll
                                for (int u = 0; u < kYBatch; ++u) v[u] += r8[u];
                            }
                        }
                    } else {
                        for (int c = 0; c < a.splits; ++c) {
                            if (c == rank) continue;
                            float r8[kYBatch];
#pragma unroll
                            for (int u = 0; u < kYBatch; ++u)
                                r8[u] = ld_dsmem_f32(mapa_shared(smem_u32(own + min(q0 + u, cnt - 1) * BM + row),
                                                                 static_cast<uint32_t>(c)));
#pragma unroll
                            for (int u = 0; u < kYBatch; ++u) v[u] += r8[u];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kYBatch; ++u)
                        if (q0 + u < min(cnt, c0 + ychunk)) Yb[(q0 + u - c0) * BM + row] = from_f32<T>(v[u]);
                }
                fence_proxy_async_smem();
            }
            named_bar_sync(1, 128);
            if (et == 0 && recv) {
                tma_store_2d(c0 + ychunk <= per ? &tmY : &tmYtail, Yb, m_tile * BM, t0 + c0);
                bulk_commit_group();
                bulk_wait_group_read1();  // the other buffer is free again
            }
        }
        if (et == 0) bulk_wait_group_read0();
    }
    tc_fence_before();
    if (!arrived) cluster_arrive();
    cluster_wait();  // no CTA leaves while its parked rows may still be copied or read
    if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
    stamp_end(a.stamp);
}

// ============================================================================================
// prefill: persistent 128 x 256 tiles, double-buffered accumulators
// ============================================================================================
// The LoRA expand of a tile runs on the tensor core as one more K block of its accumulator:
// with the tile's distinct adapters d = 0..D-1 (D * r_max <= 64), the block's operands are
//   A'[token, d * r_max + j] = s[token, j] if the token's adapter is d, else 0   (128 x 64)
//   B'[col,   d * r_max + j] = B_d[col, j]                                      (256 x 64)
// so that A' B'^T adds sum_j s[t, j] B_slot(t)[col, j] to every (token, column) of the tile
// (s rounded to the 16-bit type, float32 accumulation).  The epilogue warps write both operands
// into the pipeline stage that the block occupies, in the layout a 128-byte-swizzled TMA copy
// would leave (16-byte chunk c of row r at chunk position c ^ (r % 8)), and complete the
// stage's full barrier themselves; the producer skips that position.  Tiles with more
// adapters, or whose columns span two slices of a group, keep the epilogue's SIMT expand.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
gemm_prefill_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmY, const PrefillArgs a) {
    constexpr int BN = kPrefillBN;
    stamp_start(a.stamp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align(smem_raw, 1024);
    const int stages = a.stages;
    constexpr uint32_t x_bytes = BM * BK * 2;
    constexpr uint32_t w_bytes = BN * BK * 2;
    constexpr uint32_t stage_bytes = x_bytes + w_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
    uint64_t* empty = full + stages;
    uint64_t* acc_full = empty + stages;  // [2]
    uint64_t* acc_empty = acc_full + 2;   // [2]
    uint64_t* lora_free = acc_empty + 2;  // the LoRA block's stage is free (one phase per tile)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(lora_free + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [20]
    // y staging of the epilogue: [4 warps][2 buffers][32 rows][32 columns] 16-bit, after the barriers
    T* ystage = reinterpret_cast<T*>(smem + stages * stage_bytes + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = a.m_tiles * a.n_tiles;
    const int nkb = a.kb_total;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
        }
        mbar_init(lora_free, 1);
        flags[0] = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 2 * BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    // pipeline positions of a tile: its nkb K blocks, then (lora_mma) the LoRA block
    const int per_tile = nkb + (a.lora_mma ? 1 : 0);

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            bool waited = false;
            int deferred = 0;
            int def_kb[16], def_m[16], def_s[16];
            // first ring pass: weights first, x after the previous grid finished
            auto flush = [&]() {
                pdl_wait();
                waited = true;
                for (int d = 0; d < deferred; ++d)
                    tma_load_2d(smem + def_s[d] * stage_bytes, &tmX, &full[def_s[d]], def_kb[d] * BK, def_m[d]);
            };
            for (int tile = blockIdx.x; tile < total && !flags[0]; tile += gridDim.x) {
                int m0, n0;
                prefill_tile(tile, a.m_tiles, a.n_tiles, m0, n0);
                for (int kb = 0; kb < per_tile; ++kb, ++it) {
                    const int s = it % stages;
                    const uint32_t ph = (it / stages) & 1;
                    if (it >= stages) {
                        if (!waited) flush();
                        if (!mbar_wait(&empty[s], ph ^ 1, flags)) break;
                    }
                    if (kb == nkb) {  // the LoRA block: its stage goes to the epilogue warps
                        mbar_arrive(lora_free);
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[s], stage_bytes);
                    tma_load_2d(smem + s * stage_bytes + x_bytes, &tmW, &full[s], kb * BK, n0);
                    if (waited) {
                        tma_load_2d(smem + s * stage_bytes, &tmX, &full[s], kb * BK, m0);
                    } else {
                        def_kb[deferred] = kb;
                        def_m[deferred] = m0;
                        def_s[deferred] = s;
                        ++deferred;
                    }
                }
            }
            if (!waited) flush();
            if (flags[0]) {
                report_timeout_status(a.seg.status);
                for (int i = max(0, it - stages); i < it; ++i) {
                    if (i % per_tile == nkb) continue;  // not a copy of this thread
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&full[i % stages], (i / stages) & 1) && globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BM, BN, a.bf16 != 0);
            int it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++local) {
                const int buf = local & 1;
                const uint32_t acc = tmem + buf * BN;
                if (!mbar_wait(&acc_empty[buf], ((local >> 1) & 1) ^ 1, flags)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < per_tile; ++kb, ++it) {
                    const int s = it % stages;
                    if (!mbar_wait(&full[s], (it / stages) & 1, flags)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t xa = smem_u32(smem + s * stage_bytes);
                    const uint32_t wa = xa + x_bytes;
                    if (kb < nkb) {
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k)
                            umma_f16(acc, sdesc_sw128(xa + k * UMMA_K * 2), sdesc_sw128(wa + k * UMMA_K * 2), idesc,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                    } else {  // the LoRA block: K of its operands set by the epilogue warps (0: none)
                        const int lk = flags[1];
                        for (int k = 0; k < lk / UMMA_K; ++k)
                            umma_f16(acc, sdesc_sw128(xa + k * UMMA_K * 2), sdesc_sw128(wa + k * UMMA_K * 2), idesc, 1u);
                    }
                    umma_commit(&empty[s]);
                }
                umma_commit(&acc_full[buf]);
            }
            if (!ok) report_timeout_status(a.seg.status);
        }
    } else {
        // ---- epilogue: thread <-> token row (TMEM lane), 256 features per tile ----
        const int q = warp & 3;
        const int ldy = a.grp.ldy, R = a.pool.R, n = a.n;
        T* y = static_cast<T*>(a.y);
        bool waited = false;
        int status = LORA_OK;
        int local = 0;
        int ybuf = 0;  // this warp's staging buffer for the next 32 columns
        const int et = threadIdx.x - 64;  // 0..127
        volatile int* red = flags + 2;   // [4]: per-warp minima
        volatile int* dsl = flags + 8;   // [8]: the tile's distinct adapters
        volatile int* redx = flags + 16;  // [4]: per-warp maxima
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
            const int buf = local & 1;
            if (!waited) {
                pdl_wait();  // s, idx and the status word come from earlier kernels
                status = __ldcg(a.seg.status);
                waited = true;
            }
            int m0, n0;
            prefill_tile(tile, a.m_tiles, a.n_tiles, m0, n0);
            bool lora_done = false;  // the tile's LoRA term went through the tensor core
            if (a.lora_mma) {
                // ---- operands of the tile's LoRA block (token row et; columns et, et + 128) ----
                const int tr = m0 + et;
                const int slot_r = (status == LORA_OK && tr < n) ? __ldcg(a.seg.idx + tr) : -1;
                const int qa = group_slice_of_col(a.grp, n0);
                const int qb = group_slice_of_col(a.grp, min(n0 + BN, ldy) - 1);
                const int dmax = 64 / R;
                // distinct adapters of the tile in increasing order (uniform over the 128 threads);
                // the first round also takes the maximum, so that a tile of one adapter (the
                // common prefill case) needs no second round
                int mine = -1, D = 0;
                for (int d = 0; d <= dmax; ++d) {
                    const int cand = __reduce_min_sync(0xffffffffu, (slot_r >= 0 && mine < 0) ? slot_r : INT_MAX);
                    const int candx = d == 0 ? __reduce_max_sync(0xffffffffu, slot_r) : -1;
                    named_bar_sync(1, 128);  // the previous round has read red
                    if (lane == 0) {
                        red[q] = cand;
                        redx[q] = candx;
                    }
                    named_bar_sync(1, 128);
                    const int m = min(min(red[0], red[1]), min(red[2], red[3]));
                    if (m == INT_MAX) break;
                    D = d + 1;
                    if (d == dmax) break;  // more adapters than the block holds
                    if (slot_r == m) mine = d;
                    if (et == 0) dsl[d] = m;
                    if (d == 0 && m == max(max(redx[0], redx[1]), max(redx[2], redx[3]))) break;  // one adapter
                }
                const int lk = (D == 0 || D > dmax || qa != qb) ? 0 : (D * R + 15) / 16 * 16;
                lora_done = lk > 0;
                named_bar_sync(1, 128);  // dsl visible
                uint4 av[8], bw[2][8];
                if (lk > 0) {  // all loads first
                    const SliceRef sl = group_slice(a.grp, qa);
                    const float* srow = a.s_in + sl.s_off + (size_t)tr * R;
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        const int d = c8 * 8 / R, j = c8 * 8 - d * R;
                        av[c8] = make_uint4(0, 0, 0, 0);
                        if (c8 * 8 < lk && d == mine)
                            av[c8] = pack8<T>(__ldcg(reinterpret_cast<const float4*>(srow + j)),
                                              __ldcg(reinterpret_cast<const float4*>(srow + j + 4)));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int col = n0 + et + h * 128;
                            bw[h][c8] = make_uint4(0, 0, 0, 0);
                            if (c8 * 8 < lk && d < D && col < ldy)
                                bw[h][c8] = __ldg(reinterpret_cast<const uint4*>(
                                    static_cast<const T*>(sl.B) + ((size_t)dsl[d] * sl.h_out + (col - sl.col)) * R + j));
                        }
                    }
                }
                // the block's stage, once the producer has seen its previous use consumed (the
                // producer walks the positions in order; one lora_free phase per tile)
                const int s = (local * per_tile + nkb) % stages;
                if (et == 0) mbar_wait(lora_free, local & 1, flags);
                named_bar_sync(1, 128);
                if (flags[0]) break;
                if (lk > 0) {
                    uint8_t* As = smem + s * stage_bytes;  // [128 token rows][128 B]
                    uint8_t* Bs = As + x_bytes;            // [256 column rows][128 B]
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        if (c8 * 8 < lk) {
                            *reinterpret_cast<uint4*>(As + et * 128 + ((c8 ^ (et & 7)) << 4)) = av[c8];
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int o = et + h * 128;
                                *reinterpret_cast<uint4*>(Bs + o * 128 + ((c8 ^ (o & 7)) << 4)) = bw[h][c8];
                            }
                        }
                    }
                    fence_proxy_async_smem();  // read by the tensor core
                }
                named_bar_sync(1, 128);
                if (et == 0) {
                    flags[1] = lk;
                    mbar_arrive(&full[s]);
                }
            }
            const bool got = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (local >> 1) & 1, flags));
            if (!got) break;
            tc_fence_after();
            const int t = m0 + q * 32 + lane;
            const uint32_t taddr = tmem + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
            const int slot = (a.fuse && !lora_done && t < n) ? __ldcg(a.seg.idx + t) : -1;
            // 32 columns per round: both TMEM loads, one wait, the two 16-column pieces into
            // this warp's staging buffer (its 32 token rows), then one TMA store of the buffer
            // (rows and columns outside y are clipped; nothing is stored with an error status)
            for (int c0 = 0; c0 < BN; c0 += 32, ybuf ^= 1) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld16(taddr + c0, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
                tmem_ld16(taddr + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16]));
                tmem_ld_wait();
                T* Ys = ystage + (size_t)(q * 2 + ybuf) * 32 * 32;
                if (lane == 0) bulk_wait_group_read1();  // this buffer's previous store has read it
                __syncwarp();
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int col = n0 + c0 + 16 * hf;  // column of y
                    float v[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) v[c] = __uint_as_float(r[16 * hf + c]);
                    if (slot >= 0 && col < ldy) {
                        // the slice owning these 16 columns (slice boundaries are multiples of 16)
                        const SliceRef sl = group_slice(a.grp, group_slice_of_col(a.grp, col));
                        const float* srow = a.s_in + sl.s_off + (size_t)t * R;
                        const T* Bt = static_cast<const T*>(sl.B) + ((size_t)slot * sl.h_out + (col - sl.col)) * R;
                        const int cmax = min(16, sl.col + sl.h_out - col);
                        for (int j0 = 0; j0 < R; j0 += 8) {
                            const float4 sa = __ldg(reinterpret_cast<const float4*>(srow + j0));
                            const float4 sb = __ldg(reinterpret_cast<const float4*>(srow + j0 + 4));
                            uint4 bv[16];
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                bv[c] = c < cmax ? __ldg(reinterpret_cast<const uint4*>(Bt + (size_t)c * R + j0))
                                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                float b[8];
                                unpack8<T>(bv[c], b);
                                float acc = v[c];
                                acc = fmaf(b[0], sa.x, acc);
                                acc = fmaf(b[1], sa.y, acc);
                                acc = fmaf(b[2], sa.z, acc);
                                acc = fmaf(b[3], sa.w, acc);
                                acc = fmaf(b[4], sb.x, acc);
                                acc = fmaf(b[5], sb.y, acc);
                                acc = fmaf(b[6], sb.z, acc);
                                acc = fmaf(b[7], sb.w, acc);
                                v[c] = acc;
                            }
                        }
                    }
                    uint4* yr = reinterpret_cast<uint4*>(Ys + (size_t)lane * 32 + 16 * hf);
                    yr[0] = make_uint4(pack2<T>(v[0], v[1]), pack2<T>(v[2], v[3]), pack2<T>(v[4], v[5]),
                                       pack2<T>(v[6], v[7]));
                    yr[1] = make_uint4(pack2<T>(v[8], v[9]), pack2<T>(v[10], v[11]), pack2<T>(v[12], v[13]),
                                       pack2<T>(v[14], v[15]));
                }
                fence_proxy_async_smem();  // read by the TMA store
                __syncwarp();
                if (lane == 0 && status == LORA_OK && n0 + c0 < ldy && m0 + q * 32 < n) {
                    tma_store_2d(&tmY, Ys, n0 + c0, m0 + q * 32);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
        if (lane == 0) bulk_wait_group_read0();  // the staging buffers stay until their stores have read them
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * BN);
    stamp_end(a.stamp);
}

// ============================================================================================
// tall-tile base GEMM (no LoRA term) for grouped batches of 128-256 tokens
// ============================================================================================
// At 128-256 tokens the x tile of a stage is as large as the W tile or larger, and every row
// tile re-reads all of x.  Here a CTA owns 256 W rows: each K stage brings a [256 rows][64] W
// box and one x box, and two M=128 MMAs (rows 0-127 and 128-255, accumulators in TMEM columns
// [0, n_pad) and [n_pad, 2 n_pad)) read the same x tile, so x is re-read half as often.  Full
// K per CTA, no split, no LoRA epilogue (the segmented expand follows); y stored directly.
struct TallArgs {
    SegView seg;
    void* y;
    int n, n_pad, ldy, h_out, nkb, stages, bf16;
    int tstep;  // tokens per CTA (grid.y splits the batch when the row tiles fill few SMs)
    unsigned long long* stamp;  // benchmark instrumentation (nullptr: off)
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tall_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const TallArgs a) {
    stamp_start(a.stamp);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align(smem_raw, 1024);
    const int stages = a.stages;
    const uint32_t w_bytes = 2 * BM * BK * 2;  // 256 rows
    const uint32_t stage_bytes = w_bytes + static_cast<uint32_t>(a.n_pad) * BK * 2;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * stage_bytes);
    uint64_t* empty = full + stages;
    uint64_t* acc_full = empty + stages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // abort
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 2 * BM;  // first W row of this CTA
    const int ts = blockIdx.y * a.tstep;  // first token of this CTA
    int cols = 32;
    while (cols < 2 * a.n_pad) cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        flags[0] = 0;
        fence_barrier_init();
        prefetch_tmap(&tmW);
        prefetch_tmap(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_trigger();

    if (warp == 0) {
        // W and x are complete when this grid starts: the shrink before it releases its
        // dependents only after its own grid-dependency wait
        if (lane == 0) {
            int it = 0;
            for (; it < a.nkb && !flags[0]; ++it) {
                const int s = it % stages;
                if (it >= stages && !mbar_wait(&empty[s], ((it / stages) & 1) ^ 1, flags)) break;
                mbar_arrive_expect_tx(&full[s], stage_bytes);
                tma_load_2d_cta(smem + (size_t)s * stage_bytes, &tmW, &full[s], it * BK, m0);
                tma_load_2d_cta(smem + (size_t)s * stage_bytes + w_bytes, &tmX, &full[s], it * BK, ts);
            }
            if (flags[0]) {  // aborted: let copies already in flight land before the CTA exits
                report_timeout_status(a.seg.status);
                for (int i = max(0, it - stages); i < it; ++i) {
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(&full[i % stages], (i / stages) & 1) && globaltimer() - t0 < kWaitLimitNs) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(BM, a.n_pad, a.bf16 != 0);
            for (int i = 0; i < a.nkb; ++i) {
                const int s = i % stages;
                if (!mbar_wait(&full[s], (i / stages) & 1, flags)) {
                    report_timeout_status(a.seg.status);
                    break;
                }
                tc_fence_after();
                const uint32_t wa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint32_t xa = wa + w_bytes;
#pragma unroll
                for (int k = 0; k < BK / UMMA_K; ++k) {
                    const uint64_t xd = sdesc_sw128(xa + k * UMMA_K * 2);
                    const uint32_t acc_flag = (i > 0 || k > 0) ? 1u : 0u;
                    umma_f16(tmem, sdesc_sw128(wa + k * UMMA_K * 2), xd, idesc, acc_flag);
                    umma_f16(tmem + static_cast<uint32_t>(a.n_pad), sdesc_sw128(wa + BM * 128 + k * UMMA_K * 2), xd,
                             idesc, acc_flag);
                }
                umma_commit(&empty[s]);
            }
            umma_commit(acc_full);  // also on abort: fires once the issued MMAs have finished
        }
    } else {
        // ---- epilogue: thread <-> W row r of each 128-row half (TMEM lane) ----
        const int row = (warp & 3) * 32 + lane;
        T* y = static_cast<T*>(a.y);
        pdl_wait();  // the status word comes from an earlier kernel
        const bool st_ok = __ldcg(a.seg.status) == LORA_OK;
        const bool got = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, flags));
        if (got && st_ok) {
            tc_fence_after();
            for (int h = 0; h < 2; ++h) {
                const uint32_t taddr =
                    tmem + static_cast<uint32_t>(h * a.n_pad) + (static_cast<uint32_t>((warp & 3) * 32) << 16);
                const int o = m0 + h * BM + row;
                for (int t0 = 0; t0 < a.n_pad; t0 += 16) {
                    uint32_t r[16];
                    __syncwarp();
                    tmem_ld16(taddr + t0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (o < a.h_out && t0 + q < a.tstep && ts + t0 + q < a.n)
                            y[(size_t)(ts + t0 + q) * a.ldy + o] = from_f32<T>(__uint_as_float(r[q]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, cols);
    stamp_end(a.stamp);
}

// ============================================================================================
// host side
// ============================================================================================

struct DecodePlan {
    int n_pad, m_tiles, kb_total, splits, kb_per_split, stages, tmem_cols, dpre, push, s_parts, nacc, kc, compact;
    size_t bpre;  // room for staged B tiles: at least dpre slots in the worst case
    size_t smem;
};

// Shared-memory plan of gemm_decode_kernel (its layout comments are the reference).
static DecodePlan plan_decode(const PoolView& pv, int n, int s_parts) {
    DecodePlan p;
    p.s_parts = s_parts;
    p.n_pad = std::max(16, (n + 15) / 16 * 16);
    p.m_tiles = (pv.h_out + BM - 1) / BM;
    p.kb_total = (pv.h_in + BK - 1) / BK;
    const int sms = num_sms();
    int splits = std::max(1, sms / p.m_tiles);
    splits = std::min(splits, 8);  // portable cluster size
    splits = std::min(splits, std::max(1, p.kb_total / 4));
    p.kb_per_split = (p.kb_total + splits - 1) / splits;
    // Two 64-wide K chunks per stage (one 3-D TMA box per operand, 256 contiguous bytes per W
    // row) when every split covers whole chunk pairs.  Measured on GB300 with chained decode
    // linears (4096 x 4096, 64 tokens): 11 % less time per linear than one chunk per stage.
    // The 3-D chunk view has no ragged tail, so h_in must be a multiple of 64; batches above 64
    // tokens keep one chunk (their x boxes would leave room for too few stages).
    p.kc = (pv.h_in % BK == 0 && p.kb_per_split % 2 == 0 && p.n_pad <= 64) ? 2 : 1;
    p.splits = (p.kb_total + p.kb_per_split - 1) / p.kb_per_split;  // no empty split
    const int per = (p.n_pad + p.splits - 1) / p.splits;
    const size_t stage_bytes = ((size_t)BM * BK * 2 + (size_t)p.n_pad * BK * 2) * p.kc;
    const bool use_lsm = per <= kLsmMaxTokens;
    // dedicated region: 4 int arrays, the staged-slot table, s parts [s_parts][per][R], LoRA
    // term [per][128] (small shares), alignment, barriers
    const size_t fixed = (size_t)per * 4 * 4 + (1 + 2 * kMaxPre) * 4 + 16 + (size_t)s_parts * per * pv.R * 4 +
                         (use_lsm ? (size_t)per * BM * 4 : 0) + 128 + 2 * 1024;
    const size_t slot_b = (size_t)BM * pv.R * 2;  // one B tile at r_max (the late path's unit)
    // B tiles staged during the main loop are kept at their slots' true ranks: k slots need at
    // most this many bytes (the k largest ranks among the pool's slots, empty slots at r_max)
    auto pre_bytes = [&](int k) { return (size_t)BM * 16 * pv.top_chunks[std::min(k, kMaxPre)]; };
    const int want = std::min(std::min(per, pv.S), 32);
    const size_t limit = 225 * 1024;
    // stage area after the main loop: P [n_pad][128] + receive buffer [splits-1][per][128]
    // (exchange by bulk copies) + one late B tile
    const size_t ytile = (size_t)2 * kYChunk * BM * 2 + 128;
    const size_t park_push = (size_t)p.n_pad * BM * 4 + (size_t)(p.splits - 1) * per * BM * 4 + ytile + slot_b;
    const size_t park_pull = (size_t)p.n_pad * BM * 4 + ytile + slot_b;
    p.push = 1;
    p.stages = 0;
    p.dpre = 0;
    p.bpre = 0;
    p.compact = 0;
    for (int pass = 0; pass < 2 && !p.stages; ++pass) {
        const size_t park = pass == 0 ? park_push : park_pull;
        int min_stages = 2;
        while ((size_t)min_stages * stage_bytes < park) ++min_stages;
        for (int st = std::max(8, min_stages); st >= std::max(p.kc == 2 ? 2 : 3, min_stages); --st) {
            if ((size_t)st * stage_bytes + fixed > limit) continue;
            const size_t room = limit - st * stage_bytes - fixed;
            int dp = 0;
            while (dp < want && pre_bytes(dp + 1) <= room) ++dp;
            p.stages = st;
            p.dpre = dp;
            // tiles at r_max when the worst case fits that way (no rank reads in the kernel)
            p.compact = (size_t)want * slot_b > room;
            p.bpre = p.compact ? std::min(room, pre_bytes(want)) / 16 * 16 : std::min(room / slot_b, (size_t)want) * slot_b;
            p.push = pass == 0;
            if (dp >= want) break;
        }
    }
    if (!p.stages) p.stages = 8;  // does not fit: tc_supported rejects the shape
    // One accumulator: rotating K-blocks over several (to break the MMA dependency chain)
    // was measured and gave no gain on GB300; the mechanism stays for shapes where it might.
    p.nacc = 1;
    int cols = 32;
    while (cols < p.n_pad * p.nacc) cols <<= 1;
    p.tmem_cols = cols;
    p.smem = (size_t)p.stages * stage_bytes + fixed + p.bpre + 1024;
    return p;
}

}  // namespace tc

int tc_supported(const PoolView& pv, int n) {
    if (pv.dtype != LORA_F16 && pv.dtype != LORA_BF16) return 0;
    if (pv.h_in % 8 || pv.h_out % 8 || pv.R % 8) return 0;
    if (n > 0 && n <= tc::kDecodeMaxN && tc::plan_decode(pv, n, shrink_parts(pv, n, false)).smem > (size_t)(227 * 1024))
        return 0;
    return 1;
}

// Whether the fused decode GEMM is the faster variant: at most 32 owned tokens per CTA, and
// either the B rows of every adapter those tokens can use are staged during the main loop
// (pre-staged slots >= min(owned tokens, n_slots)) or r_max is at most 16, where the epilogue's
// late SIMT groups load little.  Measured on GB300 (32 chained 4096 x 4096 fp16 linears, us per
// linear fused / separate): r_max 8 at 64, 96, 128 tokens 13.1 / 19.4, 16.7 / 24.6, 22.2 / 25.9
// and at 192, 256 tokens (48 and 64 owned tokens) 31.0 / 31.9, 38.4 / 32.4; r_max 64 on 6
// adapters at 64, 96 tokens 18.2 / 24.9, 21.7 / 30.2 and at 128, 256 tokens (B tiles of 6
// slots at r_max 64 do not all fit beside the pipeline) 52.3 / 37.9, 84.9 / 44.7.
int decode_fused_fits(const PoolView& pv, int n) {
    if (n <= 0 || n > tc::kDecodeMaxN || !tc_supported(pv, n)) return 0;
    const tc::DecodePlan p = tc::plan_decode(pv, n, shrink_parts(pv, n, false));
    const int per = (p.n_pad + p.splits - 1) / p.splits;
    return per <= tc::kLsmMaxTokens && (p.dpre >= std::min(per, pv.S) || pv.R <= 16) ? 1 : 0;
}

template <typename T>
static int launch_tc_t(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in,
                       int s_parts, void* y, bool fuse, const void* prefetch, size_t prefetch_bytes,
                       const GroupView* grp, cudaStream_t st, int xready) {
    using namespace tc;
    const int n = sv.n;
    if (n == 0) return LORA_OK;
    const int bf16 = pv.dtype == LORA_BF16;
    const GroupView g1 = grp ? *grp : single_group(pv);
    if (g1.ldy < pv.h_out) return set_error(LORA_EINVAL, "internal: y row stride below h_out");
    if (n <= kDecodeMaxN) {
        // the decode kernel's LoRA epilogue knows one pool: a group runs it per slice, or its
        // base GEMM over the concatenated weight without the LoRA term
        if (g1.count != 1 && fuse) return set_error(LORA_EINVAL, "internal: fused decode GEMM of several slices");
        const DecodePlan p = plan_decode(pv, n, s_parts);
        CUtensorMap mW, mX, mY;
        int rc;
        if (p.kc == 2) {
            rc = make_map_chunked(&mW, W, bf16, pv.h_in, pv.h_out, BM, 2);
            if (rc) return rc;
            rc = make_map_chunked(&mX, x, bf16, pv.h_in, n, p.n_pad, 2);
        } else {
            rc = make_map(&mW, W, bf16, pv.h_in, pv.h_out, BM);
            if (rc) return rc;
            rc = make_map(&mX, x, bf16, pv.h_in, n, p.n_pad);
        }
        if (rc) return rc;
        const int per = (p.n_pad + p.splits - 1) / p.splits;
        const int ychunk = std::min(kYChunk, per);
        const int ytail = per % ychunk;
        CUtensorMap mYt;
        rc = make_map_plain(&mY, y, bf16, pv.h_out, n, BM, ychunk, g1.ldy);
        if (rc) return rc;
        rc = make_map_plain(&mYt, y, bf16, pv.h_out, n, BM, ytail ? ytail : ychunk, g1.ldy);
        if (rc) return rc;
        DecodeArgs a;
        a.pool = pv;
        a.seg = sv;
        a.s_in = s_in;
        a.y = y;
        a.n = n;
        a.n_pad = p.n_pad;
        a.kb_total = p.kb_total;
        a.splits = p.splits;
        a.kb_per_split = p.kb_per_split;
        a.stages = p.stages;
        a.tmem_cols = p.tmem_cols;
        a.nacc = p.nacc;
        a.kc = p.kc;
        a.fuse = fuse ? 1 : 0;
        a.bf16 = bf16;
        a.s_parts = s_parts;
        a.bpre_bytes = static_cast<int>(p.bpre);
        a.compact = p.compact;
        a.push = p.push;
        a.prefetch = static_cast<const char*>(prefetch);
        a.prefetch_bytes = prefetch ? prefetch_bytes : 0;
        a.stamp = take_kernel_stamp();
        // the shrink before a hand-off does not wait for x itself: only this fused single-slice
        // GEMM reads x after its published value
        if (xready && !(fuse && g1.count == 1)) return set_error(LORA_EINVAL, "internal: x-ready hand-off");
        a.xready = xready;
        a.xword = const_cast<int*>(sv.nseg) + kXreadyWord;
        static bool attr_set = false;
        if (!attr_set) {
            LORA_CUDA_TRY(cudaFuncSetAttribute(gemm_decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               227 * 1024));
            attr_set = true;
        }
        // B viewed as [n_slots * h_out rows][r_max / 8 chunks][8 columns]: one box = one chunk
        // column of 128 feature rows (staging at the slots' true ranks)
        CUtensorMap mB;
        rc = make_map_bchunks(&mB, pv.B, bf16, pv.R, (uint64_t)pv.S * pv.h_out);
        if (rc) return rc;
        void* args[] = {(void*)&mW, (void*)&mX, (void*)&mY, (void*)&mYt, (void*)&mB, (void*)&a};
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(p.m_tiles, p.splits);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = p.splits;
        attr[1].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        LORA_CUDA_TRY(cudaLaunchKernelExC(&cfg, (const void*)gemm_decode_kernel<T>, args));
        count_launch();
        return LORA_OK;
    }
    // prefill
    if (s_parts != 1) return set_error(LORA_EINVAL, "internal: prefill GEMM expects an unsplit shrink output");
    if (g1.col[g1.count] != pv.h_out) return set_error(LORA_EINVAL, "internal: slices do not cover h_out");
    PrefillArgs a;
    a.pool = pv;
    a.grp = g1;
    a.seg = sv;
    a.s_in = s_in;
    a.y = y;
    a.n = n;
    a.m_tiles = (n + BM - 1) / BM;
    a.n_tiles = (pv.h_out + kPrefillBN - 1) / kPrefillBN;
    a.kb_total = (pv.h_in + BK - 1) / BK;
    const int stage_bytes = (BM + kPrefillBN) * BK * 2;
    a.stages = std::min(4, kSmemBudget / stage_bytes);
    a.fuse = fuse ? 1 : 0;
    a.bf16 = bf16;
    a.lora_mma = fuse && pv.R <= 64 ? 1 : 0;
    a.stamp = take_kernel_stamp();
    CUtensorMap mX, mW;
    int rc = make_map(&mX, x, bf16, pv.h_in, n, BM);
    if (rc) return rc;
    rc = make_map(&mW, W, bf16, pv.h_in, pv.h_out, kPrefillBN);
    if (rc) return rc;
    // barriers (2 per stage, 4 accumulator, lora_free), the TMEM address and 20 flag words
    if ((2 * a.stages + 5) * 8 + 4 + 20 * 4 > 256) return set_error(LORA_EINVAL, "internal: prefill barrier area");
    const size_t smem = (size_t)a.stages * stage_bytes + 1024 + 256 + 4 * 2 * 32 * 32 * 2;  // + y staging
    CUtensorMap mY;
    rc = make_map_plain(&mY, y, bf16, g1.ldy, n, 32, 32, g1.ldy);
    if (rc) return rc;
    static bool attr = false;
    if (!attr) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(gemm_prefill_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           227 * 1024));
        attr = true;
    }
    const int total = a.m_tiles * a.n_tiles;
    const int grid = std::min(total, num_sms());
    void* args[] = {(void*)&mX, (void*)&mW, (void*)&mY, (void*)&a};
    LORA_CUDA_TRY(launch_pdl((const void*)gemm_prefill_kernel<T>, dim3(grid), dim3(kThreads), smem, st, args));
    return LORA_OK;
}

template <typename T>
static int launch_tall_t(const PoolView& pv, const SegView& sv, const void* W, const void* x, void* y, int ldy,
                         cudaStream_t st) {
    using namespace tc;
    const int n = sv.n;
    if (n == 0) return LORA_OK;
    if (n > kDecodeMaxN) return set_error(LORA_EINVAL, "internal: tall-tile GEMM for more than 256 tokens");
    TallArgs a;
    a.seg = sv;
    a.y = y;
    a.n = n;
    // two token halves per row tile when that still fits the SMs (q|k|v: 48 tiles -> 96 CTAs);
    // each CTA then takes in W and half of x, and writes its own tokens of y
    const int tiles = (pv.h_out + 2 * BM - 1) / (2 * BM);
    const int tsplit = (n > 128 && 2 * tiles <= num_sms()) ? 2 : 1;
    a.tstep = (n + tsplit - 1) / tsplit;
    a.n_pad = std::max(16, (a.tstep + 15) / 16 * 16);
    a.ldy = ldy;
    a.h_out = pv.h_out;
    a.nkb = (pv.h_in + BK - 1) / BK;
    a.bf16 = pv.dtype == LORA_BF16;
    a.stamp = take_kernel_stamp();
    const size_t stage_bytes = (size_t)2 * BM * BK * 2 + (size_t)a.n_pad * BK * 2;
    a.stages = std::max(2, std::min(6, (int)(kSmemBudget / stage_bytes)));
    const size_t smem = (size_t)a.stages * stage_bytes + (2 * (size_t)a.stages + 1) * 8 + 16 + 1024;
    CUtensorMap mW, mX;
    int rc = make_map(&mW, W, a.bf16, pv.h_in, pv.h_out, 2 * BM);
    if (rc) return rc;
    rc = make_map(&mX, x, a.bf16, pv.h_in, n, a.n_pad);
    if (rc) return rc;
    static bool attr_set = false;
    if (!attr_set) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(gemm_tall_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           227 * 1024));
        attr_set = true;
    }
    void* args[] = {(void*)&mW, (void*)&mX, (void*)&a};
    LORA_CUDA_TRY(launch_pdl((const void*)gemm_tall_kernel<T>, dim3(tiles, tsplit), dim3(kThreads), smem, st, args));
    return LORA_OK;
}

int launch_gemm_tall(const PoolView& pv, const SegView& sv, const void* W, const void* x, void* y, int ldy,
                     cudaStream_t st) {
    if (pv.dtype == LORA_F16) return launch_tall_t<__half>(pv, sv, W, x, y, ldy, st);
    return launch_tall_t<__nv_bfloat16>(pv, sv, W, x, y, ldy, st);
}

int launch_gemm_tc(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in, int s_parts,
                   void* y, bool fuse, cudaStream_t st, const void* prefetch, size_t prefetch_bytes,
                   const GroupView* grp, int xready) {
    if (pv.dtype == LORA_F16)
        return launch_tc_t<__half>(pv, sv, W, x, s_in, s_parts, y, fuse, prefetch, prefetch_bytes, grp, st,
                                   xready);
    return launch_tc_t<__nv_bfloat16>(pv, sv, W, x, s_in, s_parts, y, fuse, prefetch, prefetch_bytes, grp, st,
                                      xready);
}

}  // namespace lora
