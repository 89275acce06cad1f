// CUDA-core kernels of the LoRA path: the segmented shrink (x A^T), the residual expand of
// the separate variant, and a CUDA-core base GEMM with the expand fused in its epilogue
// (float32 pools and shapes the tensor-core path does not take).
//
// The execution unit of "LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排" (blog.lonae.com)
// applies the low-rank A/B product onto the base hidden state, either inside the base
// kernel (fused) or as a residual added by a second kernel (separate).  The shrink writes
// s[t, j] = (alpha_s / r_s) * sum_k x[t,k] A_s[j,k] in float32 for every token t with a slot,
// in original token order; both expands read it.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
    return v;
}

// ---- shrink, one warp per (sorted token, group of RG adapter rows) ----------------------------
// Walking tokens in sorted order keeps consecutive warps on the same adapter, so each A row
// comes from HBM once per batch and from L1/L2 afterwards.
template <typename T, int RG>
__global__ void __launch_bounds__(256)
shrink_warp_kernel(PoolView pool, SegView seg, const T* __restrict__ x, float* __restrict__ s_out) {
    pdl_wait();
    pdl_trigger();
    if (*seg.status != LORA_OK) return;
    const int lane = threadIdx.x & 31;
    const int groups = pool.R / RG;
    const long gw = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long j = gw / groups;
    const int g = (int)(gw % groups);
    if (j >= seg.n) return;
    const int t = seg.perm[j];
    const int s = seg.idx[t];
    if (s < 0) return;
    const float scale = pool.table[s].scale;
    const int h = pool.h_in;
    const T* xr = x + (size_t)t * h;
    const T* Ar = static_cast<const T*>(pool.A) + ((size_t)s * pool.R + (size_t)g * RG) * h;
    float acc[RG];
#pragma unroll
    for (int r = 0; r < RG; ++r) acc[r] = 0.f;
    if constexpr (sizeof(T) == 2) {
        for (int k = lane * 8; k < h; k += 256) {
            float xf[8];
            unpack8<T>(*reinterpret_cast<const uint4*>(xr + k), xf);
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                float af[8];
                unpack8<T>(*reinterpret_cast<const uint4*>(Ar + (size_t)r * h + k), af);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r] = fmaf(xf[e], af[e], acc[r]);
            }
        }
    } else {
        for (int k = lane; k < h; k += 32) {
            const float xv = to_f32(xr[k]);
#pragma unroll
            for (int r = 0; r < RG; ++r) acc[r] = fmaf(xv, to_f32(Ar[(size_t)r * h + k]), acc[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < RG; ++r) acc[r] = warp_sum(acc[r]);
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RG; ++r) s_out[(size_t)t * pool.R + g * RG + r] = scale * acc[r];
    }
}

// Grid-dependency wait of the decode shrinks, and the release of the base GEMM that follows.
// Without an x-ready value the dependents are released after the wait: the GEMM then knows
// that every kernel before this one has completed (x, W) and waits separately for s.  With
// one, they are released at once -- the GEMM starts streaming its weight while the previous
// linear finishes -- and the first CTA publishes the value once the wait has returned (x and
// the segments complete); the GEMM loads x after reading it and waits for s as before.
__device__ __forceinline__ void shrink_dependency_wait(const GroupView& grp, const SegView& seg) {
    if (grp.xready) {
        pdl_trigger();
        pdl_wait();
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            st_release_gpu(const_cast<int32_t*>(seg.nseg) + kXreadyWord, grp.xready);
    } else {
        pdl_wait();
        pdl_trigger();
    }
}

// ---- shrink for small batches: one CTA per (token, 8 adapter rows, K-part) -------------------
// 128 threads each own 8 consecutive input features of every 1024-feature sweep, so a sweep
// reads 2 KB of x and 16 KB of A with all nine 16-byte loads of a thread in flight; the K-parts
// (shrink_parts) are summed by the consumers.
// The whole grid is resident at once for decode batches, so tokens are taken in their original
// order (one dependent load less than walking the sorted order).
constexpr int kShrKChunk = 1024;

template <typename T>
__global__ void __launch_bounds__(128)
shrink_token_kernel(PoolView pool, GroupView grp, SegView seg, const T* __restrict__ x, float* __restrict__ s_out) {
    __shared__ float red[4][8];
    AuxStamp stamp(grp.stamp);
    shrink_dependency_wait(grp, seg);
    stamp.waited();
    const int t = blockIdx.x, ks = blockIdx.z;
    const int h = pool.h_in, R = pool.R, rg = R / 8;
    // grid rows: (slice of the group, 8-row group of r_max)
    const int qs = blockIdx.y / rg, g = blockIdx.y - qs * rg;
    const SliceRef sl = group_slice(grp, qs);
    s_out += sl.s_off;
    // this CTA's K range: part ks of gridDim.z, in sweeps of 1024 features (128 threads x 8)
    const int sweeps = ((h + kShrKChunk - 1) / kShrKChunk + gridDim.z - 1) / gridDim.z;
    const int k_beg = ks * sweeps * kShrKChunk;
    const int k_end = min(h, k_beg + sweeps * kShrKChunk);
    const int k0 = k_beg + threadIdx.x * 8;
    // independent loads first: status, slot, x; then the slot's A rows
    const int status = __ldcg(seg.status);
    const int s = __ldcg(seg.idx + t);
    uint4 xv = make_uint4(0, 0, 0, 0);
    if (k0 < k_end) xv = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)t * h + k0));
    if (s < 0 || status != LORA_OK) return;
    // rows past the adapter's true rank (only possible with several row groups): A is zero
    if (rg > 1 && g * 8 >= sl.table[s].rank) {
        if (threadIdx.x < 8) s_out[((size_t)ks * seg.n + t) * R + g * 8 + threadIdx.x] = 0.f;
        return;
    }
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.f;
    const T* Ab = static_cast<const T*>(sl.A) + ((size_t)s * R + (size_t)g * 8) * h;
    for (int k = k0; k < k_end; k += kShrKChunk) {
        if (k != k0) xv = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)t * h + k));
        uint4 av[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) av[r] = __ldg(reinterpret_cast<const uint4*>(Ab + (size_t)r * h + k));
        float xf[8];
        unpack8<T>(xv, xf);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            float af[8];
            unpack8<T>(av[r], af);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[r] = fmaf(xf[e], af[e], acc[r]);
        }
    }
    const float scale = sl.table[s].scale;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) red[warp][r] = v;
    }
    __syncthreads();
    if (threadIdx.x < 8) {
        const float v = red[0][threadIdx.x] + red[1][threadIdx.x] + red[2][threadIdx.x] + red[3][threadIdx.x];
        s_out[((size_t)ks * seg.n + t) * R + g * 8 + threadIdx.x] = scale * v;
    }
}

constexpr int kItemTok = 4;  // sorted tokens per work item (built by the segment kernel)

// Segmented shrink for short batches (16-bit).  Work item = up to 4 consecutive sorted tokens
// of one adapter segment ({slot, count, token[4]}, built once per batch by the segment
// kernel); grid (items bound, r_max/8 row groups, K parts).  A CTA loads its 8 adapter rows
// once (8 features per thread, 1024 per sweep) and applies them to the item's tokens, so an
// adapter's A rows are read once per 4 tokens of its segment rather than once per token
// (r_max 64, 64 tokens over 6 adapters: 11 MB instead of 32 MB per linear).  A thread's 32
// sums (4 tokens x 8 rows) are reduced over the warp by a reduce-scatter butterfly (31
// shuffles leave lane L the total of sum L).  Output row t (original order) of K part ks:
// s_out[(ks * n + t) * r_max + row] = scale * partial dot product.
template <typename T>
__global__ void __launch_bounds__(128, 4)
shrink_seg_kernel(PoolView pool, GroupView grp, SegView seg, const T* __restrict__ x, float* __restrict__ s_out) {
    __shared__ float red[4][32];
    AuxStamp stamp(grp.stamp);
    shrink_dependency_wait(grp, seg);
    stamp.waited();
    const int b = blockIdx.x, ks = blockIdx.z;
    const int h = pool.h_in, R = pool.R, rg = R / 8;
    // grid rows: (slice of the group, 8-row group of r_max)
    const int qs = blockIdx.y / rg, g = blockIdx.y - qs * rg;
    const SliceRef sl = group_slice(grp, qs);
    s_out += sl.s_off;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // independent loads first: status, item count, the item
    const int status = __ldcg(seg.status);
    const int n_items = __ldcg(seg.nseg + 1);
    const int4 head = __ldcg(reinterpret_cast<const int4*>(seg.items + (size_t)b * 8));      // slot, count, tok0, tok1
    const int4 tail = __ldcg(reinterpret_cast<const int4*>(seg.items + (size_t)b * 8 + 4));  // tok2, tok3, rank
    if (status != LORA_OK || b >= n_items) return;
    const int slot = head.x, nt = head.y;
    const int tok[kItemTok] = {head.z, head.w, tail.x, tail.y};
    // Rows past the adapter's true rank: A is zero there.  The item carries the rank in the
    // pool the segments were built on; segments may be shared by pools with the same slot
    // count, and this pool may hold the slot at a larger rank, so its own table decides.
    if (g * 8 >= tail.z && g * 8 >= sl.table[slot].rank) {
        const int u = threadIdx.x >> 3;
        if (threadIdx.x < kItemTok * 8 && u < nt) {
            const int t = u == 0 ? head.z : u == 1 ? head.w : u == 2 ? tail.x : tail.y;
            s_out[((size_t)ks * seg.n + t) * R + g * 8 + (threadIdx.x & 7)] = 0.f;
        }
        return;
    }
    // this CTA's K range: part ks of gridDim.z, in sweeps of 1024 features (128 threads x 8)
    const int sweeps = ((h + kShrKChunk - 1) / kShrKChunk + gridDim.z - 1) / gridDim.z;
    const int k_beg = ks * sweeps * kShrKChunk;
    const int k_end = min(h, k_beg + sweeps * kShrKChunk);
    const T* Ab = static_cast<const T*>(sl.A) + ((size_t)slot * R + (size_t)g * 8) * h;
    float v[kItemTok * 8];  // v[u * 8 + r]: token u, adapter row g*8 + r
#pragma unroll
    for (int e = 0; e < kItemTok * 8; ++e) v[e] = 0.f;
    for (int k = k_beg + threadIdx.x * 8; k < k_end; k += kShrKChunk) {
        uint4 av[8], xv[kItemTok];
#pragma unroll
        for (int u = 0; u < kItemTok; ++u) xv[u] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)tok[u] * h + k));
#pragma unroll
        for (int r = 0; r < 8; ++r) av[r] = __ldg(reinterpret_cast<const uint4*>(Ab + (size_t)r * h + k));
#pragma unroll
        for (int u = 0; u < kItemTok; ++u) {
            float xf[8];
            unpack8<T>(xv[u], xf);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float af[8];
                unpack8<T>(av[r], af);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[u * 8 + r] = fmaf(xf[e], af[e], v[u * 8 + r]);
            }
        }
    }
    // reduce-scatter over the warp: at offset o, lanes with bit o keep the upper half
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int half = 16 >> step, off = 16 >> step;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int e = 0; e < half; ++e) {
            const float send = up ? v[e] : v[e + half];
            const float keepv = up ? v[e + half] : v[e];
            v[e] = keepv + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    red[warp][lane] = v[0];
    __syncthreads();
    if (threadIdx.x < kItemTok * 8) {
        const int u = threadIdx.x >> 3, r = threadIdx.x & 7;
        if (u < nt) {
            const float sum = red[0][threadIdx.x] + red[1][threadIdx.x] + red[2][threadIdx.x] + red[3][threadIdx.x];
            const int t = u == 0 ? head.z : u == 1 ? head.w : u == 2 ? tail.x : tail.y;
            s_out[((size_t)ks * seg.n + t) * R + g * 8 + r] = sl.table[slot].scale * sum;
        }
    }
}

// ---- shrink, tiled: one CTA per (segment, 64 sorted tokens) -----------------------------------
// For long segments (prefill) x and A are staged through shared memory in K-chunks of 64 and
// every thread keeps a 4 x (R/16) register tile.
constexpr int kShrTT = 64, kShrKC = 64;

template <typename T>
__global__ void __launch_bounds__(256)
shrink_tiled_kernel(PoolView pool, SegView seg, const T* __restrict__ x, float* __restrict__ s_out) {
    extern __shared__ float sh[];
    const int R = pool.R, h = pool.h_in;
    float* xs = sh;                             // [TT][KC+1]
    float* as = sh + kShrTT * (kShrKC + 1);     // [R][KC+1]
    __shared__ int s_seg, s_j0, s_j1, s_slot;
    __shared__ int s_tok[kShrTT];
    pdl_wait();
    pdl_trigger();
    if (*seg.status != LORA_OK) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == 0) {
        // locate this CTA's (segment, tile): tiles of a segment = ceil(len / TT), none for -1
        const int nseg = *seg.nseg;
        int run = 0;
        int found = -1, ftile = 0;
        for (int base = 0; base < nseg && found < 0; base += 32) {
            const int i = base + lane;
            int ti = 0;
            if (i < nseg && seg.seg_slot[i] >= 0) ti = (seg.seg_start[i + 1] - seg.seg_start[i] + kShrTT - 1) / kShrTT;
            int v = ti;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += u;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, (int)blockIdx.x < run + v);
            if (hit) {
                const int l = __ffs(hit) - 1;
                found = base + l;
                const int vl = __shfl_sync(0xffffffffu, v, l);
                const int tl = __shfl_sync(0xffffffffu, ti, l);
                ftile = (int)blockIdx.x - (run + vl - tl);
            }
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) {
            s_seg = found;
            if (found >= 0) {
                s_slot = seg.seg_slot[found];
                s_j0 = seg.seg_start[found] + ftile * kShrTT;
                s_j1 = min(s_j0 + kShrTT, seg.seg_start[found + 1]);
            }
        }
    }
    __syncthreads();
    if (s_seg < 0) return;
    const int j0 = s_j0, cnt = s_j1 - s_j0, slot = s_slot;
    if (tid < kShrTT) s_tok[tid] = tid < cnt ? seg.perm[j0 + tid] : -1;
    __syncthreads();
    const T* A = static_cast<const T*>(pool.A) + (size_t)slot * R * h;
    const int tq = tid >> 4, tr = tid & 15;
    constexpr int MAXJ = kMaxRank / 16;
    float acc[4][MAXJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < MAXJ; ++jj) acc[i][jj] = 0.f;
    const int nj = (R + 15) / 16;
    for (int k0 = 0; k0 < h; k0 += kShrKC) {
        for (int e = tid; e < kShrTT * kShrKC; e += 256) {
            const int q = e / kShrKC, kk = e % kShrKC;
            const int t = s_tok[q];
            xs[q * (kShrKC + 1) + kk] = (t >= 0 && k0 + kk < h) ? to_f32(x[(size_t)t * h + k0 + kk]) : 0.f;
        }
        for (int e = tid; e < R * kShrKC; e += 256) {
            const int r = e / kShrKC, kk = e % kShrKC;
            as[r * (kShrKC + 1) + kk] = (k0 + kk < h) ? to_f32(A[(size_t)r * h + k0 + kk]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kShrKC; ++kk) {
            float xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = xs[(tq + 16 * i) * (kShrKC + 1) + kk];
#pragma unroll
            for (int jj = 0; jj < MAXJ; ++jj) {
                if (jj < nj && tr + 16 * jj < R) {
                    const float av = as[(tr + 16 * jj) * (kShrKC + 1) + kk];
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i][jj] = fmaf(xv[i], av, acc[i][jj]);
                }
            }
        }
        __syncthreads();
    }
    const float scale = pool.table[slot].scale;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = tq + 16 * i;
        if (q >= cnt) continue;
        const int t = s_tok[q];
#pragma unroll
        for (int jj = 0; jj < MAXJ; ++jj)
            if (jj < nj && tr + 16 * jj < R) s_out[(size_t)t * R + tr + 16 * jj] = scale * acc[i][jj];
    }
}

// ---- expand of the separate variant: y[t, o] += sum_j s[t, j] B_s[o, j] -----------------------
// One CTA per (256 outputs, 16 tokens).  y is read, the float32 LoRA term added, and y is
// rounded and written back (the residual add of the separate design).
constexpr int kExpTT = 16;

template <typename T>
__global__ void __launch_bounds__(256)
expand_kernel(PoolView pool, SegView seg, const float* __restrict__ s_in, int s_parts, T* __restrict__ y) {
    extern __shared__ float ss[];  // [TT][R]
    __shared__ int sl[kExpTT];
    pdl_wait();
    pdl_trigger();
    if (*seg.status != LORA_OK) return;
    const int R = pool.R, h_out = pool.h_out;
    const int t0 = blockIdx.y * kExpTT;
    const int nt = min(kExpTT, seg.n - t0);
    if (threadIdx.x < kExpTT) sl[threadIdx.x] = threadIdx.x < nt ? seg.idx[t0 + threadIdx.x] : -1;
    __syncthreads();
    for (int e = threadIdx.x; e < nt * R; e += blockDim.x) {
        const int q = e / R;
        float v = 0.f;
        if (sl[q] >= 0)
            for (int k = 0; k < s_parts; ++k) v += s_in[((size_t)k * seg.n + t0 + q) * R + e % R];
        ss[e] = v;
    }
    __syncthreads();
    const int o = blockIdx.x * 256 + threadIdx.x;
    if (o >= h_out) return;
    const T* B = static_cast<const T*>(pool.B);
    for (int q = 0; q < nt; ++q) {
        const int s = sl[q];
        if (s < 0) continue;
        const T* Br = B + ((size_t)s * h_out + o) * R;
        float acc = 0.f;
        if constexpr (sizeof(T) == 2) {
            for (int j = 0; j < R; j += 8) {
                float bf[8];
                unpack8<T>(*reinterpret_cast<const uint4*>(Br + j), bf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(bf[e], ss[q * R + j + e], acc);
            }
        } else {
            for (int j = 0; j < R; ++j) acc = fmaf(to_f32(Br[j]), ss[q * R + j], acc);
        }
        T* yp = y + (size_t)(t0 + q) * h_out + o;
        *yp = from_f32<T>(to_f32(*yp) + acc);
    }
}

// Segmented expand (separate variant, 16-bit): one CTA per (work item = up to 4 sorted tokens
// of one adapter segment, 256 * fpt output features of a slice).  A thread owns features o
// and, with fpt = 2, o + 256: it loads those features' B rows of the item's adapter (r_max / 8
// 16-byte loads each) and the item's y values, all before use, and adds the LoRA term of every
// token of the item.  Two features per thread pay the CTA's chain of dependent loads (item,
// shrink rows and y, B) once for twice the work; the launcher takes them when the grid still
// has two CTAs per SM (GB300: 7B layer at 256 tokens 6 % faster per step, a 6-adapter batch of
// 64 tokens at r_max 64 23 % slower with them).
template <typename T>
__global__ void __launch_bounds__(256)
expand_seg_kernel(PoolView pool, GroupView grp, SegView seg, const float* __restrict__ s_in, int s_parts,
                  T* __restrict__ y, int fpt) {
    extern __shared__ float ss[];  // [4][R]: the item's shrink rows (K parts summed)
    AuxStamp stamp(grp.stamp);
    pdl_wait();
    stamp.waited();
    pdl_trigger();
    const int b = blockIdx.x;
    // grid columns: expand blocks (256 * fpt features) of the group's slices, one after another
    int qs = 0, blk0 = 0;
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
        if (i < grp.count && (int)blockIdx.y >= grp.blk[i]) {
            qs = i;
            blk0 = grp.blk[i];
        }
    const SliceRef sl = group_slice(grp, qs);
    s_in += sl.s_off;
    const int status = __ldcg(seg.status);
    const int n_items = __ldcg(seg.nseg + 1);
    const int4 head = __ldcg(reinterpret_cast<const int4*>(seg.items + (size_t)b * 8));      // slot, count, tok0, tok1
    const int2 tail = __ldcg(reinterpret_cast<const int2*>(seg.items + (size_t)b * 8 + 4));  // tok2, tok3
    if (status != LORA_OK || b >= n_items) return;
    const int R = pool.R, h_out = sl.h_out, ldy = grp.ldy, slot = head.x, nt = head.y;
    const int tok[kItemTok] = {head.z, head.w, tail.x, tail.y};
    for (int e = threadIdx.x; e < kItemTok * R; e += blockDim.x) {
        const int u = e / R, j = e - u * R;
        const int tu = u == 0 ? head.z : u == 1 ? head.w : u == 2 ? tail.x : tail.y;  // no local array
        float v = 0.f;
        if (u < nt)
            for (int k = 0; k < s_parts; ++k) v += __ldcg(s_in + ((size_t)k * seg.n + tu) * R + j);
        ss[e] = v;
    }
    const int o = (blockIdx.y - blk0) * 256 * fpt + threadIdx.x;  // first feature within the slice
    const bool live0 = o < h_out, live1 = fpt == 2 && o + 256 < h_out;
    T* yc = y + sl.col + o;  // column of y
    float yv[2][kItemTok];
#pragma unroll
    for (int u = 0; u < kItemTok; ++u) {
        yv[0][u] = live0 && u < nt ? to_f32(yc[(size_t)tok[u] * ldy]) : 0.f;
        yv[1][u] = live1 && u < nt ? to_f32(yc[(size_t)tok[u] * ldy + 256]) : 0.f;
    }
    __syncthreads();
    if (!live0) return;
    const T* Br = static_cast<const T*>(sl.B) + ((size_t)slot * h_out + o) * R;
    // columns past the adapter's true rank are zero in B (and in s): skip them when the pool
    // has padded slots (the rank comes from this pool's own table)
    const int jmax = grp.rank_aware ? min(R, (max(sl.table[slot].rank, 1) + 7) & ~7) : R;
    float acc[2][kItemTok];
#pragma unroll
    for (int u = 0; u < kItemTok; ++u) acc[0][u] = acc[1][u] = 0.f;
    for (int j = 0; j < jmax; j += 8) {
        float b0[8], b1[8];
        unpack8<T>(__ldg(reinterpret_cast<const uint4*>(Br + j)), b0);
        unpack8<T>(live1 ? __ldg(reinterpret_cast<const uint4*>(Br + (size_t)256 * R + j)) : make_uint4(0, 0, 0, 0), b1);
#pragma unroll
        for (int u = 0; u < kItemTok; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float sv = ss[u * R + j + e];
                acc[0][u] = fmaf(b0[e], sv, acc[0][u]);
                acc[1][u] = fmaf(b1[e], sv, acc[1][u]);
            }
    }
#pragma unroll
    for (int u = 0; u < kItemTok; ++u)
        if (u < nt) {
            yc[(size_t)tok[u] * ldy] = from_f32<T>(yv[0][u] + acc[0][u]);
            if (live1) yc[(size_t)tok[u] * ldy + 256] = from_f32<T>(yv[1][u] + acc[1][u]);
        }
}

// ---- CUDA-core base GEMM, optional fused expand ---------------------------------------------
// 64 tokens x 64 outputs per CTA, 256 threads with 4 x 4 outputs each, K-chunks of 16.
template <typename T>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(PoolView pool, SegView seg, const T* __restrict__ W, const T* __restrict__ x,
                 const float* __restrict__ s_in, int s_parts, T* __restrict__ y, int fuse_lora) {
    __shared__ float xs[16][65];
    __shared__ float ws[16][65];
    pdl_wait();
    pdl_trigger();
    if (*seg.status != LORA_OK) return;
    const int n = seg.n, h_in = pool.h_in, h_out = pool.h_out, R = pool.R;
    const int t0 = blockIdx.y * 64, o0 = blockIdx.x * 64;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < h_in; k0 += 16) {
        for (int e = tid; e < 64 * 16; e += 256) {
            const int r = e >> 4, kk = e & 15;
            const int t = t0 + r, o = o0 + r, k = k0 + kk;
            xs[kk][r] = (t < n && k < h_in) ? to_f32(x[(size_t)t * h_in + k]) : 0.f;
            ws[kk][r] = (o < h_out && k < h_in) ? to_f32(W[(size_t)o * h_in + k]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty + 16 * i];
#pragma unroll
            for (int i = 0; i < 4; ++i) b[i] = ws[kk][tx + 16 * i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
        }
        __syncthreads();
    }
    const T* B = static_cast<const T*>(pool.B);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty + 16 * i;
        if (t >= n) continue;
        const int s = fuse_lora ? seg.idx[t] : -1;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int o = o0 + tx + 16 * jj;
            if (o >= h_out) continue;
            float v = acc[i][jj];
            if (s >= 0) {
                const T* Br = B + ((size_t)s * h_out + o) * R;
                float l = 0.f;
                for (int j = 0; j < R; ++j) {
                    float sj = 0.f;
                    for (int k = 0; k < s_parts; ++k) sj += s_in[((size_t)k * n + t) * R + j];
                    l = fmaf(sj, to_f32(Br[j]), l);
                }
                v += l;
            }
            y[(size_t)t * h_out + o] = from_f32<T>(v);
        }
    }
}

// ---- host launchers ----------------------------------------------------------------------------

// K-parts of the small-batch shrink: enough CTAs to keep the loads in flight (~256 CTAs per
// group of 8 adapter rows), at most 4 parts so that the consumers stage little.
int shrink_parts(const PoolView& pv, int n, bool tiled) {
    if (pv.dtype == LORA_F32 || tiled) return 1;
    int p = (pv.h_in + kShrKChunk - 1) / kShrKChunk;
    p = std::min(p, 4);
    p = std::min(p, std::max(1, 256 / std::max(n, 1)));
    return p;
}

template <typename T>
static int launch_shrink_t(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                           cudaStream_t st, bool tiled, int* s_parts) {
    const T* xp = static_cast<const T*>(x);
    *s_parts = shrink_parts(pv, sv.n, tiled);
    if constexpr (sizeof(T) == 2) {
        if (!tiled) {
            if (sv.n == 0) return LORA_OK;
            GroupView g1 = grp;
            g1.stamp = take_aux_stamp();
            void* args[] = {(void*)&pv, (void*)&g1, (void*)&sv, (void*)&xp, (void*)&s_out};
            const int rows = grp.count * (pv.R / 8);  // (slice, 8-row group) pairs
            if (shrink_segmented(pv, sv.n)) {
                // at most one item per LoRA token, and per segment one partial item beyond n / 4
                const int items = std::min(sv.n, std::min(sv.n, pv.S) + (sv.n + kItemTok - 1) / kItemTok);
                LORA_CUDA_TRY(launch_pdl((const void*)shrink_seg_kernel<T>, dim3(items, rows, *s_parts), dim3(128), 0,
                                         st, args));
            } else {
                LORA_CUDA_TRY(launch_pdl((const void*)shrink_token_kernel<T>, dim3(sv.n, rows, *s_parts), dim3(128), 0,
                                         st, args));
            }
            return LORA_OK;
        }
    }
    if (grp.count != 1) return set_error(LORA_EUNSUP, "internal: grouped shrink needs 16-bit data and <= 256 tokens");
    if (!tiled) {
        const int RG = (pv.R % 8 == 0) ? 8 : 1;
        const long warps = (long)sv.n * (pv.R / RG);
        const int blocks = (int)((warps + 7) / 8);
        if (blocks == 0) return LORA_OK;
        void* args[] = {(void*)&pv, (void*)&sv, (void*)&xp, (void*)&s_out};
        const void* fn = RG == 8 ? (const void*)shrink_warp_kernel<T, 8> : (const void*)shrink_warp_kernel<T, 1>;
        LORA_CUDA_TRY(launch_pdl(fn, dim3(blocks), dim3(256), 0, st, args));
        return LORA_OK;
    }
    const int max_tiles = (sv.n + kShrTT - 1) / kShrTT + std::min(sv.n, pv.S + 1);
    if (max_tiles == 0) return LORA_OK;
    const size_t smem = sizeof(float) * (kShrTT + pv.R) * (kShrKC + 1);
    static bool attr = false;
    if (!attr) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(shrink_tiled_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(sizeof(float) * (kShrTT + kMaxRank) * (kShrKC + 1))));
        attr = true;
    }
    void* args[] = {(void*)&pv, (void*)&sv, (void*)&xp, (void*)&s_out};
    LORA_CUDA_TRY(launch_pdl((const void*)shrink_tiled_kernel<T>, dim3(max_tiles), dim3(256), smem, st, args));
    return LORA_OK;
}

// Per token, every LoRA token re-reads its adapter's A rows: n * r_max * h_in * 2 bytes at
// most.  Past 16 MB (r_max 64 at 64 tokens, 4096 features: 33.5 MB) the segmented kernel reads
// each adapter once per 4 tokens instead (GB300, 32 chained 4096x4096 linears: r_max 64, 64
// tokens 9 % faster; r_max 8 9 % slower, since its CTAs then take up to 4 tokens each on the
// shrink's critical path).
int shrink_segmented(const PoolView& pv, int n) {
    return (double)n * pv.R * pv.h_in * 2 >= 16.0 * (1 << 20) ? 1 : 0;
}

int launch_shrink(const PoolView& pv, const SegView& sv, const void* x, float* s_out, cudaStream_t st, bool tiled,
                  int* s_parts, int xready) {
    GroupView g = single_group(pv);
    g.xready = xready;
    return launch_shrink_group(pv, g, sv, x, s_out, st, tiled, s_parts);
}

int launch_shrink_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const void* x, float* s_out,
                        cudaStream_t st, bool tiled, int* s_parts) {
    switch (pv.dtype) {
        case LORA_F32: return launch_shrink_t<float>(pv, grp, sv, x, s_out, st, tiled, s_parts);
        case LORA_F16: return launch_shrink_t<__half>(pv, grp, sv, x, s_out, st, tiled, s_parts);
        default: return launch_shrink_t<__nv_bfloat16>(pv, grp, sv, x, s_out, st, tiled, s_parts);
    }
}

template <typename T>
static int launch_expand_t(const PoolView& pv, const GroupView& grp, const SegView& sv, const float* s_in, int s_parts,
                           void* y, cudaStream_t st) {
    if (sv.n == 0) return LORA_OK;
    T* yp = static_cast<T*>(y);
    if constexpr (sizeof(T) == 2) {
        // one CTA per (work item, 256 features of a slice); items: at most one per LoRA token,
        // and per segment one partial item beyond n / 4
        const int items = std::min(sv.n, std::min(sv.n, pv.S) + (sv.n + kItemTok - 1) / kItemTok);
        // two features per thread when the grid keeps two CTAs per SM that way
        GroupView g2 = grp;
        g2.stamp = take_aux_stamp();
        int blocks512 = 0;
        for (int q = 0; q < grp.count; ++q) blocks512 += (grp.col[q + 1] - grp.col[q] + 511) / 512;
        const int fpt = (long long)items * blocks512 >= 2LL * num_sms() ? 2 : 1;
        g2.blk[0] = 0;
        for (int q = 0; q < grp.count; ++q)
            g2.blk[q + 1] = g2.blk[q] + (grp.col[q + 1] - grp.col[q] + 256 * fpt - 1) / (256 * fpt);
        void* args[] = {(void*)&pv, (void*)&g2, (void*)&sv, (void*)&s_in, (void*)&s_parts, (void*)&yp, (void*)&fpt};
        const dim3 grid(items, g2.blk[grp.count]);
        LORA_CUDA_TRY(launch_pdl((const void*)expand_seg_kernel<T>, grid, dim3(256), sizeof(float) * kItemTok * pv.R,
                                 st, args));
        return LORA_OK;
    }
    if (grp.count != 1) return set_error(LORA_EUNSUP, "internal: grouped expand needs 16-bit data");
    void* args[] = {(void*)&pv, (void*)&sv, (void*)&s_in, (void*)&s_parts, (void*)&yp};
    const dim3 grid((pv.h_out + 255) / 256, (sv.n + kExpTT - 1) / kExpTT);
    const size_t smem = sizeof(float) * kExpTT * pv.R;
    LORA_CUDA_TRY(launch_pdl((const void*)expand_kernel<T>, grid, dim3(256), smem, st, args));
    return LORA_OK;
}

int launch_expand(const PoolView& pv, const SegView& sv, const float* s_in, int s_parts, void* y, cudaStream_t st) {
    return launch_expand_group(pv, single_group(pv), sv, s_in, s_parts, y, st);
}

int launch_expand_group(const PoolView& pv, const GroupView& grp, const SegView& sv, const float* s_in, int s_parts,
                        void* y, cudaStream_t st) {
    switch (pv.dtype) {
        case LORA_F32: return launch_expand_t<float>(pv, grp, sv, s_in, s_parts, y, st);
        case LORA_F16: return launch_expand_t<__half>(pv, grp, sv, s_in, s_parts, y, st);
        default: return launch_expand_t<__nv_bfloat16>(pv, grp, sv, s_in, s_parts, y, st);
    }
}

template <typename T>
static int launch_gemm_simt_t(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in,
                              int s_parts, void* y, bool fuse, cudaStream_t st) {
    if (sv.n == 0) return LORA_OK;
    const T* Wp = static_cast<const T*>(W);
    const T* xp = static_cast<const T*>(x);
    T* yp = static_cast<T*>(y);
    int f = fuse ? 1 : 0;
    const dim3 grid((pv.h_out + 63) / 64, (sv.n + 63) / 64);
    void* args[] = {(void*)&pv, (void*)&sv, (void*)&Wp, (void*)&xp, (void*)&s_in, (void*)&s_parts, (void*)&yp, (void*)&f};
    LORA_CUDA_TRY(launch_pdl((const void*)gemm_simt_kernel<T>, grid, dim3(256), 0, st, args));
    return LORA_OK;
}

int launch_gemm_simt(const PoolView& pv, const SegView& sv, const void* W, const void* x, const float* s_in,
                     int s_parts, void* y, bool fuse, cudaStream_t st) {
    switch (pv.dtype) {
        case LORA_F32: return launch_gemm_simt_t<float>(pv, sv, W, x, s_in, s_parts, y, fuse, st);
        case LORA_F16: return launch_gemm_simt_t<__half>(pv, sv, W, x, s_in, s_parts, y, fuse, st);
        default: return launch_gemm_simt_t<__nv_bfloat16>(pv, sv, W, x, s_in, s_parts, y, fuse, st);
    }
}

}  // namespace lora
