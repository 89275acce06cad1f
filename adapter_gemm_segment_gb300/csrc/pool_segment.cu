// Adapter pool (slot table + zero-padded slabs) and the stable segment builder.
//
// Pool: "LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排" (blog.lonae.com) -- hot adapters
// stay resident in GPU memory (adapter storage pool) and low-rank adapters are zero-padded
// to the high rank so that their shapes line up (tensor-concatenation paragraph).  Mount
// refusals (slot busy, rank too large) follow the xpshop.cn article 492 case study,
// section 三 (refuse a mount rather than squeeze others; refuse mismatched versions).
//
// Segments: the adapter-level bucket of the two-level bucketing on the blog.lonae.com page,
// realised as a stable counting sort of token positions by slot (-1 first), plus the
// default-deny validation of "Multi-LoRA 在线服务隔离" (ai.codenodex.com), section
// "请求身份决定适配器，而非客户端参数": an unknown or unmounted slot is an explicit error.
#include <algorithm>
#include <functional>
#include <vector>
#include <cstdio>
#include <cstring>
#include <new>

#include "common.cuh"

namespace lora {

struct PoolLayout {
    size_t table_off, A_off, B_off, total;
};

static PoolLayout pool_layout(const lora_pool_desc& d) {
    PoolLayout L;
    const size_t es = dtype_size(d.dtype);
    L.table_off = 0;
    L.A_off = align256(sizeof(SlotEntry) * (size_t)d.n_slots);
    L.B_off = L.A_off + align256((size_t)d.n_slots * d.r_max * d.h_in * es);
    L.total = L.B_off + align256((size_t)d.n_slots * d.h_out * d.r_max * es);
    return L;
}

static int check_desc(const lora_pool_desc* d) {
    if (!d) return set_error(LORA_EINVAL, "desc is NULL");
    if (d->dtype != LORA_F32 && d->dtype != LORA_F16 && d->dtype != LORA_BF16)
        return set_error(LORA_EINVAL, "unknown dtype %d", d->dtype);
    if (d->h_in < 1 || d->h_out < 1) return set_error(LORA_EINVAL, "h_in/h_out must be >= 1");
    if (d->n_slots < 1 || d->n_slots > kMaxSlots)
        return set_error(LORA_EINVAL, "n_slots %d outside [1, %d]", d->n_slots, kMaxSlots);
    if (d->r_max < 1 || d->r_max > kMaxRank)
        return set_error(LORA_EINVAL, "r_max %d outside [1, %d]", d->r_max, kMaxRank);
    if (d->dtype != LORA_F32) {
        if (d->h_in % 8 || d->h_out % 8)
            return set_error(LORA_EINVAL, "16-bit pools need h_in and h_out multiples of 8 (got %d, %d)",
                             d->h_in, d->h_out);
        if (d->r_max % 8) return set_error(LORA_EINVAL, "16-bit pools need r_max a multiple of 8");
    }
    return LORA_OK;
}

PoolView pool_view(const lora_pool_t p) {
    PoolView v;
    v.table = static_cast<const SlotEntry*>(p->table);
    v.A = p->A;
    v.B = p->B;
    v.h_in = p->desc.h_in;
    v.h_out = p->desc.h_out;
    v.R = p->desc.r_max;
    v.S = p->desc.n_slots;
    v.dtype = p->desc.dtype;
    lora_pool* q = const_cast<lora_pool*>(p);
    if (q->top_dirty) {
        const int R8 = (p->desc.r_max + 7) / 8;
        std::vector<int> c(p->desc.n_slots, R8);
        for (int s = 0; s < p->desc.n_slots; ++s)
            if (p->mounted[s]) c[s] = std::min(R8, (p->ranks[s] + 7) / 8);
        const int k = std::min<int>(32, (int)c.size());
        std::partial_sort(c.begin(), c.begin() + k, c.end(), std::greater<int>());
        q->top_chunks[0] = 0;
        for (int i = 1; i <= 32; ++i) q->top_chunks[i] = q->top_chunks[i - 1] + (i <= k ? c[i - 1] : 0);
        q->top_dirty = false;
    }
    for (int i = 0; i <= 32; ++i) v.top_chunks[i] = p->top_chunks[i];
    return v;
}

// ---- mount kernel: copy with zero padding, then publish the slot entry ------------------------
template <typename T>
__global__ void pool_load_kernel(const T* __restrict__ A_src, const T* __restrict__ B_src, T* __restrict__ A_dst,
                                 T* __restrict__ B_dst, int r, int R, int h_in, int h_out, SlotEntry* entry,
                                 float scale) {
    const size_t nA = (size_t)R * h_in, nB = (size_t)h_out * R;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nA; i += stride) {
        const size_t j = i / h_in;
        A_dst[i] = j < (size_t)r ? A_src[i] : T(0.0f);
    }
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nB; i += stride) {
        const size_t o = i / R, j = i % R;
        B_dst[i] = j < (size_t)r ? B_src[o * r + j] : T(0.0f);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        entry->rank = r;
        entry->scale = scale;
        entry->state = kSlotReady;
    }
}

// ---- batched mount (16-bit pools): up to kLoadBatch slots per launch, 16-byte copies ---------
constexpr int kLoadBatch = 32;
struct LoadEntry {
    const void* A;  // [rank, h_in]
    const void* B;  // [h_out, rank]
    int slot, rank;
    float scale;
};
struct LoadBatch {
    LoadEntry e[kLoadBatch];
};

// grid (CTAs per slot, slots of the batch).  A slot's A rows and B rows are copied in 16-byte
// units (8 elements) with the zero padding of rank .. r_max; B rows whose rank is not a
// multiple of 8 are gathered element by element.  The source may be device memory or host
// memory the device can read.
template <typename T>
__global__ void __launch_bounds__(256)
pool_load_batch_kernel(const __grid_constant__ LoadBatch b, char* __restrict__ A_base, char* __restrict__ B_base,
                       SlotEntry* __restrict__ table, int R, int h_in, int h_out) {
    const LoadEntry& e = b.e[blockIdx.y];
    uint4* A_dst = reinterpret_cast<uint4*>(A_base + (size_t)e.slot * R * h_in * sizeof(T));
    uint4* B_dst = reinterpret_cast<uint4*>(B_base + (size_t)e.slot * h_out * R * sizeof(T));
    const size_t cpr_a = h_in / 8, cpr_b = R / 8;
    const size_t nA = (size_t)R * cpr_a, nB = (size_t)h_out * cpr_b;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < nA + nB; u += stride) {
        if (u < nA) {
            A_dst[u] = u / cpr_a < (size_t)e.rank ? static_cast<const uint4*>(e.A)[u] : zero;
        } else {
            const size_t v = u - nA, o = v / cpr_b;
            const int j0 = (int)(v - o * cpr_b) * 8;
            uint4 val = zero;
            if (j0 < e.rank) {
                const T* src = static_cast<const T*>(e.B) + o * e.rank + j0;
                if (e.rank % 8 == 0) {
                    val = *reinterpret_cast<const uint4*>(src);
                } else {
                    __align__(16) T tmp[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) tmp[k] = j0 + k < e.rank ? src[k] : T(0.0f);
                    val = *reinterpret_cast<const uint4*>(tmp);
                }
            }
            B_dst[v] = val;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        SlotEntry* t = table + e.slot;
        t->rank = e.rank;
        t->scale = e.scale;
        t->state = kSlotReady;
    }
}

// ---- segment builder -----------------------------------------------------------------------
// One CTA of 1024 threads.  Shared memory: cnt[K], off[K], rk[K], wcnt[32][K] (uint16) with
// K = S + 1 keys (key k+1 for slot k, key 0 for idx -1); rk[k] = rank of the slot of key k if
// it is mounted, else 0 (copied from the slot table once, so no token waits on a table read).
constexpr int kSegThreads = 1024;
constexpr int kItemTok = 4;  // sorted tokens per shrink work item

__global__ void __launch_bounds__(kSegThreads, 1)
segment_kernel(const int32_t* __restrict__ idx, int n, const SlotEntry* __restrict__ table, int S,
               int32_t* __restrict__ perm, int32_t* __restrict__ seg_start, int32_t* __restrict__ seg_slot,
               int32_t* __restrict__ nseg_out, int32_t* __restrict__ status, int32_t* __restrict__ idx_copy,
               int32_t* __restrict__ items) {
    extern __shared__ __align__(16) int smem_i[];
    const int K = S + 1;
    int* cnt = smem_i;
    int* off = cnt + K;
    int* rk = off + K;
    uint16_t* wcnt = reinterpret_cast<uint16_t*>(rk + K);
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int U = 4;  // tokens per thread whose loads are issued together

    pdl_wait();  // idx and the slot table may come from earlier kernels in the stream
    // hand-off words of the decode kernels (the x-ready word and its read count); each fused
    // decode GEMM leaves them at zero for the next linear over these segments
    if (tid == 0) {
        nseg_out[kXreadyWord] = 0;
        nseg_out[kXreadyCount] = 0;
    }
    for (int i = tid; i < K; i += kSegThreads) {
        cnt[i] = 0;
        const SlotEntry e = i > 0 ? table[i - 1] : SlotEntry{0, 0, 0.f, 0};
        rk[i] = (i > 0 && e.state == kSlotReady) ? max(e.rank, 1) : 0;
    }
    for (int i = tid; i < 32 * K; i += kSegThreads) wcnt[i] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();

    // 1. validate + histogram
    for (int t0 = tid; t0 < n; t0 += U * kSegThreads) {
        int kk[U];
#pragma unroll
        for (int u = 0; u < U; ++u) kk[u] = t0 + u * kSegThreads < n ? idx[t0 + u * kSegThreads] : -1;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = t0 + u * kSegThreads, k = kk[u];
            if (t >= n) continue;
            idx_copy[t] = k;
            const bool ok = (k >= -1) && (k < S) && (k < 0 || rk[k + 1] > 0);
            if (!ok) bad = 1;
            else atomicAdd(&cnt[k + 1], 1);
        }
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) {
            *status = LORA_EIDX;
            nseg_out[0] = 0;
            nseg_out[1] = 0;
            seg_start[0] = 0;
        }
        pdl_trigger();
        return;
    }

    // 2. exclusive scan of the key counts + compaction of the non-empty keys into segments
    if (warp == 0) {
        int run = 0, segs = 0;
        for (int base = 0; base < K; base += 32) {
            const int i = base + lane;
            const int c = i < K ? cnt[i] : 0;
            int v = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += u;
            }
            const int excl = run + v - c;
            if (i < K) off[i] = excl;
            const unsigned nz = __ballot_sync(0xffffffffu, c > 0);
            if (c > 0) {
                const int si = segs + __popc(nz & ((1u << lane) - 1u));
                seg_start[si] = excl;
                seg_slot[si] = i - 1;
            }
            run += __shfl_sync(0xffffffffu, v, 31);
            segs += __popc(nz);
        }
        if (lane == 0) {
            seg_start[segs] = n;
            *nseg_out = segs;
            *status = LORA_OK;
        }
    }
    __syncthreads();

    // 3. stable scatter, 1024 tokens at a time in original order.  Inside a chunk a token's
    //    rank among equal keys = (equal keys in earlier warps) + (equal keys in earlier lanes).
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int base = 0; base < n; base += kSegThreads) {
        const int t = base + tid;
        const int key = t < n ? idx[t] + 1 : K;  // K = sentinel for lanes past the end
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & lt_mask);
        const bool leader = (__ffs(peers) - 1) == lane;
        if (t < n && leader) wcnt[warp * K + key] = (uint16_t)__popc(peers);
        __syncthreads();
        if (t < n) {
            int pre = 0;
            for (int w = 0; w < warp; ++w) pre += wcnt[w * K + key];
            perm[off[key] + pre + rank] = t;
        }
        __syncthreads();
        if (t < n && leader) {
            atomicAdd(&off[key], __popc(peers));
            wcnt[warp * K + key] = 0;
        }
        __syncthreads();
    }

    // 4. shrink work items: key k >= 1 (slot k-1) gives ceil(cnt[k] / 4) runs of up to 4
    //    consecutive sorted tokens; off[k] is now the end of key k's range
    int* ibase = reinterpret_cast<int*>(wcnt);  // [K], free again
    if (warp == 0) {
        int run = 0;
        for (int base = 0; base < K; base += 32) {
            const int i = base + lane;
            const int c = (i < K && i > 0) ? (cnt[i] + kItemTok - 1) / kItemTok : 0;
            int v = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, d);
                if (lane >= d) v += u;
            }
            if (i < K) ibase[i] = run + v - c;
            run += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) nseg_out[1] = run;
    }
    __syncthreads();
    for (int j0 = tid; j0 < n; j0 += U * kSegThreads) {
        int tt[U];
#pragma unroll
        for (int u = 0; u < U; ++u) tt[u] = j0 + u * kSegThreads < n ? perm[j0 + u * kSegThreads] : 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * kSegThreads, t = tt[u];
            if (j >= n) continue;
            // the key of sorted position j: the first key whose range ends past j
            int lo = 0, hi = K - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (off[mid] > j) hi = mid;
                else lo = mid + 1;
            }
            const int key = lo;
            if (key == 0) continue;
            const int rel = j - (off[key] - cnt[key]);
            int32_t* it = items + (size_t)(ibase[key] + rel / kItemTok) * 8;
            it[2 + rel % kItemTok] = t;
            if (rel % kItemTok == 0) {
                const int nt = min(kItemTok, cnt[key] - rel);
                it[0] = key - 1;
                it[1] = nt;
                for (int v = nt; v < kItemTok; ++v) it[2 + v] = t;  // padding: a valid token
                it[6] = rk[key];                                      // the adapter's true rank
                it[7] = 0;
            }
        }
    }
    pdl_trigger();
}

struct SegLayout {
    size_t perm, seg_start, seg_slot, nseg, status, idx, items, total;
};

static SegLayout seg_layout(int n, int S) {
    SegLayout L;
    size_t o = 0;
    L.perm = o;
    o += align256(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    L.seg_start = o;
    o += align256(sizeof(int32_t) * (size_t)(S + 2));
    L.seg_slot = o;
    o += align256(sizeof(int32_t) * (size_t)(S + 1));
    L.nseg = o;
    o += 256;
    L.status = o;
    o += 256;
    L.idx = o;
    o += align256(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    L.items = o;
    o += align256(sizeof(int32_t) * 8 * (size_t)(n > 0 ? n : 1));
    L.total = o;
    return L;
}

}  // namespace lora

using namespace lora;

extern "C" {

int lora_pool_bytes(const lora_pool_desc* desc, size_t* bytes) {
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!bytes) return set_error(LORA_EINVAL, "bytes is NULL");
    *bytes = pool_layout(*desc).total;
    return LORA_OK;
}

int lora_pool_create(const lora_pool_desc* desc, void* dev_mem, size_t bytes, void* stream, lora_pool_t* out) {
    int rc = check_desc(desc);
    if (rc) return rc;
    if (!dev_mem || !out) return set_error(LORA_EINVAL, "dev_mem/out is NULL");
    if (reinterpret_cast<uintptr_t>(dev_mem) % 256) return set_error(LORA_EINVAL, "dev_mem must be 256-byte aligned");
    const PoolLayout L = pool_layout(*desc);
    if (bytes < L.total)
        return set_error(LORA_ENOSPACE, "pool needs %zu bytes, got %zu", L.total, bytes);
    LORA_CUDA_TRY(cudaMemsetAsync(dev_mem, 0, L.total, (cudaStream_t)stream));
    lora_pool* p = new (std::nothrow) lora_pool();
    if (!p) return set_error(LORA_EINVAL, "out of host memory");
    p->desc = *desc;
    p->base = static_cast<char*>(dev_mem);
    p->bytes = bytes;
    p->table = p->base + L.table_off;
    p->A = p->base + L.A_off;
    p->B = p->base + L.B_off;
    p->mounted.assign(desc->n_slots, 0);
    p->ranks.assign(desc->n_slots, 0);
    cudaPointerAttributes attr;  // the device that holds dev_mem (else the current device)
    if (cudaPointerGetAttributes(&attr, dev_mem) == cudaSuccess &&
        (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged))
        p->device = attr.device;
    else if (cudaGetDevice(&p->device) != cudaSuccess)
        p->device = -1;
    *out = p;
    return LORA_OK;
}

int lora_pool_destroy(lora_pool_t pool) {
    delete pool;
    return LORA_OK;
}

int lora_pool_load_slot(lora_pool_t pool, int slot, const void* A_dev, const void* B_dev, int rank, float alpha,
                        void* stream) {
    if (!pool) return set_error(LORA_EINVAL, "pool is NULL");
    const lora_pool_desc& d = pool->desc;
    if (slot < 0 || slot >= d.n_slots) return set_error(LORA_ESLOT, "slot %d outside [0, %d)", slot, d.n_slots);
    if (rank < 1 || rank > d.r_max) return set_error(LORA_ERANK, "rank %d outside [1, %d]", rank, d.r_max);
    if (!A_dev || !B_dev) return set_error(LORA_EINVAL, "A/B is NULL");
    if (pool->mounted[slot]) return set_error(LORA_EBUSY, "slot %d already holds an adapter", slot);
    const size_t es = dtype_size(d.dtype);
    char* A_dst = static_cast<char*>(pool->A) + (size_t)slot * d.r_max * d.h_in * es;
    char* B_dst = static_cast<char*>(pool->B) + (size_t)slot * d.h_out * d.r_max * es;
    const float scale = alpha / (float)rank;
    const size_t work = (size_t)d.r_max * d.h_in + (size_t)d.h_out * d.r_max;
    const int threads = 256;
    const int blocks = (int)std::min<size_t>((work + threads - 1) / threads, 4096);
    cudaStream_t st = (cudaStream_t)stream;
    SlotEntry* e = static_cast<SlotEntry*>(pool->table) + slot;
    int r_arg = rank, R_arg = d.r_max, hi = d.h_in, ho = d.h_out;
    float sc = scale;
    void* args[] = {(void*)&A_dev, (void*)&B_dev, (void*)&A_dst, (void*)&B_dst, (void*)&r_arg,
                    (void*)&R_arg, (void*)&hi, (void*)&ho, (void*)&e, (void*)&sc};
    const void* fn = d.dtype == LORA_F32   ? (const void*)pool_load_kernel<float>
                     : d.dtype == LORA_F16 ? (const void*)pool_load_kernel<__half>
                                           : (const void*)pool_load_kernel<__nv_bfloat16>;
    // the launch's own status (an error left over from earlier work is not reported as ours)
    LORA_CUDA_TRY(cudaLaunchKernel(fn, dim3(blocks), dim3(threads), args, 0, st));
    count_launch();
    pool->mounted[slot] = 1;
    pool->ranks[slot] = rank;
    pool->top_dirty = true;
    return LORA_OK;
}

int lora_pool_load_slots(lora_pool_t pool, int count, const int* slots, const void* const* A, const void* const* B,
                         const int* ranks, const float* alphas, void* stream) {
    if (!pool) return set_error(LORA_EINVAL, "pool is NULL");
    if (count < 0) return set_error(LORA_EINVAL, "count < 0");
    if (count == 0) return LORA_OK;
    if (!slots || !A || !B || !ranks || !alphas) return set_error(LORA_EINVAL, "slots/A/B/ranks/alphas is NULL");
    const lora_pool_desc& d = pool->desc;
    std::vector<char> seen(d.n_slots, 0);
    bool vec = d.dtype != LORA_F32;
    for (int i = 0; i < count; ++i) {  // validate everything before anything is enqueued
        const int slot = slots[i], rank = ranks[i];
        if (slot < 0 || slot >= d.n_slots) return set_error(LORA_ESLOT, "slot %d outside [0, %d)", slot, d.n_slots);
        if (rank < 1 || rank > d.r_max) return set_error(LORA_ERANK, "rank %d outside [1, %d]", rank, d.r_max);
        if (!A[i] || !B[i]) return set_error(LORA_EINVAL, "A/B of entry %d is NULL", i);
        if (pool->mounted[slot] || seen[slot]) return set_error(LORA_EBUSY, "slot %d already holds an adapter", slot);
        seen[slot] = 1;
        if ((reinterpret_cast<uintptr_t>(A[i]) | reinterpret_cast<uintptr_t>(B[i])) % 16) vec = false;
    }
    if (!vec) {  // float32 pools or unaligned sources: one mount kernel per slot
        for (int i = 0; i < count; ++i) {
            const int rc = lora_pool_load_slot(pool, slots[i], A[i], B[i], ranks[i], alphas[i], stream);
            if (rc) return rc;
        }
        return LORA_OK;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const size_t units = (size_t)d.r_max * (d.h_in / 8) + (size_t)d.h_out * (d.r_max / 8);
    const int per_slot = (int)std::min<size_t>((units + 255) / 256, 128);
    const void* fn = d.dtype == LORA_F16 ? (const void*)pool_load_batch_kernel<__half>
                                         : (const void*)pool_load_batch_kernel<__nv_bfloat16>;
    for (int c0 = 0; c0 < count; c0 += kLoadBatch) {
        const int nb = std::min(kLoadBatch, count - c0);
        LoadBatch b;
        memset(&b, 0, sizeof(b));
        for (int i = 0; i < nb; ++i)
            b.e[i] = LoadEntry{A[c0 + i], B[c0 + i], slots[c0 + i], ranks[c0 + i], alphas[c0 + i] / (float)ranks[c0 + i]};
        char* Ab = static_cast<char*>(pool->A);
        char* Bb = static_cast<char*>(pool->B);
        SlotEntry* tb = static_cast<SlotEntry*>(pool->table);
        int R = d.r_max, hi = d.h_in, ho = d.h_out;
        void* args[] = {(void*)&b, (void*)&Ab, (void*)&Bb, (void*)&tb, (void*)&R, (void*)&hi, (void*)&ho};
        LORA_CUDA_TRY(cudaLaunchKernel(fn, dim3(per_slot, nb), dim3(256), args, 0, st));
        count_launch();
        for (int i = 0; i < nb; ++i) {
            pool->mounted[slots[c0 + i]] = 1;
            pool->ranks[slots[c0 + i]] = ranks[c0 + i];
        }
        pool->top_dirty = true;
    }
    return LORA_OK;
}

int lora_pool_unload_slot(lora_pool_t pool, int slot, void* stream) {
    if (!pool) return set_error(LORA_EINVAL, "pool is NULL");
    if (slot < 0 || slot >= pool->desc.n_slots)
        return set_error(LORA_ESLOT, "slot %d outside [0, %d)", slot, pool->desc.n_slots);
    LORA_CUDA_TRY(cudaMemsetAsync(static_cast<SlotEntry*>(pool->table) + slot, 0, sizeof(SlotEntry), (cudaStream_t)stream));
    pool->mounted[slot] = 0;
    pool->ranks[slot] = 0;
    pool->top_dirty = true;
    return LORA_OK;
}

int lora_segment_workspace_bytes(int n_tokens, int n_slots, size_t* bytes) {
    if (n_tokens < 0) return set_error(LORA_EINVAL, "n_tokens < 0");
    if (n_slots < 1 || n_slots > kMaxSlots) return set_error(LORA_EINVAL, "n_slots outside [1, %d]", kMaxSlots);
    if (!bytes) return set_error(LORA_EINVAL, "bytes is NULL");
    *bytes = seg_layout(n_tokens, n_slots).total;
    return LORA_OK;
}

int lora_segment(const int32_t* idx_dev, int n_tokens, lora_pool_t pool, void* ws_dev, size_t ws_bytes,
                 lora_segments* out, void* stream) {
    if (!pool || !ws_dev || !out) return set_error(LORA_EINVAL, "pool/ws/out is NULL");
    if (n_tokens < 0) return set_error(LORA_EINVAL, "n_tokens < 0");
    if (n_tokens > 0 && !idx_dev) return set_error(LORA_EINVAL, "idx is NULL");
    if (reinterpret_cast<uintptr_t>(ws_dev) % 256) return set_error(LORA_EINVAL, "ws must be 256-byte aligned");
    const int S = pool->desc.n_slots;
    const SegLayout L = seg_layout(n_tokens, S);
    if (ws_bytes < L.total) return set_error(LORA_ENOSPACE, "segment workspace needs %zu bytes, got %zu", L.total, ws_bytes);
    char* w = static_cast<char*>(ws_dev);
    out->perm_dev = reinterpret_cast<int32_t*>(w + L.perm);
    out->seg_start_dev = reinterpret_cast<int32_t*>(w + L.seg_start);
    out->seg_slot_dev = reinterpret_cast<int32_t*>(w + L.seg_slot);
    out->nseg_dev = reinterpret_cast<int32_t*>(w + L.nseg);
    out->status_dev = reinterpret_cast<int32_t*>(w + L.status);
    out->idx_dev = reinterpret_cast<int32_t*>(w + L.idx);
    out->items_dev = reinterpret_cast<int32_t*>(w + L.items);
    out->n_tokens = n_tokens;
    out->n_slots = S;

    const int K = S + 1;
    const size_t smem = sizeof(int) * 3 * (size_t)K + sizeof(uint16_t) * 32 * (size_t)K;
    static bool attr_set = false;  // one device per process is the supported configuration
    if (!attr_set) {
        LORA_CUDA_TRY(cudaFuncSetAttribute(segment_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)(sizeof(int) * 3 * (kMaxSlots + 1) +
                                                 sizeof(uint16_t) * 32 * (kMaxSlots + 1))));
        attr_set = true;
    }
    const int32_t* idx_arg = idx_dev;
    int n_arg = n_tokens;
    const SlotEntry* table_arg = static_cast<const SlotEntry*>(pool->table);
    int S_arg = S;
    void* args[] = {(void*)&idx_arg, (void*)&n_arg, (void*)&table_arg, (void*)&S_arg, (void*)&out->perm_dev,
                    (void*)&out->seg_start_dev, (void*)&out->seg_slot_dev, (void*)&out->nseg_dev,
                    (void*)&out->status_dev, (void*)&out->idx_dev, (void*)&out->items_dev};
    LORA_CUDA_TRY(launch_pdl((const void*)segment_kernel, dim3(1), dim3(kSegThreads), smem, (cudaStream_t)stream, args));
    return LORA_OK;
}

int lora_segment_status(const lora_segments* seg, void* stream, int* status) {
    if (!seg || !status) return set_error(LORA_EINVAL, "seg/status is NULL");
    int32_t v = 0;
    LORA_CUDA_TRY(cudaMemcpyAsync(&v, seg->status_dev, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream));
    LORA_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    *status = v;
    return LORA_OK;
}

}  // extern "C"
