// Adapter loader: mounts on a copy stream that run while compute proceeds, and draining
// remounts.
//
// "LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排" (blog.lonae.com), adapter-loader
// paragraph: the loader moves adapters from the storage pool into the execution unit's buffers
// without blocking inference -- asynchronous double buffering, one copy serving the requests
// at hand while the next candidate adapter is fetched in the background (pinned host memory,
// asynchronous copies).  xpshop.cn article 492, section 三: an adapter is unloaded in
// "draining" mode -- requests already running on it finish first.
//
// Here the double buffer is the pool's slots themselves: the next adapters go into free (or
// drained) slots on the loader's copy stream while kernels on the compute streams read the
// other slots.  Mounting reads the caller's pinned host memory directly (lora_pool_load_slots;
// over NVLink-C2C on GB300), so there is no staging buffer.  Ordering is by CUDA events only,
// with no host synchronisation:
//   - every mount records a per-slot "mounted" event on the copy stream; lora_loader_acquire
//     makes a compute stream wait for it before the first batch that names the slot;
//   - lora_loader_release records, on a compute stream, a fence after the work that may read
//     a slot; a later remount of that slot first makes the copy stream wait for every fence
//     recorded since the slot's last mount (draining), then unmounts and mounts.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"

struct lora_loader {
    std::vector<lora_pool_t> pools;
    cudaStream_t copy = nullptr;
    int n_slots = 0;
    // Events are shared by every slot a call names (one record per call) and recycled once no
    // slot refers to them: a stream wait holds the record it was given, so re-recording a
    // recycled event later does not disturb waits already enqueued.
    struct Ev {
        cudaEvent_t e;
        int refs;
    };
    std::vector<Ev> evs;
    std::vector<int> mounted_ev;           // per slot: event of its last mount (-1: none)
    std::vector<std::vector<int>> fences;  // per slot: release fences since its last mount
    uint64_t mounts = 0, drained_fences = 0;
};

using namespace lora;

namespace {

// ---- one mount kernel for every (pool, slot) of a call (16-bit pools, 16-byte aligned sources)
// A call mounts an adapter into the same slot of every pool it targets (the q, k, v, ... of
// every layer): one launch covers them all instead of one per pool.  Each entry carries its
// own destination and shape; A rows and B rows are copied in 16-byte units (8 elements) with
// the zero padding of rank .. r_max, and B rows whose rank is not a multiple of 8 are gathered
// element by element.  The raw 16-bit patterns are copied, so fp16 and bf16 share the code.
constexpr int kMountBatch = 48;
struct MountEntry {
    const void* A;       // [rank, h_in] source
    const void* B;       // [h_out, rank] source
    uint4* A_dst;        // [R, h_in] slot in the pool's A slab
    uint4* B_dst;        // [h_out, R] slot in the pool's B slab
    SlotEntry* entry;    // the slot's table entry
    int rank, R, h_in, h_out;
    float scale;
};
struct MountBatch {
    MountEntry e[kMountBatch];
};
static_assert(sizeof(MountBatch) <= 4000, "kernel parameter block");

__global__ void __launch_bounds__(256) loader_mount_kernel(const __grid_constant__ MountBatch b) {
    const MountEntry& e = b.e[blockIdx.y];
    const size_t cpr_a = e.h_in / 8, cpr_b = e.R / 8;
    const size_t nA = (size_t)e.R * cpr_a, nB = (size_t)e.h_out * cpr_b;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t u = (size_t)blockIdx.x * blockDim.x + threadIdx.x; u < nA + nB; u += stride) {
        if (u < nA) {
            e.A_dst[u] = u / cpr_a < (size_t)e.rank ? static_cast<const uint4*>(e.A)[u] : zero;
        } else {
            const size_t v = u - nA, o = v / cpr_b;
            const int j0 = (int)(v - o * cpr_b) * 8;
            uint4 val = zero;
            if (j0 < e.rank) {
                const uint16_t* src = static_cast<const uint16_t*>(e.B) + o * e.rank + j0;
                if (e.rank % 8 == 0) {
                    val = *reinterpret_cast<const uint4*>(src);
                } else {
                    __align__(16) uint16_t tmp[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) tmp[k] = j0 + k < e.rank ? src[k] : uint16_t(0);
                    val = *reinterpret_cast<const uint4*>(tmp);
                }
            }
            e.B_dst[v] = val;
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        e.entry->rank = e.rank;
        e.entry->scale = e.scale;
        e.entry->state = kSlotReady;
    }
}

// Mount entry (p, i) of a validated call with one kernel per kMountBatch entries.  Returns
// LORA_EUNSUP (nothing enqueued) when a pool is float32 or a source is not 16-byte aligned.
int mount_batched(lora_loader* L, int count, const int* slots, const void* const* A, const void* const* B,
                  const int* ranks, const float* alphas) {
    const int np = static_cast<int>(L->pools.size());
    size_t max_units = 0;
    for (int p = 0; p < np; ++p) {
        const lora_pool_desc& d = L->pools[p]->desc;
        if (d.dtype == LORA_F32) return LORA_EUNSUP;
        for (int i = 0; i < count; ++i)
            if ((reinterpret_cast<uintptr_t>(A[p * count + i]) | reinterpret_cast<uintptr_t>(B[p * count + i])) % 16)
                return LORA_EUNSUP;
        max_units = std::max(max_units, (size_t)d.r_max * (d.h_in / 8) + (size_t)d.h_out * (d.r_max / 8));
    }
    const int per_slot = (int)std::min<size_t>((max_units + 255) / 256, 128);
    MountBatch b;
    int nb = 0;
    auto flush = [&]() -> int {
        if (nb == 0) return LORA_OK;
        void* args[] = {(void*)&b};
        LORA_CUDA_TRY(cudaLaunchKernel((const void*)loader_mount_kernel, dim3(per_slot, nb), dim3(256), args, 0, L->copy));
        count_launch();
        nb = 0;
        return LORA_OK;
    };
    memset(&b, 0, sizeof(b));
    for (int p = 0; p < np; ++p) {
        lora_pool_t pool = L->pools[p];
        const lora_pool_desc& d = pool->desc;
        for (int i = 0; i < count; ++i) {
            const int k = p * count + i, slot = slots[i];
            MountEntry& e = b.e[nb++];
            e.A = A[k];
            e.B = B[k];
            e.A_dst = reinterpret_cast<uint4*>(static_cast<char*>(pool->A) + (size_t)slot * d.r_max * d.h_in * 2);
            e.B_dst = reinterpret_cast<uint4*>(static_cast<char*>(pool->B) + (size_t)slot * d.h_out * d.r_max * 2);
            e.entry = static_cast<SlotEntry*>(pool->table) + slot;
            e.rank = ranks[k];
            e.R = d.r_max;
            e.h_in = d.h_in;
            e.h_out = d.h_out;
            e.scale = alphas[k] / (float)ranks[k];
            pool->mounted[slot] = 1;
            pool->ranks[slot] = ranks[k];
            pool->top_dirty = true;
            if (nb == kMountBatch) {
                const int rc = flush();
                if (rc) return rc;
            }
        }
    }
    return flush();
}

// An event no slot refers to (created on demand).
int take_event(lora_loader* L, int* id) {
    for (size_t k = 0; k < L->evs.size(); ++k)
        if (L->evs[k].refs == 0) {
            *id = static_cast<int>(k);
            return LORA_OK;
        }
    cudaEvent_t e;
    LORA_CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    L->evs.push_back({e, 0});
    *id = static_cast<int>(L->evs.size()) - 1;
    return LORA_OK;
}

int check_slots(const lora_loader* L, int count, const int* slots) {
    if (count < 0 || (count > 0 && !slots)) return set_error(LORA_EINVAL, "bad slot list");
    std::vector<uint8_t> seen(L->n_slots, 0);
    for (int i = 0; i < count; ++i) {
        if (slots[i] < 0 || slots[i] >= L->n_slots)
            return set_error(LORA_ESLOT, "slot %d outside [0, %d)", slots[i], L->n_slots);
        if (seen[slots[i]]) return set_error(LORA_EBUSY, "slot %d named twice", slots[i]);
        seen[slots[i]] = 1;
    }
    return LORA_OK;
}

// Make `stream` wait once for each distinct event among ids.
int wait_distinct(lora_loader* L, std::vector<int>& ids, cudaStream_t stream) {
    std::sort(ids.begin(), ids.end());
    ids.erase(std::unique(ids.begin(), ids.end()), ids.end());
    for (int id : ids) LORA_CUDA_TRY(cudaStreamWaitEvent(stream, L->evs[id].e, 0));
    return LORA_OK;
}

}  // namespace

extern "C" {

int lora_loader_create(int count, const lora_pool_t* pools, void* copy_stream, lora_loader_t* out) {
    if (!out) return set_error(LORA_EINVAL, "out is NULL");
    if (count < 1 || !pools) return set_error(LORA_EINVAL, "a loader needs at least one pool");
    for (int p = 0; p < count; ++p) {
        if (!pools[p]) return set_error(LORA_EINVAL, "pools[%d] is NULL", p);
        if (pools[p]->desc.n_slots != pools[0]->desc.n_slots)
            return set_error(LORA_EINVAL, "pool %d has %d slots, pool 0 has %d", p, pools[p]->desc.n_slots,
                             pools[0]->desc.n_slots);
    }
    lora_loader* L = new (std::nothrow) lora_loader();
    if (!L) return set_error(LORA_EINVAL, "out of host memory");
    L->pools.assign(pools, pools + count);
    L->copy = static_cast<cudaStream_t>(copy_stream);
    L->n_slots = pools[0]->desc.n_slots;
    L->mounted_ev.assign(L->n_slots, -1);
    L->fences.resize(L->n_slots);
    *out = L;
    return LORA_OK;
}

int lora_loader_destroy(lora_loader_t L) {
    if (!L) return LORA_OK;
    for (auto& ev : L->evs) cudaEventDestroy(ev.e);
    delete L;
    return LORA_OK;
}

int lora_loader_mount(lora_loader_t L, int count, const int* slots, const void* const* A, const void* const* B,
                      const int* ranks, const float* alphas) {
    if (!L) return set_error(LORA_EINVAL, "loader is NULL");
    int rc = check_slots(L, count, slots);
    if (rc) return rc;
    if (count == 0) return LORA_OK;
    if (!A || !B || !ranks || !alphas) return set_error(LORA_EINVAL, "A/B/ranks/alphas is NULL");
    const int np = static_cast<int>(L->pools.size());
    // validate everything before enqueueing anything
    for (int p = 0; p < np; ++p) {
        const lora_pool_desc& d = L->pools[p]->desc;
        for (int i = 0; i < count; ++i) {
            const int k = p * count + i;
            if (!A[k] || !B[k]) return set_error(LORA_EINVAL, "pool %d, slot %d: A/B is NULL", p, slots[i]);
            if (ranks[k] < 1 || ranks[k] > d.r_max)
                return set_error(LORA_ERANK, "pool %d, slot %d: rank %d outside [1, %d]", p, slots[i], ranks[k],
                                 d.r_max);
        }
    }
    int mev = -1;
    rc = take_event(L, &mev);
    if (rc) return rc;
    // drain: the copy stream waits for every fence recorded on the slots since their last mount
    std::vector<int> waits;
    for (int i = 0; i < count; ++i)
        for (int id : L->fences[slots[i]]) waits.push_back(id);
    rc = wait_distinct(L, waits, L->copy);
    if (rc) return rc;
    for (int i = 0; i < count; ++i) {
        for (int id : L->fences[slots[i]]) --L->evs[id].refs;
        L->drained_fences += L->fences[slots[i]].size();
        L->fences[slots[i]].clear();
    }
    // Remounted slots: nothing reads them any more (drained; new readers acquire the mount
    // below), and the mount kernels rewrite the whole padded slot and its table entry, so only
    // the pools' host records are reset -- no separate unmount on the device.
    for (int p = 0; p < np; ++p) {
        lora_pool_t pool = L->pools[p];
        for (int i = 0; i < count; ++i)
            if (pool->mounted[slots[i]]) {
                pool->mounted[slots[i]] = 0;
                pool->ranks[slots[i]] = 0;
                pool->top_dirty = true;
            }
    }
    rc = mount_batched(L, count, slots, A, B, ranks, alphas);
    if (rc == LORA_EUNSUP) {  // float32 pools or unaligned sources: the pools' own mounts
        for (int p = 0; p < np; ++p) {
            rc = lora_pool_load_slots(L->pools[p], count, slots, A + (size_t)p * count, B + (size_t)p * count,
                                      ranks + (size_t)p * count, alphas + (size_t)p * count, L->copy);
            if (rc) return rc;
        }
    } else if (rc) {
        return rc;
    }
    LORA_CUDA_TRY(cudaEventRecord(L->evs[mev].e, L->copy));
    for (int i = 0; i < count; ++i) {
        int& old = L->mounted_ev[slots[i]];
        if (old >= 0) --L->evs[old].refs;
        old = mev;
        ++L->evs[mev].refs;
    }
    L->mounts += (uint64_t)count;
    return LORA_OK;
}

int lora_loader_acquire(lora_loader_t L, int count, const int* slots, void* stream) {
    if (!L) return set_error(LORA_EINVAL, "loader is NULL");
    int rc = check_slots(L, count, slots);
    if (rc) return rc;
    std::vector<int> waits;
    for (int i = 0; i < count; ++i)
        if (L->mounted_ev[slots[i]] >= 0) waits.push_back(L->mounted_ev[slots[i]]);
    return wait_distinct(L, waits, static_cast<cudaStream_t>(stream));
}

int lora_loader_release(lora_loader_t L, int count, const int* slots, void* stream) {
    if (!L) return set_error(LORA_EINVAL, "loader is NULL");
    int rc = check_slots(L, count, slots);
    if (rc) return rc;
    if (count == 0) return LORA_OK;
    int id = -1;
    rc = take_event(L, &id);
    if (rc) return rc;
    LORA_CUDA_TRY(cudaEventRecord(L->evs[id].e, static_cast<cudaStream_t>(stream)));
    for (int i = 0; i < count; ++i) {
        L->fences[slots[i]].push_back(id);
        ++L->evs[id].refs;
    }
    return LORA_OK;
}

int lora_loader_stats(lora_loader_t L, uint64_t* mounts, uint64_t* drained_fences) {
    if (!L) return set_error(LORA_EINVAL, "loader is NULL");
    if (mounts) *mounts = L->mounts;
    if (drained_fences) *drained_fences = L->drained_fences;
    return LORA_OK;
}

}  // extern "C"
