// Host-tier adapter cache: the device pools' slots backed by adapters kept in pinned host
// memory, mounted on demand and evicted least-recently-used.
//
// "LLM 多 LoRA 推理服务工程 2026：从热插拔到租户编排" (blog.lonae.com) describes a tiered adapter
// store: hot adapters resident in GPU memory, warm ones in host memory, cold ones further out,
// with adapters loaded on demand and unreferenced ones evicted.  This file is the GPU/host pair
// of tiers.  One adapter identity covers all of its target modules (the registry entry of the
// ai.codenodex.com page, section "适配器先进入可信注册表"), so the cache manages a set of pools
// with the same slot count and keeps slot s of every pool holding the same adapter: one segment
// table then serves every projection of the batch.
//
// All work is host-side bookkeeping plus the pools' own stream-ordered mount and unmount calls:
// an eviction on a stream is ordered after every earlier kernel on that stream that could read
// the slot.
#include <algorithm>
#include <new>
#include <unordered_map>
#include <vector>

#include "common.cuh"

struct lora_cache {
    std::vector<lora_pool_t> pools;
    int n_slots = 0;
    struct Entry {
        std::vector<const void*> A, B;  // per pool, pinned host memory owned by the caller
        std::vector<int> ranks;
        std::vector<float> alphas;
        int slot = -1;  // device slot holding it, or -1
    };
    std::unordered_map<int64_t, Entry> reg;
    std::vector<int64_t> slot_id;    // adapter in each slot, -1 = free
    std::vector<uint64_t> last_use;  // map() call that last used each slot
    uint64_t clock = 0, hits = 0, misses = 0, evictions = 0;
};

using namespace lora;

extern "C" {

int lora_cache_create(int count, const lora_pool_t* pools, lora_cache_t* out) {
    if (!out) return set_error(LORA_EINVAL, "out is NULL");
    if (count < 1 || !pools) return set_error(LORA_EINVAL, "a cache needs at least one pool");
    for (int p = 0; p < count; ++p) {
        if (!pools[p]) return set_error(LORA_EINVAL, "pools[%d] is NULL", p);
        if (pools[p]->desc.n_slots != pools[0]->desc.n_slots)
            return set_error(LORA_EINVAL, "pool %d has %d slots, pool 0 has %d", p, pools[p]->desc.n_slots,
                             pools[0]->desc.n_slots);
        for (uint8_t m : pools[p]->mounted)
            if (m) return set_error(LORA_EBUSY, "pool %d already holds adapters: the cache owns its slots", p);
    }
    lora_cache* c = new (std::nothrow) lora_cache();
    if (!c) return set_error(LORA_EINVAL, "out of host memory");
    c->pools.assign(pools, pools + count);
    c->n_slots = pools[0]->desc.n_slots;
    c->slot_id.assign(c->n_slots, -1);
    c->last_use.assign(c->n_slots, 0);
    *out = c;
    return LORA_OK;
}

int lora_cache_destroy(lora_cache_t cache) {
    delete cache;
    return LORA_OK;
}

int lora_cache_register(lora_cache_t cache, int64_t id, const void* const* A_host, const void* const* B_host,
                        const int* ranks, const float* alphas) {
    if (!cache) return set_error(LORA_EINVAL, "cache is NULL");
    if (id < 0) return set_error(LORA_EINVAL, "adapter id %lld < 0", (long long)id);
    if (!A_host || !B_host || !ranks || !alphas) return set_error(LORA_EINVAL, "A/B/ranks/alphas is NULL");
    if (cache->reg.count(id)) return set_error(LORA_EBUSY, "adapter %lld is already registered", (long long)id);
    const int np = (int)cache->pools.size();
    lora_cache::Entry e;
    for (int p = 0; p < np; ++p) {
        const lora_pool_desc& d = cache->pools[p]->desc;
        if (!A_host[p] || !B_host[p]) return set_error(LORA_EINVAL, "A/B of pool %d is NULL", p);
        if (ranks[p] < 1 || ranks[p] > d.r_max)
            return set_error(LORA_ERANK, "pool %d: rank %d outside [1, %d]", p, ranks[p], d.r_max);
        e.A.push_back(A_host[p]);
        e.B.push_back(B_host[p]);
        e.ranks.push_back(ranks[p]);
        e.alphas.push_back(alphas[p]);
    }
    cache->reg.emplace(id, std::move(e));
    return LORA_OK;
}

static int evict_slot(lora_cache_t cache, int slot, void* stream) {
    for (lora_pool_t p : cache->pools) {
        const int rc = lora_pool_unload_slot(p, slot, stream);
        if (rc) return rc;
    }
    cache->reg[cache->slot_id[slot]].slot = -1;
    cache->slot_id[slot] = -1;
    return LORA_OK;
}

int lora_cache_unregister(lora_cache_t cache, int64_t id, void* stream) {
    if (!cache) return set_error(LORA_EINVAL, "cache is NULL");
    auto it = cache->reg.find(id);
    if (it == cache->reg.end()) return set_error(LORA_EIDX, "adapter %lld is not registered", (long long)id);
    if (it->second.slot >= 0) {
        const int rc = evict_slot(cache, it->second.slot, stream);
        if (rc) return rc;
    }
    cache->reg.erase(id);
    return LORA_OK;
}

int lora_cache_map(lora_cache_t cache, const int64_t* ids, int n, int32_t* idx_out, int* mounts_out, void* stream) {
    if (!cache) return set_error(LORA_EINVAL, "cache is NULL");
    if (n < 0) return set_error(LORA_EINVAL, "n < 0");
    if (n > 0 && (!ids || !idx_out)) return set_error(LORA_EINVAL, "ids/idx_out is NULL");
    // 1. default deny: every id is -1 or registered; nothing changes on an error
    std::vector<int64_t> distinct;
    for (int t = 0; t < n; ++t) {
        const int64_t id = ids[t];
        if (id == -1) continue;
        if (id < -1 || !cache->reg.count(id))
            return set_error(LORA_EIDX, "token %d: adapter %lld is not registered", t, (long long)id);
        distinct.push_back(id);
    }
    std::sort(distinct.begin(), distinct.end());
    distinct.erase(std::unique(distinct.begin(), distinct.end()), distinct.end());
    if ((int)distinct.size() > cache->n_slots)
        return set_error(LORA_ENOSPACE, "batch names %zu adapters, the pools have %d slots", distinct.size(),
                         cache->n_slots);
    // 2. hits: mark their slots used by this call so that no eviction below can take them
    const uint64_t now = ++cache->clock;
    std::vector<int64_t> missing;
    for (int64_t id : distinct) {
        const int s = cache->reg[id].slot;
        if (s >= 0) {
            cache->last_use[s] = now;
            ++cache->hits;
        } else {
            missing.push_back(id);
        }
    }
    // 3. misses: a free slot, else the least recently used slot this batch does not use
    //    (ties: the lowest slot)
    std::vector<int> slots;
    for (int64_t id : missing) {
        int best = -1;
        for (int s = 0; s < cache->n_slots && best < 0; ++s)
            if (cache->slot_id[s] < 0) best = s;
        if (best < 0) {
            for (int s = 0; s < cache->n_slots; ++s)
                if (cache->last_use[s] != now && (best < 0 || cache->last_use[s] < cache->last_use[best])) best = s;
            const int rc = evict_slot(cache, best, stream);
            if (rc) return rc;
            ++cache->evictions;
        }
        cache->slot_id[best] = id;
        cache->last_use[best] = now;
        cache->reg[id].slot = best;
        slots.push_back(best);
        ++cache->misses;
    }
    // 4. mount the misses: one batched mount per pool, stream-ordered before the caller's
    //    next kernels on this stream
    const int k = (int)missing.size();
    if (k > 0) {
        std::vector<const void*> A(k), B(k);
        std::vector<int> ranks(k);
        std::vector<float> alphas(k);
        for (size_t p = 0; p < cache->pools.size(); ++p) {
            for (int i = 0; i < k; ++i) {
                const lora_cache::Entry& e = cache->reg[missing[i]];
                A[i] = e.A[p];
                B[i] = e.B[p];
                ranks[i] = e.ranks[p];
                alphas[i] = e.alphas[p];
            }
            const int rc = lora_pool_load_slots(cache->pools[p], k, slots.data(), A.data(), B.data(), ranks.data(),
                                                alphas.data(), stream);
            if (rc) return rc;
        }
    }
    for (int t = 0; t < n; ++t) idx_out[t] = ids[t] < 0 ? -1 : cache->reg[ids[t]].slot;
    if (mounts_out) *mounts_out = k;
    return LORA_OK;
}

int lora_cache_slot_of(lora_cache_t cache, int64_t id, int* slot) {
    if (!cache || !slot) return set_error(LORA_EINVAL, "cache/slot is NULL");
    auto it = cache->reg.find(id);
    if (it == cache->reg.end()) return set_error(LORA_EIDX, "adapter %lld is not registered", (long long)id);
    *slot = it->second.slot;
    return LORA_OK;
}

int lora_cache_stats(lora_cache_t cache, uint64_t* hits, uint64_t* misses, uint64_t* evictions) {
    if (!cache) return set_error(LORA_EINVAL, "cache is NULL");
    if (hits) *hits = cache->hits;
    if (misses) *misses = cache->misses;
    if (evictions) *evictions = cache->evictions;
    return LORA_OK;
}

}  // extern "C"
