// Two-tier adapter residency cache (host code only).
//
// "Multi-LoRA Serving - S-LoRA/Punica Batching, Adapter Hot-Swap & Memory",
// section "Memory: slots, tiers and paging", and its adapter-cache
// simulation: adapters live in a few GPU slots, backed by a larger host-RAM
// tier, backed by disk.  A request whose adapter is in a GPU slot is served
// at once; otherwise the adapter comes from host memory (a copy) or, when the
// host tier misses too, from disk.  Each tier evicts its least recently used
// adapter when a new one would exceed its slot count.  The host tier is
// consulted (and reordered) only on a GPU miss.
//
// The cache decides residency only; it moves no data.  A server maps a GPU
// hit to "already in the pool", a host hit to an upload from pinned host
// memory (lora_pool_load_async), a disk load to a fetch plus that upload, and
// the reported GPU eviction to lora_pool_unload_async.
//
// Each tier is an intrusive doubly linked list over the key range (keys are
// adapter ids 0..n_keys-1), so a touch is O(1) with no allocation after
// creation.
#include <cstdint>
#include <new>
#include <vector>

#include "lora.h"

namespace {

class LruTier {
  public:
    bool init(int n_keys, int cap) {
        cap_ = cap;
        size_ = 0;
        head_ = tail_ = -1;
        try {
            prev_.assign(n_keys, -1);
            next_.assign(n_keys, -1);
            in_.assign(n_keys, 0);
        } catch (...) {
            return false;
        }
        return true;
    }

    // Marks `k` most recently used (inserting it on a miss) and evicts the
    // least recently used key while the tier holds more than its capacity.
    // Returns whether `k` was present; *evicted is the evicted key or -1.
    bool touch(int k, int *evicted) {
        *evicted = -1;
        const bool hit = in_[k] != 0;
        if (hit) unlink(k);
        push_back(k);
        if (size_ > cap_) {
            const int victim = head_;
            unlink(victim);
            *evicted = victim;
        }
        return hit;
    }

    bool contains(int k) const { return in_[k] != 0; }

  private:
    void unlink(int k) {
        const int p = prev_[k], n = next_[k];
        if (p >= 0) next_[p] = n; else head_ = n;
        if (n >= 0) prev_[n] = p; else tail_ = p;
        prev_[k] = next_[k] = -1;
        in_[k] = 0;
        --size_;
    }
    void push_back(int k) {
        prev_[k] = tail_;
        next_[k] = -1;
        if (tail_ >= 0) next_[tail_] = k; else head_ = k;
        tail_ = k;
        in_[k] = 1;
        ++size_;
    }

    int cap_ = 0, size_ = 0, head_ = -1, tail_ = -1;
    std::vector<int> prev_, next_;
    std::vector<uint8_t> in_;
};

}  // namespace

struct lora_tier_cache {
    int n_keys;
    LruTier gpu, host;
};

extern "C" {

int lora_tier_cache_create(lora_tier_cache **out, int n_keys, int gpu_slots, int host_slots) {
    if (!out) return LORA_ERR_ARG;
    *out = nullptr;
    if (n_keys <= 0 || gpu_slots < 0 || host_slots < 0) return LORA_ERR_ARG;
    lora_tier_cache *c = new (std::nothrow) lora_tier_cache();
    if (!c) return LORA_ERR_ARG;
    c->n_keys = n_keys;
    if (!c->gpu.init(n_keys, gpu_slots) || !c->host.init(n_keys, host_slots)) {
        delete c;
        return LORA_ERR_ARG;
    }
    *out = c;
    return LORA_OK;
}

int lora_tier_cache_destroy(lora_tier_cache *c) {
    delete c;
    return LORA_OK;
}

int lora_tier_cache_touch(lora_tier_cache *c, int adapter, int *gpu_evicted) {
    int ev = -1, ev_host = -1;
    if (gpu_evicted) *gpu_evicted = -1;
    if (!c || adapter < 0 || adapter >= c->n_keys) return LORA_ERR_ARG;
    int tier;
    if (c->gpu.touch(adapter, &ev)) tier = LORA_TIER_GPU;
    else tier = c->host.touch(adapter, &ev_host) ? LORA_TIER_HOST : LORA_TIER_DISK;
    if (gpu_evicted) *gpu_evicted = ev;
    return tier;
}

int lora_tier_cache_resident(const lora_tier_cache *c, int adapter) {
    if (!c || adapter < 0 || adapter >= c->n_keys) return LORA_ERR_ARG;
    return (c->gpu.contains(adapter) ? 1 : 0) | (c->host.contains(adapter) ? 2 : 0);
}

int lora_tier_sim(const int *trace, long long n, int n_keys, int gpu_slots, int host_slots,
                  long long *counts) {
    if (!counts || n < 0 || (n > 0 && !trace)) return LORA_ERR_ARG;
    for (long long i = 0; i < n; ++i)
        if (trace[i] < 0 || trace[i] >= n_keys) return LORA_ERR_ARG;
    lora_tier_cache *c = nullptr;
    int rc = lora_tier_cache_create(&c, n_keys, gpu_slots, host_slots);
    if (rc) return rc;
    counts[0] = counts[1] = counts[2] = 0;
    for (long long i = 0; i < n; ++i) {
        const int tier = lora_tier_cache_touch(c, trace[i], nullptr);
        ++counts[tier];
    }
    lora_tier_cache_destroy(c);
    return LORA_OK;
}

}  // extern "C"
