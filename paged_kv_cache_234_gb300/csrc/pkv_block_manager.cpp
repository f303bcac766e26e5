// pkv_block_manager.cpp -- host-side manager of the physical KV blocks:
// free-list allocator, reference counts, prefix sharing by content hash,
// copy-on-write, fill and fragmentation figures ("paged-attention-runtime"
// summary, CORE CAPABILITIES 1; "PagedAttention & KV-Cache Memory
// Management": the prefix-sharing block allocator and section 4.1.1,
// page-level reference counts with a fresh page and a copy when a shared
// page diverges).
//
// Plain C++ on the host: the block tables it produces, and the reference
// counts it exports for eviction scoring, are uploaded by the caller; the
// page copies that copy-on-write asks for run on the GPU (pkv_copy_blocks).
// Every call takes the manager's lock, so one manager may be shared by
// threads; every failing call changes nothing.
#include <stdint.h>

#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_block_manager {
    int block_size = 16;
    std::vector<int32_t> refcnt;
    std::vector<int32_t> fill;
    std::vector<uint64_t> hash_of;
    std::vector<int32_t> free_stack;  // top = back; starts handing out 0, 1, 2, ...
    std::unordered_map<uint64_t, int32_t> cache;
    std::mutex mu;

    bool in_use(int32_t b) const
    {
        return b >= 0 && b < static_cast<int32_t>(refcnt.size()) && refcnt[b] > 0;
    }

    void unregister(int32_t b)
    {
        const uint64_t h = hash_of[b];
        if (h != 0) {
            auto it = cache.find(h);
            if (it != cache.end() && it->second == b) cache.erase(it);
        }
        hash_of[b] = 0;
    }
};

namespace {

// Entries of `ids` in use, each listed at most as often as its count (when
// `respect_counts`).  Scratch map only for duplicate ids.
bool valid_ids(const pkv_block_manager *m, const int32_t *ids, int n, bool respect_counts)
{
    for (int i = 0; i < n; ++i)
        if (!m->in_use(ids[i])) return false;
    if (!respect_counts) return true;
    std::unordered_map<int32_t, int32_t> seen;
    for (int i = 0; i < n; ++i) {
        int32_t &c = seen[ids[i]];
        if (++c > m->refcnt[ids[i]]) return false;
    }
    return true;
}

}  // namespace

extern "C" pkv_status pkv_bm_create(int num_blocks, int block_size, pkv_block_manager **out)
{
    if (!out || num_blocks < 0 || block_size <= 0) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager *m = new (std::nothrow) pkv_block_manager;
    if (!m) return PKV_ERR_EXHAUSTED;
    try {
        m->block_size = block_size;
        m->refcnt.assign(num_blocks, 0);
        m->fill.assign(num_blocks, 0);
        m->hash_of.assign(num_blocks, 0);
        m->free_stack.resize(num_blocks);
        for (int i = 0; i < num_blocks; ++i) m->free_stack[i] = num_blocks - 1 - i;
        m->cache.reserve(static_cast<size_t>(num_blocks));
    } catch (...) {
        delete m;
        return PKV_ERR_EXHAUSTED;
    }
    *out = m;
    return PKV_OK;
}

extern "C" void pkv_bm_destroy(pkv_block_manager *m) { delete m; }

extern "C" pkv_status pkv_bm_allocate(pkv_block_manager *m, const uint64_t *hashes, int n,
                                      int32_t *out_ids)
{
    if (!m || n < 0 || (n > 0 && !out_ids)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    // entries needing a fresh block: no hash, or a hash neither cached nor
    // introduced by an earlier entry of this call
    int64_t fresh = 0;
    if (hashes) {
        std::unordered_map<uint64_t, int> seen;
        for (int i = 0; i < n; ++i) {
            const uint64_t h = hashes[i];
            if (h != 0 && (m->cache.count(h) || seen.count(h))) continue;
            ++fresh;
            if (h != 0) seen[h] = 1;
        }
    } else {
        fresh = n;
    }
    if (fresh > static_cast<int64_t>(m->free_stack.size())) return PKV_ERR_EXHAUSTED;
    for (int i = 0; i < n; ++i) {
        const uint64_t h = hashes ? hashes[i] : 0;
        if (h != 0) {
            auto it = m->cache.find(h);
            if (it != m->cache.end()) {
                ++m->refcnt[it->second];
                out_ids[i] = it->second;
                continue;
            }
        }
        const int32_t b = m->free_stack.back();
        m->free_stack.pop_back();
        m->refcnt[b] = 1;
        m->fill[b] = 0;
        m->hash_of[b] = h;
        if (h != 0) m->cache[h] = b;
        out_ids[i] = b;
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_free(pkv_block_manager *m, const int32_t *ids, int n)
{
    if (!m || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (!valid_ids(m, ids, n, true)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        const int32_t b = ids[i];
        if (--m->refcnt[b] == 0) {
            m->unregister(b);
            m->fill[b] = 0;
            m->free_stack.push_back(b);
        }
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_fork(pkv_block_manager *m, const int32_t *ids, int n)
{
    if (!m || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (!valid_ids(m, ids, n, false)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) ++m->refcnt[ids[i]];
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_cow(pkv_block_manager *m, const int32_t *ids, int n,
                                 int32_t *out_ids, int32_t *copy_pairs, int *num_copies)
{
    if (!m || n < 0 || (n > 0 && (!ids || !out_ids)) || !num_copies) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (!valid_ids(m, ids, n, false)) return PKV_ERR_INVALID_ARG;
    // entries processed in order; count the copies first (all-or-nothing)
    int64_t copies = 0;
    {
        std::unordered_map<int32_t, int32_t> cnt;
        for (int i = 0; i < n; ++i) {
            auto it = cnt.find(ids[i]);
            int32_t &c = it == cnt.end() ? (cnt[ids[i]] = m->refcnt[ids[i]]) : it->second;
            if (c > 1) {
                --c;
                ++copies;
            }
        }
    }
    if (copies > static_cast<int64_t>(m->free_stack.size())) return PKV_ERR_EXHAUSTED;
    int k = 0;
    for (int i = 0; i < n; ++i) {
        const int32_t b = ids[i];
        if (m->refcnt[b] == 1) {
            m->unregister(b);  // about to be written
            out_ids[i] = b;
            continue;
        }
        const int32_t nb = m->free_stack.back();
        m->free_stack.pop_back();
        --m->refcnt[b];
        m->refcnt[nb] = 1;
        m->fill[nb] = m->fill[b];
        m->hash_of[nb] = 0;
        out_ids[i] = nb;
        if (copy_pairs) {
            copy_pairs[2 * k] = b;
            copy_pairs[2 * k + 1] = nb;
        }
        ++k;
    }
    *num_copies = k;
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_set_fill(pkv_block_manager *m, const int32_t *ids,
                                      const int32_t *tokens, int n)
{
    if (!m || n < 0 || (n > 0 && (!ids || !tokens))) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (!valid_ids(m, ids, n, false)) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] > m->block_size) return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) m->fill[ids[i]] = tokens[i];
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_stats(pkv_block_manager *m, pkv_bm_stats_t *out)
{
    if (!m || !out) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    int64_t used = 0, shared = 0, logical = 0, tokens = 0;
    for (size_t b = 0; b < m->refcnt.size(); ++b) {
        const int32_t r = m->refcnt[b];
        if (r > 0) {
            ++used;
            tokens += m->fill[b];
        }
        shared += r > 1;
        logical += r;
    }
    out->free_blocks = static_cast<int64_t>(m->free_stack.size());
    out->used_blocks = used;
    out->shared_blocks = shared;
    out->logical_blocks = logical;
    out->tokens = tokens;
    out->internal_fragmentation =
        used ? 1.0 - static_cast<double>(tokens) / (static_cast<double>(used) * m->block_size)
             : 0.0;
    out->sharing_saving =
        logical ? 1.0 - static_cast<double>(used) / static_cast<double>(logical) : 0.0;
    return PKV_OK;
}

extern "C" pkv_status pkv_bm_refcounts(pkv_block_manager *m, int32_t *out, int n)
{
    if (!m || !out || n != static_cast<int>(m->refcnt.size())) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    for (int i = 0; i < n; ++i) out[i] = m->refcnt[i];
    return PKV_OK;
}
