// page_manager.cpp -- host-side page bookkeeping for the shared paged KV pool:
// refcounted, block-aligned prefix-cache pages that later requests (of any
// decoder model) reuse, and transfer pages that live only for one handoff.
//
// PrFaaS (hybrid prefix cache pool): prefix-cache blocks are reused within
// the cluster and must be block-aligned and completely filled to be reusable;
// transfer-cache blocks serve a cross-cluster transfer and are dropped once
// it is done, never occupying the pool long-term.  ICaRus (key design 2):
// because every task model's encoder is the frozen base, their caches for a
// prompt are bitwise identical, so a prefix cached by one agent is a hit for
// every later agent, whatever its decoder.
//
// A full block is identified by a hash chain over token ids, h_i =
// H(h_{i-1}, tokens of block i), and looked up with its parent hash and
// token ids compared exactly (a hash collision is never a hit).  Pages whose
// count drops to zero stay indexed, in LRU order, until a new allocation
// needs them.  No CUDA: this file only hands out page indices; the caller
// fills the pages (prefill, handoff or shkv_append_kv) and the block table.
#include <stdint.h>
#include <string.h>

#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "shkv.h"

namespace {

constexpr uint64_t kFnvOffset = 1469598103934665603ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

enum PageState : uint8_t { kFree = 0, kPrivate = 1, kPrefix = 2, kTransfer = 3 };

struct Block {
    uint64_t parent;
    std::vector<int32_t> tokens;
    int32_t page;
};

uint64_t chain_hash(uint64_t parent, const int32_t *tokens, int n)
{
    uint64_t h = kFnvOffset;
    for (int i = 0; i < 8; ++i) {
        h ^= (parent >> (8 * i)) & 0xffu;
        h *= kFnvPrime;
    }
    for (int t = 0; t < n; ++t) {
        const uint32_t v = (uint32_t)tokens[t];
        for (int i = 0; i < 4; ++i) {
            h ^= (v >> (8 * i)) & 0xffu;
            h *= kFnvPrime;
        }
    }
    return h;
}

}  // namespace

struct shkv_pages {
    int32_t num_pages, page_size;
    std::vector<int32_t> ref;
    std::vector<uint8_t> state;
    std::vector<uint64_t> key;                       // hash of the indexed block in a page
    std::vector<int32_t> free_list;                  // stack of free pages
    std::unordered_multimap<uint64_t, Block> index;  // hash -> indexed full blocks
    std::list<int32_t> lru;                          // indexed pages with ref == 0, oldest first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<uint8_t> in_lru;
    int64_t hits = 0, lookups = 0;

    Block *find(uint64_t h, uint64_t parent, const int32_t *tokens)
    {
        auto range = index.equal_range(h);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second.parent == parent &&
                memcmp(it->second.tokens.data(), tokens, sizeof(int32_t) * (size_t)page_size) == 0)
                return &it->second;
        return nullptr;
    }

    void unindex(int32_t page)
    {
        auto range = index.equal_range(key[page]);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second.page == page) {
                index.erase(it);
                return;
            }
    }

    void lru_remove(int32_t page)
    {
        if (in_lru[page]) {
            lru.erase(lru_pos[page]);
            in_lru[page] = 0;
        }
    }

    // one page for a new block: a free one, else the least recently used
    // unreferenced prefix page (dropped from the index); -1 if none
    int32_t take_page()
    {
        if (!free_list.empty()) {
            const int32_t pg = free_list.back();
            free_list.pop_back();
            return pg;
        }
        if (!lru.empty()) {
            const int32_t pg = lru.front();
            lru.pop_front();
            in_lru[pg] = 0;
            unindex(pg);
            return pg;
        }
        return -1;
    }

    void drop_ref(int32_t pg)
    {
        if (--ref[pg] > 0)
            return;
        if (state[pg] == kPrefix) {
            lru.push_back(pg);
            lru_pos[pg] = std::prev(lru.end());
            in_lru[pg] = 1;
        } else {
            state[pg] = kFree;
            free_list.push_back(pg);
        }
    }
};

extern "C" {

shkv_status shkv_pages_create(int32_t num_pages, int32_t page_size, shkv_pages **out)
{
    if (!out || num_pages < 1 || page_size < 1)
        return SHKV_ERR_INVALID_ARG;
    *out = nullptr;
    shkv_pages *m = new (std::nothrow) shkv_pages();
    if (!m)
        return SHKV_ERR_INVALID_ARG;
    m->num_pages = num_pages;
    m->page_size = page_size;
    m->ref.assign(num_pages, 0);
    m->state.assign(num_pages, kFree);
    m->key.assign(num_pages, 0);
    m->lru_pos.resize(num_pages);
    m->in_lru.assign(num_pages, 0);
    m->free_list.reserve(num_pages);
    for (int32_t p = num_pages - 1; p >= 0; --p)
        m->free_list.push_back(p);                   // page 0 is handed out first
    *out = m;
    return SHKV_OK;
}

shkv_status shkv_pages_destroy(shkv_pages *m)
{
    if (!m)
        return SHKV_ERR_INVALID_ARG;
    delete m;
    return SHKV_OK;
}

shkv_status shkv_pages_acquire(shkv_pages *m, const int32_t *tokens, int32_t n_tokens, int32_t *pages,
                               int32_t max_pages, int32_t *n_cached_tokens)
{
    if (!m || n_tokens < 0 || (n_tokens > 0 && (!tokens || !pages)) || !n_cached_tokens)
        return SHKV_ERR_INVALID_ARG;
    const int32_t P = m->page_size;
    const int32_t nblocks = (n_tokens + P - 1) / P;
    if (nblocks > max_pages)
        return SHKV_ERR_CAPACITY;
    // longest cached prefix of full blocks
    int32_t hit = 0;
    uint64_t parent = 0;
    for (; hit < n_tokens / P; ++hit) {
        const int32_t *blk = tokens + (int64_t)hit * P;
        const uint64_t h = chain_hash(parent, blk, P);
        Block *b = m->find(h, parent, blk);
        if (!b)
            break;
        pages[hit] = b->page;
        parent = h;
    }
    m->lookups += n_tokens / P;
    m->hits += hit;
    // reference the hits before taking pages, so eviction cannot take them
    for (int32_t i = 0; i < hit; ++i) {
        m->lru_remove(pages[i]);
        ++m->ref[pages[i]];
    }
    for (int32_t i = hit; i < nblocks; ++i) {
        const int32_t pg = m->take_page();
        if (pg < 0) {
            for (int32_t j = i - 1; j >= 0; --j)
                m->drop_ref(pages[j]);
            *n_cached_tokens = 0;
            return SHKV_ERR_CAPACITY;
        }
        m->state[pg] = kPrivate;
        m->ref[pg] = 1;
        pages[i] = pg;
    }
    *n_cached_tokens = hit * P;
    return SHKV_OK;
}

shkv_status shkv_pages_publish(shkv_pages *m, const int32_t *tokens, int32_t n_tokens, const int32_t *pages)
{
    if (!m || n_tokens < 0 || (n_tokens > 0 && (!tokens || !pages)))
        return SHKV_ERR_INVALID_ARG;
    const int32_t P = m->page_size;
    for (int32_t i = 0; i < n_tokens / P; ++i)
        if (pages[i] < 0 || pages[i] >= m->num_pages || m->ref[pages[i]] < 1 || m->state[pages[i]] == kTransfer)
            return SHKV_ERR_INVALID_ARG;
    uint64_t parent = 0;
    for (int32_t i = 0; i < n_tokens / P; ++i) {   // full blocks only; a partial last block is never indexed
        const int32_t *blk = tokens + (int64_t)i * P;
        const uint64_t h = chain_hash(parent, blk, P);
        const int32_t pg = pages[i];
        if (m->state[pg] == kPrivate && !m->find(h, parent, blk)) {
            Block b;
            b.parent = parent;
            b.tokens.assign(blk, blk + P);
            b.page = pg;
            m->index.emplace(h, std::move(b));
            m->state[pg] = kPrefix;
            m->key[pg] = h;
        }
        parent = h;
    }
    return SHKV_OK;
}

shkv_status shkv_pages_release(shkv_pages *m, const int32_t *pages, int32_t n_pages)
{
    if (!m || n_pages < 0 || (n_pages > 0 && !pages))
        return SHKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_pages; ++i)
        if (pages[i] < 0 || pages[i] >= m->num_pages || m->ref[pages[i]] < 1)
            return SHKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_pages; ++i)
        m->drop_ref(pages[i]);
    return SHKV_OK;
}

shkv_status shkv_pages_alloc_transfer(shkv_pages *m, int32_t n_pages, int32_t *pages)
{
    if (!m || n_pages < 0 || (n_pages > 0 && !pages))
        return SHKV_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_pages; ++i) {
        const int32_t pg = m->take_page();
        if (pg < 0) {
            for (int32_t j = i - 1; j >= 0; --j)
                m->drop_ref(pages[j]);
            return SHKV_ERR_CAPACITY;
        }
        m->state[pg] = kTransfer;
        m->ref[pg] = 1;
        pages[i] = pg;
    }
    return SHKV_OK;
}

shkv_status shkv_pages_stats(const shkv_pages *m, shkv_pages_info *info)
{
    if (!m || !info)
        return SHKV_ERR_INVALID_ARG;
    memset(info, 0, sizeof *info);
    info->num_pages = m->num_pages;
    info->free_pages = (int32_t)m->free_list.size();
    info->cached_idle_pages = (int32_t)m->lru.size();
    info->indexed_blocks = (int32_t)m->index.size();
    for (int32_t p = 0; p < m->num_pages; ++p) {
        if (m->state[p] == kTransfer)
            ++info->transfer_pages;
        if (m->ref[p] > 0)
            ++info->referenced_pages;
    }
    info->block_lookups = m->lookups;
    info->block_hits = m->hits;
    return SHKV_OK;
}

shkv_status shkv_pages_refcount(const shkv_pages *m, int32_t page, int32_t *count)
{
    if (!m || !count || page < 0 || page >= m->num_pages)
        return SHKV_ERR_INVALID_ARG;
    *count = m->ref[page];
    return SHKV_OK;
}

}  // extern "C"
