// pa_alloc.cpp -- host block allocator of libpa: free list, reference counts,
// per-sequence block tables, fork (prefix sharing), growth and copy-on-write.
//
// Rules, from the pages:
//  - blocks of B slots in one pool; token pos of a sequence is at offset pos % B
//    of table[pos / B] ("PagedAttention: Virtual Memory for the KV Cache",
//    "A block table preserves token order");
//  - a block is taken from the free pool only when a token starts a new block;
//    existing table entries never move (same page, "Growing a request");
//  - a reference count per block; a block is freed only at count zero
//    ("KV Cache Optimization and Management", answer A6);
//  - a partially filled shared last block is copied before a sequence writes
//    into it: fresh p', copy p -> p', redirect the writer's table, fix counts;
//    a full shared block needs no copy ("PagedAttention: Virtual Memory for the
//    KV Cache", "Sharing a prefix and copying a partial block"; "Paged Attention
//    and vLLM", "Continuous Batching and Scheduler").
// Policies the pages leave open (FIFO free list seeded by free_order, first
// writer copies, all-or-nothing appends, copy block taken before growth
// blocks) are documented in include/pa.h.
//
// Every operation is O(1) amortised per block touched.  Not thread-safe.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "../../include/pa.h"

#include "pa_pool.h"

namespace {

bool valid_seq(const pa_pool *p, int32_t s) {
    return p && s >= 0 && s < (int32_t)p->seqs.size() && p->seqs[s].live;
}

int64_t blocks_for(int64_t tokens, int32_t B) { return (tokens + B - 1) / B; }

using pa_pool_detail::available;
using pa_pool_detail::release_block;

int32_t take_block(pa_pool *p) {
    int32_t b = p->free_list.front();
    p->free_list.pop_front();
    p->ref[b] = 1;
    if (p->fail_budget > 0) --p->fail_budget;
    return b;
}


// Blocks one append of n tokens needs, given the refcount already given up on
// the sequence's last block by earlier copies in the same batch.
int64_t need_for(const pa_pool *p, const pa_seq_rec &s, int64_t n, int32_t ref_last) {
    if (n <= 0) return 0;
    int64_t grow = blocks_for(s.len + n, p->B) - blocks_for(s.len, p->B);
    bool cow = (s.len % p->B) != 0 && ref_last > 1;
    return grow + (cow ? 1 : 0);
}

// Apply an append whose block need has been checked.
void do_append(pa_pool *p, pa_seq_rec &s, int64_t n, int64_t *slots, int64_t *pair, int32_t *ncow) {
    const int32_t B = p->B;
    *ncow = 0;
    if (n <= 0) return;
    if (s.len % B != 0 && p->ref[s.table.back()] > 1) {
        int32_t old = s.table.back();
        int32_t fresh = take_block(p);
        --p->ref[old];  // another sequence still holds it: stays >= 1
        s.table.back() = fresh;
        pair[0] = old;
        pair[1] = fresh;
        *ncow = 1;
        ++p->cow_copies;
    }
    for (int64_t i = 0; i < n; ++i) {
        int64_t pos = s.len + i;
        int64_t logical = pos / B;
        if (logical == (int64_t)s.table.size()) s.table.push_back(take_block(p));
        if (slots) slots[i] = (int64_t)s.table[logical] * B + pos % B;
    }
    s.len += n;
}

}  // namespace

extern "C" {

pa_pool *pa_pool_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_pool *p = new (std::nothrow) pa_pool();
    if (!p) return nullptr;
    p->num_blocks = num_blocks;
    p->B = block_size;
    p->ref.assign(num_blocks, 0);
    p->given_up.assign(num_blocks, 0);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete p;
                return nullptr;
            }
            seen[b] = 1;
            p->free_list.push_back(b);
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) p->free_list.push_back(i);
    }
    return p;
}

void pa_pool_destroy(pa_pool *pool) { delete pool; }

int32_t pa_seq_create(pa_pool *pool) {
    if (!pool) return -PA_ERR_INVALID;
    pool->seqs.emplace_back();
    pool->seqs.back().live = true;
    ++pool->live;
    return (int32_t)pool->seqs.size() - 1;
}

int32_t pa_seq_fork(pa_pool *pool, int32_t parent) {
    if (!valid_seq(pool, parent)) return -PA_ERR_BAD_INDEX;
    pa_seq_rec child;
    child.table = pool->seqs[parent].table;
    child.len = pool->seqs[parent].len;
    child.live = true;
    for (int32_t b : child.table) ++pool->ref[b];
    pool->seqs.push_back(std::move(child));
    ++pool->live;
    return (int32_t)pool->seqs.size() - 1;
}

int32_t pa_seq_append(pa_pool *pool, int32_t seq, int32_t n_tokens, int64_t *slots_out,
                      int64_t *cow_pairs_out, int32_t *n_cow) {
    if (!pool || n_tokens < 0 || !cow_pairs_out || !n_cow || (n_tokens > 0 && !slots_out))
        return PA_ERR_INVALID;
    if (!valid_seq(pool, seq)) return PA_ERR_BAD_INDEX;
    pa_seq_rec &s = pool->seqs[seq];
    int32_t ref_last = s.table.empty() ? 0 : pool->ref[s.table.back()];
    if (need_for(pool, s, n_tokens, ref_last) > available(pool)) return PA_ERR_OOM;
    do_append(pool, s, n_tokens, slots_out, cow_pairs_out, n_cow);
    return PA_OK;
}

int32_t pa_seq_append_batch(pa_pool *pool, const int32_t *seqs, int32_t n, int32_t tokens_each,
                            int64_t *slots_out, int64_t *cow_pairs_out, int32_t *n_cow) {
    if (!pool || n < 0 || tokens_each < 0 || !n_cow || (n > 0 && (!seqs || !cow_pairs_out)) ||
        (n > 0 && tokens_each > 0 && !slots_out))
        return PA_ERR_INVALID;
    // each sequence at most once: mark it with this call's epoch
    if (++pool->batch_epoch == 0) {  // the counter wrapped: forget every old mark
        for (auto &rec : pool->seqs) rec.batch_mark = 0;
        pool->batch_epoch = 1;
    }
    const uint32_t epoch = pool->batch_epoch;
    for (int32_t i = 0; i < n; ++i) {
        if (!valid_seq(pool, seqs[i])) return PA_ERR_BAD_INDEX;
        pa_seq_rec &s = pool->seqs[seqs[i]];
        if (s.batch_mark == epoch) return PA_ERR_INVALID;
        s.batch_mark = epoch;
    }
    // Dry run: copies made earlier in the batch lower the count of the block
    // they left, which can spare a later sharer its own copy.
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        const pa_seq_rec &s = pool->seqs[seqs[i]];
        int32_t ref_last = 0;
        if (!s.table.empty()) {
            const int32_t last = s.table.back();
            ref_last = pool->ref[last] - pool->given_up[last];
        }
        need += need_for(pool, s, tokens_each, ref_last);
        if (tokens_each > 0 && s.len % pool->B != 0 && ref_last > 1) {
            const int32_t last = s.table.back();
            if (pool->given_up[last]++ == 0) pool->touched.push_back(last);
        }
    }
    for (int32_t b : pool->touched) pool->given_up[b] = 0;
    pool->touched.clear();
    if (need > available(pool)) return PA_ERR_OOM;
    int32_t pairs = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t c = 0;
        do_append(pool, pool->seqs[seqs[i]], tokens_each,
                  slots_out ? slots_out + (int64_t)i * tokens_each : nullptr,
                  cow_pairs_out + 2 * pairs, &c);
        pairs += c;
    }
    *n_cow = pairs;
    return PA_OK;
}

int32_t pa_seq_free(pa_pool *pool, int32_t seq) {
    if (!valid_seq(pool, seq)) return PA_ERR_BAD_INDEX;
    pa_seq_rec &s = pool->seqs[seq];
    for (int32_t b : s.table) release_block(pool, b);
    s.table.clear();
    s.table.shrink_to_fit();
    s.len = 0;
    s.live = false;
    --pool->live;
    return PA_OK;
}

int32_t pa_seq_table(const pa_pool *pool, int32_t seq, int32_t *out, int32_t cap) {
    if (!valid_seq(pool, seq)) return -PA_ERR_BAD_INDEX;
    const auto &t = pool->seqs[seq].table;
    int32_t n = (int32_t)t.size();
    if (out && cap > 0) std::memcpy(out, t.data(), sizeof(int32_t) * (size_t)(n < cap ? n : cap));
    return n;
}

int32_t pa_seq_len(const pa_pool *pool, int32_t seq) {
    if (!valid_seq(pool, seq)) return -PA_ERR_BAD_INDEX;
    return (int32_t)pool->seqs[seq].len;
}

int32_t pa_pool_export(const pa_pool *pool, const int32_t *seqs, int32_t n, int32_t max_blocks,
                       int32_t pad, int32_t *tables_out, int32_t *lens_out) {
    if (!pool || n < 0 || max_blocks <= 0 || (n > 0 && (!seqs || !tables_out || !lens_out)))
        return PA_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i)
        if (!valid_seq(pool, seqs[i])) return PA_ERR_BAD_INDEX;
    for (int32_t i = 0; i < n; ++i) {
        const auto &s = pool->seqs[seqs[i]];
        if ((int64_t)s.table.size() > max_blocks) return PA_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        const auto &s = pool->seqs[seqs[i]];
        int32_t *row = tables_out + (int64_t)i * max_blocks;
        const size_t k = s.table.size();
        if (k) std::memcpy(row, s.table.data(), k * sizeof(int32_t));
        std::fill(row + k, row + max_blocks, pad);
        lens_out[i] = (int32_t)s.len;
    }
    return PA_OK;
}

int32_t pa_pool_num_free(const pa_pool *pool) {
    return pool ? (int32_t)pool->free_list.size() : -PA_ERR_INVALID;
}

int32_t pa_block_refcount(const pa_pool *pool, int32_t block) {
    if (!pool || block < 0 || block >= pool->num_blocks) return -PA_ERR_BAD_INDEX;
    return pool->ref[block];
}

int32_t pa_pool_get_stats(const pa_pool *pool, pa_pool_stats *out) {
    if (!pool || !out) return PA_ERR_INVALID;
    pa_pool_stats st{};
    st.num_blocks = pool->num_blocks;
    st.block_size = pool->B;
    st.free_blocks = (int32_t)pool->free_list.size();
    for (int32_t r : pool->ref) {
        if (r >= 1) ++st.used_blocks;
        if (r >= 2) ++st.shared_blocks;
    }
    st.live_seqs = pool->live;
    st.cow_copies = pool->cow_copies;
    for (const auto &s : pool->seqs) {
        if (!s.live) continue;
        st.tokens += s.len;
        st.table_slots += (int64_t)s.table.size() * pool->B;
    }
    st.padded_slots = st.table_slots - st.tokens;
    *out = st;
    return PA_OK;
}

int32_t pa_seq_swap_out(pa_pool *dev, pa_pool *host, int32_t seq, int32_t *host_seq, int64_t *pairs_out,
                        int32_t *n_pairs) {
    if (!dev || !host || !host_seq || !n_pairs || dev == host || dev->B != host->B) return PA_ERR_INVALID;
    if (!valid_seq(dev, seq)) return PA_ERR_BAD_INDEX;
    const pa_seq_rec &s = dev->seqs[seq];
    const int64_t nb = (int64_t)s.table.size();
    if (nb > 0 && !pairs_out) return PA_ERR_INVALID;
    if (nb > available(host)) return PA_ERR_OOM;
    // host copy of the sequence: one private host slot per block, same length
    const int32_t h = pa_seq_create(host);
    pa_seq_rec &hs = host->seqs[h];
    for (int64_t j = 0; j < nb; ++j) {
        const int32_t hb = take_block(host);
        hs.table.push_back(hb);
        pairs_out[2 * j] = s.table[j];
        pairs_out[2 * j + 1] = hb;
    }
    hs.len = s.len;
    *host_seq = h;
    *n_pairs = (int32_t)nb;
    pa_seq_free(dev, seq);  // blocks still used by other sequences stay on the device
    return PA_OK;
}

int32_t pa_seq_swap_in(pa_pool *dev, pa_pool *host, int32_t host_seq, int32_t *dev_seq, int64_t *pairs_out,
                       int32_t *n_pairs) {
    if (!dev || !host || !dev_seq || !n_pairs || dev == host || dev->B != host->B) return PA_ERR_INVALID;
    if (!valid_seq(host, host_seq)) return PA_ERR_BAD_INDEX;
    const pa_seq_rec &hs = host->seqs[host_seq];
    const int64_t nb = (int64_t)hs.table.size();
    if (nb > 0 && !pairs_out) return PA_ERR_INVALID;
    if (nb > available(dev)) return PA_ERR_OOM;
    const int32_t d = pa_seq_create(dev);
    pa_seq_rec &ds = dev->seqs[d];
    for (int64_t j = 0; j < nb; ++j) {
        const int32_t db = take_block(dev);
        ds.table.push_back(db);
        pairs_out[2 * j] = hs.table[j];
        pairs_out[2 * j + 1] = db;
    }
    ds.len = hs.len;
    *dev_seq = d;
    *n_pairs = (int32_t)nb;
    pa_seq_free(host, host_seq);
    return PA_OK;
}

int32_t pa_copy_pairs_check(const int64_t *pairs, int32_t num_pairs, int32_t num_blocks) {
    if (num_pairs < 0 || num_blocks <= 0 || (num_pairs > 0 && !pairs)) return PA_ERR_INVALID;
    std::vector<int64_t> dst;
    try {
        dst.reserve((size_t)num_pairs);
    } catch (const std::bad_alloc &) {
        return PA_ERR_OOM;
    }
    for (int32_t i = 0; i < num_pairs; ++i) {
        const int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PA_ERR_BAD_INDEX;
        dst.push_back(d);
    }
    std::sort(dst.begin(), dst.end());
    if (std::adjacent_find(dst.begin(), dst.end()) != dst.end()) return PA_ERR_INVALID;
    for (int32_t i = 0; i < num_pairs; ++i)
        if (std::binary_search(dst.begin(), dst.end(), pairs[2 * i])) return PA_ERR_INVALID;
    return PA_OK;
}

int32_t pa_pool_set_fail_after(pa_pool *pool, int32_t n) {
    if (!pool) return PA_ERR_INVALID;
    pool->fail_budget = n < 0 ? -1 : n;
    return PA_OK;
}

}  // extern "C"
