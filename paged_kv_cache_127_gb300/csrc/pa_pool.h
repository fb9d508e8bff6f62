// pa_pool.h -- internal layout of the host block pool, shared by the
// allocator (pa_alloc.cpp) and the prefix cache (pa_prefix.cpp).
#pragma once

#include <cstdint>
#include <deque>
#include <vector>

#include "../../include/pa.h"

struct pa_seq_rec {
    std::vector<int32_t> table;
    int64_t len = 0;
    bool live = false;
    uint32_t batch_mark = 0;  // batch calls: the call that last listed this sequence
};

struct pa_pool {
    int32_t num_blocks = 0;
    int32_t B = 0;
    std::deque<int32_t> free_list;
    std::vector<int32_t> ref;
    std::vector<pa_seq_rec> seqs;
    int32_t live = 0;
    int64_t cow_copies = 0;
    int64_t fail_budget = -1;  // < 0: unlimited
    // scratch of pa_seq_append_batch, kept between calls so a call allocates nothing
    uint32_t batch_epoch = 0;
    std::vector<int32_t> given_up;   // per block: copies made earlier in the batch (zero outside a call)
    std::vector<int32_t> touched;    // blocks whose given_up count is nonzero
};


namespace pa_pool_detail {

inline int64_t available(const pa_pool *p) {
    int64_t f = (int64_t)p->free_list.size();
    if (p->fail_budget >= 0 && p->fail_budget < f) f = p->fail_budget;
    return f;
}

// Drop one reference; a block reaching zero goes to the back of the free list.
inline void release_block(pa_pool *p, int32_t b) {
    if (--p->ref[b] == 0) p->free_list.push_back(b);
}

}  // namespace pa_pool_detail
