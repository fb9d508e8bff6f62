// host_stress.cpp -- random operation streams over the host side of libpa (the
// block allocator, copy-on-write, swap pools and the prefix cache), for builds
// with AddressSanitizer / UndefinedBehaviorSanitizer.  Links the allocator and
// prefix-cache sources directly; no GPU or CUDA runtime is involved.
//
// After every operation it checks the pool's bookkeeping against a plain model
// of what the sequences hold:
//   - each block's refcount = its occurrences in the live tables (+1 while the
//     prefix cache keeps it), so sum(refcount) = sum(table lengths) + cached;
//   - the free count = the number of blocks with refcount 0;
//   - a table has ceil(len / B) entries, every entry a block in range;
//   - appends return slots in the sequence's own blocks, and a failed
//     (out-of-memory) call leaves tables, lengths and the free count unchanged.
// Usage: host_stress <seed> <operations>; exit status 0 when every check holds.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "pa.h"

namespace {

struct Rng {  // xorshift64*
    uint64_t s;
    explicit Rng(uint64_t seed) : s(seed * 0x9E3779B97F4A7C15ull + 1) {}
    uint64_t next() {
        s ^= s >> 12;
        s ^= s << 25;
        s ^= s >> 27;
        return s * 0x2545F4914F6CDD1Dull;
    }
    int below(int n) { return n <= 0 ? 0 : (int)(next() % (uint64_t)n); }
};

int g_failures = 0;
#define CHECK(cond, ...)                                                    \
    do {                                                                    \
        if (!(cond)) {                                                      \
            std::fprintf(stderr, "check failed at line %d: ", __LINE__);     \
            std::fprintf(stderr, __VA_ARGS__);                              \
            std::fprintf(stderr, "\n");                                     \
            if (++g_failures > 20) std::exit(1);                            \
        }                                                                   \
    } while (0)

struct Seq {
    int32_t id;
    std::vector<int32_t> tokens;  // one token id per stored position
};

struct World {
    int32_t N, B, host_N;
    pa_pool *dev = nullptr;
    pa_pool *host = nullptr;
    pa_prefix_cache *cache = nullptr;
    std::vector<Seq> live;      // device sequences
    std::vector<Seq> swapped;   // host sequences (ids in the host pool)
    std::vector<std::vector<int32_t>> prompts;
};

std::vector<int32_t> table_of(const pa_pool *p, int32_t id) {
    int32_t n = pa_seq_table(p, id, nullptr, 0);
    std::vector<int32_t> t(n > 0 ? n : 0);
    if (n > 0) pa_seq_table(p, id, t.data(), n);
    return t;
}

// Refcounts of `pool` against the tables of `seqs`, plus `cached` blocks held elsewhere.
void check_pool(const pa_pool *pool, int32_t N, int32_t B, const std::vector<Seq> &seqs, int32_t cached,
                const char *what) {
    std::vector<int64_t> uses(N, 0);
    int64_t entries = 0;
    for (const Seq &s : seqs) {
        const int32_t len = pa_seq_len(pool, s.id);
        CHECK(len == (int32_t)s.tokens.size(), "%s: seq %d len %d, model %zu", what, s.id, len, s.tokens.size());
        const std::vector<int32_t> t = table_of(pool, s.id);
        CHECK((int64_t)t.size() == ((int64_t)len + B - 1) / B, "%s: seq %d has %zu blocks for %d tokens", what, s.id,
              t.size(), len);
        for (int32_t b : t) {
            CHECK(b >= 0 && b < N, "%s: seq %d holds block %d", what, s.id, b);
            if (b >= 0 && b < N) ++uses[b];
        }
        entries += (int64_t)t.size();
    }
    int64_t refsum = 0, zero = 0;
    for (int32_t b = 0; b < N; ++b) {
        const int32_t r = pa_block_refcount(pool, b);
        CHECK(r >= 0, "%s: refcount(%d) = %d", what, b, r);
        CHECK(r >= uses[b], "%s: block %d refcount %d below its %lld table uses", what, b, r, (long long)uses[b]);
        CHECK(r <= uses[b] + 1, "%s: block %d refcount %d above uses %lld + 1", what, b, r, (long long)uses[b]);
        refsum += r;
        if (r == 0) ++zero;
    }
    CHECK(refsum == entries + cached, "%s: refcounts sum to %lld, tables %lld + cached %d", what, (long long)refsum,
          (long long)entries, cached);
    CHECK(pa_pool_num_free(pool) == zero, "%s: %d free, %lld blocks at refcount 0", what, pa_pool_num_free(pool),
          (long long)zero);
    pa_pool_stats st{};
    CHECK(pa_pool_get_stats(pool, &st) == PA_OK, "%s: stats", what);
    CHECK(st.free_blocks == pa_pool_num_free(pool), "%s: stats free %d", what, st.free_blocks);
}

void check_all(World &w) {
    const int32_t cached = pa_prefix_cached_blocks(w.cache);
    check_pool(w.dev, w.N, w.B, w.live, cached, "device");
    check_pool(w.host, w.host_N, w.B, w.swapped, 0, "host");
}

// Slots of the last n positions of a sequence must lie in its own blocks.
void check_slots(const pa_pool *p, int32_t B, const Seq &s, const int64_t *slots, int32_t n) {
    const std::vector<int32_t> t = table_of(p, s.id);
    const int32_t len = (int32_t)s.tokens.size();
    for (int32_t i = 0; i < n; ++i) {
        const int32_t pos = len - n + i;
        const int64_t want = (int64_t)t[pos / B] * B + pos % B;
        CHECK(slots[i] == want, "slot of seq %d pos %d: %lld, want %lld", s.id, pos, (long long)slots[i],
              (long long)want);
    }
}

}  // namespace

namespace {

std::vector<int32_t> random_tokens(Rng &r, int32_t n) {
    std::vector<int32_t> t(n);
    for (int32_t &x : t) x = r.below(3);
    return t;
}

// Append n tokens to s; on success its model grows, on out-of-memory nothing may change.
bool append(World &w, Rng &r, Seq &s, int32_t n) {
    const std::vector<int32_t> before = table_of(w.dev, s.id);
    const int32_t free_before = pa_pool_num_free(w.dev);
    std::vector<int64_t> slots(n > 0 ? n : 1);
    int64_t pair[2] = {-1, -1};
    int32_t n_cow = -1;
    const int32_t rc = pa_seq_append(w.dev, s.id, n, slots.data(), pair, &n_cow);
    if (rc == PA_ERR_OOM) {
        CHECK(table_of(w.dev, s.id) == before, "failed append changed seq %d's table", s.id);
        CHECK(pa_pool_num_free(w.dev) == free_before, "failed append changed the free count");
        return false;
    }
    CHECK(rc == PA_OK, "append returned %d", rc);
    if (rc != PA_OK) return false;
    const int32_t len0 = (int32_t)s.tokens.size();
    const std::vector<int32_t> extra = random_tokens(r, n);
    s.tokens.insert(s.tokens.end(), extra.begin(), extra.end());
    check_slots(w.dev, w.B, s, slots.data(), n);
    const std::vector<int32_t> after = table_of(w.dev, s.id);
    if (n_cow == 1) {  // the partial last block was copied: old id out, new id in its place
        const int32_t j = len0 / w.B;
        CHECK(len0 % w.B != 0 && j < (int32_t)before.size(), "copy without a partial last block");
        if (len0 % w.B != 0 && j < (int32_t)before.size()) {
            CHECK(pair[0] == before[j] && pair[1] == after[j], "copy pair (%lld, %lld) for block %d -> %d",
                  (long long)pair[0], (long long)pair[1], before[j], after[j]);
        }
    } else {
        CHECK(n_cow == 0, "n_cow %d", n_cow);
        for (size_t j = 0; j < before.size(); ++j) CHECK(after[j] == before[j], "table entry %zu moved", j);
    }
    return true;
}

void op_create(World &w, Rng &r) {
    if (w.live.size() >= 48) return;
    const std::vector<int32_t> &prompt = w.prompts[r.below((int)w.prompts.size())];
    const int32_t L = 1 + r.below((int32_t)prompt.size());
    std::vector<int32_t> matched(L / w.B + 1);
    const int32_t n = pa_prefix_match(w.cache, prompt.data(), L, matched.data(), (int32_t)matched.size());
    CHECK(n >= 0 && (int64_t)n * w.B <= L, "match returned %d for %d tokens", n, L);
    Seq s;
    s.id = n > 0 ? pa_seq_create_from_prefix(w.dev, matched.data(), n) : pa_seq_create(w.dev);
    CHECK(s.id >= 0, "create returned %d", s.id);
    if (s.id < 0) return;
    s.tokens.assign(prompt.begin(), prompt.begin() + (int64_t)n * w.B);
    w.live.push_back(s);
    Seq &t = w.live.back();
    const int32_t rest = L - n * w.B;
    if (rest > 0 && append(w, r, t, rest)) {
        // the prompt's tokens, not random ones, so later requests can match them
        for (int32_t i = n * w.B; i < L; ++i) t.tokens[i] = prompt[i];
    }
}

void op_fork(World &w, Rng &r) {
    if (w.live.empty() || w.live.size() >= 48) return;
    const Seq &p = w.live[r.below((int)w.live.size())];
    const int32_t id = pa_seq_fork(w.dev, p.id);
    CHECK(id >= 0, "fork returned %d", id);
    if (id >= 0) w.live.push_back(Seq{id, p.tokens});
}

void op_append(World &w, Rng &r) {
    if (w.live.empty()) return;
    append(w, r, w.live[r.below((int)w.live.size())], 1 + r.below(2 * w.B));
}

void op_batch(World &w, Rng &r) {
    if (w.live.empty()) return;
    std::vector<int> pick;
    for (int i = 0; i < (int)w.live.size(); ++i)
        if (r.below(3) == 0) pick.push_back(i);
    if (pick.empty()) return;
    const int32_t each = 1 + r.below(2);
    std::vector<int32_t> ids;
    std::vector<std::vector<int32_t>> before;
    for (int i : pick) {
        ids.push_back(w.live[i].id);
        before.push_back(table_of(w.dev, w.live[i].id));
    }
    const int32_t free_before = pa_pool_num_free(w.dev);
    std::vector<int64_t> slots(ids.size() * each), pairs(2 * ids.size());
    int32_t n_cow = -1;
    const int32_t rc = pa_seq_append_batch(w.dev, ids.data(), (int32_t)ids.size(), each, slots.data(), pairs.data(),
                                           &n_cow);
    if (rc == PA_ERR_OOM) {
        for (size_t k = 0; k < ids.size(); ++k)
            CHECK(table_of(w.dev, ids[k]) == before[k], "failed batch changed seq %d", ids[k]);
        CHECK(pa_pool_num_free(w.dev) == free_before, "failed batch changed the free count");
        return;
    }
    CHECK(rc == PA_OK, "batch append returned %d", rc);
    if (rc != PA_OK) return;
    CHECK(n_cow >= 0 && n_cow <= (int32_t)ids.size(), "batch n_cow %d", n_cow);
    CHECK(pa_copy_pairs_check(pairs.data(), n_cow, w.N) == PA_OK,
          "batch copy pairs fail the host check");
    for (size_t k = 0; k < pick.size(); ++k) {
        Seq &s = w.live[pick[k]];
        const std::vector<int32_t> extra = random_tokens(r, each);
        s.tokens.insert(s.tokens.end(), extra.begin(), extra.end());
        check_slots(w.dev, w.B, s, slots.data() + k * each, each);
    }
    // a duplicate id is refused and changes nothing
    if (ids.size() >= 1) {
        const int32_t dup[2] = {ids[0], ids[0]};
        const int32_t f = pa_pool_num_free(w.dev);
        CHECK(pa_seq_append_batch(w.dev, dup, 2, 1, slots.data(), pairs.data(), &n_cow) == PA_ERR_INVALID,
              "duplicate ids accepted");
        CHECK(pa_pool_num_free(w.dev) == f, "refused batch changed the free count");
    }
}

void op_free(World &w, Rng &r) {
    if (w.live.empty()) return;
    const int i = r.below((int)w.live.size());
    CHECK(pa_seq_free(w.dev, w.live[i].id) == PA_OK, "free");
    w.live.erase(w.live.begin() + i);
}

void op_swap_out(World &w, Rng &r) {
    if (w.live.empty()) return;
    const int i = r.below((int)w.live.size());
    const int32_t nb = (int32_t)table_of(w.dev, w.live[i].id).size();
    std::vector<int64_t> pairs(2 * (nb > 0 ? nb : 1));
    int32_t host_id = -1, n = -1;
    const int32_t rc = pa_seq_swap_out(w.dev, w.host, w.live[i].id, &host_id, pairs.data(), &n);
    if (rc == PA_ERR_OOM) return;
    CHECK(rc == PA_OK && n == nb, "swap out rc %d, %d pairs for %d blocks", rc, n, nb);
    if (rc != PA_OK) return;
    w.swapped.push_back(Seq{host_id, w.live[i].tokens});
    w.live.erase(w.live.begin() + i);
}

void op_swap_in(World &w, Rng &r) {
    if (w.swapped.empty() || w.live.size() >= 48) return;
    const int i = r.below((int)w.swapped.size());
    const int32_t nb = (int32_t)table_of(w.host, w.swapped[i].id).size();
    std::vector<int64_t> pairs(2 * (nb > 0 ? nb : 1));
    int32_t dev_id = -1, n = -1;
    const int32_t rc = pa_seq_swap_in(w.dev, w.host, w.swapped[i].id, &dev_id, pairs.data(), &n);
    if (rc == PA_ERR_OOM) return;
    CHECK(rc == PA_OK && n == nb, "swap in rc %d, %d pairs for %d blocks", rc, n, nb);
    if (rc != PA_OK) return;
    w.live.push_back(Seq{dev_id, w.swapped[i].tokens});
    w.swapped.erase(w.swapped.begin() + i);
}

void op_insert(World &w, Rng &r) {
    if (w.live.empty()) return;
    const Seq &s = w.live[r.below((int)w.live.size())];
    const std::vector<int32_t> t = table_of(w.dev, s.id);
    const int32_t rc = pa_prefix_insert(w.cache, s.tokens.data(), (int32_t)s.tokens.size(), t.data(),
                                        (int32_t)t.size());
    CHECK(rc >= 0 || rc == -PA_ERR_INVALID, "insert returned %d", rc);
}

void op_evict(World &w, Rng &r) {
    const int32_t before = pa_prefix_cached_blocks(w.cache);
    const int32_t n = pa_prefix_evict(w.cache, 1 + r.below(8));
    CHECK(n >= 0 && pa_prefix_cached_blocks(w.cache) == before - n, "evict %d of %d", n, before);
}

void op_fail_after(World &w, Rng &r) { pa_pool_set_fail_after(w.dev, r.below(4) == 0 ? -1 : r.below(6)); }

void op_export(World &w, Rng &r) {
    if (w.live.empty()) return;
    std::vector<int32_t> ids;
    int32_t longest = 0;
    for (const Seq &s : w.live)
        if (r.below(2) == 0) {
            ids.push_back(s.id);
            const int32_t nb = (int32_t)table_of(w.dev, s.id).size();
            longest = nb > longest ? nb : longest;
        }
    if (ids.empty()) return;
    const int32_t cols = (longest > 0 ? longest : 1) + r.below(3);  // at least one column
    std::vector<int32_t> tables(ids.size() * cols), lens(ids.size());
    CHECK(pa_pool_export(w.dev, ids.data(), (int32_t)ids.size(), 0, -1, tables.data(), lens.data()) == PA_ERR_INVALID,
          "export into zero columns accepted");
    CHECK(pa_pool_export(w.dev, ids.data(), (int32_t)ids.size(), cols, -1, tables.data(), lens.data()) == PA_OK,
          "export");
    for (size_t k = 0; k < ids.size(); ++k) {
        const std::vector<int32_t> t = table_of(w.dev, ids[k]);
        CHECK(lens[k] == pa_seq_len(w.dev, ids[k]), "exported length");
        for (int32_t j = 0; j < cols; ++j)
            CHECK(tables[k * cols + j] == (j < (int32_t)t.size() ? t[j] : -1), "exported table");
    }
    if (longest > 0)
        CHECK(pa_pool_export(w.dev, ids.data(), (int32_t)ids.size(), longest - 1, -1, tables.data(), lens.data()) ==
                  PA_ERR_INVALID, "export into too few columns accepted");
}

}  // namespace

int main(int argc, char **argv) {
    const uint64_t seed = argc > 1 ? std::strtoull(argv[1], nullptr, 10) : 1;
    const long ops = argc > 2 ? std::strtol(argv[2], nullptr, 10) : 20000;
    Rng r(seed);
    const int32_t block_sizes[4] = {1, 2, 4, 16};
    World w;
    w.B = block_sizes[r.below(4)];
    w.N = 48 + r.below(96);
    w.host_N = w.N / 2;
    std::vector<int32_t> order(w.N);
    for (int32_t i = 0; i < w.N; ++i) order[i] = i;
    for (int32_t i = w.N - 1; i > 0; --i) std::swap(order[i], order[r.below(i + 1)]);
    w.dev = pa_pool_create(w.N, w.B, order.data());
    w.host = pa_pool_create(w.host_N, w.B, nullptr);
    w.cache = pa_prefix_cache_create(w.dev);
    if (!w.dev || !w.host || !w.cache) {
        std::fprintf(stderr, "set-up failed\n");
        return 1;
    }
    CHECK(pa_pool_create(0, w.B, nullptr) == nullptr && pa_pool_create(4, 0, nullptr) == nullptr, "bad pool accepted");
    for (int p = 0; p < 4; ++p) w.prompts.push_back(random_tokens(r, 1 + r.below(6 * w.B)));
    void (*table[])(World &, Rng &) = {op_create, op_create, op_fork,   op_append,   op_append,  op_append,
                                       op_batch,  op_free,   op_free,   op_swap_out, op_swap_in, op_insert,
                                       op_insert, op_evict,  op_export, op_fail_after};
    const int kinds = (int)(sizeof(table) / sizeof(table[0]));
    for (long i = 0; i < ops && g_failures == 0; ++i) {
        table[r.below(kinds)](w, r);
        check_all(w);
    }
    // tear down: every block returns to its pool
    pa_pool_set_fail_after(w.dev, -1);
    pa_prefix_cache_destroy(w.cache);
    w.cache = nullptr;
    for (const Seq &s : w.live) CHECK(pa_seq_free(w.dev, s.id) == PA_OK, "final free");
    for (const Seq &s : w.swapped) CHECK(pa_seq_free(w.host, s.id) == PA_OK, "final host free");
    CHECK(pa_pool_num_free(w.dev) == w.N && pa_pool_num_free(w.host) == w.host_N, "blocks lost: %d/%d and %d/%d free",
          pa_pool_num_free(w.dev), w.N, pa_pool_num_free(w.host), w.host_N);
    pa_pool_stats st{};
    pa_pool_get_stats(w.dev, &st);
    pa_pool_destroy(w.dev);
    pa_pool_destroy(w.host);
    std::printf("seed %llu: %ld operations, B=%d N=%d, %lld copy-on-write copies, %d failures\n",
                (unsigned long long)seed, ops, w.B, w.N, (long long)st.cow_copies, g_failures);
    return g_failures == 0 ? 0 : 1;
}
