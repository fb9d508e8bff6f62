// pa_chunk_umma.cuh -- chunk attention for long query chunks (chunked prefill)
// on the 5th-generation tensor cores: tcgen05.mma with operands in shared
// memory and the accumulators in tensor memory (TMEM).
//
// What is computed is what pa_chunk_mma.cuh computes (the query at position
// pos = len_s - n_s + t attends to keys 0..pos; "Paged Attention and vLLM",
// "KV Cache Fundamentals" and "Block Table and Logical-to-Physical Mapping"),
// for chunks whose (query token, query head) rows fill 128-row tiles.
//
// Work: a work item is (MT 128-row tiles, KV head, sequence); the rows of a
// KV head are r = t * G + gq.  The item's CTA walks the visible context in
// steps of PA_CHUNK_UMMA_KEYS keys, with no split across CTAs (a tile has
// enough rows to keep the tensor cores busy), so there is no merge.  MT = 2
// tiles share every K/V load and give the softmax two warpgroups.  The kernel
// is persistent, one CTA per SM: each CTA claims items from the plan's
// longest-first list one at a time and keeps TMEM, barriers and rings from
// item to item; the next item's query tiles (a second set) and first S overlap
// the finished item's epilogue, whose output leaves by TMA stores.  Warp roles:
//   warps 0, 2   producers of K and of V: 16-row TMA boxes (one KV head, both
//                128-byte halves of D) into two 3-stage rings, so that a K
//                stage is refilled as soon as its S MMAs complete, well before
//                the P V that frees the V stage; table entries outside the pool,
//                or keys past the context, are not loaded and are marked in a
//                per-stage mask;
//   warps 1, 3   issue tile 0's MMAs (lane 0), S in warp 1 (which also
//   (4, 5)       allocates TMEM, 256 columns per tile), P V in warp 3; warps 4
//                and 5 do the same for tile 1, so a tile waits only on itself:
//                  S_u,j = Q_u K_j^T   M 128, N = keys, K = D     -> TMEM S[u][j % kSB]
//                  O_u  += P_u,j V_j   M 128, N = D,    K = keys  -> TMEM O[u]
//                with P split into P_hi + P_lo (two bf16 / f16 operands) so
//                the probabilities keep ~16 significant bits;
//   warps 4.. (6.. with two tiles)  one softmax warpgroup per tile, one thread per row (TMEM
//                lane 32 * (warp % 4) + lane): read S, mask (causal and
//                not-loaded keys), online softmax in log2 units, write P_hi /
//                P_lo into TMEM over the S just read (the P V MMA takes its A
//                operand from TMEM), zero the V rows of keys that must not
//                contribute (their slots may hold anything); epilogue O / l.
// The running maximum is only moved when a row's new maximum exceeds it by
// more than 2^8 (exp2 units): until then the weights are exp2(x - m) <= 256,
// exact in fp32, and O and l share the stale maximum, so the result is the
// same softmax; moving it costs a read-modify-write of the row of O in TMEM.
//
// Synchronisation is by mbarriers only, every wait bounded: on a timeout the
// kernel sets PA_DEVERR_TIMEOUT, waits (bounded) for the MMAs and copies it
// issued, frees its TMEM and returns.
#pragma once

#include <cuda.h>

#include <cmath>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_mma.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

// Keys per step (PA_CHUNK_UMMA_KEYS): each tile has 128 TMEM columns for S/P
// buffers, so 128 / keys of them (a step's S may run that many steps minus one
// ahead of the P V that frees its buffer).

template <int D, int MT>
struct UmmaCfg {
    static constexpr int kM = 128;                         // rows per tile (TMEM lanes)
    static constexpr int kMT = MT;                         // tiles per CTA
    static constexpr int kN = PA_CHUNK_UMMA_KEYS;          // keys per step
    static constexpr int kSB = 128 / kN;                   // S/P buffers per tile
    static constexpr int kBoxes = kN / 16;                 // 16-row TMA boxes per step
    static constexpr int kSub = D / 64;                    // 128-byte halves of a row
    static constexpr int kKS = D / 16;                     // k-steps of S = Q K^T
    static constexpr int kStages = kN == 64 ? 3 : 6;
    // warps: 0 K producer, 2 V producer; per tile u an S issuer (warp 1, 4) and a
    // P V issuer (warp 3, 5); then one softmax warpgroup per tile
    static constexpr int kSoftWarp0 = MT == 2 ? 6 : 4;
    static constexpr int kThreads = 32 * (kSoftWarp0 + 4 * MT);
    static constexpr int kHalf = kN * 128;                 // one half of K (or V) of a step
    static constexpr int kTile = kSub * kHalf;             // K (or V) of a step
    static constexpr int kStageBytes = 2 * kTile;
    static constexpr int kQTile = kSub * kM * 128;         // Q of one tile (kSub halves of kM x 128 bytes)
    static constexpr int kQHalf = kM * 128;
    // two sets of query tiles: a CTA loads the next work item's while its
    // epilogue stages the finished item's output through the other set
    static constexpr size_t kQOff = 0;
    static constexpr size_t kKVOff = kQOff + (size_t)2 * MT * kQTile;
    static constexpr size_t kBarOff = kKVOff + (size_t)kStages * kStageBytes;
    // k_full, k_empty, v_full, v_empty, v_zeroed [kStages] | per tile: s_full, p_full, o_done [kSB],
    // q_full [2], q_free [2], drain_s, drain_p, item_ready [2]
    static constexpr int kTileBars = 3 * kSB + 8;
    static constexpr int kNumBars = 5 * kStages + MT * kTileBars;
    static constexpr size_t kMaskOff = kBarOff + 8 * kNumBars;
    static constexpr size_t kSlotOff = kMaskOff + 4 * kStages;
    // published work items: per tile and query-tile set, 16 ints (UmmaSlot)
    static constexpr size_t kItemOff = kSlotOff + 16;
    static constexpr size_t kSmem = kItemOff + (size_t)MT * 2 * 64 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 256 * MT;
    static constexpr uint32_t kOCol = 128 * MT;            // S[u][b] at 128 u + kN b; O[u] at kOCol + D u
    // P[u][b] aliases S[u][b]: P_hi in its first kN / 2 columns, P_lo in the next
    // kN / 2 (two 16-bit values per column)
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(MT == 1 || MT == 2, "tiles per CTA");
    static_assert(kN == 32 || kN == 64, "keys per step");
    static_assert(kOCol + MT * D <= kTmemCols, "TMEM budget");
    static_assert(kKVOff % 1024 == 0, "swizzle atoms 1024-byte aligned");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert(kQTile % 16384 == 0, "query tile holds whole 16 KB output boxes");
};

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// TMA store of one box from shared memory (bulk-group completion), and the
// waits on this thread's stores: until at most N are still reading shared
// memory, and until all have completed.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int x, int y, int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3}], [%4], %5;" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(src), "l"(policy)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Barrier over the 128 threads of one softmax warpgroup (ids 1 and 2; 0 is __syncthreads).
__device__ __forceinline__ void warpgroup_sync(int id) {
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}
// The same barrier, returning whether `pred` holds in all 128 threads.
__device__ __forceinline__ bool warpgroup_all(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id)
        : "memory");
    return r != 0;
}

// One work item of the tcgen05 path: KV head kvh of the plan's entry (sequence
// s, tile group), i.e. rows r0 .. r0 + 128 MT - 1 of that head's
// (query token, query head) rows, and the steps of keys those rows see.
struct UmmaItem {
    int s, kvh, r0, qs, n, len, tiles, nch;
};
// A work item as the K producer publishes it to a tile's roles, or the end
// mark (no more items).
struct UmmaSlot {
    UmmaItem it;
    int end;
};

// Work index w = entry * Hkv + kvh of the plan's longest-first list; false
// past the list's end or when the entry has no rows (every role skips it alike).
template <typename C>
__device__ __forceinline__ bool umma_item(const ChunkArgs &a, int w, int nwork, UmmaItem &it) {
    if (w >= nwork) return false;
    const int4 e = a.plan_list[w / a.Hkv];
    const int G = a.Hq / a.Hkv;
    it.s = e.x;
    it.kvh = w % a.Hkv;
    it.r0 = e.y * C::kM * C::kMT;
    it.qs = a.query_start[it.s];
    it.n = a.query_start[it.s + 1] - it.qs;
    if (it.n <= 0 || it.r0 >= it.n * G) return false;
    it.len = a.context_lens[it.s];
    it.tiles = min(C::kMT, (it.n * G - it.r0 + C::kM - 1) / C::kM);  // tiles with at least one row
    const int t_last = min(it.n - 1, (it.r0 + C::kM * it.tiles - 1) / G);
    it.nch = (it.len - it.n + t_last) / C::kN + 1;                // kN-key steps up to the last position
    return true;
}

// Persistent: each CTA's K producer claims the entries of the plan's
// longest-first list one at a time (an atomic counter, so an SM takes the next
// longest item as soon as it is ready for one) and publishes each to the roles
// of every tile, through a shared-memory slot per tile and query-tile set; the
// CTA keeps its TMEM, barriers and K/V ring across items.
// Every tile's roles see every item, and those of a tile without rows in it
// only release its ring stages.  The ring's stage and phase follow the count g
// of steps so far, the S/P buffers and their phases the count c of the tile's
// own steps, the slots and query-tile sets the count of items published.
template <typename T, int D, int B, int MT>
__global__ void __launch_bounds__(UmmaCfg<D, MT>::kThreads, 1)
    chunk_umma_kernel(const ChunkArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmo) {
    using C = UmmaCfg<D, MT>;
    using M = Mma16<T>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *basep = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    griddep_wait();  // the plan kernel's list of (sequence, tile group), longest first
    const int nwork = a.plan_hdr[0] * a.Hkv;
    if ((int)blockIdx.x >= nwork) return;
    const int G = a.Hq / a.Hkv;

    const uint32_t qb = base + (uint32_t)C::kQOff;
    const uint32_t kvb = base + (uint32_t)C::kKVOff;
    const uint32_t bars = base + (uint32_t)C::kBarOff;
    auto k_full = [&](int i) { return bars + 8u * (uint32_t)i; };
    auto k_empty = [&](int i) { return bars + 8u * (uint32_t)(C::kStages + i); };
    auto v_full = [&](int i) { return bars + 8u * (uint32_t)(2 * C::kStages + i); };
    auto v_empty = [&](int i) { return bars + 8u * (uint32_t)(3 * C::kStages + i); };
    // tile 0's softmax has zeroed this step's V rows that must not contribute
    auto v_zeroed = [&](int i) { return bars + 8u * (uint32_t)(4 * C::kStages + i); };
    auto tbar = [&](int u, int i) { return bars + 8u * (uint32_t)(5 * C::kStages + u * C::kTileBars + i); };
    constexpr int kSB = C::kSB;
    auto s_full = [&](int u, int b) { return tbar(u, b); };
    auto p_full = [&](int u, int b) { return tbar(u, kSB + b); };
    // P V of a step on buffer b complete: O is up to date and S/P[u][b] may be rewritten
    auto o_done = [&](int u, int b) { return tbar(u, 2 * kSB + b); };
    auto q_full = [&](int u, int x) { return tbar(u, 3 * kSB + x); };
    // the epilogue has finished with query-tile set x of tile u (its staging area)
    auto q_free = [&](int u, int x) { return tbar(u, 3 * kSB + 2 + x); };
    auto drain_s = [&](int u) { return tbar(u, 3 * kSB + 4); };
    auto drain_p = [&](int u) { return tbar(u, 3 * kSB + 5); };
    // the K producer has published tile u's next item in slot x
    auto item_ready = [&](int u, int x) { return tbar(u, 3 * kSB + 6 + x); };
    UmmaSlot *slots = reinterpret_cast<UmmaSlot *>(basep + C::kItemOff);
    auto slot = [&](int u, int x) -> UmmaSlot & { return slots[2 * u + x]; };
    // wait for tile u's k-th published item (slot k & 1) and read it
    auto take = [&](int u, int k, UmmaSlot &out) {
        const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(item_ready(u, k & 1), (uint32_t)(k >> 1) & 1u, kWaitLimit));
        if (got) out = slot(u, k & 1);
        return got;
    };
    auto qtile = [&](int x, int u) { return qb + (uint32_t)((x * MT + u) * C::kQTile); };
    auto s_col = [&](int u, int b) { return (uint32_t)(128 * u + C::kN * b); };
    auto o_col = [&](int u) { return C::kOCol + (uint32_t)(D * u); };
    int *vmask = reinterpret_cast<int *>(basep + C::kMaskOff);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(basep + C::kSlotOff);

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), MT);  // one arrival per tile's S issuer (a commit, or a plain
            mbar_init(v_full(i), 1);    // arrival when the item has no rows in that tile)
            mbar_init(v_empty(i), MT);  // likewise from each tile's P V issuer
            mbar_init(v_zeroed(i), 4);
        }
        for (int u = 0; u < MT; ++u) {
            for (int b = 0; b < kSB; ++b) {
                mbar_init(s_full(u, b), 1);
                mbar_init(p_full(u, b), 4);
                mbar_init(o_done(u, b), 1);
            }
            for (int x = 0; x < 2; ++x) {
                mbar_init(q_full(u, x), 1);
                mbar_init(q_free(u, x), 4 + 2);  // the softmax warps, and both MMA issuers once they have read the slot
                mbar_init(item_ready(u, x), 1);
            }
            mbar_init(drain_s(u), 1);
            mbar_init(drain_p(u), 1);
        }
        fence_mbar_init();
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmo);
    }
    if (warp == 1) tc::tmem_alloc(smem_addr(tslot), C::kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers: K (warp 0), V (warp 2)
        const bool is_v = warp == 2;
        const uint64_t pol = policy_evict_last();  // the other row tiles of this head reread these keys
        const uint64_t qpol = policy_evict_first();
        const CUtensorMap *map = is_v ? &tmv : &tmk;
        const uint32_t ring = kvb + (is_v ? (uint32_t)C::kTile : 0u);
        int g = 0;                  // ring steps issued
        int ku[MT];                 // items published to each tile so far (query-tile sets)
#pragma unroll
        for (int u = 0; u < MT; ++u) ku[u] = 0;
        int k0 = 0;                 // V producer: tile 0's items taken so far
        bool ok = true;
        for (;;) {
            UmmaItem it;
            if (!is_v) {
                // claim the next entry of the longest-first list (skipping entries
                // without rows); past its end, publish the end mark to every tile
                bool have = false;
                while (!have) {
                    int w = 0;
                    if (lane == 0) w = atomicAdd(&a.plan_hdr[1], 1);
                    w = __shfl_sync(0xffffffffu, w, 0);
                    if (w >= nwork) break;
                    have = umma_item<C>(a, w, nwork, it);
                }
                // every tile's roles see every item (a tile without rows in it releases
                // its ring stages); slot x of tile u is free once the tile's roles are
                // done with the item before last
                for (int u = 0; ok && u < MT; ++u) {
                    const int x = ku[u] & 1;
                    if (ku[u] >= 2) ok = mbar_wait_bounded(q_free(u, x), (uint32_t)((ku[u] >> 1) - 1) & 1u, kWaitLimit);
                    if (ok && lane == 0) {
                        UmmaSlot &sl = slot(u, x);
                        if (have) sl.it = it;
                        sl.end = have ? 0 : 1;
                        mbar_arrive(item_ready(u, x));
                        if (have && u >= it.tiles) {
                            mbar_arrive(q_full(u, x));  // no query tile: keep the set's phases in step
                        } else if (have) {
                            // the query tile: tile u holds rows r0 + 128 u .., i.e. tokens
                            // (r0 + 128 u) / G .. of the sequence's chunk, G heads each; rows
                            // of tokens past the chunk are never used (their keys are all masked)
                            mbar_arrive_expect_tx(q_full(u, x), (uint32_t)C::kQTile);
#pragma unroll
                            for (int sb = 0; sb < C::kSub; ++sb)
                                tma_load_3d(qtile(x, u) + (uint32_t)(sb * C::kQHalf), &tmq, sb * 64, it.kvh * G,
                                            it.qs + (it.r0 + C::kM * u) / G, q_full(u, x), qpol);
                        }
                    }
                    ++ku[u];
                }
                __syncwarp();
                if (!ok || !have) break;
            } else {
                // the V producer follows tile 0's items (tile 0 has rows in every item)
                UmmaSlot sl;
                ok = take(0, k0++, sl);
                if (!ok || sl.end) break;
                it = sl.it;
            }
            const int32_t *row = a.block_tables + (size_t)it.s * a.max_blocks;
            for (int j = 0; j < it.nch; ++j, ++g) {
                const int st = g % C::kStages;
                if (g >= C::kStages &&
                    !mbar_wait_bounded(is_v ? v_empty(st) : k_empty(st), (uint32_t)((g / C::kStages) - 1) & 1u,
                                       kWaitLimit)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    int mask = 0, blk[C::kBoxes];
#pragma unroll
                    for (int i = 0; i < C::kBoxes; ++i) {
                        const int tok = j * C::kN + 16 * i;
                        blk[i] = -1;
                        if (tok < it.len) {
                            const int pbk = row[tok / B];
                            if (pbk >= 0 && pbk < a.N) {
                                blk[i] = pbk;
                                mask |= 1 << i;
                            } else if (!is_v) {
                                set_error(a.err, PA_DEVERR_BAD_BLOCK);
                            }
                        }
                    }
                    if (is_v) vmask[st] = mask;  // read by the softmax after v_full (released with v_empty)
                    const uint32_t bar = is_v ? v_full(st) : k_full(st);
                    const uint32_t bytes = (uint32_t)__popc(mask) * C::kSub * 2048u;
                    if (bytes == 0) {
                        mbar_arrive(bar);
                    } else {
                        mbar_arrive_expect_tx(bar, bytes);
                        const uint32_t dst = ring + (uint32_t)(st * C::kStageBytes);
#pragma unroll
                        for (int i = 0; i < C::kBoxes; ++i) {
                            if (!(mask >> i & 1)) continue;
                            const int y = (j * C::kN + 16 * i) % B;
                            const int z = blk[i] * a.Hkv + it.kvh;
#pragma unroll
                            for (int sb = 0; sb < C::kSub; ++sb)
                                tma_load_3d(dst + (uint32_t)(sb * C::kHalf + i * 2048), map, sb * 64, y, z, bar, pol);
                        }
                    }
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (!ok && lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
        // copies still in flight must land before the CTA's shared memory is released
        for (int k = max(0, g - C::kStages); k < g; ++k)
            mbar_wait_bounded(is_v ? v_full(k % C::kStages) : k_full(k % C::kStages), (uint32_t)(k / C::kStages) & 1u,
                              kWaitLimit);
    } else if (warp == 1 || (MT == 2 && warp == 4)) {
        // ------------------------------------------------------------ S = Q K^T issuer of tile u
        // One issuer per tile: a tile waits for its own P V, not the other tile's.
        const int u = warp == 1 ? 0 : 1;
        constexpr uint32_t idesc_s = tc::f16_idesc(kBf16, false, C::kM, C::kN);
        // Descriptors built once: a step's operands are these plus compile-time
        // offsets (tc::desc_add), which keeps the issue loop to the MMAs themselves.
        const uint64_t kdesc0 = tc::sw128_desc(kvb, 16u, 1024u);
        int g = 0, c = 0, ku = 0;  // ring steps, this tile's steps, this tile's items
        bool ok = true;
        for (;;) {
            UmmaSlot sl;
            ok = take(u, ku, sl);
            if (!ok || sl.end) break;
            const UmmaItem it = sl.it;
            const int x = ku & 1;
            const uint32_t qpar = (uint32_t)(ku >> 1) & 1u;
            ++ku;
            if (lane == 0) mbar_arrive(q_free(u, x));  // done with the slot
            if (u >= it.tiles) {
                // no rows in this tile: release each K stage as it lands
                for (int j = 0; ok && j < it.nch; ++j, ++g) {
                    const int st = g % C::kStages;
                    ok = mbar_wait_bounded(k_full(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit);
                    if (ok && lane == 0) mbar_arrive(k_empty(st));
                    __syncwarp();
                }
                if (!ok) break;
                continue;
            }
            ok = mbar_wait_bounded(q_full(u, x), qpar, kWaitLimit);
            const uint64_t qdesc = tc::sw128_desc(qtile(x, u), 16u, 1024u);
            for (int j = 0; ok && j < it.nch; ++j, ++g, ++c) {
                const int st = g % C::kStages;
                const int b = c % kSB;
                ok = mbar_wait_bounded(k_full(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit);
                // S/P[u][b] is free once the P V of this tile's step c - kSB has read P from it
                if (ok && c >= kSB) ok = mbar_wait_bounded(o_done(u, b), (uint32_t)((c / kSB) - 1) & 1u, kWaitLimit);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint64_t kdesc = tc::desc_add(kdesc0, (uint32_t)(st * C::kStageBytes));
                    const uint32_t sd = tbase + s_col(u, b);
#pragma unroll
                    for (int k = 0; k < C::kKS; ++k) {
                        tc::mma_f16_ss(sd, tc::desc_add(qdesc, (uint32_t)((k >> 2) * C::kQHalf + 32 * (k & 3))),
                                       tc::desc_add(kdesc, (uint32_t)((k >> 2) * C::kHalf + 32 * (k & 3))), idesc_s,
                                       k > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(s_full(u, b));
                    tc::mma_commit(k_empty(st));  // the K stage is free once every tile's S MMAs complete
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (!ok && lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
        // every MMA issued by this thread has completed before TMEM is freed
        if (lane == 0) tc::mma_commit(drain_s(u));
        __syncwarp();
        mbar_wait_bounded(drain_s(u), 0u, kWaitLimit);
    } else if (warp == 3 || (MT == 2 && warp == 5)) {
        // ------------------------------------------------------------ O += P V issuer of tile u
        // Threads of their own: issuing S MMAs may block while the tensor pipe is
        // busy, and must not hold back a P V whose P is ready.  An item's first
        // P V overwrites O: its P is published after the softmax warps have read
        // the previous item's O out in their epilogue.
        const int u = warp == 3 ? 0 : 1;
        constexpr uint32_t idesc_o = tc::f16_idesc(kBf16, true, C::kM, D);
        const uint64_t vdesc0 = tc::sw128_desc(kvb + (uint32_t)C::kTile, (uint32_t)C::kHalf, 1024u);
        const uint32_t od = tbase + o_col(u);
        int g = 0, c = 0, ku = 0;
        bool ok = true;
        for (;;) {
            UmmaSlot sl;
            ok = take(u, ku, sl);
            if (!ok || sl.end) break;
            const UmmaItem it = sl.it;
            if (lane == 0) mbar_arrive(q_free(u, ku & 1));  // done with the slot
            ++ku;
            if (u >= it.tiles) {
                // no rows in this tile: release each V stage as it lands
                for (int j = 0; ok && j < it.nch; ++j, ++g) {
                    const int st = g % C::kStages;
                    ok = mbar_wait_bounded(v_full(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit);
                    if (ok && lane == 0) mbar_arrive(v_empty(st));
                    __syncwarp();
                }
                if (!ok) break;
                continue;
            }
            for (int j = 0; ok && j < it.nch; ++j, ++g, ++c) {
                const int b = c % kSB;
                const int st = g % C::kStages;
                ok = mbar_wait_bounded(v_full(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit);
                // tile 0's softmax zeroes the V rows that must not contribute; tile 0's own
                // P V is issued after that (its P is published after the zeroing)
                if (ok && u > 0) ok = mbar_wait_bounded(v_zeroed(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit);
                if (ok) ok = mbar_wait_bounded(p_full(u, b), (uint32_t)(c / kSB) & 1u, kWaitLimit);
                if (!ok) break;
                tc::fence_after_sync();
                if (lane == 0) {
                    const uint64_t vdesc = tc::desc_add(vdesc0, (uint32_t)(st * C::kStageBytes));
                    const uint32_t pa0 = tbase + s_col(u, b);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int k = 0; k < C::kN / 16; ++k)
                            tc::mma_f16_ts(od, pa0 + (uint32_t)((C::kN / 2) * part + 8 * k), tc::desc_add(vdesc, 2048u * k),
                                           idesc_o, (j > 0 || part > 0 || k > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(o_done(u, b));
                    tc::mma_commit(v_empty(st));
                }
                __syncwarp();
            }
            if (!ok) break;
        }
        if (!ok && lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
        if (lane == 0) tc::mma_commit(drain_p(u));
        __syncwarp();
        mbar_wait_bounded(drain_p(u), 0u, kWaitLimit);
    } else if (warp >= C::kSoftWarp0) {
        // ------------------------------------------------------------ softmax (one row per thread)
        const int u = (warp - C::kSoftWarp0) / 4;  // tile of this warpgroup
        const int wq = warp & 3;                 // TMEM lanes 32 * wq .. 32 * wq + 31
        const int r = 32 * wq + lane;            // row within the tile
        const float sl = a.scale * 1.4426950408889634f;
        const uint32_t tl = tbase + ((uint32_t)(wq * 32) << 16);
        int g = 0, c = 0, ku = 0;
        bool ok = true;
        for (;;) {
            UmmaSlot item;
            ok = take(u, ku, item);
            if (!ok || item.end) break;
            const UmmaItem it = item.it;
            const int x = ku & 1;
            ++ku;
            if (u >= it.tiles) {
                // no rows in this tile: only the ring's step count moves on
                g += it.nch;
                __syncwarp();
                if (lane == 0) mbar_arrive(q_free(u, x));
                continue;
            }
            const int n = it.n, len = it.len, nch = it.nch;
            const int R = it.r0 + C::kM * u + r;
            const int t = R / G;
            const bool valid = t < n;
            const int pos = len - n + t;
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < nch; ++j, ++g, ++c) {
                const int b = c % kSB;
                const int st = g % C::kStages;
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(s_full(u, b), (uint32_t)(c / kSB) & 1u, kWaitLimit));
                if (!ok) break;
                tc::fence_after_sync();
                uint32_t sv[C::kN / 32][32];
#pragma unroll
                for (int q = 0; q < C::kN / 32; ++q) tc::tmem_ld32(tl + s_col(u, b) + 32u * q, sv[q]);
                tc::tmem_wait_ld();
                ok = __all_sync(0xffffffffu, mbar_wait_bounded(v_full(st), (uint32_t)(g / C::kStages) & 1u, kWaitLimit));
                if (!ok) break;
                const int mask = vmask[st];
                const int lim = valid ? pos - j * C::kN : -1;  // last visible key of this step
                // raw logits; the softmax scale is folded into the exponent's FFMA
                float f[C::kN];
#pragma unroll
                for (int cc = 0; cc < C::kN; ++cc) f[cc] = __uint_as_float(sv[cc >> 5][cc & 31]);
                float mul = sl;
                if (!(sl > 0.f)) {
                    // a non-positive scale: scale first, mask to -inf
#pragma unroll
                    for (int cc = 0; cc < C::kN; ++cc)
                        f[cc] = (cc <= lim && (mask >> (cc >> 4) & 1)) ? f[cc] * sl : -INFINITY;
                    mul = 1.f;
                } else if (!(__all_sync(0xffffffffu, lim >= C::kN - 1) && mask == (1 << C::kBoxes) - 1)) {
                    // a step on the diagonal, past the context or over a block not loaded
#pragma unroll
                    for (int cc = 0; cc < C::kN; ++cc)
                        if (!(cc <= lim && (mask >> (cc >> 4) & 1))) f[cc] = -INFINITY;
                }
                // row maximum as 8 independent chains (a single 64-long chain of
                // dependent max operations would sit on the critical path)
                float mx[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mx[i] = f[i];
#pragma unroll
                for (int cc = 8; cc < C::kN; ++cc) mx[cc & 7] = fmaxf(mx[cc & 7], f[cc]);
                const float mr = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                const float mc = mr * mul;  // -inf when nothing is visible
                const bool need = mc > m_used + 8.f;
                const float alpha = (need && j > 0) ? ex2(m_used - mc) : 1.f;
                if (need) m_used = mc;
                const float mu = m_used == -INFINITY ? 0.f : m_used;
                // P = exp2(x - m) split into P_hi + P_lo, in registers before waiting,
                // two keys per packed f32x2 operation; the row sum in 4 pair accumulators
                uint32_t hw[C::kN / 2], lw[C::kN / 2];
                uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
                const uint64_t mul2 = tc::f2(mul, mul), nmu2 = tc::f2(-mu, -mu);
#pragma unroll
                for (int v = 0; v < C::kN / 2; ++v) {
                    const float2 xa = tc::f2split(tc::fma2(tc::f2(f[2 * v], f[2 * v + 1]), mul2, nmu2));
                    const float p0 = ex2(xa.x), p1 = ex2(xa.y);
                    const uint64_t pp = tc::f2(p0, p1);
                    ls[v & 3] = tc::add2(ls[v & 3], pp);
                    hw[v] = M::pack(p0, p1);
                    const float2 hf = M::unpack(hw[v]);
                    const float2 d = tc::f2split(tc::sub2(pp, tc::f2(hf.x, hf.y)));
                    lw[v] = M::pack(d.x, d.y);
                }
                const float2 s01 = tc::f2split(tc::add2(ls[0], ls[1])), s23 = tc::f2split(tc::add2(ls[2], ls[3]));
                l = l * alpha + ((s01.x + s01.y) + (s23.x + s23.y));
                // O may be rescaled only once the P V of step j - 1 has landed in it
                const bool rescale = j > 0 && __any_sync(0xffffffffu, need);
                if (rescale) {
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(o_done(u, (c - 1) % kSB),
                                                                    (uint32_t)((c - 1) / kSB) & 1u, kWaitLimit));
                    if (!ok) break;
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int q = 0; q < D / 16; ++q) {
                        uint32_t ov[16];
                        tc::tmem_ld16(tl + o_col(u) + 16u * q, ov);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tc::tmem_st16(tl + o_col(u) + 16u * q, ov);
                    }
                    tc::tmem_wait_st();
                }
                // P into TMEM over this step's S (already read): P_hi, then P_lo
                if constexpr (C::kN == 64) {
                    tc::tmem_st32(tl + s_col(u, b), hw);
                    tc::tmem_st32(tl + s_col(u, b) + 32u, lw);
                } else {
                    tc::tmem_st16(tl + s_col(u, b), hw);
                    tc::tmem_st16(tl + s_col(u, b) + 16u, lw);
                }
                tc::tmem_wait_st();
                // V rows of keys that were not loaded or lie past the context hold
                // anything: tile 0's warpgroup zeroes them (row r < kN of this step's
                // V, whole 128-byte rows) before it publishes its P and v_zeroed, which
                // the other tile's P V issuer waits for.
                if (u == 0 && r < C::kN && (j * C::kN + r >= len || !(mask >> (r >> 4) & 1))) {
                    const uint32_t vrow = kvb + (uint32_t)(st * C::kStageBytes + C::kTile + r * 128);
#pragma unroll
                    for (int sb = 0; sb < C::kSub; ++sb)
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc)
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + sb * C::kHalf + cc * 16),
                                         "r"(0u)
                                         : "memory");
                }
                tc::fence_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(p_full(u, b));
                    if (u == 0) mbar_arrive(v_zeroed(st));
                }
            }
            const int last = c - 1;  // this tile's last step of the item
            if (ok)
                ok = __all_sync(0xffffffffu,
                                mbar_wait_bounded(o_done(u, last % kSB), (uint32_t)(last / kSB) & 1u, kWaitLimit));
            // One decision for the warpgroup: every warp reaches this barrier (all
            // its waits above are bounded), so the epilogue's barriers below are
            // entered by all four warps or by none.
            ok = warpgroup_all(1 + u, ok);
            if (!ok) break;
            // ---- epilogue: out = O / l, staged through the item's query tile (its S
            // MMAs are complete, so it is free).
            tc::fence_after_sync();
            tc::fence_async_smem();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const uint32_t qt = qtile(x, u);
            if (it.r0 + C::kM * (u + 1) <= n * G) {
                // A tile whose 128 rows all belong to the chunk: 32-column blocks, each
                // staged as one TMA box (rows in (token, head) order, 128-byte
                // swizzle) and stored by one thread while the warpgroup moves on;
                // consecutive blocks take turns in the query tile's 16 KB parts.
                constexpr int kParts = C::kQTile / 16384;  // 2 (D 128) or 1 (D 64)
                const bool issuer = wq == 0 && lane == 0;
                const uint64_t spol = policy_evict_first();
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    const uint32_t half = qt + (uint32_t)((cb % kParts) * 16384);
                    if (cb >= kParts) {
                        if (issuer) bulk_wait_read<kParts - 1>();  // the store of block cb - kParts has read this part
                        warpgroup_sync(1 + u);
                    }
                    uint32_t ov[32];
                    tc::tmem_ld32(tl + o_col(u) + (uint32_t)(32 * cb), ov);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(half + (uint32_t)(r * 128) +
                                                                                      ((uint32_t)(i ^ (r & 7)) << 4)),
                                     "f"(__uint_as_float(ov[4 * i]) * inv), "f"(__uint_as_float(ov[4 * i + 1]) * inv),
                                     "f"(__uint_as_float(ov[4 * i + 2]) * inv), "f"(__uint_as_float(ov[4 * i + 3]) * inv)
                                     : "memory");
                    tc::fence_async_smem();
                    warpgroup_sync(1 + u);
                    if (issuer) tma_store_3d(&tmo, half, 32 * cb, it.kvh * G, it.qs + (it.r0 + C::kM * u) / G, spol);
                }
                if (issuer) bulk_wait_read<0>();
                warpgroup_sync(1 + u);
            } else {
                // A tile with rows past the chunk: each warp stages its 32 rows, W
                // columns at a time (rows of W floats, 16-byte chunks swizzled by row),
                // then writes whole rows of the chunk's tokens to global memory,
                // lanes_per_row lanes per row, instead of one 16-byte piece of 32
                // different rows per store.
                constexpr int W = D / 2;                       // columns per pass
                constexpr int kRowBytes = W * 4;               // 256 (D 128) or 128 (D 64)
                constexpr int kRowsPerPiece = 4096 / kRowBytes;  // rows in one 4 KB piece of the warp's Q slice
                constexpr int kLanesPerRow = kRowBytes / 16;
                constexpr int kRowsPerStore = 32 / kLanesPerRow;
                const int lg = __ffs(G) - 1;
                const int rbase = it.r0 + C::kM * u + 32 * wq;  // tile row of this warp's first row
                auto stage = [&](int rr, int cc) {  // staging address of 16-byte chunk cc of row rr
                    return qt + (uint32_t)((rr / kRowsPerPiece) * C::kQHalf + wq * 32 * 128) +
                           (uint32_t)((rr % kRowsPerPiece) * kRowBytes) + ((uint32_t)(cc ^ (rr & 7)) << 4);
                };
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
                    for (int q = 0; q < W / 32; ++q) {
                        uint32_t ov[32];
                        tc::tmem_ld32(tl + o_col(u) + (uint32_t)(pass * W + 32 * q), ov);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(stage(lane, 8 * q + i / 4)),
                                         "f"(__uint_as_float(ov[i]) * inv), "f"(__uint_as_float(ov[i + 1]) * inv),
                                         "f"(__uint_as_float(ov[i + 2]) * inv), "f"(__uint_as_float(ov[i + 3]) * inv)
                                         : "memory");
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 32 / kRowsPerStore; ++i) {
                        const int rr = i * kRowsPerStore + lane / kLanesPerRow;  // row of this warp's 32
                        const int cc = lane % kLanesPerRow;
                        const int Rr = rbase + rr;
                        const int tr = Rr >> lg;  // G is a power of two
                        const float4 v = *reinterpret_cast<const float4 *>(smem_raw + (stage(rr, cc) - raw));
                        if (tr < n)
                            __stcs(reinterpret_cast<float4 *>(a.out + ((size_t)(it.qs + tr) * a.Hq + it.kvh * G +
                                                                       (Rr & (G - 1))) * D + pass * W + 4 * cc),
                                   v);
                    }
                    __syncwarp();
                }
            }
            // the query-tile set may be reloaded (async proxy) after these generic-proxy reads
            tc::fence_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_free(u, x));
        }
        if (!ok && lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
        if (wq == 0 && lane == 0) bulk_wait_all();  // this thread's output stores have completed
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, C::kTmemCols);
    }
}

template <typename T, int D, int B, int MT>
cudaError_t launch_chunk_umma_t(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st) {
    using C = UmmaCfg<D, MT>;
    static std::atomic<int> sms_of[kMaxLaunchDevices];
    int sms = 0;
    cudaError_t e = per_device_value(sms_of, &sms, [](int dev, int *v) {
        cudaError_t r = cudaFuncSetAttribute(chunk_umma_kernel<T, D, B, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::kSmem);
        if (r != cudaSuccess) return r;
        return cudaDeviceGetAttribute(v, cudaDevAttrMultiProcessorCount, dev);
    });
    if (e != cudaSuccess) return e;
    const int G = a.Hq / a.Hkv;
    const long long rows = (long long)a.max_query_len * G;
    const long long groups = (rows + C::kM * MT - 1) / (C::kM * MT);  // tile groups per sequence, at most
    const long long work = groups * a.S * a.Hkv;                       // list entries x KV heads, at most
    if (work > 0x7fffffffLL) return cudaErrorInvalidValue;
    // persistent: one CTA per SM (the shared memory admits no second one)
    const long long ctas = work < sms ? work : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ctas > 0 ? ctas : 1));
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_umma_kernel<T, D, B, MT>, a, tmk, tmv, tmq, tmo);
}

// Two tiles per CTA once a sequence can fill them (chunk_umma_rows).
template <typename T, int D, int B>
cudaError_t dispatch_chunk_umma_mt(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st) {
    return a.umma_rows == 256 ? launch_chunk_umma_t<T, D, B, 2>(a, tmk, tmv, tmq, tmo, st)
                              : launch_chunk_umma_t<T, D, B, 1>(a, tmk, tmv, tmq, tmo, st);
}

template <typename T>
cudaError_t dispatch_chunk_umma(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st) {
    if (a.D == 64 && a.B == 16) return dispatch_chunk_umma_mt<T, 64, 16>(a, tmk, tmv, tmq, tmo, st);
    if (a.D == 64 && a.B == 32) return dispatch_chunk_umma_mt<T, 64, 32>(a, tmk, tmv, tmq, tmo, st);
    if (a.D == 128 && a.B == 16) return dispatch_chunk_umma_mt<T, 128, 16>(a, tmk, tmv, tmq, tmo, st);
    if (a.D == 128 && a.B == 32) return dispatch_chunk_umma_mt<T, 128, 32>(a, tmk, tmv, tmq, tmo, st);
    return cudaErrorNotSupported;
}

}  // namespace pa
