// pa_chunk_mma.cuh -- paged attention for a chunk of query tokens per sequence
// (a prefill chunk, or drafted tokens being verified) on sm_103a, with q.k and
// p.v on the tensor cores.
//
// What is computed: the n_s query rows of sequence s are its last n_s
// positions (their keys and values already in the cache); the query at
// position pos = len_s - n_s + t attends to keys 0 .. pos:
//
//   out[i, h] = softmax(scale * q[i, h] . K_s[0..pos]^T) . V_s[0..pos]
//
// ("Paged Attention and vLLM", "KV Cache Fundamentals": the cache of a
// sequence at length t holds tokens 1..t; "Block Table and Logical-to-Physical
// Mapping" for the paged read; "Paged Attention CUDA Kernel" for the
// per-partition m_b / l_b / v_b^acc terms merged across partitions.)
//
// Work: an item is (sequence, context partition, group of HG KV heads, row
// block).  For one KV head the query rows are the (query token, query head of
// the group) pairs r = t * G + gq, cut into 16-row tiles; a row block is RW
// tiles.  A CTA has HG x RW consumer warps: warp w takes KV head g0 + w % HG
// and tile w / HG of the block.  The producer is the decode kernel's: one more
// warp claims items from the plan's list and streams 16-token chunks of the HG
// heads into a shared-memory ring with 3-D TMA copies; here all HG x RW
// consumer warps read each stage, so a partition's K/V is read once per row
// block, not once per query.
//
// Per chunk and warp:
//   S = Q K^T    mma.m16n8k16, A = the tile's 16 query rows (rows g and g + 8
//                of the fragment belong to this lane);
//   causal mask: row r sees partition-local key kk iff kk <= its position
//                minus the partition start;
//   online softmax per row in log2 units (a row with no visible key yet keeps
//                m = -inf and contributes nothing);
//   O += P V     P split as P_hi + P_lo, both 16-bit, as two MMAs, so the
//                weights are near-fp32; V read with ldmatrix.trans.  V rows past
//                the partition's tokens may hold anything (NaN included), so
//                their B-fragment halves are zeroed in registers -- RW warps
//                share one head's tile in shared memory and must not write it.
// A warp whose rows all end before a chunk skips that chunk's arithmetic.
//
// Eight consumer warps (HG 4, RW 2): the CTA is launched as three warpgroups
// at 168 registers a thread, the most that lets 12 warps fit one SM.  The
// producer's warpgroup hands all but 40 of its registers to the two consumer
// warpgroups (setmaxnreg: 8 x 232 + 4 x 40 = 12 x 168); one of its warps
// produces, the other three exit.  With 232 registers a consumer warp takes
// two full chunks that its rows see in one step: S for all 32 keys, one row
// maximum and rescale, then P V for both chunks (the second chunk's V
// fragments loaded over the first's).  Measured on 256 sequences x 5 query
// tokens: 5.22 TB/s with 9 warps at 168 registers, 5.79 with the register
// split, 5.99 with the paired chunks.
//
// Finish: a row whose context fits in one partition writes out[] directly;
// otherwise each partition stores (m, l, acc) and the merge kernel combines
// the row's partitions 0 .. pos / partition_size.
#pragma once

#include <cuda.h>

#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_mma.cuh"

namespace pa {

// Shared-memory ring budget of one SM: one CTA per SM when RW == 2 (eight
// warps), two when RW == 1.
#ifndef PA_CHUNK_STAGE_BUDGET
#define PA_CHUNK_STAGE_BUDGET (192 * 1024)
#endif

template <int D, int HG, int RW>
struct ChunkCfg {
    static constexpr int kKS = D / 16;                   // k-steps of q.k
    static constexpr int kNT = D / 8;                    // 8-wide n-tiles of p.v
    static constexpr int kSub = D / 64;                  // 128-byte halves of a row
    static constexpr int kHeadSub = kChunkRows * 128;    // one head's half-rows of a chunk
    static constexpr int kBoxBytes = HG * kHeadSub;      // one TMA box: that, for HG heads
    static constexpr int kTileBytes = kSub * kBoxBytes;  // K (or V) of a chunk, all HG heads
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kConsumers = HG * RW;              // warp w < HG * RW: head w % HG, row tile w / HG
    // eight consumer warps: a whole warpgroup around the producer warp, so its
    // registers can be handed to the consumers (setmaxnreg)
    static constexpr bool kRegSplit = kConsumers == 8;
    static constexpr int kThreads = (kConsumers + (kRegSplit ? 4 : 1)) * 32;
    static constexpr int kMinBlocks = RW == 1 ? 2 : 1;
    static constexpr int kStagesRaw = PA_CHUNK_STAGE_BUDGET / kMinBlocks / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kSlots = 3;                     // work items in flight per CTA
    static constexpr int kTblCap = kMaxPartitionBlocks;  // table entries per item slot
    static constexpr size_t kFullOff = (size_t)kStages * kStageBytes;
    static constexpr size_t kEmptyOff = kFullOff + 8 * kStages;
    static constexpr size_t kItemFullOff = kEmptyOff + 8 * kStages;
    static constexpr size_t kItemEmptyOff = kItemFullOff + 8 * kSlots;
    static constexpr size_t kInfoOff = kItemEmptyOff + 8 * kSlots;  // kSlots x 3 int4
    static constexpr size_t kTblOff = kInfoOff + 48 * kSlots;
    static constexpr size_t kSmem = kTblOff + (size_t)kSlots * kTblCap * 4 + 1024;  // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(RW == 1 || RW == 2, "row tiles per KV head");
    static_assert(kChunkRows == 16, "one chunk is one m16n8k16 k-extent of tokens");
    static_assert(kHeadSub % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static_assert(kInfoOff % 16 == 0, "int4 slot info");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

template <typename T, int D, int B, int HG, int RW>
__global__ void __launch_bounds__(ChunkCfg<D, HG, RW>::kThreads, ChunkCfg<D, HG, RW>::kMinBlocks)
    chunk_mma_kernel(const ChunkArgs a, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    using C = ChunkCfg<D, HG, RW>;
    using M = Mma16<T>;
    constexpr int kCPB = B / 16;  // chunks per block
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned: the 128-byte swizzle repeats every 1 KB
    unsigned char *basep = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;
    const int Pt = a.partition_size;
    const int ngroups = a.Hkv / HG;
    const int cap = a.max_blocks * a.B;

    const uint32_t full0 = base + (uint32_t)C::kFullOff;
    const uint32_t empty0 = base + (uint32_t)C::kEmptyOff;
    const uint32_t ifull0 = base + (uint32_t)C::kItemFullOff;
    const uint32_t iempty0 = base + (uint32_t)C::kItemEmptyOff;
    // [slot * 3]: (s, p, tokens, row block), (g0, chunks, valid, query_start[s]), (n_s, len_s, -, -)
    int4 *info = reinterpret_cast<int4 *>(basep + C::kInfoOff);
    int32_t *tbl = reinterpret_cast<int32_t *>(basep + C::kTblOff);  // [slot][kTblCap]

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, C::kConsumers);
        }
        for (int i = 0; i < C::kSlots; ++i) {
            mbar_init(ifull0 + 8 * i, 1);
            mbar_init(iempty0 + 8 * i, C::kConsumers);
        }
        fence_mbar_init();
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    __syncthreads();
    griddep_wait();  // the plan kernel's work list must be complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_items = a.plan_hdr[0];

    // ---- lane roles in the MMA fragments
    const int g = lane >> 2;         // fragment rows g and g + 8
    const int c2 = (lane & 3) * 2;   // fragment column pair
    const int lm = lane >> 3;        // ldmatrix: which 8x8 matrix this lane addresses
    const int lr = lane & 7;         // ldmatrix: which row of it
    const uint32_t kx = (uint32_t)(lm ^ lr);          // swizzled chunk bits for K reads
    const uint32_t vx = (uint32_t)((lm >> 1) ^ lr);   // and for V reads
    const float sl = a.scale * 1.4426950408889634f;   // logits in log2 units
    const int head = warp % HG;      // KV head of the item's group
    const int tile_of = warp / HG;   // row tile within the item's row block

    // ------------------------------------------------------------ producer warp
    // The last warp claims items, fills the item slots and issues the TMA loads,
    // up to kStages chunks ahead of the consumer warps and across item
    // boundaries; it never consumes, so a claim overlaps the chunks already in
    // the ring instead of stalling it.  First item: list entry blockIdx.x; later
    // ones are claimed from the counter when the issue cursor reaches them, not
    // earlier, so each CTA's last item is taken as late as possible and the
    // largest-first order bounds the tail.
    if (warp >= C::kConsumers) {
        if constexpr (C::kRegSplit) {
            // launched at 168 registers a thread (3 warps per scheduler): the
            // producer warpgroup gives up all but 40, the two consumer warpgroups
            // take 232 (8 x 232 + 4 x 40 = 12 x 168); one warp of the group produces
            asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory");
            if (warp > C::kConsumers) return;
        }
        const uint64_t pol = policy_evict_first();
        int iss = 0;  // chunks issued
        bool ok = true;
        for (int seq = 0; ok; ++seq) {
            const int slot = seq % C::kSlots;
            // every consumer warp must be done with the item that used this slot
            if (seq >= C::kSlots &&
                !mbar_wait_bounded(iempty0 + 8 * slot, (uint32_t)((seq / C::kSlots) - 1) & 1u, kWaitLimit)) {
                if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                break;
            }
            int idx = 0;
            if (lane == 0) idx = seq == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(a.plan_hdr + 1, 1);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            int4 e0 = make_int4(0, 0, 0, 0), e1 = make_int4(0, 0, 0, 0), e2 = make_int4(0, 0, 0, 0);
            int32_t *tb = tbl + slot * C::kTblCap;
            if (idx < n_items) {
                const int4 e = a.plan_list[idx / ngroups];
                e0 = e;
                const int qs = a.query_start[e.x];
                const int n = a.query_start[e.x + 1] - qs;
                int len = a.context_lens[e.x];
                len = len < 0 ? 0 : (len > cap ? cap : len);
                e1 = make_int4((idx % ngroups) * HG, (e.z + 15) >> 4, 1, qs);
                e2 = make_int4(n, len, 0, 0);
                const int nblk = (e.z + B - 1) / B;
                const int32_t *row = a.block_tables + (size_t)e.x * a.max_blocks + (size_t)e.y * (Pt / B);
                for (int i = lane; i < nblk; i += 32) {
                    int pb = row[i];
                    if (pb < 0 || pb >= a.N) {
                        set_error(a.err, PA_DEVERR_BAD_BLOCK);
                        pb = -1;
                    }
                    tb[i] = pb;
                }
            }
            if (lane == 0) {
                info[3 * slot] = e0;
                info[3 * slot + 1] = e1;
                info[3 * slot + 2] = e2;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ifull0 + 8 * slot);  // release: info and table visible
            if (idx >= n_items) break;
            for (int c = 0; c < e1.y; ++c) {
                const int st = iss % C::kStages;
                // every consumer warp has released this stage's previous chunk
                if (iss >= C::kStages &&
                    !mbar_wait_bounded(empty0 + 8 * st, (uint32_t)((iss / C::kStages) - 1) & 1u, kWaitLimit)) {
                    if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t bar = full0 + 8 * st;
                    const int pb = tb[c / kCPB];
                    if (pb < 0) {
                        mbar_arrive(bar);  // bad table entry: complete the phase without data
                    } else {
                        const uint32_t dst = base + (uint32_t)(st * C::kStageBytes);
                        const int y = (c % kCPB) * kChunkRows;
                        const int z = pb * a.Hkv + e1.x;
                        mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
                        for (int sb = 0; sb < C::kSub; ++sb) {
                            tma_load_3d(dst + sb * C::kBoxBytes, &tmk, sb * 64, y, z, bar, pol);
                            tma_load_3d(dst + C::kTileBytes + sb * C::kBoxBytes, &tmv, sb * 64, y, z, bar, pol);
                        }
                    }
                }
                ++iss;
            }
        }
        // The CTA's shared memory outlives its copies: wait for the last
        // kStages chunks issued (one pending phase per stage at most, so the
        // parities are unambiguous); they have normally landed long ago.
        for (int k = iss > C::kStages ? iss - C::kStages : 0; k < iss; ++k)
            mbar_wait_bounded(full0 + 8 * (k % C::kStages), (uint32_t)(k / C::kStages) & 1u, kWaitLimit);
        return;
    }

    // ------------------------------------------------------------ consumer warps
    // Every consumer warp walks the same items (slot by slot) and chunks
    // (stage by stage).
    if constexpr (C::kRegSplit) asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory");
    uint32_t qa[C::kKS][4];
    int cons = 0;  // chunks consumed by this warp
    for (int seq = 0;; ++seq) {
        const int slot = seq % C::kSlots;
        if (!mbar_wait_bounded(ifull0 + 8 * slot, (uint32_t)(seq / C::kSlots) & 1u, kWaitLimit)) {
            if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
            break;
        }
        const int4 e0 = info[3 * slot];
        const int4 e1 = info[3 * slot + 1];
        const int4 e2 = info[3 * slot + 2];
        if (!e1.z) break;  // no more work
        const int p = e0.y, ntok = e0.z;
        const int kvh = e1.x + head;
        const int nchunk = e1.y;
        const int qs = e1.w;
        const int n = e2.x, len = e2.y;
        const int32_t *ctb = tbl + slot * C::kTblCap;

        // this lane's two query rows
        const int r0 = (e0.w * RW + tile_of) * 16 + g;
        const int r1 = r0 + 8;
        const int t0 = r0 / G, t1 = r1 / G;
        const bool v0 = t0 < n, v1 = t1 < n;
        const int h0 = kvh * G + r0 % G, h1 = kvh * G + r1 % G;
        const int pos0 = len - n + t0, pos1 = len - n + t1;
        const int lim0 = v0 ? pos0 - p * Pt : -1;  // last visible partition-local key
        const int lim1 = v1 ? pos1 - p * Pt : -1;
        const int wlim = __reduce_max_sync(0xffffffffu, max(lim0, lim1));
        {
            const uint16_t *qb = static_cast<const uint16_t *>(a.q);
            const uint16_t *q0 = qb + ((size_t)(qs + (v0 ? t0 : 0)) * a.Hq + h0) * D;
            const uint16_t *q1 = qb + ((size_t)(qs + (v1 ? t1 : 0)) * a.Hq + h1) * D;
#pragma unroll
            for (int ks = 0; ks < C::kKS; ++ks) {
                qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + ks * 16 + c2) : 0u;
                qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + ks * 16 + c2) : 0u;
                qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t *>(q0 + ks * 16 + 8 + c2) : 0u;
                qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t *>(q1 + ks * 16 + 8 + c2) : 0u;
            }
        }
        float o[C::kNT][4];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        bool timed_out = false;

        for (int j = 0; j < nchunk; ++j) {
            const int st = cons % C::kStages;
            const uint32_t parity = (uint32_t)(cons / C::kStages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st, parity, kWaitLimit))) {
                if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                timed_out = true;
                break;
            }
            const int nv = ctb[j / kCPB] < 0 ? 0 : min(16, ntok - j * 16);
            // two full chunks that some row of this warp sees: one softmax step over 32 keys
            const bool pair = C::kRegSplit && j + 1 < nchunk && nv == 16 && ctb[(j + 1) / kCPB] >= 0 && ntok - (j + 1) * 16 >= 16 &&
                              (j + 1) * 16 <= wlim;
            if (pair) {
                const int st2 = (cons + 1) % C::kStages;
                const uint32_t parity2 = (uint32_t)((cons + 1) / C::kStages) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * st2, parity2, kWaitLimit))) {
                    if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                    timed_out = true;
                    break;
                }
                const uint32_t kstp[2] = {base + (uint32_t)(st * C::kStageBytes) + (uint32_t)(head * C::kHeadSub),
                                          base + (uint32_t)(st2 * C::kStageBytes) + (uint32_t)(head * C::kHeadSub)};
                uint32_t bv[C::kNT / 2][4];
#pragma unroll
                for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                    const uint32_t addr = kstp[0] + C::kTileBytes + (uint32_t)((ntp >> 2) * C::kBoxBytes) +
                                          (uint32_t)(((lm & 1) * 8 + lr) * 128) +
                                          (((uint32_t)(2 * (ntp & 3)) ^ vx) << 4);
                    ldsm_x4_t(addr, bv[ntp][0], bv[ntp][1], bv[ntp][2], bv[ntp][3]);
                }
                float sc[2][2][2][4];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            sc[c][nt][hh][0] = sc[c][nt][hh][1] = sc[c][nt][hh][2] = sc[c][nt][hh][3] = 0.f;
#pragma unroll
                for (int ks2 = 0; ks2 < C::kKS / 2; ++ks2) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const uint32_t addr = kstp[c] + (uint32_t)((ks2 >> 1) * C::kBoxBytes) +
                                                  (uint32_t)((nt * 8 + lr) * 128) +
                                                  (((uint32_t)(4 * (ks2 & 1)) ^ kx) << 4);
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(addr, b0, b1, b2, b3);
                            const int k0 = 2 * ks2, k1 = 2 * ks2 + 1;
                            M::mma(sc[c][nt][0], qa[k0][0], qa[k0][1], qa[k0][2], qa[k0][3], b0, b1);
                            M::mma(sc[c][nt][1], qa[k1][0], qa[k1][1], qa[k1][2], qa[k1][3], b2, b3);
                        }
                    }
                }
                // logits of the 32 keys: chunk c, keys c2, c2+1, 8+c2, 9+c2 at [4c .. 4c+3]
                float x0[8], x1[8];
                const int koff[4] = {0, 1, 8, 9};
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    x0[4 * c + 0] = (sc[c][0][0][0] + sc[c][0][1][0]) * sl;
                    x0[4 * c + 1] = (sc[c][0][0][1] + sc[c][0][1][1]) * sl;
                    x0[4 * c + 2] = (sc[c][1][0][0] + sc[c][1][1][0]) * sl;
                    x0[4 * c + 3] = (sc[c][1][0][1] + sc[c][1][1][1]) * sl;
                    x1[4 * c + 0] = (sc[c][0][0][2] + sc[c][0][1][2]) * sl;
                    x1[4 * c + 1] = (sc[c][0][0][3] + sc[c][0][1][3]) * sl;
                    x1[4 * c + 2] = (sc[c][1][0][2] + sc[c][1][1][2]) * sl;
                    x1[4 * c + 3] = (sc[c][1][0][3] + sc[c][1][1][3]) * sl;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kk = (j + c) * 16 + c2 + koff[i];
                        if (kk > lim0) x0[4 * c + i] = -INFINITY;
                        if (kk > lim1) x1[4 * c + i] = -INFINITY;
                    }
                }
                float mx0 = x0[0], mx1 = x1[0];
#pragma unroll
                for (int i = 1; i < 8; ++i) {
                    mx0 = fmaxf(mx0, x0[i]);
                    mx1 = fmaxf(mx1, x1[i]);
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                if (__any_sync(0xffffffffu, mx0 > m0 || mx1 > m1)) {
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float al0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
                    const float al1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt) {
                        o[nt][0] *= al0;
                        o[nt][1] *= al0;
                        o[nt][2] *= al1;
                        o[nt][3] *= al1;
                    }
                    m0 = mn0;
                    m1 = mn1;
                }
                const float mu0 = m0 == -INFINITY ? 0.f : m0;
                const float mu1 = m1 == -INFINITY ? 0.f : m1;
                float p0[8], p1[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    p0[i] = ex2(x0[i] - mu0);
                    p1[i] = ex2(x1[i] - mu1);
                }
                l0 += ((p0[0] + p0[1]) + (p0[2] + p0[3])) + ((p0[4] + p0[5]) + (p0[6] + p0[7]));
                l1 += ((p1[0] + p1[1]) + (p1[2] + p1[3])) + ((p1[4] + p1[5]) + (p1[6] + p1[7]));
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    if (c == 1) {  // the second chunk's V fragments, over the first chunk's
#pragma unroll
                        for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                            const uint32_t addr = kstp[1] + C::kTileBytes + (uint32_t)((ntp >> 2) * C::kBoxBytes) +
                                                  (uint32_t)(((lm & 1) * 8 + lr) * 128) +
                                                  (((uint32_t)(2 * (ntp & 3)) ^ vx) << 4);
                            ldsm_x4_t(addr, bv[ntp][0], bv[ntp][1], bv[ntp][2], bv[ntp][3]);
                        }
                    }
                    const uint32_t h0a = M::pack(p0[4 * c], p0[4 * c + 1]), h1a = M::pack(p1[4 * c], p1[4 * c + 1]);
                    const uint32_t h0b = M::pack(p0[4 * c + 2], p0[4 * c + 3]);
                    const uint32_t h1b = M::pack(p1[4 * c + 2], p1[4 * c + 3]);
                    const float2 f0a = M::unpack(h0a), f1a = M::unpack(h1a);
                    const float2 f0b = M::unpack(h0b), f1b = M::unpack(h1b);
                    const uint32_t l0a = M::pack(p0[4 * c] - f0a.x, p0[4 * c + 1] - f0a.y);
                    const uint32_t l1a = M::pack(p1[4 * c] - f1a.x, p1[4 * c + 1] - f1a.y);
                    const uint32_t l0b = M::pack(p0[4 * c + 2] - f0b.x, p0[4 * c + 3] - f0b.y);
                    const uint32_t l1b = M::pack(p1[4 * c + 2] - f1b.x, p1[4 * c + 3] - f1b.y);
#pragma unroll
                    for (int ntq = 0; ntq < C::kNT / 4; ++ntq) {
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int ntp = 2 * ntq + u;
                            M::mma(o[4 * ntq + 2 * u], h0a, h1a, h0b, h1b, bv[ntp][0], bv[ntp][1]);
                            M::mma(o[4 * ntq + 2 * u + 1], h0a, h1a, h0b, h1b, bv[ntp][2], bv[ntp][3]);
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int ntp = 2 * ntq + u;
                            M::mma(o[4 * ntq + 2 * u], l0a, l1a, l0b, l1b, bv[ntp][0], bv[ntp][1]);
                            M::mma(o[4 * ntq + 2 * u + 1], l0a, l1a, l0b, l1b, bv[ntp][2], bv[ntp][3]);
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty0 + 8 * st);
                    mbar_arrive(empty0 + 8 * st2);
                }
                cons += 2;
                ++j;
                continue;
            }
            if (nv > 0 && j * 16 <= wlim) {
                const uint32_t kst = base + (uint32_t)(st * C::kStageBytes) + (uint32_t)(head * C::kHeadSub);
                const uint32_t vst = kst + C::kTileBytes;
                // V fragments first: they do not depend on P, so their shared-memory
                // latency hides behind S and the softmax instead of stalling P V
                uint32_t bv[C::kNT / 2][4];
#pragma unroll
                for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                    const uint32_t addr = vst + (uint32_t)((ntp >> 2) * C::kBoxBytes) +
                                          (uint32_t)(((lm & 1) * 8 + lr) * 128) +
                                          (((uint32_t)(2 * (ntp & 3)) ^ vx) << 4);
                    ldsm_x4_t(addr, bv[ntp][0], bv[ntp][1], bv[ntp][2], bv[ntp][3]);
                }
                // ---- S = Q K^T for 16 tokens (two n-tiles of 8), even / odd k-steps apart
                float sc[2][2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) sc[nt][hh][0] = sc[nt][hh][1] = sc[nt][hh][2] = sc[nt][hh][3] = 0.f;
#pragma unroll
                for (int ks2 = 0; ks2 < C::kKS / 2; ++ks2) {
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt) {
                        const uint32_t addr = kst + (uint32_t)((ks2 >> 1) * C::kBoxBytes) +
                                              (uint32_t)((nt * 8 + lr) * 128) +
                                              (((uint32_t)(4 * (ks2 & 1)) ^ kx) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        const int k0 = 2 * ks2, k1 = 2 * ks2 + 1;
                        M::mma(sc[nt][0], qa[k0][0], qa[k0][1], qa[k0][2], qa[k0][3], b0, b1);
                        M::mma(sc[nt][1], qa[k1][0], qa[k1][1], qa[k1][2], qa[k1][3], b2, b3);
                    }
                }
                // ---- causal mask and online softmax; tokens c2, c2+1, 8+c2, 9+c2 of rows g, g+8
                const int kb = j * 16 + c2;
                float x0[4] = {(sc[0][0][0] + sc[0][1][0]) * sl, (sc[0][0][1] + sc[0][1][1]) * sl,
                               (sc[1][0][0] + sc[1][1][0]) * sl, (sc[1][0][1] + sc[1][1][1]) * sl};
                float x1[4] = {(sc[0][0][2] + sc[0][1][2]) * sl, (sc[0][0][3] + sc[0][1][3]) * sl,
                               (sc[1][0][2] + sc[1][1][2]) * sl, (sc[1][0][3] + sc[1][1][3]) * sl};
                const int koff[4] = {0, 1, 8, 9};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (kb + koff[i] > lim0) x0[i] = -INFINITY;
                    if (kb + koff[i] > lim1) x1[i] = -INFINITY;
                }
                float mx0 = fmaxf(fmaxf(x0[0], x0[1]), fmaxf(x0[2], x0[3]));
                float mx1 = fmaxf(fmaxf(x1[0], x1[1]), fmaxf(x1[2], x1[3]));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                if (__any_sync(0xffffffffu, mx0 > m0 || mx1 > m1)) {
                    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                    const float al0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
                    const float al1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
                    l0 *= al0;
                    l1 *= al1;
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt) {
                        o[nt][0] *= al0;
                        o[nt][1] *= al0;
                        o[nt][2] *= al1;
                        o[nt][3] *= al1;
                    }
                    m0 = mn0;
                    m1 = mn1;
                }
                // a row with no visible key so far has m = -inf and all logits -inf: weights 0
                const float mu0 = m0 == -INFINITY ? 0.f : m0;
                const float mu1 = m1 == -INFINITY ? 0.f : m1;
                float p0[4], p1[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p0[i] = ex2(x0[i] - mu0);
                    p1[i] = ex2(x1[i] - mu1);
                }
                l0 += (p0[0] + p0[1]) + (p0[2] + p0[3]);
                l1 += (p1[0] + p1[1]) + (p1[2] + p1[3]);
                // A fragments of P: a0 row g tokens c2.., a1 row g+8 tokens c2.., a2 / a3 tokens 8+c2..
                const uint32_t h0a = M::pack(p0[0], p0[1]), h1a = M::pack(p1[0], p1[1]);
                const uint32_t h0b = M::pack(p0[2], p0[3]), h1b = M::pack(p1[2], p1[3]);
                const float2 f0a = M::unpack(h0a), f1a = M::unpack(h1a);
                const float2 f0b = M::unpack(h0b), f1b = M::unpack(h1b);
                const uint32_t l0a = M::pack(p0[0] - f0a.x, p0[1] - f0a.y);
                const uint32_t l1a = M::pack(p1[0] - f1a.x, p1[1] - f1a.y);
                const uint32_t l0b = M::pack(p0[2] - f0b.x, p0[3] - f0b.y);
                const uint32_t l1b = M::pack(p1[2] - f1b.x, p1[3] - f1b.y);
                // V rows at or past the partition's last token: zero their halves of the
                // B fragments (b0 / b2 hold tokens c2, c2+1; b1 / b3 tokens 8+c2, 9+c2)
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (nv < 16) {
                    mlo = (c2 < nv ? 0x0000ffffu : 0u) | (c2 + 1 < nv ? 0xffff0000u : 0u);
                    mhi = (c2 + 8 < nv ? 0x0000ffffu : 0u) | (c2 + 9 < nv ? 0xffff0000u : 0u);
                }
                // ---- O += P_hi V + P_lo V, two 16-column groups at a time so that the
                // two MMAs into one accumulator are four issues apart
#pragma unroll
                for (int ntq = 0; ntq < C::kNT / 4; ++ntq) {
                    uint32_t b[2][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int ntp = 2 * ntq + u;
                        b[u][0] = bv[ntp][0] & mlo;
                        b[u][1] = bv[ntp][1] & mhi;
                        b[u][2] = bv[ntp][2] & mlo;
                        b[u][3] = bv[ntp][3] & mhi;
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        M::mma(o[4 * ntq + 2 * u], h0a, h1a, h0b, h1b, b[u][0], b[u][1]);
                        M::mma(o[4 * ntq + 2 * u + 1], h0a, h1a, h0b, h1b, b[u][2], b[u][3]);
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        M::mma(o[4 * ntq + 2 * u], l0a, l1a, l0b, l1b, b[u][0], b[u][1]);
                        M::mma(o[4 * ntq + 2 * u + 1], l0a, l1a, l0b, l1b, b[u][2], b[u][3]);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            ++cons;
        }
        if (timed_out) break;

        // ---- finish this warp's two rows per lane
        float lt0 = l0, lt1 = l1;
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 1);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const bool vr = rr == 0 ? v0 : v1;
            const int tr = rr == 0 ? t0 : t1;
            const int hr = rr == 0 ? h0 : h1;
            const int npr = vr ? (rr == 0 ? pos0 : pos1) / Pt + 1 : 0;  // partitions this row sees
            const float lt = rr == 0 ? lt0 : lt1;
            const float mr = rr == 0 ? m0 : m1;
            if (!vr || p >= npr) continue;
            const size_t row = (size_t)(qs + tr) * a.Hq + hr;
            if (npr == 1) {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                float *orow = a.out + row * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(orow + nt * 8 + c2) =
                        make_float2(o[nt][2 * rr] * inv, o[nt][2 * rr + 1] * inv);
            } else {
                const size_t r = row * a.max_parts + p;
                float *acc = a.ws_acc + r * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(acc + nt * 8 + c2) = make_float2(o[nt][2 * rr], o[nt][2 * rr + 1]);
                if ((lane & 3) == 0) *reinterpret_cast<float2 *>(a.ws_ml + 2 * r) = make_float2(mr, lt);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(iempty0 + 8 * slot);  // this warp is done with the item slot
    }
}

template <typename T, int D, int B, int HG, int RW>
cudaError_t launch_chunk_mma_t(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                               cudaStream_t st) {
    using C = ChunkCfg<D, HG, RW>;
    static std::atomic<int> grid_for[kMaxLaunchDevices];
    int grid = 0;
    cudaError_t e = per_device_value(grid_for, &grid, [](int dev, int *v) {
        cudaError_t r = cudaFuncSetAttribute(chunk_mma_kernel<T, D, B, HG, RW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
        if (r != cudaSuccess) return r;
        int sms = 0, per_sm = 0;
        r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r != cudaSuccess) return r;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_mma_kernel<T, D, B, HG, RW>, C::kThreads,
                                                          C::kSmem);
        if (r != cudaSuccess) return r;
        *v = sms * (per_sm > 0 ? per_sm : 1);
        return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_mma_kernel<T, D, B, HG, RW>, a, tmk, tmv);
}

template <typename T, int D, int B, int HG>
cudaError_t dispatch_chunk_rw(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv, cudaStream_t st) {
    return a.row_warps == 2 ? launch_chunk_mma_t<T, D, B, HG, 2>(a, tmk, tmv, st)
                            : launch_chunk_mma_t<T, D, B, HG, 1>(a, tmk, tmv, st);
}

template <typename T, int D, int B>
cudaError_t dispatch_chunk_hg(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv, cudaStream_t st) {
    switch (a.head_group) {
#if PA_MMA_HEAD_GROUP >= 8
        case 8: return dispatch_chunk_rw<T, D, B, 8>(a, tmk, tmv, st);
#endif
        case 4: return dispatch_chunk_rw<T, D, B, 4>(a, tmk, tmv, st);
        case 2: return dispatch_chunk_rw<T, D, B, 2>(a, tmk, tmv, st);
        default: return dispatch_chunk_rw<T, D, B, 1>(a, tmk, tmv, st);
    }
}

template <typename T>
cudaError_t dispatch_chunk_mma(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv, cudaStream_t st) {
    if (a.D == 64 && a.B == 16) return dispatch_chunk_hg<T, 64, 16>(a, tmk, tmv, st);
    if (a.D == 64 && a.B == 32) return dispatch_chunk_hg<T, 64, 32>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 16) return dispatch_chunk_hg<T, 128, 16>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 32) return dispatch_chunk_hg<T, 128, 32>(a, tmk, tmv, st);
    return cudaErrorNotSupported;
}

}  // namespace pa
