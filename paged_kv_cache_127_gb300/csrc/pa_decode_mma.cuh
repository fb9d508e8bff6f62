// pa_decode_mma.cuh -- PagedAttention decode for f16 / bf16 caches on sm_103a,
// with q.k and p.v on the tensor cores.
//
// What is computed ("Paged Attention and vLLM", "Block Table and
// Logical-to-Physical Mapping", the a_t equation; "Paged Attention CUDA Kernel",
// the per-partition m_b / l_b / v_b^acc terms and their log-sum-exp merge):
//
//   out[s, h] = softmax(scale * q[s, h] . K_s^T) . V_s
//
// over the context_lens[s] tokens of s, gathered through its block table.
//
// Work: a work item is one (sequence, context partition, group of HG KV heads).
// A small plan kernel lists the (sequence, partition) pairs, largest first, in
// the workspace.  The kernel is persistent: in each CTA a producer warp claims
// items from a global counter and streams their 16-token chunks into a ring of
// shared-memory stages with TMA tensor copies (cp.async.bulk.tensor, 128-byte
// swizzle) -- one 3-D box covers 16 rows of all HG heads, so a copy is 8 KB
// rather than one head's 2 KB -- running ahead across item boundaries, and
// consumer warp w computes the item's KV head g0 + w.  Full barriers
// (transaction counts) signal data; empty barriers (one arrival per consumer
// warp) return stages to the producer.
//
// Per 16-token chunk, with G = Hq / Hkv query heads sharing the KV head:
//   S = Q K^T   mma.m16n8k16, A = the G query rows (padded to 16 with zeros),
//               B = K rows read with ldmatrix from the swizzled tile;
//   online softmax in log2 units on the S fragments (row max over 4 lanes);
//   O += P V    mma.m16n8k16 with P split as P_hi + P_lo (both 16-bit): rows
//               0-7 of A carry P_hi, rows 8-15 carry P_lo, so the padding rows
//               buy near-fp32 weights; V read with ldmatrix.trans.  O's row g
//               plus row g + 8 is the head's output.
// Only the context's tokens are used: masked logits are -inf, and V rows past
// the context in a tail block are zeroed in shared memory before the P V MMA
// (so NaN in unused slots cannot leak through 0 * NaN).
//
// Finish: an item that covers its whole sequence writes out[] directly;
// otherwise it stores (m, l, acc) for its partition and the merge kernel,
// launched right after this one, combines the partitions.  (Merging in the
// last-finishing warp instead needs a device-wide fence per partial and
// stalls the CTA's stage ring while that warp merges; measured slower.)
#pragma once

#include <cuda.h>

#include <cmath>
#include <cstring>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_mma.cuh"

namespace pa {

// ------------------------------------------------------------------ configuration
// A CTA owns HG consecutive KV heads of one (sequence, partition) work item --
// one warp per head.  A stage holds one 16-token chunk of the item for all HG
// heads: K rows then V rows, each split into 128-byte-wide halves of D; one TMA
// box is one half for the HG heads (HG x 16 rows x 128 bytes, 8 KB at HG = 4),
// written with the 128-byte swizzle.  Bigger boxes than one head's 2 KB keep
// the bulk-copy engine at HBM speed.
// Build-time switch: 1 computes q.k and p.v of the 16-bit decode on the CUDA
// cores instead of the tensor cores, everything else unchanged (for comparing
// the two on otherwise identical sources; the build takes it from the
// environment variable of the same name).
#ifndef PA_DECODE_CUDA_CORE
#define PA_DECODE_CUDA_CORE 0
#endif

#ifndef PA_MMA_STAGE_BUDGET
#define PA_MMA_STAGE_BUDGET (96 * 1024)
#endif

template <int D, int HG>
struct MmaCfg {
    static constexpr int kKS = D / 16;                   // k-steps of q.k
    static constexpr int kNT = D / 8;                    // 8-wide n-tiles of p.v
    static constexpr int kSub = D / 64;                  // 128-byte halves of a row
    static constexpr int kHeadSub = kChunkRows * 128;    // one head's half-rows of a chunk
    static constexpr int kBoxBytes = HG * kHeadSub;      // one TMA box: that, for HG heads
    static constexpr int kTileBytes = kSub * kBoxBytes;  // K (or V) of a chunk, all HG heads
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kConsumers = HG;                   // warp w < HG computes head g0 + w of an item
    static constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
    static constexpr int kStagesRaw = PA_MMA_STAGE_BUDGET / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kSlots = 3;                     // work items in flight per CTA
    static constexpr int kTblCap = kMaxPartitionBlocks;  // table entries per item slot
    // shared-memory layout from a 1024-aligned base
    static constexpr size_t kFullOff = (size_t)kStages * kStageBytes;
    static constexpr size_t kEmptyOff = kFullOff + 8 * kStages;
    static constexpr size_t kItemFullOff = kEmptyOff + 8 * kStages;
    static constexpr size_t kItemEmptyOff = kItemFullOff + 8 * kSlots;
    static constexpr size_t kInfoOff = kItemEmptyOff + 8 * kSlots;   // kSlots x int4 (s, p, ntok, np) + int4 (g0, ...)
    static constexpr size_t kTblOff = kInfoOff + 32 * kSlots;
    static constexpr size_t kSmem = kTblOff + (size_t)kSlots * kTblCap * 4 + 1024;  // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(kChunkRows == 16, "one chunk is one m16n8k16 k-extent of tokens");
    static_assert(kHeadSub % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

#if PA_DECODE_CUDA_CORE
// Build-time alternative (PA_DECODE_CUDA_CORE=1) for a same-sources comparison
// of the tensor-core choice: the consumer warps compute q.k and p.v with fp32
// FMAs on the CUDA cores; the producer warp, the stage ring, the work items,
// the masking and the finish are those of the tensor-core consumer.
//   q.k   lane (t = lane % 16, half = lane / 16) takes token t of the chunk and
//         one half of D for each of the G query heads (q read through L1), and
//         one shuffle adds the two halves;
//   softmax  per query head over the chunk's 16 tokens (shuffle max / sum);
//   p.v   lane takes D / 32 consecutive columns of every head and the
//         weights of each token by shuffle.
template <typename T>
__device__ __forceinline__ float2 widen2(uint32_t w) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    else {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
}

template <typename T, int D, int B, int HG>
__device__ __forceinline__ void consumer_cuda_core(const DecodeArgs &a, uint32_t base, uint32_t full0, uint32_t empty0,
                                                   uint32_t ifull0, uint32_t iempty0, const int4 *info,
                                                   const int32_t *tbl, int warp, int lane) {
    using C = MmaCfg<D, HG>;
    using E = Elem<T>;
    constexpr int kCPB = B / 16;
    constexpr int kHalf = D / 2;      // dims of one lane's q.k half
    constexpr int kPer = D / 32;      // output columns per lane
    const unsigned full = 0xffffffffu;
    const int G = a.Hq / a.Hkv;
    const float sl = a.scale * 1.4426950408889634f;
    const int t = lane & 15, hf = lane >> 4;
    const int d0 = kPer * lane;
    int cons = 0;
    for (int seq = 0;; ++seq) {
        const int slot = seq % C::kSlots;
        if (!mbar_wait_bounded(ifull0 + 8 * slot, (uint32_t)(seq / C::kSlots) & 1u, kWaitLimit)) {
            if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
            break;
        }
        const int4 e0 = info[2 * slot];
        const int4 e1 = info[2 * slot + 1];
        if (!e1.z) break;  // no more work
        const int s = e0.x, p = e0.y, ntok = e0.z, np = e0.w;
        const int kvh = e1.x + warp;
        const int nchunk = e1.y;
        const int32_t *ctb = tbl + slot * C::kTblCap;
        const T *qb = static_cast<const T *>(a.q) + ((size_t)s * a.Hq + (size_t)kvh * G) * D;
        float o[8][kPer], m_run[8], l_run[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            m_run[g] = -INFINITY;
            l_run[g] = 0.f;
#pragma unroll
            for (int i = 0; i < kPer; ++i) o[g][i] = 0.f;
        }
        bool timed_out = false;
        for (int j = 0; j < nchunk; ++j) {
            const int st = cons % C::kStages;
            const uint32_t parity = (uint32_t)(cons / C::kStages) & 1u;
            if (!__all_sync(full, mbar_wait_bounded(full0 + 8 * st, parity, kWaitLimit))) {
                if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                timed_out = true;
                break;
            }
            const int nv = ctb[j / kCPB] < 0 ? 0 : min(16, ntok - j * 16);
            const uint32_t kst = base + (uint32_t)(st * C::kStageBytes) + (uint32_t)(warp * C::kHeadSub);
            const uint32_t vst = kst + C::kTileBytes;
            if (nv > 0) {
                // ---- S = q K^T: token t, half hf of D
                float sd[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) sd[g] = 0.f;
#pragma unroll
                for (int c = 0; c < kHalf / 8; ++c) {
                    const int e = hf * kHalf + 8 * c;  // first element of this 16-byte chunk
                    const uint32_t addr = kst + (uint32_t)((e / 64) * C::kBoxBytes) + (uint32_t)(t * 128) +
                                          ((uint32_t)(((e % 64) / 8) ^ (t & 7)) << 4);
                    float kf[8];
                    E::unpack(lds128(addr), kf);
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        if (g < G) {
                            float qf[8];
                            E::unpack(__ldg(reinterpret_cast<const uint4 *>(qb + (size_t)g * D + e)), qf);
#pragma unroll
                            for (int i = 0; i < 8; ++i) sd[g] = fmaf(qf[i], kf[i], sd[g]);
                        }
                    }
                }
                // ---- online softmax per head over the chunk's tokens (lanes t and t + 16 agree)
                float pw[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    pw[g] = 0.f;
                    if (g < G) {
                        const float dot = sd[g] + __shfl_xor_sync(full, sd[g], 16);
                        const float x = t < nv ? dot * sl : -INFINITY;
                        float mx = x;
                        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 1));
                        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 2));
                        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
                        if (mx > m_run[g]) {  // the same in every lane
                            const float al = ex2(m_run[g] - mx);
                            l_run[g] *= al;
#pragma unroll
                            for (int i = 0; i < kPer; ++i) o[g][i] *= al;
                            m_run[g] = mx;
                        }
                        const float pv = ex2(x - m_run[g]);  // 0 past the context
                        float ps = pv;
                        ps += __shfl_xor_sync(full, ps, 1);
                        ps += __shfl_xor_sync(full, ps, 2);
                        ps += __shfl_xor_sync(full, ps, 4);
                        ps += __shfl_xor_sync(full, ps, 8);
                        l_run[g] += ps;
                        pw[g] = pv;
                    }
                }
                // ---- O += p V: columns d0 .. d0 + kPer of every head; tokens past the context are not read
#pragma unroll
                for (int tt = 0; tt < 16; ++tt) {
                    if (tt < nv) {
                        const uint32_t vaddr = vst + (uint32_t)((d0 / 64) * C::kBoxBytes) + (uint32_t)(tt * 128) +
                                               ((uint32_t)(((d0 % 64) / 8) ^ (tt & 7)) << 4) + (uint32_t)((d0 % 8) * 2);
                        float vf[kPer];
                        if constexpr (kPer == 4) {
                            uint32_t w0, w1;
                            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(vaddr));
                            const float2 a0 = widen2<T>(w0), a1 = widen2<T>(w1);
                            vf[0] = a0.x, vf[1] = a0.y, vf[2] = a1.x, vf[3] = a1.y;
                        } else {
                            uint32_t w0;
                            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w0) : "r"(vaddr));
                            const float2 a0 = widen2<T>(w0);
                            vf[0] = a0.x, vf[1] = a0.y;
                        }
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            if (g < G) {
                                const float pg = __shfl_sync(full, pw[g], tt);
#pragma unroll
                                for (int i = 0; i < kPer; ++i) o[g][i] = fmaf(pg, vf[i], o[g][i]);
                            }
                        }
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            ++cons;
        }
        if (timed_out) break;
        // ---- finish: whole-sequence items write out[], partitions their (m, l, acc)
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            if (g < G) {
                const int h = kvh * G + g;
                if (np == 1) {
                    const float inv = l_run[g] > 0.f ? 1.f / l_run[g] : 0.f;
                    float *orow = a.out + ((size_t)s * a.Hq + h) * D + d0;
#pragma unroll
                    for (int i = 0; i < kPer; ++i) orow[i] = o[g][i] * inv;
                } else {
                    const size_t r = ((size_t)s * a.Hq + h) * a.max_parts + p;
                    float *acc = a.ws_acc + r * D + d0;
#pragma unroll
                    for (int i = 0; i < kPer; ++i) acc[i] = o[g][i];
                    if (lane == 0) *reinterpret_cast<float2 *>(a.ws_ml + 2 * r) = make_float2(m_run[g], l_run[g]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(iempty0 + 8 * slot);
    }
}
#endif  // PA_DECODE_CUDA_CORE

template <typename T, int D, int B, int HG>
__global__ void __launch_bounds__(MmaCfg<D, HG>::kThreads, 2)
    decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    using C = MmaCfg<D, HG>;
    using M = Mma16<T>;
    constexpr int kCPB = B / 16;  // chunks per block
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-aligned: the 128-byte swizzle repeats every 1 KB
    unsigned char *basep = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = a.Hq / a.Hkv;
    const int ngroups = a.Hkv / HG;

    const uint32_t full0 = base + (uint32_t)C::kFullOff;
    const uint32_t empty0 = base + (uint32_t)C::kEmptyOff;
    const uint32_t ifull0 = base + (uint32_t)C::kItemFullOff;
    const uint32_t iempty0 = base + (uint32_t)C::kItemEmptyOff;
    int4 *info = reinterpret_cast<int4 *>(basep + C::kInfoOff);     // [slot * 2]: (s, p, ntok, np), (g0, nchunk, valid, -)
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
    // Right after this call's own plan kernel (a.early), everything before the
    // plan is complete when this grid starts, so the caches, tables and lengths
    // may be read at once; only the producer waits, for the plan's list, before
    // its first claim.  Otherwise wait here for the kernel before this one.
    if (!a.early) griddep_wait();
    // The merge kernel may be scheduled now: it only waits (griddepcontrol.wait)
    // beside this grid, which already fills every SM, and starts on completion.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- lane roles in the MMA fragments
    const int g = lane >> 2;         // fragment row = query head within the group (rows 8-15: P_lo)
    const int c2 = (lane & 3) * 2;   // fragment column pair
    const int lm = lane >> 3;        // ldmatrix: which 8x8 matrix this lane addresses
    const int lr = lane & 7;         // ldmatrix: which row of it
    const uint32_t kx = (uint32_t)(lm ^ lr);          // swizzled chunk bits for K reads
    const uint32_t vx = (uint32_t)((lm >> 1) ^ lr);   // and for V reads
    const float sl = a.scale * 1.4426950408889634f;   // logits in log2 units

    // ------------------------------------------------------------ producer warp
    // The last warp claims work items, fills the item slots, and issues the TMA
    // loads, up to kStages chunks ahead of the consumer warps and across item
    // boundaries; it never consumes, so a claim (an atomic, the list entry and
    // the item's table slice) overlaps the chunks already in the ring instead
    // of stalling it.  CTA b's first item is partition 0 of sequence
    // b / ngroups, head group b % ngroups, for the first min(S, grid / ngroups)
    // sequences (b < nstatic), else list entry b - nstatic; the plan's list
    // holds every item but the direct ones, and each later item is claimed
    // from the counter only when the issue cursor reaches it (a few chunks
    // before it is consumed).  Claiming any earlier would fix each CTA's last
    // item while the list still holds bigger ones, and the largest-first order
    // would no longer bound the tail.
    if (warp == C::kConsumers) {
        const uint64_t pol = policy_evict_first();
        const int nstatic = min(a.S, (int)gridDim.x / ngroups) * ngroups;  // items taken without the list
        const int cap = a.max_blocks * B;
        bool listed = false;  // the plan's list is complete and visible
        int n_items = 0;
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
            int4 e = make_int4(0, 0, 0, 0);
            int g0 = 0;
            bool have = false;
            if (seq == 0 && (int)blockIdx.x < nstatic) {
                const int s = blockIdx.x / ngroups;
                int len = a.context_lens[s];
                len = len < 0 ? 0 : (len > cap ? cap : len);  // the plan flags bad lengths
                if (len > 0) {
                    e = make_int4(s, 0, min(a.partition_size, len), (len + a.partition_size - 1) / a.partition_size);
                    g0 = (blockIdx.x % ngroups) * HG;
                    have = true;
                }
            }
            if (!have) {
                if (!listed) {
                    griddep_wait();
                    n_items = a.plan_hdr[0];
                    listed = true;
                }
                // CTAs past the directly taken items start with list entry
                // b - nstatic, without an atomic; later claims follow them
                int idx = 0;
                if (seq == 0 && (int)blockIdx.x >= nstatic) idx = blockIdx.x - nstatic;
                else if (lane == 0) idx = (int)gridDim.x - nstatic + atomicAdd(a.plan_hdr + 1, 1);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                if (idx < n_items) {
                    e = a.plan_list[idx / ngroups];
                    g0 = (idx % ngroups) * HG;
                    have = true;
                }
            }
            int4 e0 = make_int4(0, 0, 0, 0), e1 = make_int4(0, 0, 0, 0);
            int32_t *tb = tbl + slot * C::kTblCap;
            if (have) {
                e0 = e;
                e1 = make_int4(g0, (e.z + 15) >> 4, 1, 0);
                const int nblk = (e.z + B - 1) / B;
                const int32_t *row = a.block_tables + (size_t)e.x * a.max_blocks + (size_t)e.y * (a.partition_size / B);
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
                info[2 * slot] = e0;
                info[2 * slot + 1] = e1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ifull0 + 8 * slot);  // release: info and table visible
            if (!have) break;
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
        // This warp made every claim of the CTA.  The last CTA to get here
        // resets the counters, so the plan's list can serve the next launch
        // (after the plan itself, which resets them first, has completed).
        if (!listed) griddep_wait();
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(a.plan_hdr + 2, 1) == (int)gridDim.x - 1) {
                a.plan_hdr[1] = 0;
                a.plan_hdr[2] = 0;
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumer warps
    // Every consumer warp walks the same sequence of items (slot by slot) and
    // chunks (stage by stage); warp w computes the item's KV head g0 + w.
#if PA_DECODE_CUDA_CORE
    consumer_cuda_core<T, D, B, HG>(a, base, full0, empty0, ifull0, iempty0, info, tbl, warp, lane);
    return;
#endif
    uint32_t qa[C::kKS][2];
    int cons = 0;  // chunks consumed by this warp
    for (int seq = 0;; ++seq) {
        const int slot = seq % C::kSlots;
        if (!mbar_wait_bounded(ifull0 + 8 * slot, (uint32_t)(seq / C::kSlots) & 1u, kWaitLimit)) {
            if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
            break;
        }
        const int4 e0 = info[2 * slot];
        const int4 e1 = info[2 * slot + 1];
        if (!e1.z) break;  // no more work
        const int s = e0.x, p = e0.y, ntok = e0.z, np = e0.w;
        const int kvh = e1.x + warp;
        const int nchunk = e1.y;
        const int32_t *ctb = tbl + slot * C::kTblCap;
        {
            const int h = kvh * G + g;
            const uint16_t *qrow = static_cast<const uint16_t *>(a.q) + ((size_t)s * a.Hq + h) * D;
#pragma unroll
            for (int ks = 0; ks < C::kKS; ++ks) {
                qa[ks][0] = g < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + c2) : 0u;
                qa[ks][1] = g < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + c2) : 0u;
            }
        }
        float o[C::kNT][4];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
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
            const uint32_t kst = base + (uint32_t)(st * C::kStageBytes) + (uint32_t)(warp * C::kHeadSub);
            const uint32_t vst = kst + C::kTileBytes;
            if (nv > 0) {
                if (nv < 16) {
                    // tail chunk: zero this head's V rows past the context (whole
                    // 128-byte rows, so the swizzle does not matter)
                    const int nz = (16 - nv) * C::kSub * 8;
                    for (int i = lane; i < nz; i += 32) {
                        const int chunk = i & 7;
                        const int rowi = i >> 3;
                        const int sb = rowi / (16 - nv);
                        const int r = nv + rowi % (16 - nv);
                        const uint32_t addr = vst + sb * C::kBoxBytes + r * 128 + chunk * 16;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
                    }
                    __syncwarp();
                }
                // ---- S = Q K^T for 16 tokens (two n-tiles of 8), two accumulators
                // per n-tile (even / odd k-steps) to halve the MMA dependency chain
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
                        M::mma(sc[nt][0], qa[2 * ks2][0], 0u, qa[2 * ks2][1], 0u, b0, b1);
                        M::mma(sc[nt][1], qa[2 * ks2 + 1][0], 0u, qa[2 * ks2 + 1][1], 0u, b2, b3);
                    }
                }
                // ---- online softmax on this lane's row g, tokens c2, c2+1, 8+c2, 9+c2
                float x[4] = {(sc[0][0][0] + sc[0][1][0]) * sl, (sc[0][0][1] + sc[0][1][1]) * sl,
                              (sc[1][0][0] + sc[1][1][0]) * sl, (sc[1][0][1] + sc[1][1][1]) * sl};
                if (nv < 16) {
                    if (c2 >= nv) x[0] = -INFINITY;
                    if (c2 + 1 >= nv) x[1] = -INFINITY;
                    if (c2 + 8 >= nv) x[2] = -INFINITY;
                    if (c2 + 9 >= nv) x[3] = -INFINITY;
                }
                float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (__any_sync(0xffffffffu, mx > m_run)) {
                    const float mn = fmaxf(m_run, mx);
                    const float al = ex2(m_run - mn);
                    l_run *= al;
#pragma unroll
                    for (int nt = 0; nt < C::kNT; ++nt) {
                        o[nt][0] *= al;
                        o[nt][1] *= al;
                        o[nt][2] *= al;
                        o[nt][3] *= al;
                    }
                    m_run = mn;
                }
                float pr[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) pr[i] = ex2(x[i] - m_run);
                l_run += (pr[0] + pr[1]) + (pr[2] + pr[3]);
                // P = P_hi + P_lo, both 16-bit: rows 0-7 of A carry P_hi, rows 8-15 P_lo
                const uint32_t h01 = M::pack(pr[0], pr[1]);
                const uint32_t h23 = M::pack(pr[2], pr[3]);
                const float2 f01 = M::unpack(h01);
                const float2 f23 = M::unpack(h23);
                const uint32_t l01 = M::pack(pr[0] - f01.x, pr[1] - f01.y);
                const uint32_t l23 = M::pack(pr[2] - f23.x, pr[3] - f23.y);
                // ---- O += P V
#pragma unroll
                for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                    const uint32_t addr = vst + (uint32_t)((ntp >> 2) * C::kBoxBytes) +
                                          (uint32_t)(((lm & 1) * 8 + lr) * 128) +
                                          (((uint32_t)(2 * (ntp & 3)) ^ vx) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    M::mma(o[2 * ntp], h01, l01, h23, l23, b0, b1);
                    M::mma(o[2 * ntp + 1], h01, l01, h23, l23, b2, b3);
                }
            }
            // release the stage: order these generic shared-memory accesses before
            // the next bulk copy into it, then count this warp out
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            ++cons;
        }
        if (timed_out) break;

        // ---- finish this warp's head of the item
        float lt = l_run;
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        const int h = kvh * G + g;
        if (np == 1) {
            if (g < G) {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                float *orow = a.out + ((size_t)s * a.Hq + h) * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(orow + nt * 8 + c2) =
                        make_float2((o[nt][0] + o[nt][2]) * inv, (o[nt][1] + o[nt][3]) * inv);
            }
        } else {
            if (g < G) {
                const size_t r = ((size_t)s * a.Hq + h) * a.max_parts + p;
                float *acc = a.ws_acc + r * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(acc + nt * 8 + c2) =
                        make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
                if ((lane & 3) == 0) *reinterpret_cast<float2 *>(a.ws_ml + 2 * r) = make_float2(m_run, lt);
            }

        }
        __syncwarp();
        if (lane == 0) mbar_arrive(iempty0 + 8 * slot);  // this warp is done with the item slot
    }
}

// Grid of the persistent kernel on the current device: SMs x resident CTAs
// per SM (the shared-memory attribute is set on first use per device).
template <typename T, int D, int B, int HG>
cudaError_t decode_mma_grid(int *grid) {
    using C = MmaCfg<D, HG>;
    static std::atomic<int> grid_for[kMaxLaunchDevices];
    return per_device_value(grid_for, grid, [](int dev, int *v) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<T, D, B, HG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel<T, D, B, HG>, C::kThreads,
                                                          C::kSmem);
        if (e != cudaSuccess) return e;
        *v = sms * (per_sm > 0 ? per_sm : 1);
        return cudaSuccess;
    });
}

template <typename T, int D, int B, int HG>
cudaError_t launch_decode_mma_t(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t st) {
    using C = MmaCfg<D, HG>;
    int grid = 0;
    cudaError_t e = decode_mma_grid<T, D, B, HG>(&grid);
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
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<T, D, B, HG>, a, tmk, tmv);
}

template <typename T, int D, int B>
cudaError_t dispatch_decode_mma_hg(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   cudaStream_t st) {
    switch (a.head_group) {
#if PA_MMA_HEAD_GROUP >= 8
        case 8: return launch_decode_mma_t<T, D, B, 8>(a, tmk, tmv, st);
#endif
        case 4: return launch_decode_mma_t<T, D, B, 4>(a, tmk, tmv, st);
        case 2: return launch_decode_mma_t<T, D, B, 2>(a, tmk, tmv, st);
        default: return launch_decode_mma_t<T, D, B, 1>(a, tmk, tmv, st);
    }
}

template <typename T>
cudaError_t dispatch_decode_mma(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t st) {
    if (a.D == 64 && a.B == 16) return dispatch_decode_mma_hg<T, 64, 16>(a, tmk, tmv, st);
    if (a.D == 64 && a.B == 32) return dispatch_decode_mma_hg<T, 64, 32>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 16) return dispatch_decode_mma_hg<T, 128, 16>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 32) return dispatch_decode_mma_hg<T, 128, 32>(a, tmk, tmv, st);
    return cudaErrorNotSupported;
}

template <typename T, int D, int B>
cudaError_t decode_mma_grid_hg(const DecodeArgs &a, int *grid) {
    switch (a.head_group) {
#if PA_MMA_HEAD_GROUP >= 8
        case 8: return decode_mma_grid<T, D, B, 8>(grid);
#endif
        case 4: return decode_mma_grid<T, D, B, 4>(grid);
        case 2: return decode_mma_grid<T, D, B, 2>(grid);
        default: return decode_mma_grid<T, D, B, 1>(grid);
    }
}

template <typename T>
cudaError_t dispatch_decode_mma_grid(const DecodeArgs &a, int *grid) {
    if (a.D == 64 && a.B == 16) return decode_mma_grid_hg<T, 64, 16>(a, grid);
    if (a.D == 64 && a.B == 32) return decode_mma_grid_hg<T, 64, 32>(a, grid);
    if (a.D == 128 && a.B == 16) return decode_mma_grid_hg<T, 128, 16>(a, grid);
    if (a.D == 128 && a.B == 32) return decode_mma_grid_hg<T, 128, 32>(a, grid);
    return cudaErrorNotSupported;
}

}  // namespace pa
