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
// Work: a work item is one (sequence, KV head, context partition).  A small
// plan kernel lists the items, largest first, in the workspace.  Every warp of
// this persistent kernel is an independent decode engine: it claims items
// from a global counter, keeps the next item's block-table slice in shared
// memory, and streams the item's KV tiles through its own ring of shared-
// memory stages.  Lane 0 fills a stage with TMA tensor copies
// (cp.async.bulk.tensor, 128-byte swizzle): the K rows and the V rows of one
// (physical block, KV head).  The ring runs across item boundaries, so HBM
// stays busy while a warp finishes an item.
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
// otherwise it stores (m, l, acc) for its partition, and the warp that
// completes the last partition of a (sequence, KV head) merges them.
#pragma once

#include <cuda.h>

#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename T>
struct Mma16;

template <>
struct Mma16<__nv_bfloat16> {
    static __device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // x0 goes to the low half (the lower-indexed element of a fragment pair)
    static __device__ __forceinline__ uint32_t pack(float x0, float x1) {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
        return d;
    }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
};

template <>
struct Mma16<__half> {
    static __device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    static __device__ __forceinline__ uint32_t pack(float x0, float x1) {
        uint32_t d;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
        return d;
    }
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
};

// ------------------------------------------------------------------ configuration
// A stage holds one 16-token chunk of one (physical block, KV head): its K rows
// and its V rows, each split into 128-byte-wide swizzled sub-tiles.  A 32-slot
// block is two chunks.
template <int D>
struct MmaCfg {
    static constexpr int kKS = D / 16;          // k-steps of q.k
    static constexpr int kNT = D / 8;           // 8-wide n-tiles of p.v
    static constexpr int kSub = D / 64;         // 128-byte swizzled sub-tiles per row
    static constexpr int kSubBytes = kChunkRows * 128;  // one sub-tile of a 16-token chunk
    static constexpr int kTileBytes = kSub * kSubBytes;  // K (or V) rows of a chunk
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kWarps = 8;
    static constexpr int kStages = (192 * 1024) / (kWarps * kStageBytes);
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kTblCap = kMaxPartitionBlocks;  // table entries per item slot
    static constexpr size_t kBarsOff = (size_t)kWarps * kStages * kStageBytes;
    static constexpr size_t kTblOff = kBarsOff + (size_t)kWarps * kStages * 8;
    static constexpr size_t kSmem = kTblOff + (size_t)kWarps * 2 * kTblCap * 4 + 1024;  // + alignment slack
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(kChunkRows == 16, "one chunk is one m16n8k16 k-extent of tokens");
    static_assert(kStages >= 2, "stages");
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// One work item: partition p of sequence s, for one KV head.  ntok tokens from
// p * partition_size; np = partitions of the sequence.
struct WorkItem {
    int s, kvh, p, np, ntok, nchunk;
};

template <typename T, int D, int B>
__global__ void __launch_bounds__(MmaCfg<D>::kThreads, 1)
    decode_mma_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    using C = MmaCfg<D>;
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

    const uint32_t st0 = base + (uint32_t)(warp * C::kStages * C::kStageBytes);
    const uint32_t bar0 = base + (uint32_t)C::kBarsOff + (uint32_t)(warp * C::kStages * 8);
    int32_t *tbl = reinterpret_cast<int32_t *>(basep + C::kTblOff) + warp * 2 * C::kTblCap;

    if (lane == 0) {
        for (int i = 0; i < C::kStages; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
        if (warp == 0) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
        }
    }
    __syncwarp();
    griddep_wait();  // the plan kernel's work list must be complete (no-op without PDL)
    const int n_items = a.plan_hdr[0];

    // ---- lane roles in the MMA fragments
    const int g = lane >> 2;         // fragment row = query head within the group (rows 8-15: P_lo)
    const int c2 = (lane & 3) * 2;   // fragment column pair
    const int lm = lane >> 3;        // ldmatrix: which 8x8 matrix this lane addresses
    const int lr = lane & 7;         // ldmatrix: which row of it
    const uint32_t kx = (uint32_t)(lm ^ lr);          // swizzled chunk bits for K reads
    const uint32_t vx = (uint32_t)((lm >> 1) ^ lr);   // and for V reads
    const float sl = a.scale * 1.4426950408889634f;   // logits in log2 units

    // Claims are pipelined: the counter is bumped one item ahead, so the atomic's
    // latency is hidden behind the current item's work.
    int ticket = 0;
    if (lane == 0) ticket = atomicAdd(a.plan_hdr + 1, 1);
    // Turn the pending ticket into a work item: its plan entry, its block-table
    // slice (into tb) and its query fragments (into qf); then take the next ticket.
    auto claim = [&](WorkItem &it, int32_t *tb, uint32_t (&qf)[C::kKS][2]) -> bool {
        const int idx = __shfl_sync(0xffffffffu, ticket, 0);
        if (lane == 0) ticket = atomicAdd(a.plan_hdr + 1, 1);
        if (idx >= n_items) return false;
        const int4 e = a.plan_list[idx / a.Hkv];
        it.s = e.x;
        it.p = e.y;
        it.ntok = e.z;
        it.np = e.w;
        it.kvh = idx % a.Hkv;
        it.nchunk = (it.ntok + 15) >> 4;
        const int nblk = (it.ntok + B - 1) / B;
        const int32_t *row = a.block_tables + (size_t)it.s * a.max_blocks + (size_t)it.p * (Pt / B);
        int pbv[(kMaxPartitionBlocks + 31) / 32];
#pragma unroll
        for (int k = 0; k < (kMaxPartitionBlocks + 31) / 32; ++k) {
            const int i = lane + 32 * k;
            pbv[k] = i < nblk ? row[i] : 0;
            if (32 * (k + 1) >= nblk) break;
        }
        const int h = it.kvh * G + g;
        const uint16_t *qrow = static_cast<const uint16_t *>(a.q) + ((size_t)it.s * a.Hq + h) * D;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
            qf[ks][0] = g < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + c2) : 0u;
            qf[ks][1] = g < G ? *reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8 + c2) : 0u;
        }
#pragma unroll
        for (int k = 0; k < (kMaxPartitionBlocks + 31) / 32; ++k) {
            const int i = lane + 32 * k;
            if (i < nblk) {
                int pb = pbv[k];
                if (pb < 0 || pb >= a.N) {
                    set_error(a.err, PA_DEVERR_BAD_BLOCK);
                    pb = -1;
                }
                tb[i] = pb;
            }
            if (32 * (k + 1) >= nblk) break;
        }
        __syncwarp();
        return true;
    };

    int iss = 0, cons = 0;
    auto issue_chunk = [&](const int32_t *tb, int ci, int kvh) {
        const int slot = iss % C::kStages;
        const uint32_t bar = bar0 + 8 * slot;
        if (lane == 0) {
            const int pb = tb[ci / kCPB];
            if (pb < 0) {
                mbar_arrive(bar);  // bad table entry: complete the phase without data
            } else {
                const uint32_t dst = st0 + (uint32_t)(slot * C::kStageBytes);
                const int y = (pb * a.Hkv + kvh) * B + (ci % kCPB) * 16;
                mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
                for (int sb = 0; sb < C::kSub; ++sb) {
                    tma_load_2d(dst + sb * C::kSubBytes, &tmk, sb * 64, y, bar);
                    tma_load_2d(dst + C::kTileBytes + sb * C::kSubBytes, &tmv, sb * 64, y, bar);
                }
            }
        }
        ++iss;
    };

    WorkItem cur, nxt;
    uint32_t qa[C::kKS][2], qn[C::kKS][2];
    int cs = 0;  // table slot of cur
    if (!claim(cur, tbl, qa)) return;
    bool has_nxt = claim(nxt, tbl + C::kTblCap, qn);
    int iss_sel = 0, iss_j = 0;  // issue cursor: item (0 = cur, 1 = nxt) and chunk within it
    auto top_up = [&]() {
        while (iss - cons < C::kStages) {
            if (iss_sel == 0) {
                if (iss_j < cur.nchunk) {
                    issue_chunk(tbl + cs * C::kTblCap, iss_j, cur.kvh);
                    ++iss_j;
                    continue;
                }
                if (!has_nxt) break;
                iss_sel = 1;
                iss_j = 0;
            }
            if (iss_j < nxt.nchunk) {
                issue_chunk(tbl + (cs ^ 1) * C::kTblCap, iss_j, nxt.kvh);
                ++iss_j;
                continue;
            }
            break;
        }
    };

    while (true) {
        float o[C::kNT][4];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        const int32_t *ctb = tbl + cs * C::kTblCap;

        for (int j = 0; j < cur.nchunk; ++j) {
            top_up();
            const int slot = cons % C::kStages;
            const uint32_t parity = (uint32_t)(cons / C::kStages) & 1u;
            const bool got = mbar_wait_bounded(bar0 + 8 * slot, parity, kWaitLimit);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
                for (int k = cons + 1; k < iss; ++k)  // drain this warp's copies in flight
                    mbar_wait_bounded(bar0 + 8 * (k % C::kStages), (uint32_t)(k / C::kStages) & 1u, kWaitLimit);
                return;
            }
            const int nv = ctb[j / kCPB] < 0 ? 0 : min(16, cur.ntok - j * 16);
            const uint32_t kst = st0 + (uint32_t)(slot * C::kStageBytes);
            const uint32_t vst = kst + C::kTileBytes;
            if (nv > 0) {
                if (nv < 16) {
                    // tail chunk: zero the V rows past the context (whole 128-byte rows,
                    // so the swizzle does not matter)
                    const int nz = (16 - nv) * C::kSub * 8;
                    for (int i = lane; i < nz; i += 32) {
                        const int chunk = i & 7;
                        const int rowi = i >> 3;
                        const int sb = rowi / (16 - nv);
                        const int r = nv + rowi % (16 - nv);
                        const uint32_t addr = vst + sb * C::kSubBytes + r * 128 + chunk * 16;
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
                        const uint32_t addr = kst + (uint32_t)((ks2 >> 1) * C::kSubBytes) +
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
                float p[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) p[i] = ex2(x[i] - m_run);
                l_run += (p[0] + p[1]) + (p[2] + p[3]);
                // P = P_hi + P_lo, both 16-bit: rows 0-7 of A carry P_hi, rows 8-15 P_lo
                const uint32_t h01 = M::pack(p[0], p[1]);
                const uint32_t h23 = M::pack(p[2], p[3]);
                const float2 f01 = M::unpack(h01);
                const float2 f23 = M::unpack(h23);
                const uint32_t l01 = M::pack(p[0] - f01.x, p[1] - f01.y);
                const uint32_t l23 = M::pack(p[2] - f23.x, p[3] - f23.y);
                // ---- O += P V
#pragma unroll
                for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                    const uint32_t addr = vst + (uint32_t)((ntp >> 2) * C::kSubBytes) +
                                          (uint32_t)(((lm & 1) * 8 + lr) * 128) +
                                          (((uint32_t)(2 * (ntp & 3)) ^ vx) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    M::mma(o[2 * ntp], h01, l01, h23, l23, b0, b1);
                    M::mma(o[2 * ntp + 1], h01, l01, h23, l23, b2, b3);
                }
            }
            // the stage is consumed: order these generic shared-memory accesses
            // before the next bulk copy into it, then let lane 0 reuse it
            fence_proxy_async_smem();
            __syncwarp();
            ++cons;
        }

        // ---- finish the item
        float lt = l_run;
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        const int h = cur.kvh * G + g;
        if (cur.np == 1) {
            if (g < G) {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                float *orow = a.out + ((size_t)cur.s * a.Hq + h) * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(orow + nt * 8 + c2) =
                        make_float2((o[nt][0] + o[nt][2]) * inv, (o[nt][1] + o[nt][3]) * inv);
            }
        } else {
            if (g < G) {
                const size_t r = ((size_t)cur.s * a.Hq + h) * a.max_parts + cur.p;
                float *acc = a.ws_acc + r * D;
#pragma unroll
                for (int nt = 0; nt < C::kNT; ++nt)
                    *reinterpret_cast<float2 *>(acc + nt * 8 + c2) =
                        make_float2(o[nt][0] + o[nt][2], o[nt][1] + o[nt][3]);
                if ((lane & 3) == 0) *reinterpret_cast<float2 *>(a.ws_ml + 2 * r) = make_float2(m_run, lt);
            }
            __threadfence();
            __syncwarp();
            int done = 0;
            if (lane == 0) done = atomicAdd(a.plan_cnt + (size_t)cur.s * a.Hkv + cur.kvh, 1);
            done = __shfl_sync(0xffffffffu, done, 0);
            if (done == cur.np - 1) {  // last partition of this (sequence, KV head): merge
                __threadfence();
                constexpr int kPer = D / 32;
                for (int gg = 0; gg < G; ++gg) {
                    const size_t r0 = ((size_t)cur.s * a.Hq + cur.kvh * G + gg) * a.max_parts;
                    float Mx = -INFINITY;
                    for (int pp = lane; pp < cur.np; pp += 32) Mx = fmaxf(Mx, __ldcg(a.ws_ml + 2 * (r0 + pp)));
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
                    float L = 0.f, acc[kPer];
#pragma unroll
                    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
                    if (Mx != -INFINITY) {
                        for (int pp = 0; pp < cur.np; ++pp) {
                            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.ws_ml + 2 * (r0 + pp)));
                            const float w = ex2(ml.x - Mx);
                            L += w * ml.y;
                            const float *src = a.ws_acc + (r0 + pp) * D + lane * kPer;
                            if constexpr (kPer == 4) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                                acc[0] += w * v.x;
                                acc[1] += w * v.y;
                                acc[2] += w * v.z;
                                acc[3] += w * v.w;
                            } else {
                                const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                                acc[0] += w * v.x;
                                acc[1] += w * v.y;
                            }
                        }
                    }
                    const float inv = L > 0.f ? 1.f / L : 0.f;
                    float *dst = a.out + ((size_t)cur.s * a.Hq + cur.kvh * G + gg) * D + lane * kPer;
#pragma unroll
                    for (int i = 0; i < kPer; ++i) dst[i] = acc[i] * inv;
                }
            }
        }

        if (!has_nxt) break;
        cur = nxt;
        cs ^= 1;
#pragma unroll
        for (int ks = 0; ks < C::kKS; ++ks) {
            qa[ks][0] = qn[ks][0];
            qa[ks][1] = qn[ks][1];
        }
        if (iss_sel == 1)
            iss_sel = 0;  // the cursor was already streaming the new current item
        else
            iss_j = 0;
        has_nxt = claim(nxt, tbl + (cs ^ 1) * C::kTblCap, qn);
    }
}

template <typename T, int D, int B>
cudaError_t launch_decode_mma_t(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t st) {
    using C = MmaCfg<D>;
    static bool configured[64] = {};
    static int grid_for[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(decode_mma_kernel<T, D, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::kSmem);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_mma_kernel<T, D, B>, C::kThreads,
                                                          C::kSmem);
        if (e != cudaSuccess) return e;
        grid_for[dev] = sms * (per_sm > 0 ? per_sm : 1);
        configured[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid_for[dev]);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<T, D, B>, a, tmk, tmv);
}

template <typename T>
cudaError_t dispatch_decode_mma(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t st) {
    if (a.D == 64 && a.B == 16) return launch_decode_mma_t<T, 64, 16>(a, tmk, tmv, st);
    if (a.D == 64 && a.B == 32) return launch_decode_mma_t<T, 64, 32>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 16) return launch_decode_mma_t<T, 128, 16>(a, tmk, tmv, st);
    if (a.D == 128 && a.B == 32) return launch_decode_mma_t<T, 128, 32>(a, tmk, tmv, st);
    return cudaErrorNotSupported;
}

}  // namespace pa
