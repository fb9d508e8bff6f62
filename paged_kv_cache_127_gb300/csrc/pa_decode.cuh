// pa_decode.cuh -- PagedAttention decode kernels for sm_103a.
//
// What is computed ("Paged Attention and vLLM", "Block Table and
// Logical-to-Physical Mapping", the a_t equation; "Paged Attention CUDA Kernel",
// the per-partition m_b / l_b / v_b^acc terms and the log-sum-exp merge):
//
//   out[s, h] = softmax(scale * q[s, h] . [K_tau(0) || K_tau(1) || ...]^T) . V
//
// over the context_lens[s] tokens of sequence s, gathered through its block
// table inside the kernel (no contiguous K/V is ever built).
//
// Work decomposition
//   grid.x = S * Hkv (sequence, KV head), grid.y = context partition.  A CTA
//   handles the G = Hq / Hkv query heads that share one KV head, so every K/V
//   byte of the pool is read from HBM once per decode ("grouped-query
//   attention stores fewer KV heads than query heads").  Partitions of
//   partition_size tokens split long contexts across CTAs (split-K); a
//   sequence that fits in one partition is finished in place, otherwise each
//   CTA leaves (m, l, acc[D]) per query head in the workspace for the merge
//   kernel.
//
// Inside a CTA
//   kWarps warps share the partition's blocks round-robin.  Each warp owns a
//   private ring of kStages shared-memory stages; lane 0 fills a stage with
//   two 1-D bulk copies (cp.async.bulk, the TMA engine) -- the K rows and the
//   V rows of one (physical block, KV head), each B*D contiguous elements --
//   signalled through an mbarrier with a transaction count.  While a warp
//   computes on one stage the next ones are in flight.
//   K phase: a token row (D elements = LPT 16-byte chunks) is spread over LPT
//   lanes; each lane multiplies its chunk by the G query chunks it keeps in
//   registers, for TL tokens at once, then the partial dot products are
//   reduced across the LPT lanes with a transposing butterfly: the lane's
//   token order is permuted (XOR with a lane-dependent mask) so each step sends
//   the upper half of the registers and adds into the lower half, with no
//   selects.
//   Softmax: per warp, online max / sum in log2 units (q is pre-scaled by
//   scale * log2 e, so exp is one ex2); the running sums are rescaled only
//   when the warp's maximum grows.
//   V phase: each lane accumulates p * v for its chunk of D over the tile's
//   tokens; masked (tail) tokens are skipped, never multiplied by p = 0, so
//   NaN in unused slots cannot leak.
//   The warps' (m, l, acc) are merged in shared memory at the end.
#pragma once

#include <cmath>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <typename T, int D, int B, int G>
struct DecodeCfg {
    static constexpr int kEB = Elem<T>::kBytes;
    static constexpr int kVec = Elem<T>::kVec;        // elements per 16-byte chunk
    static constexpr int kLPT = D / kVec;             // lanes per token row
    static_assert(kLPT >= 8 && kLPT <= 32 && (kLPT & (kLPT - 1)) == 0, "unsupported D/dtype");
    static constexpr int kTPP = 32 / kLPT;            // token rows per warp pass
    static constexpr int kTLraw = B / kTPP;
    static constexpr int kTL = kTLraw < 8 ? kTLraw : 8;  // tokens per lane per tile
    static_assert(kTL >= 1 && kTL <= kLPT, "tile shape");
    static constexpr int kLogTL = ilog2(kTL);
    static constexpr int kLogLPT = ilog2(kLPT);
    static constexpr int kTT = kTL * kTPP;            // tokens per tile
    static constexpr int kTiles = B / kTT;            // tiles per block
    static_assert(kTiles * kTT == B, "tile shape");
    static constexpr int kRowBytes = D * kEB;
    static constexpr int kBlkBytes = B * kRowBytes;   // K (or V) rows of one (block, head)
    static constexpr int kStageBytes = 2 * kBlkBytes;
    static constexpr int kWarps = (4 * 2 * kStageBytes <= 200 * 1024) ? 4 : 2;
    static constexpr int kStagesRaw = (96 * 1024) / (kWarps * kStageBytes);
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 4 ? 4 : kStagesRaw);
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kWarpStageBytes = kStages * kStageBytes;
    static constexpr int kRecFloats = G * D + 2 * G;  // a warp's (acc, m, l) record
    static_assert(kRecFloats * 4 <= kWarpStageBytes, "record must fit in the warp's stages");
    static constexpr size_t kSmemStages = (size_t)kWarps * kWarpStageBytes;
    static constexpr size_t kSmemBars = (size_t)kWarps * kStages * 8;
    static constexpr size_t kSmemTable = (size_t)kMaxPartitionBlocks * 4;
    static constexpr size_t kSmemP = (size_t)kWarps * kTT * G * 4;
    static constexpr size_t kSmem = kSmemStages + kSmemBars + kSmemTable + kSmemP + 16;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

template <typename T, int D, int B, int G>
__global__ void __launch_bounds__(DecodeCfg<T, D, B, G>::kThreads)
    decode_partition_kernel(const DecodeArgs a) {
    using C = DecodeCfg<T, D, B, G>;
    extern __shared__ __align__(128) unsigned char smem[];

    const int kvh = blockIdx.x % a.Hkv;
    const int s = blockIdx.x / a.Hkv;
    const int part = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    int len = a.context_lens[s];
    const int cap = a.max_blocks * B;
    if (len < 0 || len > cap) {
        if (threadIdx.x == 0 && part == 0 && kvh == 0) set_error(a.err, PA_DEVERR_BAD_LEN);
        len = len < 0 ? 0 : cap;
    }
    const int Pt = a.partition_size;
    const int nparts = (len + Pt - 1) / Pt;
    if (len == 0) {  // empty context: zero output rows
        if (part == 0)
            for (int i = threadIdx.x; i < G * D; i += C::kThreads)
                a.out[((size_t)s * a.Hq + kvh * G) * D + i] = 0.f;
        return;
    }
    if (part >= nparts) return;

    const int tok0 = part * Pt;              // multiple of B
    const int tok1 = min(len, tok0 + Pt);
    const int blk0 = tok0 / B;
    const int nblk = (tok1 - tok0 + B - 1) / B;

    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kSmemStages);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + C::kSmemStages + C::kSmemBars);
    float *pbuf = reinterpret_cast<float *>(smem + C::kSmemStages + C::kSmemBars + C::kSmemTable);
    volatile int &s_abort = *reinterpret_cast<int *>(smem + C::kSmem - 16);

    // bulk copies need 16-byte aligned destinations; the stage offsets are
    // multiples of 16, so only the base needs checking
    if (smem_addr(smem) & 15u) {
        if (threadIdx.x == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
        return;
    }
    if (threadIdx.x == 0) s_abort = 0;
    const int32_t *trow = a.block_tables + (size_t)s * a.max_blocks + blk0;
    for (int i = threadIdx.x; i < nblk; i += C::kThreads) {
        int p = trow[i];
        if (p < 0 || p >= a.N) {
            set_error(a.err, PA_DEVERR_BAD_BLOCK);
            p = -1;
        }
        tbl[i] = p;
    }
    const uint32_t bar0 = smem_addr(bars + warp * C::kStages);
    if (lane == 0) {
        for (int i = 0; i < C::kStages; ++i) mbar_init(bar0 + 8 * i, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // this warp's blocks: jb = warp + k * kWarps, k = 0 .. nk-1
    const int nk = warp < nblk ? (nblk - warp + C::kWarps - 1) / C::kWarps : 0;
    const uint32_t wst = smem_addr(stages + warp * C::kWarpStageBytes);
    const char *kbase = static_cast<const char *>(a.k_cache);
    const char *vbase = static_cast<const char *>(a.v_cache);

    auto issue = [&](int k) {  // lane 0 only
        const int jb = warp + k * C::kWarps;
        const int slot = k % C::kStages;
        const uint32_t bar = bar0 + 8 * slot;
        const int p = tbl[jb];
        if (p < 0) {  // bad table entry: complete the phase with no data
            mbar_arrive(bar);
            return;
        }
        const size_t off = ((size_t)p * a.Hkv + kvh) * C::kBlkBytes;
        const uint32_t dst = wst + slot * C::kStageBytes;
        mbar_arrive_expect_tx(bar, 2 * C::kBlkBytes);
        bulk_g2s(dst, kbase + off, C::kBlkBytes, bar);
        bulk_g2s(dst + C::kBlkBytes, vbase + off, C::kBlkBytes, bar);
    };
    if (lane == 0) {
        const int npro = nk < C::kStages ? nk : C::kStages;
        for (int k = 0; k < npro; ++k) issue(k);
    }

    // lane roles
    const int sub = lane / C::kLPT;  // token row within a pass
    const int li = lane % C::kLPT;   // 16-byte chunk of the row
    int mask = 0;                    // token permutation for the transposing reduction
#pragma unroll
    for (int k = 0; k < C::kLogTL; ++k)
        mask |= ((li >> (C::kLogLPT - 1 - k)) & 1) << (C::kLogTL - 1 - k);
    const bool leader = (li & ((1 << (C::kLogLPT - C::kLogTL)) - 1)) == 0;

    // the G query chunks, pre-scaled so that logits come out in log2 units
    float qf[G][C::kVec];
    {
        const float qs = a.scale * 1.4426950408889634f;
        const char *qb = static_cast<const char *>(a.q);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 c = *reinterpret_cast<const uint4 *>(
                qb + (((size_t)s * a.Hq + kvh * G + g) * D + li * C::kVec) * C::kEB);
            Elem<T>::unpack(c, qf[g]);
#pragma unroll
            for (int e = 0; e < C::kVec; ++e) qf[g][e] *= qs;
        }
    }

    float m_run[G], l_run[G], acc[G][C::kVec];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int e = 0; e < C::kVec; ++e) acc[g][e] = 0.f;
    }
    float *wp = pbuf + warp * C::kTT * G;

    int kfail = nk;
    for (int k = 0; k < nk; ++k) {
        const int slot = k % C::kStages;
        const uint32_t parity = (k / C::kStages) & 1;
        const bool got = mbar_wait_bounded(bar0 + 8 * slot, parity, kWaitLimit);
        if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) set_error(a.err, PA_DEVERR_TIMEOUT);
            kfail = k;
            break;
        }
        const int jb = warp + k * C::kWarps;
        const int nvalid = tbl[jb] < 0 ? 0 : min(B, tok1 - (tok0 + jb * B));
        const uint32_t kst = wst + slot * C::kStageBytes;
        const uint32_t vst = kst + C::kBlkBytes;

#pragma unroll
        for (int tt = 0; tt < C::kTiles; ++tt) {
            const int tbase = tt * C::kTT;
            if (tbase >= nvalid) break;

            // ---- K phase: partial dots for kTL tokens, G heads
            float pd[C::kTL][G];
#pragma unroll
            for (int r = 0; r < C::kTL; ++r) {
                const int t = tbase + (r ^ mask) * C::kTPP + sub;
                const uint4 c = lds128(kst + t * C::kRowBytes + li * 16);
                float kf[C::kVec];
                Elem<T>::unpack(c, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float d = 0.f;
#pragma unroll
                    for (int e = 0; e < C::kVec; ++e) d = fmaf(qf[g][e], kf[e], d);
                    pd[r][g] = d;
                }
            }
            // transposing reduction across the LPT lanes of a row
#pragma unroll
            for (int st = 0; st < C::kLogTL; ++st) {
                const int half = C::kTL >> (st + 1);
                const int off = C::kLPT >> (st + 1);
#pragma unroll
                for (int r = 0; r < half; ++r)
#pragma unroll
                    for (int g = 0; g < G; ++g)
                        pd[r][g] += __shfl_xor_sync(0xffffffffu, pd[r + half][g], off);
            }
#pragma unroll
            for (int off = C::kLPT >> (C::kLogTL + 1); off >= 1; off >>= 1)
#pragma unroll
                for (int g = 0; g < G; ++g) pd[0][g] += __shfl_xor_sync(0xffffffffu, pd[0][g], off);

            // ---- online softmax (log2 domain)
            const int tmine = mask * C::kTPP + sub;  // this lane's token within the tile
            const bool valid = tbase + tmine < nvalid;
            float sc[G], mx[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                sc[g] = valid ? pd[0][g] : -INFINITY;
                mx[g] = sc[g];
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
                for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], off));
            bool grow = false;
#pragma unroll
            for (int g = 0; g < G; ++g) grow |= mx[g] > m_run[g];
            if (grow) {  // warp-uniform
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float mn = fmaxf(m_run[g], mx[g]);
                    const float alpha = ex2(m_run[g] - mn);
                    l_run[g] *= alpha;
#pragma unroll
                    for (int e = 0; e < C::kVec; ++e) acc[g][e] *= alpha;
                    m_run[g] = mn;
                }
            }
            if (leader) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = ex2(sc[g] - m_run[g]);
                    l_run[g] += p;
                    wp[tmine * G + g] = p;
                }
            }
            __syncwarp();

            // ---- V phase: acc += p * v over the tile's valid tokens
#pragma unroll
            for (int r = 0; r < C::kTL; ++r) {
                const int ti = r * C::kTPP + sub;
                if (tbase + ti < nvalid) {
                    const uint4 c = lds128(vst + (tbase + ti) * C::kRowBytes + li * 16);
                    float vf[C::kVec];
                    Elem<T>::unpack(c, vf);
                    float pv[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) pv[g] = wp[ti * G + g];
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < C::kVec; ++e) acc[g][e] = fmaf(pv[g], vf[e], acc[g][e]);
                }
            }
            __syncwarp();
        }
        // stage consumed: refill it with the block kStages ahead
        if (lane == 0 && k + C::kStages < nk) {
            fence_proxy_async_smem();
            issue(k + C::kStages);
        }
        __syncwarp();
    }

    if (kfail < nk) {  // timed out: drain what is still in flight, then give up
        const int kend = min(nk, kfail + C::kStages);
        for (int k = kfail; k < kend; ++k)
            mbar_wait_bounded(bar0 + 8 * (k % C::kStages), (k / C::kStages) & 1, kWaitLimit);
        if (lane == 0) s_abort = 1;
    }

    // ---- warp result: sum acc over the kTPP rows, l over the warp
#pragma unroll
    for (int off = C::kLPT; off < 32; off <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::kVec; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], off);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int g = 0; g < G; ++g) l_run[g] += __shfl_xor_sync(0xffffffffu, l_run[g], off);

    // the warp's stages are all consumed: reuse them for its record
    float *rec = reinterpret_cast<float *>(stages + warp * C::kWarpStageBytes);
    if (sub == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::kVec; e += 4)
                *reinterpret_cast<float4 *>(rec + g * D + li * C::kVec + e) =
                    make_float4(acc[g][e], acc[g][e + 1], acc[g][e + 2], acc[g][e + 3]);
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            rec[G * D + g] = m_run[g];
            rec[G * D + G + g] = l_run[g];
        }
    }
    __syncthreads();
    if (s_abort) return;

    // ---- merge the warps; finish in place or leave a partial for the merge kernel
    for (int it = threadIdx.x; it < G * D / 4; it += C::kThreads) {
        const int g = it / (D / 4);
        const int d = (it % (D / 4)) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
            const float *rw = reinterpret_cast<const float *>(stages + w * C::kWarpStageBytes);
            M = fmaxf(M, rw[G * D + g]);
        }
        float L = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < C::kWarps; ++w) {
                const float *rw = reinterpret_cast<const float *>(stages + w * C::kWarpStageBytes);
                const float sw = ex2(rw[G * D + g] - M);
                L += sw * rw[G * D + G + g];
                const float4 x = *reinterpret_cast<const float4 *>(rw + g * D + d);
                A.x += sw * x.x;
                A.y += sw * x.y;
                A.z += sw * x.z;
                A.w += sw * x.w;
            }
        }
        const int h = kvh * G + g;
        if (nparts == 1) {
            const float inv = L > 0.f ? 1.f / L : 0.f;
            *reinterpret_cast<float4 *>(a.out + ((size_t)s * a.Hq + h) * D + d) =
                make_float4(A.x * inv, A.y * inv, A.z * inv, A.w * inv);
        } else {
            const size_t r = ((size_t)s * a.Hq + h) * a.max_parts + part;
            *reinterpret_cast<float4 *>(a.ws_acc + r * D + d) = A;
            if (d == 0) {
                a.ws_ml[2 * r] = M;
                a.ws_ml[2 * r + 1] = L;
            }
        }
    }
}

template <typename T, int D, int B, int G>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t st) {
    using C = DecodeCfg<T, D, B, G>;
    static std::atomic<int> configured[kMaxLaunchDevices];
    int one = 0;
    cudaError_t e = per_device_value(configured, &one, [](int, int *v) {
        *v = 1;
        return cudaFuncSetAttribute(decode_partition_kernel<T, D, B, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::kSmem);
    });
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(a.S * a.Hkv), (unsigned)a.max_parts);
    decode_partition_kernel<T, D, B, G><<<grid, C::kThreads, C::kSmem, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_decode(const DecodeArgs &a, cudaStream_t st) {
    const int G = a.Hq / a.Hkv;
#define PA_DECODE_CASE(D_, B_, G_) \
    if (a.D == D_ && a.B == B_ && G == G_) return launch_decode_t<T, D_, B_, G_>(a, st);
#define PA_DECODE_CASES_DB(D_, B_) \
    PA_DECODE_CASE(D_, B_, 1) PA_DECODE_CASE(D_, B_, 2) PA_DECODE_CASE(D_, B_, 4) PA_DECODE_CASE(D_, B_, 8)
    PA_DECODE_CASES_DB(64, 16)
    PA_DECODE_CASES_DB(64, 32)
    PA_DECODE_CASES_DB(128, 16)
    PA_DECODE_CASES_DB(128, 32)
#undef PA_DECODE_CASES_DB
#undef PA_DECODE_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
