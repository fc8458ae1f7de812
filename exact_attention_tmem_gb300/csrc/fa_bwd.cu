// fa_bwd.cu — backward pass of exact attention on sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes ("FlashAttention" deep dive, section "How it works": the backward
// pass recomputes P = exp(Q K^T * scale - L) per tile from the saved L, then uses
// D = rowsum(dO o O) and dS = P o (dP - D) to form dQ, dK and dV).  With the scale
// inside S, the chain rule gives dV = P^T dO, dP = dO V^T, dK = scale * dS^T Q and
// dQ = scale * dS K.
//
// Three kernels on the caller's stream:
//  1. bwd_pre:  D_i = sum_t dO_it O_it (fp32), the negated logsumexp in base 2
//               (-L * log2 e), both padded to whole 128-row tiles (padding rows get
//               D = 0 and -L = -inf, so their probabilities are exactly 0), and the
//               fp32 dQ accumulator cleared.
//  2. bwd_main: one CTA per (batch*head, 128-key block j).  K_j and V_j stay in
//               shared memory; the CTA walks the query blocks i (i >= j when causal:
//               blocks above the diagonal are skipped) and per block runs five
//               tcgen05 products:
//                 S^T  = K_j Q_i^T          (TMEM)        -> P^T = 2^(S^T*scale*log2e - L2_i)
//                 dP^T = V_j dO_i^T         (TMEM)        -> dS^T = P^T o (dP^T - D_i)
//                 dV  += P^T dO_i           (A = P^T from TMEM)
//                 dQ_i = dS K_j             (A = dS from shared memory, MN-major)
//                 dK  += dS^T Q_i           (A = the same tile, K-major)
//               dQ_i leaves tensor memory in 32-column boxes through a ring of two
//               16 KB shared buffers (one box is written while the previous one is
//               being reduced) and TMA bulk reduce-add (fp32) into the dQ accumulator;
//               dK and dV accumulate in TMEM for the whole walk and are written once.
//  3. bwd_post: dQ = bf16(scale * accumulator).
//
// Tensor memory (512 columns): dK [0, d) | dV [d, 2d) | S^T [2d, 2d+128) | dP^T [2d+128,
// 2d+256).  P^T (bf16) is written over the first 64 S^T columns, and dQ_i accumulates in
// the dP^T columns once the softmax warps have read dP^T.  Per query block the MMA warp
// issues dQ_i | dK_i | dP^T_{i+1} (after the dQ_i read-out) | dV_{i+1}, and the S^T
// warp S^T_{i+2} once Q_{i+2} has landed: the read-out gates only the next dP^T.
//
// Warp roles (352 threads): warps 0-3 own one key row each (softmax recompute and dS),
// warps 4-7 own one query row each (dQ read-out, staging and bulk reduce), warp 8
// issues the MMAs, warp 9 issues the TMA loads, and warp 10 issues the S^T products
// of the single-pass kernel (the MMA warp issues them in the dK/dV-only kernel, where
// warp 10 has nothing to do).  Every wait is time-limited (see
// ptx.cuh).  The shared-memory budget at d = 128 is within 1 KB of the 227 KB limit,
// so the kernel relies on the dynamic shared window starting 1024-byte aligned and
// checks it instead of over-allocating (a misaligned start is reported, not used).
#include <climits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// Both tiled kernels: warp 8 issues the MMAs, warp 9 the TMA loads.  The key-block
// kernel (bwd_main_kernel) has an eleventh warp that issues the S^T products of the
// single-pass variant, so that the MMA warp never blocks on a Q tile while dS_i is
// ready; the query-block kernel (bwd_dq_kernel) has ten warps.
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kSWarp = 10;
constexpr int kMainThreads = 352;
constexpr int kDqThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

// kDQ = false (the dK/dV-only kernel) needs neither the dS tile nor the dQ staging
// tile, and spends the room on a third Q stage and a second dO stage, so that the
// loads run far enough ahead to hide their latency.  The base-2 logsumexp and D of
// query block i have their own ring of two slots: they are read until dS_i is done.
template <int D, bool kDQ>
struct BwdCfg {
    static constexpr int kBoxes = D * 2 / kBoxBytes;
    static constexpr int kBoxTileBytes = kTileRows * kBoxBytes;    // 16 KB
    static constexpr int kTileBytes = kBoxes * kBoxTileBytes;
    static constexpr int kQStages = kDQ ? 2 : 3;
    static constexpr int kDOStages = (D == 128 && kDQ) ? 1 : 2;
    static constexpr int kVecStages = 2;
    static constexpr int kVecBytes = kTileRows * 4;                 // 128 fp32
    static constexpr int kDSBytes = kDQ ? 2 * kBoxTileBytes : 0;    // 128 x 128 bf16
    // dQ staging: a ring of two box buffers of 32 fp32 columns x 128 rows (16 KB each)
    static constexpr int kDQStageBytes = kDQ ? 2 * kTileRows * 32 * 4 : 0;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kKOff + kTileBytes;
    static constexpr int kQOff = kVOff + kTileBytes;
    static constexpr int kDOOff = kQOff + kQStages * kTileBytes;
    static constexpr int kDSOff = kDOOff + kDOStages * kTileBytes;
    static constexpr int kDQOff = kDSOff + kDSBytes;
    static constexpr int kLOff = kDQOff + kDQStageBytes;
    static constexpr int kDOff = kLOff + kVecStages * kVecBytes;
    static constexpr int kBarOff = kDOff + kVecStages * kVecBytes;
    static constexpr int kNumBars = 1 + 2 * kQStages + 2 * kDOStages + kVecStages + 10;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16;
    // tensor memory
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kDKCol = 0;
    static constexpr uint32_t kDVCol = D;
    static constexpr uint32_t kSCol = 2 * D;
    static constexpr uint32_t kDPCol = 2 * D + 128;
    static constexpr int kKSteps = D / 16;          // K steps over the head dim
    static constexpr int kRowSteps = kTileRows / 16; // K steps over 128 rows
    static constexpr uint32_t kIdescSS = make_idesc(kFormatBF16, 128, 128, false, false);
    static constexpr uint32_t kIdescTS = make_idesc(kFormatBF16, 128, D, false, true);

    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(2 * D + 256 <= 512, "tensor memory budget");
};

template <int QS, int DS, int VS>
struct BwdBars {
    static constexpr int kKV = 0;
    static constexpr int kQFull = 1;                 // + stage
    static constexpr int kQEmpty = 1 + QS;           // + stage
    static constexpr int kDOFull = 1 + 2 * QS;       // + stage
    static constexpr int kDOEmpty = 1 + 2 * QS + DS; // + stage
    static constexpr int kVecFull = 1 + 2 * QS + 2 * DS;  // + slot
    static constexpr int kSFull = 1 + 2 * QS + 2 * DS + VS;
    static constexpr int kDPFull = kSFull + 1;
    static constexpr int kPFull = kSFull + 2;
    static constexpr int kDSFull = kSFull + 3;
    static constexpr int kDQFull = kSFull + 4;
    static constexpr int kDQFree = kSFull + 5;
    static constexpr int kDrain = kSFull + 6;
    static constexpr int kDVIssued = kSFull + 7;   // dV_i handed to the tensor pipe (S^T_{i+1} may follow)
    static constexpr int kSDrain = kSFull + 8;     // the S^T warp's products have completed
    static constexpr int kDVDone = kSFull + 9;     // the last dV product has completed
};

enum : int {
    kSiteBLoadQ = 31, kSiteBLoadDO = 32, kSiteBMmaKV = 33, kSiteBMmaQ = 34, kSiteBMmaDO = 35,
    kSiteBMmaP = 36, kSiteBMmaDS = 37, kSiteBMmaDQ = 38, kSiteBSoftS = 39, kSiteBSoftL = 40,
    kSiteBSoftDP = 41, kSiteBMisaligned = 42, kSiteBDQ = 43, kSiteBEpi = 44, kSiteBDrain = 45
};

// ------------------------------------------------------------------------------------
// 1. pre-processing: D, base-2 logsumexp (padded), cleared dQ accumulator
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
bwd_pre_kernel(const __nv_bfloat16 *__restrict__ o, const __nv_bfloat16 *__restrict__ dout,
               const float *__restrict__ lse, float *__restrict__ delta, float *__restrict__ lse2,
               float *__restrict__ dq_acc, int N, int Npad, int BH) {
    // The main kernel is launched as this grid's dependent: it may start its set-up (and
    // its loads of Q, K, V, dO) as soon as every CTA of this grid is running, and waits
    // for this grid's results before it reads D, L or the accumulator.
    grid_launch_dependents();
    constexpr int kLanesPerRow = D / 8;              // 16-byte chunks per row
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    constexpr int kUnroll = 4;                       // row groups in flight per warp
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanesPerRow;
    const int part = lane % kLanesPerRow;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long total_rows = static_cast<long long>(BH) * Npad;
    for (long long base = warp_global * kRowsPerWarp * kUnroll; base < total_rows;
         base += nwarps * kRowsPerWarp * kUnroll) {
        // all loads of the group first, then the sums
        uint4 a[kUnroll], b[kUnroll];
        float lv[kUnroll];
        bool valid[kUnroll];
        long long rr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            rr[u] = base + u * kRowsPerWarp + sub;
            valid[u] = false;
            a[u] = make_uint4(0u, 0u, 0u, 0u);
            b[u] = a[u];
            lv[u] = 0.f;
            if (rr[u] < total_rows) {
                const long long bh = rr[u] / Npad;
                const int i = static_cast<int>(rr[u] - bh * Npad);
                valid[u] = i < N;
                if (valid[u]) {
                    const long long src_row = bh * N + i;
                    a[u] = reinterpret_cast<const uint4 *>(o + src_row * D)[part];
                    b[u] = reinterpret_cast<const uint4 *>(dout + src_row * D)[part];
                    if (part == 0) lv[u] = lse[src_row];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            float acc = 0.f;
            const __nv_bfloat162 *pa = reinterpret_cast<const __nv_bfloat162 *>(&a[u]);
            const __nv_bfloat162 *pb = reinterpret_cast<const __nv_bfloat162 *>(&b[u]);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 fa = __bfloat1622float2(pa[t]);
                const float2 fb = __bfloat1622float2(pb[t]);
                acc = fmaf(fa.x, fb.x, acc);
                acc = fmaf(fa.y, fb.y, acc);
            }
#pragma unroll
            for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (rr[u] < total_rows && part == 0) {
                delta[rr[u]] = valid[u] ? acc : 0.f;
                lse2[rr[u]] = valid[u] ? -lv[u] * kLog2e : -INFINITY;
            }
        }
    }
    if (dq_acc == nullptr) return;   // the deterministic backward has no accumulator
    const long long n4 = static_cast<long long>(BH) * N * D / 4;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    float4 *acc4 = reinterpret_cast<float4 *>(dq_acc);
    for (long long x = tid; x < n4; x += nthreads) acc4[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ------------------------------------------------------------------------------------
// 3. post-processing: dQ = bf16(scale * accumulator)
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
bwd_post_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dq, long long n8, float scale) {
    grid_dependency_wait();   // launched as the main kernel's dependent: its reductions are in
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const float4 *src = reinterpret_cast<const float4 *>(dq_acc);
    uint4 *dst = reinterpret_cast<uint4 *>(dq);
    for (long long x = tid; x < n8; x += nthreads) {
        const float4 a = src[2 * x], b = src[2 * x + 1];
        uint4 w;
        w.x = pack_bf16(a.x * scale, a.y * scale);
        w.y = pack_bf16(a.z * scale, a.w * scale);
        w.z = pack_bf16(b.x * scale, b.y * scale);
        w.w = pack_bf16(b.z * scale, b.w * scale);
        dst[x] = w;
    }
}

// ------------------------------------------------------------------------------------
// 2. main kernel
// ------------------------------------------------------------------------------------
// kDQ = false: the key-block kernel of the deterministic backward, which computes dK and
// dV only (dQ comes from bwd_dq_kernel); per query block the MMA warp then issues
// dV_i | S^T_{i+1} | dK_i | dP^T_{i+1}, and dS is not staged in shared memory.
template <int D, bool kDQ>
__global__ void __launch_bounds__(kMainThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const float *__restrict__ lse2,
                const float *__restrict__ delta,
                __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, int N, int Npad, int nkv,
                int group, float scale, float scale_log2, int causal, unsigned int *status) {
    using C = BwdCfg<D, kDQ>;
    using B = BwdBars<C::kQStages, C::kDOStages, C::kVecStages>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if ((base & 1023u) != 0) {  // see the note at the top of this file
        if (threadIdx.x == 0 && atomicOr(&status[0], kStatusTimeout) == 0u) status[1] = kSiteBMisaligned;
        return;
    }
    uint8_t *smem = smem_raw;
    const uint32_t sK = base + C::kKOff, sV = base + C::kVOff, sQ = base + C::kQOff;
    const uint32_t sDO = base + C::kDOOff, sDS = base + C::kDSOff, sDQ = base + C::kDQOff;
    const uint32_t sL = base + C::kLOff, sD = base + C::kDOff, sBar = base + C::kBarOff;
    uint8_t *dS_ptr = smem + C::kDSOff;
    uint8_t *dQ_stage = smem + C::kDQOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx wc{abort_flag, status};
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int bh, j;                               // key/value head, key block
    heavy_first_order(blockIdx.x, nkv, bh, j);   // j = 0 (the longest causal walk) first
    const int nq = Npad / kTileRows;
    const int i0 = causal ? j : 0;
    const int n_q = nq - i0;                 // query blocks per query head (>= 1)
    // The walk covers the query blocks of every query head that shares this key/value
    // head (grouped-query attention; group = 1 is plain multi-head attention):
    // iteration `it` is query head bh*group + it / n_q, query block i0 + it % n_q.
    const int n_it = group * n_q;
    auto q_head = [&](int it) { return bh * group + it / n_q; };
    auto q_block = [&](int it) { return i0 + it % n_q; };

    if (threadIdx.x == 0) {
        mbar_init(bar(B::kKV), 1);
        for (int s = 0; s < C::kQStages; ++s) {
            mbar_init(bar(B::kQFull + s), 1);
            mbar_init(bar(B::kQEmpty + s), 1);
        }
        for (int s = 0; s < C::kDOStages; ++s) {
            mbar_init(bar(B::kDOFull + s), 1);
            mbar_init(bar(B::kDOEmpty + s), 1);
        }
        for (int s = 0; s < C::kVecStages; ++s) mbar_init(bar(B::kVecFull + s), 1);
        mbar_init(bar(B::kSFull), 1);
        mbar_init(bar(B::kDPFull), 1);
        mbar_init(bar(B::kPFull), 128);
        mbar_init(bar(B::kDSFull), 128);
        mbar_init(bar(B::kDQFull), 1);
        mbar_init(bar(B::kDQFree), 128);
        mbar_init(bar(B::kDrain), 1);
        mbar_init(bar(B::kDVIssued), 1);
        mbar_init(bar(B::kSDrain), 1);
        mbar_init(bar(B::kDVDone), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kLoadWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            if constexpr (kDQ) tma_prefetch_desc(&tm_dq);
            mbar_arrive_expect_tx(bar(B::kKV), 2 * C::kTileBytes);
            for (int b = 0; b < C::kBoxes; ++b) {
                tma_load_3d(sK + b * C::kBoxTileBytes, &tm_k, bar(B::kKV), b * 64, j * kTileRows, bh);
                tma_load_3d(sV + b * C::kBoxTileBytes, &tm_v, bar(B::kKV), b * 64, j * kTileRows, bh);
            }
            int q_loads = 0, do_loads = 0, vec_loads = 0;
            for (int it = 0; it < n_it; ++it) {
                const int i = q_block(it), hq = q_head(it);
                const float *lrow = lse2 + static_cast<int64_t>(hq) * Npad;
                const float *drow = delta + static_cast<int64_t>(hq) * Npad;
                const int qs = it % C::kQStages, qu = it / C::kQStages;
                if (qu > 0 && !mbar_wait(bar(B::kQEmpty + qs), (qu - 1) & 1, wc, kSiteBLoadQ)) break;
                mbar_arrive_expect_tx(bar(B::kQFull + qs), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sQ + qs * C::kTileBytes + b * C::kBoxTileBytes, &tm_q, bar(B::kQFull + qs),
                                b * 64, i * kTileRows, hq);
                ++q_loads;
                // the vectors of block it - kVecStages are free once dK of that block (the
                // end of its dS phase) has been issued and completed
                const int vs = it % C::kVecStages;
                if (it >= C::kVecStages) {
                    const int r = it - C::kVecStages;
                    if (!mbar_wait(bar(B::kQEmpty + r % C::kQStages), (r / C::kQStages) & 1, wc, kSiteBLoadQ)) break;
                }
                // D and L come from the pre-processing grid (this kernel may have started before it
                // finished): wait for that grid before the first vector load
                if (it == 0) grid_dependency_wait();
                mbar_arrive_expect_tx(bar(B::kVecFull + vs), 2 * C::kVecBytes);
                bulk_load(sL + vs * C::kVecBytes, lrow + i * kTileRows, C::kVecBytes, bar(B::kVecFull + vs));
                bulk_load(sD + vs * C::kVecBytes, drow + i * kTileRows, C::kVecBytes, bar(B::kVecFull + vs));
                ++vec_loads;
                const int ds = it % C::kDOStages, du = it / C::kDOStages;
                if (du > 0 && !mbar_wait(bar(B::kDOEmpty + ds), (du - 1) & 1, wc, kSiteBLoadDO)) break;
                mbar_arrive_expect_tx(bar(B::kDOFull + ds), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sDO + ds * C::kTileBytes + b * C::kBoxTileBytes, &tm_do, bar(B::kDOFull + ds),
                                b * 64, i * kTileRows, hq);
                ++do_loads;
            }
            // Every copy issued above must land before this CTA may exit: wait for the
            // last fill of every stage.
            mbar_wait_drain(bar(B::kKV), 0, wc, kSiteBDrain);
            for (int s = 0; s < C::kQStages && s < q_loads; ++s) {
                const int last = s + ((q_loads - 1 - s) / C::kQStages) * C::kQStages;
                mbar_wait_drain(bar(B::kQFull + s), (last / C::kQStages) & 1, wc, kSiteBDrain);
            }
            for (int s = 0; s < C::kDOStages && s < do_loads; ++s) {
                const int last = s + ((do_loads - 1 - s) / C::kDOStages) * C::kDOStages;
                mbar_wait_drain(bar(B::kDOFull + s), (last / C::kDOStages) & 1, wc, kSiteBDrain);
            }
            for (int s = 0; s < C::kVecStages && s < vec_loads; ++s) {
                const int last = s + ((vec_loads - 1 - s) / C::kVecStages) * C::kVecStages;
                mbar_wait_drain(bar(B::kVecFull + s), (last / C::kVecStages) & 1, wc, kSiteBDrain);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (every wait is warp-uniform) and lane 0 issues.
        {
            auto mbar_wait_w = [&](uint32_t b, uint32_t parity, int site) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
            };
            const uint32_t tDK = tmem + C::kDKCol, tDV = tmem + C::kDVCol;
            const uint32_t tS = tmem + C::kSCol, tDP = tmem + C::kDPCol;
            auto wait_q = [&](int it) -> int {
                const int s = it % C::kQStages;
                if (!mbar_wait_w(bar(B::kQFull + s), (it / C::kQStages) & 1, kSiteBMmaQ)) return -1;
                tc_fence_after();
                return s;
            };
            auto wait_do = [&](int it) -> int {
                const int s = it % C::kDOStages;
                if (!mbar_wait_w(bar(B::kDOFull + s), (it / C::kDOStages) & 1, kSiteBMmaDO)) return -1;
                tc_fence_after();
                return s;
            };
            // K-major x K-major product over the head dim: D[128 x 128] = A B^T (each
            // product goes out from one asm block; see umma_f16_ss_x8)
            auto mma_kk = [&](uint32_t d_tmem, uint32_t a_s, uint32_t b_s) {
                const uint64_t a0 = sdesc_sw128(a_s, 16, 1024), b0 = sdesc_sw128(b_s, 16, 1024);
                uint64_t a[C::kKSteps], b[C::kKSteps];
#pragma unroll
                for (int kk = 0; kk < C::kKSteps; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32;
                    a[kk] = sdesc_step(a0, off);
                    b[kk] = sdesc_step(b0, off);
                }
                if constexpr (C::kKSteps == 8) umma_f16_ss_x8(d_tmem, a, b, C::kIdescSS, 0u);
                else umma_f16_ss_x4(d_tmem, a, b, C::kIdescSS, 0u);
            };
            // A from TMEM (128 x 128, bf16 packed), B MN-major [128 rows x D], 16 rows per step
            auto mma_tn = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t b_s, bool acc) {
                const uint64_t b0 = sdesc_sw128(b_s, C::kBoxTileBytes, 1024);
                uint64_t b[C::kRowSteps];
#pragma unroll
                for (int kk = 0; kk < C::kRowSteps; ++kk) b[kk] = sdesc_step(b0, kk * 16 * kBoxBytes);
                umma_f16_ts_x8(d_tmem, a_tmem, b, C::kIdescTS, acc ? 1u : 0u);
            };
            bool ok = mbar_wait_w(bar(B::kKV), 0, kSiteBMmaKV);
            tc_fence_after();
            int qs = -1, dos = -1;
            if constexpr (!kDQ) {   // single pass: the S^T products come from the S^T warp
                if (ok) {
                    qs = wait_q(0);
                    ok = qs >= 0;
                }
                if (ok) {
                    mma_kk(tS, sK, sQ + qs * C::kTileBytes);
                    umma_commit(bar(B::kSFull));
                }
            }
            if (ok) {
                dos = wait_do(0);
                ok = dos >= 0;
            }
            if (ok) {
                mma_kk(tDP, sV, sDO + dos * C::kTileBytes);
                umma_commit(bar(B::kDPFull));
            }
            if constexpr (kDQ) {
                // dS_i is in shared memory only (the dS^T tile read K-major is dK's A
                // operand, read MN-major it is dQ's), so dQ_i goes first, into the dP^T
                // columns the softmax warps have finished reading.  Per query block:
                // dQ_i | dK_i | dP^T_{i+1} (after the dQ_i read-out) | dV_{i+1}, and the
                // S^T warp adds S^T_{i+2} once Q_{i+2} has landed and dV_{i+1} (which
                // reads P^T_{i+1} from the S^T columns) is in the pipe ahead of it.  The
                // chain from dS_i to dS_{i+1} is dQ, dK, the read-out and dP^T; dK_i
                // completes before dP^T_{i+1}, so the softmax warps overwrite the dS tile
                // only after both products have read it.
                if (ok) {  // dV_0
                    ok = mbar_wait_w(bar(B::kPFull), 0, kSiteBMmaP);
                    if (ok) {
                        tc_fence_after();
                        mma_tn(tDV, tS, sDO + dos * C::kTileBytes, false);
                        umma_commit(bar(B::kDOEmpty + dos));     // dP^T_0 and dV_0 have read dO_0
                        if (n_it == 1) umma_commit(bar(B::kDVDone));
                        if (lane == 0) mbar_arrive(bar(B::kDVIssued));
                    }
                }
                for (int it = 0; ok && it < n_it; ++it) {
                    const int qs_it = it % C::kQStages;
                    if (!mbar_wait_w(bar(B::kDSFull), it & 1, kSiteBMmaDS)) { ok = false; break; }
                    tc_fence_after();
                    {   // dQ_i = dS K_j (A = dS, MN-major) into the dP^T columns
                        const uint64_t a0 = sdesc_sw128(sDS, C::kBoxTileBytes, 1024);
                        const uint64_t b0 = sdesc_sw128(sK, C::kBoxTileBytes, 1024);
                        uint64_t a[C::kRowSteps], b[C::kRowSteps];
#pragma unroll
                        for (int kk = 0; kk < C::kRowSteps; ++kk) {
                            a[kk] = sdesc_step(a0, kk * 16 * kBoxBytes);
                            b[kk] = sdesc_step(b0, kk * 16 * kBoxBytes);
                        }
                        // A (dS) and B (K_j) both MN-major
                        constexpr uint32_t kIdescDQ = make_idesc(kFormatBF16, 128, D, true, true);
                        umma_f16_ss_x8(tDP, a, b, kIdescDQ, 0u);
                    }
                    umma_commit(bar(B::kDQFull));
                    {   // dK += dS^T Q_i (A = the same tile, K-major over the query rows)
                        const uint64_t a0 = sdesc_sw128(sDS, 16, 1024);
                        const uint64_t b0 = sdesc_sw128(sQ + qs_it * C::kTileBytes, C::kBoxTileBytes, 1024);
                        uint64_t a[C::kRowSteps], b[C::kRowSteps];
#pragma unroll
                        for (int kk = 0; kk < C::kRowSteps; ++kk) {
                            a[kk] = sdesc_step(a0, (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32);
                            b[kk] = sdesc_step(b0, kk * 16 * kBoxBytes);
                        }
                        umma_f16_ss_x8(tDK, a, b, C::kIdescTS, it > 0 ? 1u : 0u);
                    }
                    umma_commit(bar(B::kQEmpty + qs_it));
                    if (it + 1 < n_it) {
                        const int dn = wait_do(it + 1);
                        if (dn < 0) { ok = false; break; }
                        // dP^T_{i+1} once dQ_i has left the dP^T columns; it goes ahead of
                        // dV_{i+1}, so the softmax warps' P_{i+1} is off the path from dS_i
                        // to dS_{i+1} (it overlaps dQ_i, dK_i and dP^T_{i+1})
                        if (!mbar_wait_w(bar(B::kDQFree), it & 1, kSiteBMmaDQ)) { ok = false; break; }
                        tc_fence_after();
                        mma_kk(tDP, sV, sDO + dn * C::kTileBytes);
                        umma_commit(bar(B::kDPFull));
                        // dV += P^T dO_{i+1} (P^T from the S^T columns)
                        if (!mbar_wait_w(bar(B::kPFull), (it + 1) & 1, kSiteBMmaP)) { ok = false; break; }
                        tc_fence_after();
                        mma_tn(tDV, tS, sDO + dn * C::kTileBytes, true);
                        umma_commit(bar(B::kDOEmpty + dn));
                        if (it + 2 == n_it) umma_commit(bar(B::kDVDone));
                        if (lane == 0) mbar_arrive(bar(B::kDVIssued));
                    }
                }
            } else {
                for (int it = 0; ok && it < n_it; ++it) {
                    if (!mbar_wait_w(bar(B::kPFull), it & 1, kSiteBMmaP)) { ok = false; break; }
                    tc_fence_after();
                    mma_tn(tDV, tS, sDO + dos * C::kTileBytes, it > 0);
                    umma_commit(bar(B::kDOEmpty + dos));
                    if (it + 1 == n_it) umma_commit(bar(B::kDVDone));
                    int qs_next = -1;
                    if (it + 1 < n_it) {  // S^T_{i+1}: the S^T columns are free after dV_i
                        qs_next = wait_q(it + 1);
                        if (qs_next < 0) { ok = false; break; }
                        mma_kk(tS, sK, sQ + qs_next * C::kTileBytes);
                        umma_commit(bar(B::kSFull));
                    }
                    if (!mbar_wait_w(bar(B::kDSFull), it & 1, kSiteBMmaDS)) { ok = false; break; }
                    tc_fence_after();
                    mma_tn(tDK, tDP, sQ + qs * C::kTileBytes, it > 0);
                    umma_commit(bar(B::kQEmpty + qs));
                    qs = qs_next;
                    if (it + 1 < n_it) {  // dP^T_{i+1}: its columns are free after dK_i
                        dos = wait_do(it + 1);
                        if (dos < 0) { ok = false; break; }
                        mma_kk(tDP, sV, sDO + dos * C::kTileBytes);
                        umma_commit(bar(B::kDPFull));
                    }
                }
            }
            // Drain the tensor pipe before tensor memory can be released; the dK/dV
            // epilogue waits on the same commit (it follows the last dK product).
            umma_commit(bar(B::kDrain));
            mbar_wait_drain(bar(B::kDrain), 0, wc, kSiteBDrain);
        }
    } else if (warp == kSWarp) {
        // ------------------------------------------------------------ S^T issuer (single pass)
        // S^T_i = K_j Q_i^T once Q_i has landed and dV_{i-1} has been issued: the
        // product overwrites the S^T columns that dV_{i-1} reads, and the tensor pipe
        // runs products in the order they were issued.  The whole warp runs the loop;
        // lane 0 issues.
        if constexpr (kDQ) {
            auto wait_w = [&](uint32_t b, uint32_t parity, int site) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
            };
            const uint32_t tS = tmem + C::kSCol;
            bool ok = wait_w(bar(B::kKV), 0, kSiteBMmaKV);
            int issued = 0;
            for (int it = 0; ok && it < n_it; ++it) {
                const int qs = it % C::kQStages;
                if (!wait_w(bar(B::kQFull + qs), (it / C::kQStages) & 1, kSiteBMmaQ)) { ok = false; break; }
                if (it > 0 && !wait_w(bar(B::kDVIssued), (it - 1) & 1, kSiteBMmaP)) { ok = false; break; }
                tc_fence_after();
                const uint64_t a0 = sdesc_sw128(sK, 16, 1024);
                const uint64_t b0 = sdesc_sw128(sQ + qs * C::kTileBytes, 16, 1024);
                uint64_t a[C::kKSteps], b[C::kKSteps];
#pragma unroll
                for (int kk = 0; kk < C::kKSteps; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32;
                    a[kk] = sdesc_step(a0, off);
                    b[kk] = sdesc_step(b0, off);
                }
                if constexpr (C::kKSteps == 8) umma_f16_ss_x8(tS, a, b, C::kIdescSS, 0u);
                else umma_f16_ss_x4(tS, a, b, C::kIdescSS, 0u);
                umma_commit(bar(B::kSFull));
                ++issued;
            }
            // tensor memory is released after the final barrier: let this warp's
            // products finish first (they normally have long before)
            if (issued > 0) {
                umma_commit(bar(B::kSDrain));
                mbar_wait_drain(bar(B::kSDrain), 0, wc, kSiteBDrain);
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ key rows: P^T and dS^T
        const int c = warp * 32 + lane;                     // key row within the block
        const int kg = j * kTileRows + c;                   // global key index
        const bool key_valid = kg < N;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tSr = tmem + lane_off + C::kSCol;
        const uint32_t tDPr = tmem + lane_off + C::kDPCol;
        // this thread's row of dS^T in the MN-major, 128-byte swizzled shared tile
        uint8_t *ds_row0 = dS_ptr + c * kBoxBytes;
        const int swz = c & 7;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int i = q_block(it);
            const int vs = it % C::kVecStages;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull), it & 1, wc, kSiteBSoftS) &&
                                             mbar_wait(bar(B::kVecFull + vs), (it / C::kVecStages) & 1, wc, kSiteBSoftL));
            if (!ok) break;
            tc_fence_after();
            // P^T = 2^(S^T * scale*log2e - L2) in fp32, kept as packed bf16: the same values
            // feed the dV product (from TMEM) and dS below.
            uint32_t pk[64];
            {
                uint32_t sr[128];
                tmem_ld_x128(tSr, sr);
                const uint32_t nL = sL + vs * C::kVecBytes;   // -L * log2 e, 4 queries per load
                const float2 sl2 = make_float2(scale_log2, scale_log2);
                // causal: query q sees key c iff c <= q (same block offsets on the diagonal)
                const int qmin = (causal && i == j) ? c : 0;
                if (key_valid && qmin == 0) {
#pragma unroll
                    for (int u = 0; u < 64; u += 2) {
                        const float4 l4 = lds_f4(nL + 8 * u);
                        const float2 x0 = fma2(make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])),
                                               sl2, make_float2(l4.x, l4.y));
                        const float2 x1 = fma2(make_float2(__uint_as_float(sr[2 * u + 2]), __uint_as_float(sr[2 * u + 3])),
                                               sl2, make_float2(l4.z, l4.w));
                        pk[u] = pack_bf16(ex2(x0.x), ex2(x0.y));
                        pk[u + 1] = pack_bf16(ex2(x1.x), ex2(x1.y));
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 64; u += 2) {
                        const float4 l4 = lds_f4(nL + 8 * u);
                        const float2 x0 = fma2(make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])),
                                               sl2, make_float2(l4.x, l4.y));
                        const float2 x1 = fma2(make_float2(__uint_as_float(sr[2 * u + 2]), __uint_as_float(sr[2 * u + 3])),
                                               sl2, make_float2(l4.z, l4.w));
                        pk[u] = pack_bf16((key_valid && 2 * u >= qmin) ? ex2(x0.x) : 0.f,
                                          (key_valid && 2 * u + 1 >= qmin) ? ex2(x0.y) : 0.f);
                        pk[u + 1] = pack_bf16((key_valid && 2 * u + 2 >= qmin) ? ex2(x1.x) : 0.f,
                                              (key_valid && 2 * u + 3 >= qmin) ? ex2(x1.y) : 0.f);
                    }
                }
            }
            tmem_st_x64(tSr, pk);
            tc_fence_before();
            mbar_arrive(bar(B::kPFull));
            // dS^T = P^T o (dP^T - D)
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kDPFull), it & 1, wc, kSiteBSoftDP));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sDv = sD + vs * C::kVecBytes;   // D, 4 queries per load
            // 32 query columns at a time; the load of the next chunk is in flight while
            // this chunk is computed and stored
            uint32_t rbuf[2][32];
            tmem_ld_x32_nowait(tDPr, rbuf[0]);
            tmem_wait_ld_fence(rbuf[0]);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t (&r)[32] = rbuf[ch & 1];
                if (ch < 3) tmem_ld_x32_nowait(tDPr + 32u * (ch + 1), rbuf[(ch + 1) & 1]);
                uint32_t dk2[16];
#pragma unroll
                for (int t = 0; t < 16; t += 2) {
                    const float4 d4 = lds_f4(sDv + 4 * (32 * ch + 2 * t));
                    const uint32_t pp0 = pk[16 * ch + t], pp1 = pk[16 * ch + t + 1];
                    const float2 p0 = make_float2(__uint_as_float(pp0 << 16), __uint_as_float(pp0 & 0xffff0000u));
                    const float2 p1 = make_float2(__uint_as_float(pp1 << 16), __uint_as_float(pp1 & 0xffff0000u));
                    const float2 ds0 = mul2(p0, sub2(make_float2(__uint_as_float(r[2 * t]), __uint_as_float(r[2 * t + 1])),
                                                     make_float2(d4.x, d4.y)));
                    const float2 ds1 = mul2(p1, sub2(make_float2(__uint_as_float(r[2 * t + 2]),
                                                                 __uint_as_float(r[2 * t + 3])),
                                                     make_float2(d4.z, d4.w)));
                    dk2[t] = pack_bf16(ds0.x, ds0.y);
                    dk2[t + 1] = pack_bf16(ds1.x, ds1.y);
                }
                // shared: query columns 32*ch .. 32*ch+31 = box (ch / 2), 16-byte chunks
                // 4*(ch % 2) .. 4*(ch % 2)+3 of this key's row (read by the dQ and dK products)
                if constexpr (kDQ) {
                    uint8_t *box = ds_row0 + (ch >> 1) * C::kBoxTileBytes;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int chunk = 4 * (ch & 1) + u;
                        *reinterpret_cast<uint4 *>(box + ((chunk ^ swz) << 4)) =
                            make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
                    }
                }
                // tensor memory (the dK/dV-only kernel: dK reads dS^T from there): dS^T
                // packed over the first 64 dP^T columns (chunk ch writes columns 16ch..,
                // all of which have been read by now)
                if constexpr (!kDQ) asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                    "%12, %13, %14, %15, %16};\n\t" ::"r"(tDPr + 16u * ch),
                    "r"(dk2[0]), "r"(dk2[1]), "r"(dk2[2]), "r"(dk2[3]), "r"(dk2[4]), "r"(dk2[5]),
                    "r"(dk2[6]), "r"(dk2[7]), "r"(dk2[8]), "r"(dk2[9]), "r"(dk2[10]), "r"(dk2[11]),
                    "r"(dk2[12]), "r"(dk2[13]), "r"(dk2[14]), "r"(dk2[15])
                    : "memory");
                if (ch < 3) tmem_wait_ld_fence(rbuf[(ch + 1) & 1]);
            }
            if constexpr (!kDQ) asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            if constexpr (kDQ) fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(B::kDSFull));
        }
        // ------------------------------------------------------------ epilogue: dV row
        // dV is final once the last dV product has completed (dQ and dK of the last query
        // block may still be running)
        if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kDVDone), 0, wc, kSiteBEpi));
        }
        if (ok) {
            tc_fence_after();
            __nv_bfloat16 *row = dv + (static_cast<int64_t>(bh) * N + (key_valid ? kg : 0)) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t r[32];
                tmem_ld_x32(tmem + lane_off + C::kDVCol + 32u * ch, r);
                if (key_valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(row + 32 * ch);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(pack_bf16(__uint_as_float(r[8 * u]), __uint_as_float(r[8 * u + 1])),
                                            pack_bf16(__uint_as_float(r[8 * u + 2]), __uint_as_float(r[8 * u + 3])),
                                            pack_bf16(__uint_as_float(r[8 * u + 4]), __uint_as_float(r[8 * u + 5])),
                                            pack_bf16(__uint_as_float(r[8 * u + 6]), __uint_as_float(r[8 * u + 7])));
                }
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ query rows: dQ read-out
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                   // query row within the block
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tDQr = tmem + lane_off + C::kDPCol;  // dQ_i accumulates in the dP^T columns
        bool ok = true;
        int g = 0;   // dQ boxes issued so far
        // the accumulator is cleared by the pre-processing grid: wait for it before reducing
        if (kDQ && threadIdx.x == 128) grid_dependency_wait();
        for (int it = 0; kDQ && it < n_it; ++it) {
            const int i = q_block(it);
            // all 128 threads leave together, so none is left waiting at a named barrier
            ok = named_barrier_and(1, 128, mbar_wait(bar(B::kDQFull), it & 1, wc, kSiteBDQ));
            if (!ok) break;
            tc_fence_after();
            uint32_t v[D / 32][32];
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) tmem_ld_x32(tDQr + 32u * ch, v[ch]);
            tc_fence_before();
            mbar_arrive(bar(B::kDQFree));
            // dQ_i leaves in 32-column boxes (128 rows x 128 bytes, 128-byte swizzled)
            // through a ring of two box buffers: box g is written while the bulk
            // reduction of box g - 1 still reads the other buffer.  Rows past N fall
            // outside the tensor map and are dropped by the reduction.
#pragma unroll
            for (int b = 0; b < D / 32; ++b, ++g) {
                if (g >= 2) {   // buffer g & 1 was last read by box g - 2
                    if (threadIdx.x == 128) bulk_wait_group_read1();
                    named_barrier_sync(1, 128);
                }
                uint8_t *row = dQ_stage + (g & 1) * C::kBoxTileBytes + r * kBoxBytes;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4 *>(row + ((u ^ (r & 7)) << 4)) =
                        make_uint4(v[b][4 * u], v[b][4 * u + 1], v[b][4 * u + 2], v[b][4 * u + 3]);
                fence_proxy_async_smem();
                named_barrier_sync(1, 128);
                if (threadIdx.x == 128) {
                    tma_reduce_add_3d(&tm_dq, sDQ + (g & 1) * C::kBoxTileBytes, 32 * b, i * kTileRows, q_head(it));
                    bulk_commit_group();
                }
            }
        }
        // the staging buffers must have been read before the CTA releases its shared memory
        if (threadIdx.x == 128) bulk_wait_group_read0();
        // ------------------------------------------------------------ epilogue: dK row
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kDrain), 0, wc, kSiteBEpi));
        }
        if (ok) {
            tc_fence_after();
            const int kg = j * kTileRows + r;
            const bool key_valid = kg < N;
            __nv_bfloat16 *row = dk + (static_cast<int64_t>(bh) * N + (key_valid ? kg : 0)) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t v[32];
                tmem_ld_x32(tmem + lane_off + C::kDKCol + 32u * ch, v);
                if (key_valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(row + 32 * ch);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(
                            pack_bf16(__uint_as_float(v[8 * u]) * scale, __uint_as_float(v[8 * u + 1]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 2]) * scale, __uint_as_float(v[8 * u + 3]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 4]) * scale, __uint_as_float(v[8 * u + 5]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 6]) * scale, __uint_as_float(v[8 * u + 7]) * scale));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------------------------
// 4. query-block kernel of the deterministic backward: dQ with one writer per row
// ------------------------------------------------------------------------------------
// One CTA per (query head, pair of 128-row query tiles), the forward kernel's layout:
// Q_t and dO_t of both tiles stay in shared memory while K_j and V_j stream through
// their own rings (two K stages, so K_{j+1} is resident while dQ_t(j) still reads
// K_j).  Per key block j and tile t the tensor cores compute
//     S_t  = Q_t K_j^T           (TMEM, SD_t columns)   -> P = 2^(S*scale*log2e - L2)
//     dP_t = dO_t V_j^T          (TMEM, the same columns once S has been read)
//     dQ_t += dS_t K_j           (A = dS_t, packed bf16 over the first 64 SD_t columns)
// and dQ_t accumulates in TMEM across the whole walk in key-block order, so the
// result is the same bits on every run.  dQ = scale * dQ_t is written once.
// Tensor memory: SD_0 [0,128) | SD_1 [128,256) | dQ_0 [256,256+d) | dQ_1 [256+d,256+2d).
template <int D>
struct DqCfg {
    static constexpr int kBoxes = D * 2 / kBoxBytes;
    static constexpr int kBoxTileBytes = kTileRows * kBoxBytes;
    static constexpr int kTileBytes = kBoxes * kBoxTileBytes;
    static constexpr int kKStages = 2;
    static constexpr int kVStages = D == 128 ? 1 : 2;
    static constexpr int kQOff = 0;                          // Q_0, Q_1
    static constexpr int kDOOff = 2 * kTileBytes;            // dO_0, dO_1
    static constexpr int kKOff = 4 * kTileBytes;
    static constexpr int kVOff = kKOff + kKStages * kTileBytes;
    static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 8 + 1;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kDQCol = 256;
    static constexpr int kKSteps = D / 16;
    static constexpr int kRowSteps = kTileRows / 16;
    static constexpr uint32_t kIdescS = make_idesc(kFormatBF16, 128, 128, false, false);
    static constexpr uint32_t kIdescDQ = make_idesc(kFormatBF16, 128, D, false, true);
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(256 + 2 * D <= 512, "tensor memory budget");
};

template <int KS, int VS>
struct DqBars {
    static constexpr int kQ = 0;
    static constexpr int kKFull = 1;                  // + stage
    static constexpr int kKEmpty = 1 + KS;            // + stage
    static constexpr int kVFull = 1 + 2 * KS;         // + stage
    static constexpr int kVEmpty = 1 + 2 * KS + VS;   // + stage
    static constexpr int kSFull = 1 + 2 * KS + 2 * VS;  // + tile
    static constexpr int kSRead = kSFull + 2;         // + tile
    static constexpr int kDPFull = kSFull + 4;        // + tile
    static constexpr int kDSFull = kSFull + 6;        // + tile
    static constexpr int kDone = kSFull + 8;
};

enum : int {
    kSiteQLoadK = 51, kSiteQLoadV = 52, kSiteQMmaQ = 53, kSiteQMmaK = 54, kSiteQMmaV = 55, kSiteQMmaS = 56,
    kSiteQMmaDS = 57, kSiteQSoftS = 58, kSiteQSoftDP = 59, kSiteQEpi = 60, kSiteQDrain = 61,
    kSiteQMisaligned = 62
};

template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const float *__restrict__ lse2, const float *__restrict__ delta, __nv_bfloat16 *__restrict__ dq,
              int N, int Npad, int num_pairs, int group, float scale, float scale_log2, int causal,
              unsigned int *status) {
    using C = DqCfg<D>;
    using B = DqBars<C::kKStages, C::kVStages>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    if ((base & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned window
        if (threadIdx.x == 0 && atomicOr(&status[0], kStatusTimeout) == 0u) status[1] = kSiteQMisaligned;
        return;
    }
    uint8_t *smem = smem_raw;
    const uint32_t sQ = base + C::kQOff, sDO = base + C::kDOOff;
    const uint32_t sK = base + C::kKOff, sV = base + C::kVOff, sBar = base + C::kBarOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx wc{abort_flag, status};
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int bh, rank;                                     // query head, pair rank
    heavy_first_order(blockIdx.x, num_pairs, bh, rank);
    const int bh_kv = bh / group;                     // its key/value head
    const int pair = causal ? (num_pairs - 1 - rank) : rank;   // longest walks first
    const int nkv = (N + kTileRows - 1) / kTileRows;
    int ntile[2];                                     // key blocks each query tile visits
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = 2 * pair + t;
        ntile[t] = qt * kTileRows >= N ? 0 : (causal ? min(qt + 1, nkv) : nkv);
    }
    const int nmax = max(ntile[0], ntile[1]);

    if (threadIdx.x == 0) {
        mbar_init(bar(B::kQ), 1);
        for (int s = 0; s < C::kKStages; ++s) {
            mbar_init(bar(B::kKFull + s), 1);
            mbar_init(bar(B::kKEmpty + s), 1);
        }
        for (int s = 0; s < C::kVStages; ++s) {
            mbar_init(bar(B::kVFull + s), 1);
            mbar_init(bar(B::kVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B::kSFull + t), 1);
            mbar_init(bar(B::kSRead + t), 128);
            mbar_init(bar(B::kDPFull + t), 1);
            mbar_init(bar(B::kDSFull + t), 128);
        }
        mbar_init(bar(B::kDone), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kLoadWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_do);
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t) qbytes += ntile[t] > 0 ? 2 * C::kTileBytes : 0;
            mbar_arrive_expect_tx(bar(B::kQ), qbytes);
            for (int t = 0; t < 2; ++t) {
                if (ntile[t] == 0) continue;
                for (int b = 0; b < C::kBoxes; ++b) {
                    tma_load_3d(sQ + t * C::kTileBytes + b * C::kBoxTileBytes, &tm_q, bar(B::kQ), b * 64,
                                (2 * pair + t) * kTileRows, bh);
                    tma_load_3d(sDO + t * C::kTileBytes + b * C::kBoxTileBytes, &tm_do, bar(B::kQ), b * 64,
                                (2 * pair + t) * kTileRows, bh);
                }
            }
            int k_loads = 0, v_loads = 0;
            for (int j = 0; j < nmax; ++j) {
                const int ks = j % C::kKStages, ku = j / C::kKStages;
                if (ku > 0 && !mbar_wait(bar(B::kKEmpty + ks), (ku - 1) & 1, wc, kSiteQLoadK)) break;
                mbar_arrive_expect_tx(bar(B::kKFull + ks), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sK + ks * C::kTileBytes + b * C::kBoxTileBytes, &tm_k, bar(B::kKFull + ks), b * 64,
                                j * kTileRows, bh_kv);
                ++k_loads;
                const int vs = j % C::kVStages, vu = j / C::kVStages;
                if (vu > 0 && !mbar_wait(bar(B::kVEmpty + vs), (vu - 1) & 1, wc, kSiteQLoadV)) break;
                mbar_arrive_expect_tx(bar(B::kVFull + vs), C::kTileBytes);
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sV + vs * C::kTileBytes + b * C::kBoxTileBytes, &tm_v, bar(B::kVFull + vs), b * 64,
                                j * kTileRows, bh_kv);
                ++v_loads;
            }
            // Every copy issued above must land before this CTA may exit.
            mbar_wait_drain(bar(B::kQ), 0, wc, kSiteQDrain);
            for (int s = 0; s < C::kKStages && s < k_loads; ++s) {
                const int last = s + ((k_loads - 1 - s) / C::kKStages) * C::kKStages;
                mbar_wait_drain(bar(B::kKFull + s), (last / C::kKStages) & 1, wc, kSiteQDrain);
            }
            for (int s = 0; s < C::kVStages && s < v_loads; ++s) {
                const int last = s + ((v_loads - 1 - s) / C::kVStages) * C::kVStages;
                mbar_wait_drain(bar(B::kVFull + s), (last / C::kVStages) & 1, wc, kSiteQDrain);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (every wait is warp-uniform) and lane 0 issues.
        {
            auto mbar_wait_w = [&](uint32_t b, uint32_t parity, int site) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
            };
            const uint32_t tSD[2] = {tmem, tmem + 128u};
            const uint32_t tDQ[2] = {tmem + C::kDQCol, tmem + C::kDQCol + D};
            auto active = [&](int t, int j) { return j < ntile[t]; };
            // S_t = A_t B^T over the head dim; A_t = Q_t or dO_t, B = K_j or V_j (both K-major)
            auto mma_rows = [&](uint32_t d_tmem, uint32_t a_tile, uint32_t b_tile) {
                const uint64_t a0 = sdesc_sw128(a_tile, 16, 1024), b0 = sdesc_sw128(b_tile, 16, 1024);
                uint64_t a[C::kKSteps], b[C::kKSteps];
#pragma unroll
                for (int kk = 0; kk < C::kKSteps; ++kk) {
                    const uint32_t off = (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32;
                    a[kk] = sdesc_step(a0, off);
                    b[kk] = sdesc_step(b0, off);
                }
                if constexpr (C::kKSteps == 8) umma_f16_ss_x8(d_tmem, a, b, C::kIdescS, 0u);
                else umma_f16_ss_x4(d_tmem, a, b, C::kIdescS, 0u);
            };
            auto wait_k = [&](int j) -> int {
                const int s = j % C::kKStages;
                if (!mbar_wait_w(bar(B::kKFull + s), (j / C::kKStages) & 1, kSiteQMmaK)) return -1;
                tc_fence_after();
                return s;
            };
            auto wait_v = [&](int j) -> int {
                const int s = j % C::kVStages;
                if (!mbar_wait_w(bar(B::kVFull + s), (j / C::kVStages) & 1, kSiteQMmaV)) return -1;
                tc_fence_after();
                return s;
            };
            // dP_t(j) for both tiles once their S has been read; then V_j's stage is free
            auto issue_dp = [&](int j) -> bool {
                const int vs = wait_v(j);
                if (vs < 0) return false;
                for (int t = 0; t < 2; ++t) {
                    if (!active(t, j)) continue;
                    if (!mbar_wait_w(bar(B::kSRead + t), j & 1, kSiteQMmaS)) return false;
                    tc_fence_after();
                    mma_rows(tSD[t], sDO + t * C::kTileBytes, sV + vs * C::kTileBytes);
                    umma_commit(bar(B::kDPFull + t));
                }
                umma_commit(bar(B::kVEmpty + vs));
                return true;
            };
            bool ok = nmax > 0 && mbar_wait_w(bar(B::kQ), 0, kSiteQMmaQ);
            if (ok) {
                tc_fence_after();
                int ks = wait_k(0);
                ok = ks >= 0;
                if (ok) {
                    for (int t = 0; t < 2; ++t) {
                        if (!active(t, 0)) continue;
                        mma_rows(tSD[t], sQ + t * C::kTileBytes, sK + ks * C::kTileBytes);
                        umma_commit(bar(B::kSFull + t));
                    }
                    ok = issue_dp(0);
                }
            }
            for (int j = 0; ok && j < nmax; ++j) {
                const int ks = j % C::kKStages;
                int ks_next = -1;
                for (int t = 0; ok && t < 2; ++t) {
                    if (!active(t, j)) continue;
                    // dQ_t += dS_t K_j, then S_t for the next key block into the same columns
                    if (!mbar_wait_w(bar(B::kDSFull + t), j & 1, kSiteQMmaDS)) { ok = false; break; }
                    tc_fence_after();
                    {
                        const uint64_t b0 = sdesc_sw128(sK + ks * C::kTileBytes, C::kBoxTileBytes, 1024);
                        uint64_t b[C::kRowSteps];
#pragma unroll
                        for (int kk = 0; kk < C::kRowSteps; ++kk) b[kk] = sdesc_step(b0, kk * 16 * kBoxBytes);
                        umma_f16_ts_x8(tDQ[t], tSD[t], b, C::kIdescDQ, j > 0 ? 1u : 0u);
                    }
                    if (active(t, j + 1)) {
                        if (ks_next < 0) ks_next = wait_k(j + 1);
                        if (ks_next < 0) { ok = false; break; }
                        mma_rows(tSD[t], sQ + t * C::kTileBytes, sK + ks_next * C::kTileBytes);
                        umma_commit(bar(B::kSFull + t));
                    }
                }
                if (!ok) break;
                umma_commit(bar(B::kKEmpty + ks));
                if (j + 1 < nmax) ok = issue_dp(j + 1);
            }
            // Both tiles' dQ are complete once everything issued so far has retired.
            umma_commit(bar(B::kDone));
            mbar_wait_drain(bar(B::kDone), 0, wc, kSiteQDrain);
        }
    } else {
        // ------------------------------------------------------------ query rows (warps 0-7)
        const int t = warp >> 2;                            // query tile of this warpgroup
        const int r = (warp & 3) * 32 + lane;               // row within the tile
        const int qt = 2 * pair + t;
        const int q = qt * kTileRows + r;                   // query index (< Npad)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tSDr = tmem + lane_off + 128u * t;
        const uint32_t tDQr = tmem + lane_off + C::kDQCol + D * t;
        const int n_j = ntile[t];
        float nL = 0.f, Dr = 0.f;
        if (n_j > 0) {
            nL = lse2[static_cast<int64_t>(bh) * Npad + q];   // -L * log2 e (-inf on padding rows)
            Dr = delta[static_cast<int64_t>(bh) * Npad + q];
        }
        const float2 nL2 = make_float2(nL, nL), D2 = make_float2(Dr, Dr);
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        bool ok = true;
        for (int j = 0; j < n_j; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull + t), j & 1, wc, kSiteQSoftS));
            if (!ok) break;
            tc_fence_after();
            // P = 2^(S * scale*log2e - L2), kept as packed bf16 in registers
            uint32_t pk[64];
            {
                uint32_t sr[128];
                tmem_ld_x128(tSDr, sr);
                // S is in registers: dP may overwrite its columns while P is computed
                tc_fence_before();
                mbar_arrive(bar(B::kSRead + t));
                // keys past N, and (causal) keys after this query, get probability 0
                const int kmax = min(N - 1 - j * kTileRows, causal ? q - j * kTileRows : kTileRows - 1);
                if (kmax >= kTileRows - 1) {
#pragma unroll
                    for (int u = 0; u < 64; ++u) {
                        const float2 x = fma2(make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])),
                                              sl2, nL2);
                        pk[u] = pack_bf16(ex2(x.x), ex2(x.y));
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 64; ++u) {
                        const float2 x = fma2(make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])),
                                              sl2, nL2);
                        pk[u] = pack_bf16(2 * u <= kmax ? ex2(x.x) : 0.f, 2 * u + 1 <= kmax ? ex2(x.y) : 0.f);
                    }
                }
            }
            // dS = P o (dP - D), packed bf16 over the first 64 columns
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kDPFull + t), j & 1, wc, kSiteQSoftDP));
            if (!ok) break;
            tc_fence_after();
            uint32_t rbuf[2][32];
            tmem_ld_x32_nowait(tSDr, rbuf[0]);
            tmem_wait_ld_fence(rbuf[0]);
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t (&rr)[32] = rbuf[ch & 1];
                if (ch < 3) tmem_ld_x32_nowait(tSDr + 32u * (ch + 1), rbuf[(ch + 1) & 1]);
                uint32_t d2[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const uint32_t pp = pk[16 * ch + u];
                    const float2 p = make_float2(__uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u));
                    const float2 ds = mul2(p, sub2(make_float2(__uint_as_float(rr[2 * u]), __uint_as_float(rr[2 * u + 1])),
                                                   D2));
                    d2[u] = pack_bf16(ds.x, ds.y);
                }
                // chunk ch writes columns 16ch .. 16ch+15, all of which have been read
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                    "%12, %13, %14, %15, %16};\n\t" ::"r"(tSDr + 16u * ch),
                    "r"(d2[0]), "r"(d2[1]), "r"(d2[2]), "r"(d2[3]), "r"(d2[4]), "r"(d2[5]), "r"(d2[6]), "r"(d2[7]),
                    "r"(d2[8]), "r"(d2[9]), "r"(d2[10]), "r"(d2[11]), "r"(d2[12]), "r"(d2[13]), "r"(d2[14]),
                    "r"(d2[15])
                    : "memory");
                if (ch < 3) tmem_wait_ld_fence(rbuf[(ch + 1) & 1]);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            mbar_arrive(bar(B::kDSFull + t));
        }
        // ------------------------------------------------------------ epilogue: dQ row
        if (ok && n_j > 0) ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kDone), 0, wc, kSiteQEpi));
        if (ok && n_j > 0) {
            tc_fence_after();
            __nv_bfloat16 *row = dq + (static_cast<int64_t>(bh) * N + (q < N ? q : 0)) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t v[32];
                tmem_ld_x32(tDQr + 32u * ch, v);
                if (q < N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(row + 32 * ch);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        dst[u] = make_uint4(
                            pack_bf16(__uint_as_float(v[8 * u]) * scale, __uint_as_float(v[8 * u + 1]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 2]) * scale, __uint_as_float(v[8 * u + 3]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 4]) * scale, __uint_as_float(v[8 * u + 5]) * scale),
                            pack_bf16(__uint_as_float(v[8 * u + 6]) * scale, __uint_as_float(v[8 * u + 7]) * scale));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

int grid_for(long long work_items, int per_block) {
    long long g = (work_items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    if (g > 152LL * 16) g = 152LL * 16;
    return static_cast<int>(g);
}

template <int D>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t stream) {
    const long long rows = static_cast<long long>(a.BH) * a.Npad;
    bwd_pre_kernel<D><<<grid_for(rows, 64), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(a.o), static_cast<const __nv_bfloat16 *>(a.dout), a.lse, a.delta,
        a.lse2, a.dq_acc, a.N, a.Npad, a.BH);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    auto kern = a.deterministic ? bwd_main_kernel<D, false> : bwd_main_kernel<D, true>;
    const int smem_bytes = a.deterministic ? BwdCfg<D, false>::kSmemBytes : BwdCfg<D, true>::kSmemBytes;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    const int nkv = a.Npad / kTileRows;
    const long long blocks = static_cast<long long>(a.BH / a.group) * nkv;
    if (blocks <= 0 || blocks > INT_MAX) return cudaErrorInvalidValue;
    const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    // programmatic dependent launch: the main kernel's set-up overlaps the end of the
    // pre-processing grid (it waits for that grid's results before using them)
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kMainThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dq, static_cast<const float *>(a.lse2),
                           static_cast<const float *>(a.delta), static_cast<__nv_bfloat16 *>(a.dk),
                           static_cast<__nv_bfloat16 *>(a.dv), a.N, a.Npad, nkv, a.group, a.scale, scale_log2,
                           a.causal, a.status);
    if (e != cudaSuccess) return e;

    if (a.deterministic) {
        using CQ = DqCfg<D>;
        auto qkern = bwd_dq_kernel<D>;
        e = cudaFuncSetAttribute(qkern, cudaFuncAttributeMaxDynamicSharedMemorySize, CQ::kSmemBytes);
        if (e != cudaSuccess) return e;
        const int num_pairs = (nkv + 1) / 2;
        const long long qblocks = static_cast<long long>(a.BH) * num_pairs;
        if (qblocks > INT_MAX) return cudaErrorInvalidValue;
        qkern<<<static_cast<unsigned>(qblocks), kDqThreads, CQ::kSmemBytes, stream>>>(
            a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.lse2, a.delta, static_cast<__nv_bfloat16 *>(a.dq), a.N, a.Npad,
            num_pairs, a.group, a.scale, scale_log2, a.causal, a.status);
        return cudaGetLastError();
    }

    const long long n8 = static_cast<long long>(a.BH) * a.N * D / 8;
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3(static_cast<unsigned>(grid_for(n8, 256)));
    pcfg.blockDim = dim3(256);
    pcfg.stream = stream;
    pcfg.attrs = pdl;
    pcfg.numAttrs = 1;
    return cudaLaunchKernelEx(&pcfg, bwd_post_kernel, static_cast<const float *>(a.dq_acc),
                              static_cast<__nv_bfloat16 *>(a.dq), n8, a.scale);
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdArgs &a, cudaStream_t stream) {
    if (a.d == 64) return launch_bwd_t<64>(a, stream);
    if (a.d == 128) return launch_bwd_t<128>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
