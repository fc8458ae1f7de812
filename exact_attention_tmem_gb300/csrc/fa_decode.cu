// fa_decode.cu — decoding: one query row per head against a long key/value sequence.
//
// What it computes ("FlashAttention" deep dive, section "Implementation notes",
// decoding): with a single query row there is too little work per head to fill the
// GPU, so the keys are split into chunks processed in parallel; each chunk reduces to
// a partial (m, l, acc) triple (running max, denominator, unnormalised output) and the
// triples are merged with the same rescaling rule the tiled forward pass uses.  The
// query is the newest position, so it sees every key; no mask applies.
//
// The work is a matrix-vector product per head (4 Nk d FLOP against 4 Nk d bytes of
// bf16 K and V): bound by HBM bandwidth, not by the tensor cores, so it runs on the
// CUDA cores and is organised around the memory stream:
//  1. decode_split_kernel: one CTA per (batch, key/value head, chunk).  All G query
//     heads that share the key/value head (grouped-query attention) are handled by the
//     same CTA, so K and V are read from HBM once per key/value head.  K and V rows
//     stream through a 3-stage shared-memory ring filled by bulk copies (one thread
//     issues; 64 keys per stage).  Each group of D/8 lanes takes one key at a time
//     (16 bytes of the row per lane, so a warp reads whole 256-byte rows), reduces the
//     dot products with shuffles, and keeps its own (m, l, acc) per query head; the
//     rescale is applied once per stage (a block of keys), as in the forward kernel.
//     With several query heads per key/value head the work per byte grows with the
//     group, so the CTA has 8 warps (two CTAs per SM up to 4 heads per group) and the
//     products and the output update run on packed pairs (fma.rn.f32x2): the stream
//     of dependent shuffles, exponentials and FMAs needs the warps to hide latency.
//     At the end the lane groups' triples are merged through shared memory and the
//     CTA writes one partial triple per query head to the workspace.
//  2. decode_combine_kernel: one CTA per (batch, query head) merges the chunks'
//     triples: O = acc / l in bf16 and L = (m + log2 l) ln 2.
// Scores are kept in base 2 (log2 e folded into the scale), like the forward kernel.
#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecStageKeys = 64;
constexpr int kDecStages = 3;
constexpr float kDecLn2 = 0.6931471805599453f;

enum : int { kSiteDecFull = 71, kSiteDecDrain = 72 };

template <int D, int G>
struct DecCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kTileBytes = kDecStageKeys * kRowBytes;      // K or V of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kLanesPerKey = D / 8;                        // 16 bytes per lane
    static constexpr int kKeysPerStep = 32 / kLanesPerKey;            // keys per warp per step
    static constexpr int kGroups = kDecWarps * kKeysPerStep;          // lane groups per CTA
    static constexpr int kSteps = kDecStageKeys / kGroups;            // keys per lane group per stage
    static constexpr int kRingBytes = kDecStages * kStageBytes;
    // the lane groups' (m, l, acc) triples, merged through shared memory after the loop
    static constexpr int kMergeBytes = (2 * kGroups * G + kGroups * G * D) * 4;
    static constexpr int kBarOff = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kMiscOff = kBarOff + 8 * kDecStages;
    static constexpr int kSmemBytes = kMiscOff + 16;
    // two CTAs per SM (16 warps) while the registers allow it
    static constexpr int kMinBlocks = G <= 4 ? 2 : 1;
    static_assert(kDecStageKeys % kGroups == 0, "whole steps per stage");
};

__device__ __forceinline__ float2 bf2f(uint32_t x) {
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

// Partials layout in the workspace, per (query head bh, chunk c): m[bh][c], l[bh][c],
// acc[bh][c][D] (fp32; m in base-2 units).
template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, DecCfg<D, G>::kMinBlocks)
decode_split_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                    const __nv_bfloat16 *__restrict__ v, float *__restrict__ part_m, float *__restrict__ part_l,
                    float *__restrict__ part_acc, int Nk, int chunk_keys, int num_chunks, int max_chunks,
                    int group, float scale_log2, unsigned int *status) {
    using C = DecCfg<D, G>;
    grid_launch_dependents();   // the merge kernel may launch now; it waits for this grid
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t base = smem_u32(smem);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff);
    const WaitCtx wc{abort_flag, status};
    auto full_bar = [&](int s) -> uint32_t { return base + C::kBarOff + 8u * static_cast<uint32_t>(s); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int grp = warp * C::kKeysPerStep + lane / C::kLanesPerKey;   // lane group in the CTA
    const int sl = lane % C::kLanesPerKey;                            // 16-byte column chunk
    // The `group` query heads of a key/value head are split into group / G sub-groups
    // of G heads; the CTAs of one chunk's sub-groups are adjacent in the launch order,
    // so all but the first read the chunk's K and V from L2.
    const int nsub = group / G;
    const int sub = blockIdx.x % nsub;
    const int c = (blockIdx.x / nsub) % num_chunks;
    const int bkv = blockIdx.x / (nsub * num_chunks);                 // batch * Hkv + kv head
    const int64_t qh0 = static_cast<int64_t>(bkv) * group + sub * G;  // first query head of the CTA
    const int key0 = c * chunk_keys;
    const int key1 = min(Nk, key0 + chunk_keys);
    const int n_tiles = (key1 - key0 + kDecStageKeys - 1) / kDecStageKeys;
    const __nv_bfloat16 *kh = k + static_cast<int64_t>(bkv) * Nk * D;
    const __nv_bfloat16 *vh = v + static_cast<int64_t>(bkv) * Nk * D;

    if (tid == 0) {
        for (int s = 0; s < kDecStages; ++s) mbar_init(full_bar(s), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int t) {
        const int s = t % kDecStages;
        const int k_first = key0 + t * kDecStageKeys;
        const uint32_t bytes = static_cast<uint32_t>(min(kDecStageKeys, key1 - k_first)) * C::kRowBytes;
        mbar_arrive_expect_tx(full_bar(s), 2 * bytes);
        bulk_load(base + s * C::kStageBytes, kh + static_cast<int64_t>(k_first) * D, bytes, full_bar(s));
        bulk_load(base + s * C::kStageBytes + C::kTileBytes, vh + static_cast<int64_t>(k_first) * D, bytes,
                  full_bar(s));
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < kDecStages && issued < n_tiles; ++issued) issue(issued);

    // this lane's 8 query elements of each head (as 4 pairs), pre-scaled into base-2
    // score units; products and the output update run on packed pairs (fma.rn.f32x2)
    float2 qf[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(q + (qh0 + g) * D + sl * 8);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = bf2f(w[e]);
            qf[g][e] = make_float2(f.x * scale_log2, f.y * scale_log2);
        }
    }
    float m[G], l[G];
    float2 acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = make_float2(0.f, 0.f);
    }

    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kDecStages;
        ok = __syncthreads_and(mbar_wait(full_bar(s), (t / kDecStages) & 1, wc, kSiteDecFull)) != 0;
        if (!ok) break;
        // every thread is past tile t - 1: its stage can be refilled
        if (tid == 0 && t >= 1 && issued < n_tiles) issue(issued++);
        const uint8_t *sk = smem + s * C::kStageBytes;
        const uint8_t *sv = sk + C::kTileBytes;
        const int n_keys = min(kDecStageKeys, key1 - (key0 + t * kDecStageKeys));
        // scores of this lane group's keys in the stage (key = st * kGroups + grp)
        float sc[C::kSteps][G];
#pragma unroll
        for (int st = 0; st < C::kSteps; ++st) {
            const int key = st * C::kGroups + grp;
            const uint4 raw = *reinterpret_cast<const uint4 *>(sk + key * C::kRowBytes + sl * 16);
            const float2 kf[4] = {bf2f(raw.x), bf2f(raw.y), bf2f(raw.z), bf2f(raw.w)};
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float2 a = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 4; ++e) a = fma2(qf[g][e], kf[e], a);
                sc[st][g] = a.x + a.y;
            }
        }
#pragma unroll
        for (int off = C::kLanesPerKey / 2; off > 0; off >>= 1)
#pragma unroll
            for (int st = 0; st < C::kSteps; ++st)
#pragma unroll
                for (int g = 0; g < G; ++g) sc[st][g] += __shfl_xor_sync(0xffffffffu, sc[st][g], off);
        // one rescale per stage, then the stage's keys
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = m[g];
#pragma unroll
            for (int st = 0; st < C::kSteps; ++st)
                if (st * C::kGroups + grp < n_keys) mx = fmaxf(mx, sc[st][g]);
            if (mx > m[g]) {   // m = -inf on the first keys: the factor is 0 and acc, l are 0
                const float a = ex2(m[g] - mx);
                const float2 a2 = make_float2(a, a);
                l[g] *= a;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[g][e] = mul2(acc[g][e], a2);
                m[g] = mx;
            }
        }
#pragma unroll
        for (int st = 0; st < C::kSteps; ++st) {
            const int key = st * C::kGroups + grp;
            if (key >= n_keys) continue;   // keys past the chunk: no contribution
            const uint4 raw = *reinterpret_cast<const uint4 *>(sv + key * C::kRowBytes + sl * 16);
            const float2 vf[4] = {bf2f(raw.x), bf2f(raw.y), bf2f(raw.z), bf2f(raw.w)};
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float p = ex2(sc[st][g] - m[g]);
                const float2 p2 = make_float2(p, p);
                l[g] += p;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[g][e] = fma2(p2, vf[e], acc[g][e]);
            }
        }
    }
    if (!ok) {
        // every copy issued must land before the CTA exits
        if (tid == 0)
            for (int s = 0; s < kDecStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / kDecStages) * kDecStages;
                mbar_wait_drain(full_bar(s), (last / kDecStages) & 1, wc, kSiteDecDrain);
            }
        return;
    }

    // ---- merge the lane groups' triples through shared memory (the ring is idle now)
    __syncthreads();
    float *mg = reinterpret_cast<float *>(smem);                 // [kGroups][G]
    float *lg = mg + C::kGroups * G;                             // [kGroups][G]
    float *ag = lg + C::kGroups * G;                             // [kGroups][G][D]
    if (sl == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            mg[grp * G + g] = m[g];
            lg[grp * G + g] = l[g];
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            *reinterpret_cast<float2 *>(&ag[(grp * G + g) * D + sl * 8 + 2 * e]) = acc[g][e];
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kDecThreads) {
        const int g = idx / D, e = idx % D;
        float M = -INFINITY;
        for (int r = 0; r < C::kGroups; ++r) M = fmaxf(M, mg[r * G + g]);
        float L = 0.f, A = 0.f;
        for (int r = 0; r < C::kGroups; ++r) {
            const float mr = mg[r * G + g];
            const float wgt = mr == -INFINITY ? 0.f : ex2(mr - M);   // groups that saw no key weigh 0
            L = fmaf(lg[r * G + g], wgt, L);
            A = fmaf(ag[(r * G + g) * D + e], wgt, A);
        }
        const int64_t slot = (qh0 + g) * max_chunks + c;
        part_acc[slot * D + e] = A;
        if (e == 0) {
            part_m[slot] = M;
            part_l[slot] = L;
        }
    }
}

// ------------------------------------------------------------------------------------
// Tensor-core variant for groups of query heads (grouped-query attention).  With G query
// heads per key/value head every K and V element feeds G dot products, which on the CUDA
// cores costs more issue slots than the memory stream allows once G reaches a few heads.
// Here the G query rows (padded to 16) are the M dimension of mma.sync m16n8k16 (bf16
// in, fp32 accumulate):
//   S (16 x 16 keys) = Q (16 x d) K^T      B fragments of K read with ldmatrix
//   O (16 x d)      += P (16 x 16 keys) V  P = the S accumulator fragment repacked as the
//                                          A fragment; V read with ldmatrix.trans
// One CTA of 4 warps per (batch, key/value head, chunk); a stage holds 64 keys (K and V,
// loaded by TMA with 128-byte swizzle so that the ldmatrix rows hit distinct banks) and
// each warp takes 16 of them, keeping its own (m, l, O) per query row; the warps' triples
// are merged through shared memory into one partial triple per query head and chunk,
// the layout decode_combine_kernel merges.
constexpr int kMmaDecThreads = 128;
constexpr int kMmaDecStages = 3;

template <int D>
struct DecMmaCfg {
    static constexpr int kBoxes = D * 2 / 128;                   // 128-byte boxes per row
    static constexpr int kBoxBytes = kDecodeBoxRows * 128;       // 64 keys x 128 bytes
    static constexpr int kTileBytes = kBoxes * kBoxBytes;        // K or V of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRingBytes = kMmaDecStages * kStageBytes;
    static constexpr int kMergeBytes = 4 * (2 * 16 + 16 * D) * 4;    // per warp: m, l, O (16 rows)
    static constexpr int kBarOff = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
    static constexpr int kMiscOff = kBarOff + 8 * kMmaDecStages;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;      // + room to align the base to 1 KB
    static_assert(kDecodeBoxRows == 4 * 16, "four warps of 16 keys per stage");
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

template <int D>
__global__ void __launch_bounds__(kMmaDecThreads, 2)
decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __nv_bfloat16 *__restrict__ q, float *__restrict__ part_m, float *__restrict__ part_l,
                  float *__restrict__ part_acc, int Nk, int chunk_keys, int num_chunks, int max_chunks, int group,
                  float scale_log2, unsigned int *status) {
    using C = DecMmaCfg<D>;
    grid_launch_dependents();   // the merge kernel may launch now; it waits for this grid
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;     // 128-byte swizzle repeats every 1 KB
    uint8_t *smem = smem_raw + (base - raw);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff);
    const WaitCtx wc{abort_flag, status};
    auto full_bar = [&](int s) -> uint32_t { return base + C::kBarOff + 8u * static_cast<uint32_t>(s); };

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int bkv = blockIdx.x / num_chunks;          // batch * Hkv + key/value head
    const int c = blockIdx.x % num_chunks;
    const int key0 = c * chunk_keys;
    const int key1 = min(Nk, key0 + chunk_keys);
    const int n_tiles = (key1 - key0 + kDecodeBoxRows - 1) / kDecodeBoxRows;

    if (tid == 0) {
        for (int s = 0; s < kMmaDecStages; ++s) mbar_init(full_bar(s), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int t) {
        const int s = t % kMmaDecStages;
        const uint32_t dst = base + s * C::kStageBytes;
        mbar_arrive_expect_tx(full_bar(s), C::kStageBytes);   // rows past Nk arrive zero-filled
        for (int b = 0; b < C::kBoxes; ++b) {
            tma_load_3d(dst + b * C::kBoxBytes, &tm_k, full_bar(s), b * 64, key0 + t * kDecodeBoxRows, bkv);
            tma_load_3d(dst + C::kTileBytes + b * C::kBoxBytes, &tm_v, full_bar(s), b * 64,
                        key0 + t * kDecodeBoxRows, bkv);
        }
    };
    int issued = 0;
    if (tid == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        for (; issued < kMmaDecStages && issued < n_tiles; ++issued) issue(issued);
    }

    // Q fragments: rows g0 = lane / 4 and g1 = g0 + 8 of the group (zero past it),
    // columns 16k + 2(lane % 4) (+1, +8, +9)
    const int g0 = lane >> 2, g1 = g0 + 8;
    const int cc = 2 * (lane & 3);
    auto q2 = [&](int g, int col) -> uint32_t {
        if (g >= group) return 0u;
        return *reinterpret_cast<const uint32_t *>(q + (static_cast<int64_t>(bkv) * group + g) * D + col);
    };
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
        qa[k][0] = q2(g0, 16 * k + cc);
        qa[k][1] = q2(g1, 16 * k + cc);
        qa[k][2] = q2(g0, 16 * k + cc + 8);
        qa[k][3] = q2(g1, 16 * k + cc + 8);
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;   // running max of rows g0, g1 (base-2 units)
    float l0 = 0.f, l1 = 0.f;               // this thread's part of the running sums
    // a 16-byte chunk `ch` (8 elements of d) of stage row `key` in a swizzled tile
    auto chunk_addr = [&](uint32_t tile, int key, int ch) -> uint32_t {
        return tile + (ch >> 3) * C::kBoxBytes + key * 128 + (((ch & 7) ^ (key & 7)) << 4);
    };
    const int kw = 16 * warp;               // this warp's keys in a stage

    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kMmaDecStages;
        ok = __syncthreads_and(mbar_wait(full_bar(s), (t / kMmaDecStages) & 1, wc, kSiteDecFull)) != 0;
        if (!ok) break;
        // every thread is past tile t - 1: its stage can be refilled
        if (tid == 0 && t >= 1 && issued < n_tiles) issue(issued++);
        const uint32_t sk = base + s * C::kStageBytes, sv = sk + C::kTileBytes;
        const int n_keys = min(kDecodeBoxRows, key1 - (key0 + t * kDecodeBoxRows));
        // S = Q K^T over this warp's 16 keys (two 8-key column tiles)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const int key = kw + 8 * n + (lane & 7);
#pragma unroll
            for (int kp = 0; kp < D / 32; ++kp) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(chunk_addr(sk, key, 4 * kp + (lane >> 3)), r0, r1, r2, r3);
                mma_bf16_16816(sc[n], qa[2 * kp], r0, r1);
                mma_bf16_16816(sc[n], qa[2 * kp + 1], r2, r3);
            }
        }
        // scaled scores, keys past the chunk masked; online softmax per row
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool valid = kw + 8 * n + cc + e < n_keys;
                sc[n][e] = valid ? sc[n][e] * scale_log2 : -INFINITY;
                sc[n][2 + e] = valid ? sc[n][2 + e] * scale_log2 : -INFINITY;
                mx0 = fmaxf(mx0, sc[n][e]);
                mx1 = fmaxf(mx1, sc[n][2 + e]);
            }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        // a row that has seen no key yet keeps m = -inf, l = 0, O = 0
        const float a0 = mn0 == -INFINITY ? 1.f : ex2(m0 - mn0);
        const float a1 = mn1 == -INFINITY ? 1.f : ex2(m1 - mn1);
        const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
        m0 = mn0;
        m1 = mn1;
        float p[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                p[n][e] = ex2(sc[n][e] - base0);
                p[n][2 + e] = ex2(sc[n][2 + e] - base1);
            }
        l0 = l0 * a0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
        l1 = l1 * a1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
        if (a0 != 1.f || a1 != 1.f) {
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] *= a0;
                o[n][1] *= a0;
                o[n][2] *= a1;
                o[n][3] *= a1;
            }
        }
        // P as the A fragment (rows g0, g1; keys cc, cc + 1, cc + 8, cc + 9 of the 16)
        const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]),
                                pack_bf16(p[1][0], p[1][1]), pack_bf16(p[1][2], p[1][3])};
        // O += P V: V read transposed, two 8-column tiles of d per ldmatrix
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
            const int key = kw + 8 * ((lane >> 3) & 1) + (lane & 7);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(chunk_addr(sv, key, 2 * np + (lane >> 4)), r0, r1, r2, r3);
            mma_bf16_16816(o[2 * np], pa, r0, r1);
            mma_bf16_16816(o[2 * np + 1], pa, r2, r3);
        }
    }
    if (!ok) {
        // every copy issued must land before the CTA exits
        if (tid == 0)
            for (int s = 0; s < kMmaDecStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / kMmaDecStages) * kMmaDecStages;
                mbar_wait_drain(full_bar(s), (last / kMmaDecStages) & 1, wc, kSiteDecDrain);
            }
        return;
    }

    // ---- merge the four warps' triples through shared memory (the ring is idle now)
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    __syncthreads();
    float *mw = reinterpret_cast<float *>(smem);        // [4][16]
    float *lw = mw + 4 * 16;                            // [4][16]
    float *ow = lw + 4 * 16;                            // [4][16][D]
    if ((lane & 3) == 0) {
        mw[warp * 16 + g0] = m0;
        mw[warp * 16 + g1] = m1;
        lw[warp * 16 + g0] = l0;
        lw[warp * 16 + g1] = l1;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        *reinterpret_cast<float2 *>(&ow[(warp * 16 + g0) * D + 8 * n + cc]) = make_float2(o[n][0], o[n][1]);
        *reinterpret_cast<float2 *>(&ow[(warp * 16 + g1) * D + 8 * n + cc]) = make_float2(o[n][2], o[n][3]);
    }
    __syncthreads();
    for (int idx = tid; idx < group * D; idx += kMmaDecThreads) {
        const int g = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * 16 + g]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float mr = mw[w * 16 + g];
            const float wgt = mr == -INFINITY ? 0.f : ex2(mr - M);   // warps that saw no key weigh 0
            L = fmaf(lw[w * 16 + g], wgt, L);
            A = fmaf(ow[(w * 16 + g) * D + e], wgt, A);
        }
        const int64_t slot = (static_cast<int64_t>(bkv) * group + g) * max_chunks + c;
        part_acc[slot * D + e] = A;
        if (e == 0) {
            part_m[slot] = M;
            part_l[slot] = L;
        }
    }
}

// One CTA of D threads per (batch, query head); thread e owns output column e.  The
// merge is latency-bound (a few KB per head), so every load it needs is issued before
// any arithmetic: the chunks' m and l (one chunk per thread) and thread e's
// accumulator column of the first kCombinePre chunks.  The sums run in chunk order,
// as a plain sequential merge would.
constexpr int kCombinePre = 32;
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float *__restrict__ part_m, const float *__restrict__ part_l,
                      const float *__restrict__ part_acc, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                      int num_chunks, int max_chunks) {
    constexpr int kPer = kDecodeMaxChunks / D;   // chunks per thread for m and l
    constexpr int kWarps = D / 32;
    __shared__ float m_sh[kDecodeMaxChunks], l_sh[kDecodeMaxChunks];
    __shared__ float red[kWarps];
    grid_dependency_wait();     // launched as the split kernel's dependent: its partials are in
    const int bh = blockIdx.x;
    const int e = threadIdx.x;
    const int64_t base = static_cast<int64_t>(bh) * max_chunks;
    float a[kCombinePre];
#pragma unroll
    for (int j = 0; j < kCombinePre; ++j) a[j] = j < num_chunks ? part_acc[(base + j) * D + e] : 0.f;
    float mv[kPer], lv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int c = e + j * D;
        mv[j] = c < num_chunks ? part_m[base + c] : -INFINITY;
        lv[j] = c < num_chunks ? part_l[base + c] : 0.f;
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int c = e + j * D;
        if (c < num_chunks) {
            m_sh[c] = mv[j];
            l_sh[c] = lv[j];
        }
        mx = fmaxf(mx, mv[j]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if ((e & 31) == 0) red[e >> 5] = mx;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int c = 0; c < kCombinePre; ++c) {
        if (c < num_chunks) {
            const float mc = m_sh[c];
            const float wgt = mc == -INFINITY ? 0.f : ex2(mc - M);   // chunks that saw no key weigh 0
            L = fmaf(l_sh[c], wgt, L);
            A = fmaf(a[c], wgt, A);
        }
    }
    for (int c = kCombinePre; c < num_chunks; ++c) {
        const float mc = m_sh[c];
        const float wgt = mc == -INFINITY ? 0.f : ex2(mc - M);
        L = fmaf(l_sh[c], wgt, L);
        A = fmaf(part_acc[(base + c) * D + e], wgt, A);
    }
    o[static_cast<int64_t>(bh) * D + e] = __float2bfloat16_rn(A / L);
    if (e == 0) lse[bh] = (M + __log2f(L)) * kDecLn2;
}

// The merge of the chunks' triples, launched as the split kernel's programmatic
// dependent: its CTAs can be scheduled once every split CTA is running (during the split
// grid's last wave) and start merging the moment that grid completes.
template <int D>
cudaError_t launch_combine(const DecodeArgs &a, cudaStream_t stream) {
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.BHkv * a.group));
    cfg.blockDim = dim3(D);
    cfg.stream = stream;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, static_cast<const float *>(a.part_m),
                              static_cast<const float *>(a.part_l), static_cast<const float *>(a.part_acc),
                              static_cast<__nv_bfloat16 *>(a.o), a.lse, a.num_chunks, a.max_chunks);
}

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t stream) {
    using C = DecCfg<D, G>;
    auto kern = decode_split_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.BHkv) * (a.group / G) * a.num_chunks;
    if (blocks <= 0 || blocks > INT_MAX) return cudaErrorInvalidValue;
    const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(blocks), kDecThreads, C::kSmemBytes, stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.part_m, a.part_l, a.part_acc, a.Nk, a.chunk_keys, a.num_chunks,
        a.max_chunks, a.group, scale_log2, a.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine<D>(a, stream);
}

template <int D>
cudaError_t launch_decode_mma(const DecodeArgs &a, cudaStream_t stream) {
    using C = DecMmaCfg<D>;
    auto kern = decode_mma_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = static_cast<long long>(a.BHkv) * a.num_chunks;
    if (blocks <= 0 || blocks > INT_MAX) return cudaErrorInvalidValue;
    const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(blocks), kMmaDecThreads, C::kSmemBytes, stream>>>(
        a.tm_k, a.tm_v, static_cast<const __nv_bfloat16 *>(a.q), a.part_m, a.part_l, a.part_acc, a.Nk,
        a.chunk_keys, a.num_chunks, a.max_chunks, a.group, scale_log2, a.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine<D>(a, stream);
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t stream) {
    if (a.group >= kDecodeMmaMinGroup) return launch_decode_mma<D>(a, stream);
    switch (decode_subgroup(a.group)) {   // 1..5 or 7
        case 1: return launch_decode_t<D, 1>(a, stream);
        case 2: return launch_decode_t<D, 2>(a, stream);
        case 3: return launch_decode_t<D, 3>(a, stream);
        case 4: return launch_decode_t<D, 4>(a, stream);
        case 5: return launch_decode_t<D, 5>(a, stream);
        case 7: return launch_decode_t<D, 7>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t decode_ctas_per_sm_d(int group, int *out) {
    if (group >= kDecodeMmaMinGroup) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             DecMmaCfg<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, decode_mma_kernel<D>, kMmaDecThreads,
                                                             DecMmaCfg<D>::kSmemBytes);
    }
    group = decode_subgroup(group);
    auto q = [out](auto kern, int smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, kern, kDecThreads, smem);
    };
    switch (group) {
        case 1: return q(decode_split_kernel<D, 1>, DecCfg<D, 1>::kSmemBytes);
        case 2: return q(decode_split_kernel<D, 2>, DecCfg<D, 2>::kSmemBytes);
        case 3: return q(decode_split_kernel<D, 3>, DecCfg<D, 3>::kSmemBytes);
        case 4: return q(decode_split_kernel<D, 4>, DecCfg<D, 4>::kSmemBytes);
        case 5: return q(decode_split_kernel<D, 5>, DecCfg<D, 5>::kSmemBytes);
        case 7: return q(decode_split_kernel<D, 7>, DecCfg<D, 7>::kSmemBytes);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_subgroup(int group) {
    if (group >= kDecodeMmaMinGroup) return group;   // the tensor-core kernel takes the whole group
    if (group <= 4) return group;
    if (group % 4 == 0) return 4;
    if (group % 3 == 0) return 3;
    return group;
}

cudaError_t decode_ctas_per_sm(int d, int group, int *out) {
    if (d == 64) return decode_ctas_per_sm_d<64>(group, out);
    if (d == 128) return decode_ctas_per_sm_d<128>(group, out);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t stream) {
    // the merge keeps one table entry per chunk in shared memory (checked before any launch)
    if (a.num_chunks < 1 || a.num_chunks > kDecodeMaxChunks || a.num_chunks > a.max_chunks)
        return cudaErrorInvalidValue;
    if (a.d == 64) return launch_decode_d<64>(a, stream);
    if (a.d == 128) return launch_decode_d<128>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
