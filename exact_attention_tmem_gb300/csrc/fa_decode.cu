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

template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const float *__restrict__ part_m, const float *__restrict__ part_l,
                      const float *__restrict__ part_acc, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse,
                      int num_chunks, int max_chunks) {
    const int bh = blockIdx.x;
    const int e = threadIdx.x;
    const int64_t base = static_cast<int64_t>(bh) * max_chunks;
    float M = -INFINITY;
    for (int c = 0; c < num_chunks; ++c) M = fmaxf(M, part_m[base + c]);
    float L = 0.f, A = 0.f;
    for (int c = 0; c < num_chunks; ++c) {
        const float mc = part_m[base + c];
        const float wgt = mc == -INFINITY ? 0.f : ex2(mc - M);
        L = fmaf(part_l[base + c], wgt, L);
        A = fmaf(part_acc[(base + c) * D + e], wgt, A);
    }
    o[static_cast<int64_t>(bh) * D + e] = __float2bfloat16_rn(A / L);
    if (e == 0) lse[bh] = (M + __log2f(L)) * kDecLn2;
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
    decode_combine_kernel<D><<<static_cast<unsigned>(a.BHkv * a.group), D, 0, stream>>>(
        a.part_m, a.part_l, a.part_acc, static_cast<__nv_bfloat16 *>(a.o), a.lse, a.num_chunks, a.max_chunks);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t stream) {
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
    if (a.d == 64) return launch_decode_d<64>(a, stream);
    if (a.d == 128) return launch_decode_d<128>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
