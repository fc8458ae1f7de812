// fa_fp8.cu — FP8 (e4m3) forward pass with incoherent processing, and the kernels that
// quantize its inputs.
//
// The pages say only that the third-generation kernel has a low-precision FP8 mode
// "with incoherent processing" ("FlashAttention" deep dive, section "How it works";
// "FlashAttention Explained", section "Later versions").  The reading taken here:
//  * codes are e4m3 (round to nearest even, saturating at +-448), one scale per
//    (batch, head) slice of Q, K and V (descale = amax / 448);
//  * incoherent processing rotates every row of Q and of K by the same orthogonal
//    matrix diag(s) H / sqrt(d) (H the Sylvester Hadamard matrix, s random signs the
//    caller draws), which leaves Q K^T unchanged and spreads outlier coordinates over
//    the row before rounding; V is not rotated;
//  * the forward pass is the bf16 kernel's algorithm with both products of
//    tcgen05.mma kind::f8f6f4 (twice the bf16 rate): S = Q8 K8^T, P rounded to e4m3
//    in tensor memory, O += P8 V8; the row sum l stays in fp32.  The per-head scales
//    enter the exponent (dq * dk * scale * log2 e) and the epilogue (dv / l).
//
// Kernels:
//  * qk_amax_kernel / v_amax (the same kernel, no rotation): per-head max |x| of the
//    (rotated) rows, one warp per row, atomicMax on the float bits;
//  * qk_quant_kernel: rotate again, scale by 448 / amax, round to e4m3;
//  * v_quant_t_kernel: V codes transposed to [B*Hkv, d, Npad] (keys contiguous, N padded
//    to a multiple of 16 with zero codes): the K-major B operand of the P V product;
//  * finalize_scales_kernel: amax -> descale in place;
//  * fwd_fp8_kernel: one CTA per (batch, head, two 128-row query tiles), the layout of
//    the bf16 forward kernel (warps 0-7 softmax, 8 MMA, 9 TMA), d = 128.
#include <climits>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kE4M3Max = 448.0f;
constexpr float kLn2f = 0.6931471805599453f;

// ------------------------------------------------------------------------------------
// quantization
// ------------------------------------------------------------------------------------
// One warp per row; lane l holds elements EPL*l .. EPL*l + EPL-1.  With kRot the row is
// multiplied by the signs, run through the Walsh-Hadamard butterflies (strides 1, 2, 4,
// ...: lower element x + partner, upper element partner - x) and scaled by the fp32
// value of 1/sqrt(D).
template <int D, bool kRot>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *row, const float *signs, int lane,
                                         float (&x)[D / 32]) {
    constexpr int EPL = D / 32;
    if constexpr (EPL == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(row + 4 * lane);
        x[0] = __uint_as_float(w.x << 16);
        x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16);
        x[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + 2 * lane);
        x[0] = __uint_as_float(w << 16);
        x[1] = __uint_as_float(w & 0xffff0000u);
    }
    if constexpr (kRot) {
#pragma unroll
        for (int r = 0; r < EPL; ++r) x[r] *= signs[EPL * lane + r];
        // strides inside the lane
#pragma unroll
        for (int s = 1; s < EPL; s <<= 1) {
#pragma unroll
            for (int r = 0; r < EPL; ++r) {
                if (r & s) continue;
                const float a = x[r], b = x[r + s];
                x[r] = a + b;
                x[r + s] = a - b;
            }
        }
        // strides across lanes: element bit s <-> lane bit s / EPL
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
            for (int r = 0; r < EPL; ++r) {
                const float p = __shfl_xor_sync(0xffffffffu, x[r], m);
                x[r] = (lane & m) ? p - x[r] : x[r] + p;
            }
        }
        const float inv_sqrt_d = D == 128 ? 0.08838834764831845f : 0.125f;
#pragma unroll
        for (int r = 0; r < EPL; ++r) x[r] *= inv_sqrt_d;
    }
}

// amax_bits must be zero on entry; afterwards it holds the per-head max |x| as float bits.
template <int D, bool kRot>
__global__ void __launch_bounds__(256)
amax_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ signs, unsigned int *amax_bits,
            long long rows, int N) {
    const int lane = threadIdx.x & 31;
    const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long per = (rows + nwarps - 1) / nwarps;
    const long long r0 = warp_g * per, r1 = min(rows, r0 + per);
    float m = 0.f;
    long long head = r0 / N;
    for (long long r = r0; r < r1; ++r) {
        if (r / N != head) {   // flush the previous head's max
            if (lane == 0) atomicMax(&amax_bits[head], __float_as_uint(m));
            head = r / N;
            m = 0.f;
        }
        float v[D / 32];
        load_row<D, kRot>(x + r * D, signs, lane, v);
#pragma unroll
        for (int e = 0; e < D / 32; ++e) m = fmaxf(m, fabsf(v[e]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    }
    if (r0 < r1 && lane == 0) atomicMax(&amax_bits[head], __float_as_uint(m));
}

__device__ __forceinline__ float head_inv_scale(unsigned int amax_bits) {
    float a = __uint_as_float(amax_bits);
    if (!(a > 0.f)) a = 1.f;   // an all-zero head
    return kE4M3Max / a;
}

template <int D, bool kRot>
__global__ void __launch_bounds__(256)
qk_quant_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ signs,
                const unsigned int *__restrict__ amax_bits, uint8_t *__restrict__ x8, long long rows, int N) {
    constexpr int EPL = D / 32;
    const int lane = threadIdx.x & 31;
    const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long r = warp_g; r < rows; r += nwarps) {
        const float inv = head_inv_scale(amax_bits[r / N]);
        float v[EPL];
        load_row<D, kRot>(x + r * D, signs, lane, v);
        if constexpr (EPL == 4) {
            *reinterpret_cast<uint32_t *>(x8 + r * D + 4 * lane) =
                pack_e4m3x4(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
        } else {
            *reinterpret_cast<uint16_t *>(x8 + r * D + 2 * lane) =
                static_cast<uint16_t>(pack_e4m3x4(v[0] * inv, v[1] * inv, 0.f, 0.f) & 0xffffu);
        }
    }
}

// V codes transposed: one CTA per (head, 64 keys); keys N .. Npad-1 get code 0.
template <int D>
__global__ void __launch_bounds__(256)
v_quant_t_kernel(const __nv_bfloat16 *__restrict__ v, const unsigned int *__restrict__ amax_bits,
                 uint8_t *__restrict__ vt8, int N, int Npad, int tiles) {
    __shared__ uint8_t tile[D][64 + 4];
    const int bh = blockIdx.x / tiles;
    const int k0 = (blockIdx.x % tiles) * 64;
    const float inv = head_inv_scale(amax_bits[bh]);
    const __nv_bfloat16 *vh = v + static_cast<int64_t>(bh) * N * D;
    for (int idx = threadIdx.x; idx < 64 * D; idx += blockDim.x) {
        const int key = idx / D, c = idx % D;
        const int kg = k0 + key;
        uint8_t code = 0;
        if (kg < N) code = static_cast<uint8_t>(pack_e4m3x4(__bfloat162float(vh[static_cast<int64_t>(kg) * D + c]) * inv,
                                                            0.f, 0.f, 0.f) & 0xffu);
        tile[c][key] = code;
    }
    __syncthreads();
    uint8_t *dst = vt8 + static_cast<int64_t>(bh) * D * Npad;
    for (int idx = threadIdx.x; idx < D * 16; idx += blockDim.x) {
        const int c = idx / 16, k4 = (idx % 16) * 4;
        if (k0 + k4 < Npad) {
            const uint32_t w = tile[c][k4] | (tile[c][k4 + 1] << 8) | (tile[c][k4 + 2] << 16) |
                               (static_cast<uint32_t>(tile[c][k4 + 3]) << 24);
            *reinterpret_cast<uint32_t *>(dst + static_cast<int64_t>(c) * Npad + k0 + k4) = w;
        }
    }
}

__global__ void finalize_scales_kernel(unsigned int *amax_descale, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        float a = __uint_as_float(amax_descale[i]);
        if (!(a > 0.f)) a = 1.f;
        reinterpret_cast<float *>(amax_descale)[i] = a / kE4M3Max;
    }
}

int blocks_for(long long rows, int rows_per_block) {
    long long g = (rows + rows_per_block - 1) / rows_per_block;
    if (g < 1) g = 1;
    if (g > 152LL * 8) g = 152LL * 8;
    return static_cast<int>(g);
}

// ------------------------------------------------------------------------------------
// FP8 forward
// ------------------------------------------------------------------------------------
struct F8Cfg {
    static constexpr int D = 128;
    static constexpr int kTileBytes = kTileRows * D;                // 16 KB: one 128-byte box of 128 rows
    static constexpr int kStages = 8;                               // K and V^T tiles alternate
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
    static constexpr int kNumBars = 8 + 2 * kStages;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static constexpr int kThreads = 320;
    static constexpr int kMmaWarp = 8, kLoadWarp = 9;
    static constexpr uint32_t kOCol = 256;
    static constexpr int kKSteps = D / 32;                          // 32-byte K steps over d
    static constexpr int kPVSteps = kTileRows / 32;                 // 32-key K steps
    static constexpr uint32_t kIdescQK = make_idesc(kFormatE4M3, 128, 128, false, false);
    static constexpr uint32_t kIdescPV = make_idesc(kFormatE4M3, 128, D, false, false);
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct F8Bars {
    static constexpr int kQ = 0;
    static constexpr int kKVFull = 1;                          // + stage
    static constexpr int kKVEmpty = 1 + F8Cfg::kStages;        // + stage
    static constexpr int kSFull = 1 + 2 * F8Cfg::kStages;      // + tile
    static constexpr int kPFull = kSFull + 2;                  // + tile
    static constexpr int kODone = kSFull + 4;                  // + tile
    static constexpr int kMmaDone = kSFull + 6;
};

enum : int {
    kSite8LoadEmpty = 81, kSite8MmaQ = 82, kSite8MmaKV = 83, kSite8MmaP = 84, kSite8SoftS = 85,
    kSite8SoftO = 86, kSite8EpiO = 87, kSite8Drain = 88, kSite8MmaDrain = 89
};

constexpr float kRescaleThreshold8 = 8.0f;
constexpr float kRescaleBound8 = 256.0f;

__global__ void __launch_bounds__(F8Cfg::kThreads, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_vt, const float *__restrict__ dsc_q,
               const float *__restrict__ dsc_k, const float *__restrict__ dsc_v, __nv_bfloat16 *__restrict__ out,
               float *__restrict__ lse, int N, int num_pairs, int group, float scale_log2, int causal,
               unsigned int *status) {
    using C = F8Cfg;
    using B = F8Bars;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kQOff, sKV = base + C::kKVOff, sBar = base + C::kBarOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx wc{abort_flag, status};
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int bh, rank;
    heavy_first_order(blockIdx.x, num_pairs, bh, rank);
    const int bh_kv = bh / group;
    const int pair = causal ? (num_pairs - 1 - rank) : rank;
    const int nkv = (N + kTileRows - 1) / kTileRows;
    int ntile[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = 2 * pair + t;
        ntile[t] = qt * kTileRows >= N ? 0 : (causal ? min(qt + 1, nkv) : nkv);
    }
    const int nmax = max(ntile[0], ntile[1]);

    if (threadIdx.x == 0) {
        mbar_init(bar(B::kQ), 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(B::kKVFull + s), 1);
            mbar_init(bar(B::kKVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(B::kSFull + t), 1);
            mbar_init(bar(B::kPFull + t), 128);
            mbar_init(bar(B::kODone + t), 1);
        }
        mbar_init(bar(B::kMmaDone), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == C::kLoadWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_vt);
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t) qbytes += ntile[t] > 0 ? C::kTileBytes : 0;
            mbar_arrive_expect_tx(bar(B::kQ), qbytes);
            for (int t = 0; t < 2; ++t)
                if (ntile[t] > 0) tma_load_3d(sQ + t * C::kTileBytes, &tm_q, bar(B::kQ), 0, (2 * pair + t) * kTileRows, bh);
            int seq = 0;
            for (; seq < 2 * nmax; ++seq) {
                const int s = seq % C::kStages, use = seq / C::kStages;
                if (use > 0 && !mbar_wait(bar(B::kKVEmpty + s), (use - 1) & 1, wc, kSite8LoadEmpty)) break;
                mbar_arrive_expect_tx(bar(B::kKVFull + s), C::kTileBytes);
                const int j = seq >> 1;
                if (seq & 1)   // V^T_j: d rows of 128 key bytes
                    tma_load_3d(sKV + s * C::kTileBytes, &tm_vt, bar(B::kKVFull + s), j * kTileRows, 0, bh_kv);
                else           // K_j: 128 key rows of d bytes
                    tma_load_3d(sKV + s * C::kTileBytes, &tm_k, bar(B::kKVFull + s), 0, j * kTileRows, bh_kv);
            }
            mbar_wait_drain(bar(B::kQ), 0, wc, kSite8Drain);
            for (int s = 0; s < C::kStages && s < seq; ++s) {
                const int last = s + ((seq - 1 - s) / C::kStages) * C::kStages;
                mbar_wait_drain(bar(B::kKVFull + s), (last / C::kStages) & 1, wc, kSite8Drain);
            }
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer (whole warp, lane 0 issues)
        {
            auto mbar_wait_w = [&](uint32_t b, uint32_t parity, int site) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
            };
            const uint32_t tS[2] = {tmem, tmem + 128u};
            const uint32_t tO[2] = {tmem + C::kOCol, tmem + C::kOCol + D};
            auto wait_kv = [&](int seq) -> int {
                const int s = seq % C::kStages;
                if (!mbar_wait_w(bar(B::kKVFull + s), (seq / C::kStages) & 1, kSite8MmaKV)) return -1;
                tc_fence_after();
                return s;
            };
            static_assert(C::kKSteps == 4 && C::kPVSteps == 4, "4-step products");
            auto issue_qk = [&](int t, int s) {
                const uint64_t a0 = sdesc_sw128(sQ + t * C::kTileBytes, 16, 1024);
                const uint64_t b0 = sdesc_sw128(sKV + s * C::kTileBytes, 16, 1024);
                uint64_t a[4], b[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    a[kk] = sdesc_step(a0, kk * 32);
                    b[kk] = sdesc_step(b0, kk * 32);
                }
                umma_f8_ss_x4(tS[t], a, b, C::kIdescQK, 0u);
            };
            auto issue_pv = [&](int t, int s, bool acc) {
                const uint64_t b0 = sdesc_sw128(sKV + s * C::kTileBytes, 16, 1024);
                uint64_t b[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) b[kk] = sdesc_step(b0, kk * 32);
                umma_f8_ts_x4(tO[t], tS[t], b, C::kIdescPV, acc ? 1u : 0u);
            };
            bool ok = mbar_wait_w(bar(B::kQ), 0, kSite8MmaQ);
            if (ok) {
                const int sk = wait_kv(0);
                ok = sk >= 0;
                if (ok) {
                    for (int t = 0; t < 2; ++t) {
                        if (ntile[t] == 0) continue;
                        issue_qk(t, sk);
                        umma_commit(bar(B::kSFull + t));
                    }
                    umma_commit(bar(B::kKVEmpty + sk));
                }
            }
            for (int j = 0; ok && j < nmax; ++j) {
                const int sv = wait_kv(2 * j + 1);
                if (sv < 0) { ok = false; break; }
                int skn = -1;
                for (int t = 0; t < 2; ++t) {
                    if (j >= ntile[t]) continue;
                    if (!mbar_wait_w(bar(B::kPFull + t), j & 1, kSite8MmaP)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(t, sv, j > 0);
                    umma_commit(bar(B::kODone + t));
                    if (j + 1 < ntile[t]) {
                        if (skn < 0) {
                            skn = wait_kv(2 * (j + 1));
                            if (skn < 0) { ok = false; break; }
                        }
                        issue_qk(t, skn);
                        umma_commit(bar(B::kSFull + t));
                    }
                }
                if (!ok) break;
                umma_commit(bar(B::kKVEmpty + sv));
                if (skn >= 0) umma_commit(bar(B::kKVEmpty + skn));
            }
            umma_commit(bar(B::kMmaDone));
            mbar_wait_drain(bar(B::kMmaDone), 0, wc, kSite8MmaDrain);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int row_g = (2 * pair + t) * kTileRows + row;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tSr = tmem + lane_off + 128u * t;
        const uint32_t tOr = tmem + lane_off + C::kOCol + D * t;
        // base-2 exponent scale of this head: softmax scale * log2 e * descale_q * descale_k
        const float sl = scale_log2 * dsc_q[bh] * dsc_k[bh_kv];
        const float2 sl2 = make_float2(sl, sl);
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < ntile[t]; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull + t), j & 1, wc, kSite8SoftS));
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld_x128(tSr, sr);
            const int kv0 = j * kTileRows;
            const int lim = min(causal ? row_g - kv0 : kTileRows - 1, N - 1 - kv0);
            auto apply_mask = [&]() {
                if (lim < kTileRows - 1) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c > lim) sr[c] = __float_as_uint(-INFINITY);
                }
            };
            apply_mask();
            auto row_max = [&]() -> float {
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    mx0 = max3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                    mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    mx2 = max3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                    mx3 = max3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
                }
                return fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl;
            };
            // P = 2^(s * sl - m) in fp32 for the row sum, e4m3 (four per column) for P V
            uint32_t pk[32];
            auto exp_pass = [&](float m) -> float {
                const float neg = (m == -INFINITY) ? 0.f : -m;
                const float2 ng2 = make_float2(neg, neg);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const float2 x0 =
                        fma2(make_float2(__uint_as_float(sr[4 * u]), __uint_as_float(sr[4 * u + 1])), sl2, ng2);
                    const float2 x1 =
                        fma2(make_float2(__uint_as_float(sr[4 * u + 2]), __uint_as_float(sr[4 * u + 3])), sl2, ng2);
                    const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
                    const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                    acc0 = add2(acc0, p0);
                    acc1 = add2(acc1, p1);
                    pk[u] = pack_e4m3x4(p0.x, p0.y, p1.x, p1.y);
                }
                const float2 accs = add2(acc0, acc1);
                return accs.x + accs.y;
            };
            float alpha = 1.f;
            bool upd = false;
            float blk;
            if (__any_sync(0xffffffffu, m_run == -INFINITY)) {
                const float mx = row_max();
                upd = mx > m_run + (m_run == -INFINITY ? 0.f : kRescaleThreshold8);
                if (upd) {
                    alpha = ex2(m_run - mx);
                    m_run = mx;
                }
                blk = exp_pass(m_run);
            } else {
                blk = exp_pass(m_run);
                // P must stay below 2^8 (e4m3 holds up to 448): the block sum bounds every P.
                // Otherwise take the row max from S, still in tensor memory (re-read in
                // chunks so that S need not stay in registers), and recompute if it grew.
                if (__any_sync(0xffffffffu, !(blk < kRescaleBound8))) {
                    float m4 = -INFINITY;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t r[32];
                        tmem_ld_x32(tSr + 32u * ch, r);
                        float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
                        for (int c = 0; c < 32; c += 4) {
                            const int cc = 32 * ch + c;
                            a0 = max3(a0, cc > lim ? -INFINITY : __uint_as_float(r[c]),
                                      cc + 1 > lim ? -INFINITY : __uint_as_float(r[c + 1]));
                            a1 = max3(a1, cc + 2 > lim ? -INFINITY : __uint_as_float(r[c + 2]),
                                      cc + 3 > lim ? -INFINITY : __uint_as_float(r[c + 3]));
                        }
                        m4 = max3(m4, a0, a1);
                    }
                    const float mx = m4 * sl;
                    upd = mx > m_run + kRescaleThreshold8;
                    if (upd) {
                        alpha = ex2(m_run - mx);
                        m_run = mx;
                    }
                    if (__any_sync(0xffffffffu, upd)) {
                        tmem_ld_x128(tSr, sr);
                        apply_mask();
                        blk = exp_pass(m_run);
                    }
                }
            }
            tmem_st_x32(tSr, pk);
            l_run = l_run * alpha + blk;
            if (j > 0 && __any_sync(0xffffffffu, upd)) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kODone + t), (j - 1) & 1, wc, kSite8SoftO));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_x32(tOr + 32u * c, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st_x32(tOr + 32u * c, o);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B::kPFull + t));
        }
        // ------------------------------------------------------------ epilogue
        if (ok && ntile[t] > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kODone + t), (ntile[t] - 1) & 1, wc, kSite8EpiO));
            if (ok) {
                tc_fence_after();
                const float f = l_run > 0.f ? dsc_v[bh_kv] / l_run : 0.f;
                const bool valid = row_g < N;
                __nv_bfloat16 *orow = out + (static_cast<int64_t>(bh) * N + (valid ? row_g : 0)) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_x32(tOr + 32u * c, o);
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint4 w;
                            w.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * f, __uint_as_float(o[8 * i + 1]) * f);
                            w.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * f, __uint_as_float(o[8 * i + 3]) * f);
                            w.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * f, __uint_as_float(o[8 * i + 5]) * f);
                            w.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * f, __uint_as_float(o[8 * i + 7]) * f);
                            dst[i] = w;
                        }
                    }
                }
                if (valid)
                    lse[static_cast<int64_t>(bh) * N + row_g] =
                        l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2f : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == C::kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_quantize_qk_fp8(const void *x, const float *signs, void *x8, float *descale, int BH, int N,
                                   int d, cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * N;
    unsigned int *amax = reinterpret_cast<unsigned int *>(descale);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * BH, stream);
    if (e != cudaSuccess) return e;
    const int g = blocks_for(rows, 64);
    const auto *xb = static_cast<const __nv_bfloat16 *>(x);
    auto *x8b = static_cast<uint8_t *>(x8);
    if (d == 128) {
        if (signs) amax_kernel<128, true><<<g, 256, 0, stream>>>(xb, signs, amax, rows, N);
        else amax_kernel<128, false><<<g, 256, 0, stream>>>(xb, signs, amax, rows, N);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (signs) qk_quant_kernel<128, true><<<g, 256, 0, stream>>>(xb, signs, amax, x8b, rows, N);
        else qk_quant_kernel<128, false><<<g, 256, 0, stream>>>(xb, signs, amax, x8b, rows, N);
    } else if (d == 64) {
        if (signs) amax_kernel<64, true><<<g, 256, 0, stream>>>(xb, signs, amax, rows, N);
        else amax_kernel<64, false><<<g, 256, 0, stream>>>(xb, signs, amax, rows, N);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (signs) qk_quant_kernel<64, true><<<g, 256, 0, stream>>>(xb, signs, amax, x8b, rows, N);
        else qk_quant_kernel<64, false><<<g, 256, 0, stream>>>(xb, signs, amax, x8b, rows, N);
    } else {
        return cudaErrorInvalidValue;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    finalize_scales_kernel<<<(BH + 255) / 256, 256, 0, stream>>>(amax, BH);
    return cudaGetLastError();
}

cudaError_t launch_quantize_v_fp8(const void *v, void *vt8, float *descale, int BH, int N, int Npad, int d,
                                  cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * N;
    unsigned int *amax = reinterpret_cast<unsigned int *>(descale);
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * BH, stream);
    if (e != cudaSuccess) return e;
    const int g = blocks_for(rows, 64);
    const auto *vb = static_cast<const __nv_bfloat16 *>(v);
    const int tiles = (Npad + 63) / 64;
    const long long vblocks = static_cast<long long>(BH) * tiles;
    if (vblocks > INT_MAX) return cudaErrorInvalidValue;
    if (d == 128) {
        amax_kernel<128, false><<<g, 256, 0, stream>>>(vb, nullptr, amax, rows, N);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        v_quant_t_kernel<128><<<static_cast<unsigned>(vblocks), 256, 0, stream>>>(vb, amax, static_cast<uint8_t *>(vt8),
                                                                                 N, Npad, tiles);
    } else if (d == 64) {
        amax_kernel<64, false><<<g, 256, 0, stream>>>(vb, nullptr, amax, rows, N);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        v_quant_t_kernel<64><<<static_cast<unsigned>(vblocks), 256, 0, stream>>>(vb, amax, static_cast<uint8_t *>(vt8),
                                                                                N, Npad, tiles);
    } else {
        return cudaErrorInvalidValue;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    finalize_scales_kernel<<<(BH + 255) / 256, 256, 0, stream>>>(amax, BH);
    return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const Fp8FwdArgs &a, cudaStream_t stream) {
    using C = F8Cfg;
    if (a.d != 128) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int num_pairs = (a.N + 2 * kTileRows - 1) / (2 * kTileRows);
    const long long blocks = static_cast<long long>(a.BH) * num_pairs;
    if (blocks <= 0 || blocks > INT_MAX) return cudaErrorInvalidValue;
    const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    fwd_fp8_kernel<<<static_cast<unsigned>(blocks), C::kThreads, C::kSmemBytes, stream>>>(
        a.tm_q, a.tm_k, a.tm_vt, a.dsc_q, a.dsc_k, a.dsc_v, static_cast<__nv_bfloat16 *>(a.o), a.lse, a.N,
        num_pairs, a.group, scale_log2, a.causal, a.status);
    return cudaGetLastError();
}

}  // namespace fa
