// fa_fwd.cu — forward pass of exact attention on sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes ("FlashAttention" deep dive, section "How it works"): for each
// query tile Q_i and each key/value tile K_j, V_j in turn, S = Q_i K_j^T * scale,
// m_new = max(m, rowmax S), P = exp(S - m_new), alpha = exp(m - m_new),
// l = alpha*l + rowsum P, acc = alpha*acc + P V_j; at the end O_i = acc / l and
// L_i = m + log l.  Causal tiles above the diagonal are never loaded or multiplied
// ("tm_flash_attention_arch_2k", section "The architecture: every step explained";
// deep dive, section "Implementation notes"), and only the diagonal tile is masked.
//
// GB300 design (differs from the pages' A100/H100 kernels):
//  * One CTA owns two 128-row query tiles of one (batch, head) and streams K/V
//    tiles through a multi-stage shared-memory ring filled by TMA.
//  * Both contractions run on the 5th-generation tensor cores: S_t = Q_t K_j^T with
//    both operands in shared memory, O_t += P_t V_j with P_t read from tensor
//    memory, where the softmax warps wrote it over S_t.  S and O live in tensor
//    memory (TMEM): S0 | S1 | O0 | O1 = 128 + 128 + d + d of its 512 columns.
//  * Warp roles: warps 0-3 and 4-7 are the softmax warpgroups of tile 0 and tile 1
//    (thread r owns row r: tcgen05.ld gives it its whole row, so row max and row
//    sum need no shuffles); warp 8 issues every MMA from one thread; warp 9 issues
//    every TMA load from one thread.  The two tiles ping-pong: the tensor cores
//    work on one tile's products while the other tile's softmax runs.
//  * Base-2 exponentials with log2(e) folded into the scale (deep dive,
//    "Implementation notes").  The running max is updated lazily: only when a row's
//    max grows by more than 2^8 in the base-2 domain are l and the TMEM accumulator
//    rescaled.  Exact: l and acc always refer to the same stale max, and the final
//    O = acc / l and L = m + log2(l) use it too.
//  * Every wait is time-limited; see ptx.cuh.
#include <cfloat>
#include <climits>
#include <type_traits>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

template <typename T, int D, int QT>
struct FwdCfg {
    static constexpr bool kTF32 = std::is_same<T, float>::value;
    // QT query tiles of 128 rows per CTA: 4 softmax warps per tile, then the MMA warp
    // and the TMA warp.  With QT = 1 two CTAs share an SM (half the shared memory and
    // tensor memory each); with QT = 2 one CTA owns the SM.
    static constexpr int kMmaWarp = 4 * QT;
    static constexpr int kLoadWarp = 4 * QT + 1;
    static constexpr int kThreads = 32 * (4 * QT + 2);
    static constexpr int kMinBlocks = QT == 1 ? 2 : 1;
    static constexpr int kSmemBudget = QT == 1 ? 100 * 1024 : 200 * 1024;
    static constexpr int kEB = static_cast<int>(sizeof(T));
    static constexpr int kRowBytes = D * kEB;
    static constexpr int kBoxCols = kBoxBytes / kEB;        // elements per 128-byte box row
    static constexpr int kBoxes = kRowBytes / kBoxBytes;     // boxes per tile
    static constexpr int kBoxTileBytes = kTileRows * kBoxBytes;
    static constexpr int kTileBytes = kBoxes * kBoxTileBytes;
    static constexpr int kKStep = 32 / kEB;                  // K elements per MMA instruction
    static constexpr int kQKSteps = kRowBytes / 32;
    static constexpr int kPVSteps = kTileRows / kKStep;
    static constexpr int kStagesFit = (kSmemBudget - QT * kTileBytes) / kTileBytes;
    // TF32: two stages, so K always lands in stage 0 and V in stage 1 (see kVtOff)
    static constexpr int kStages = kTF32 ? 2 : (kStagesFit > 8 ? 8 : kStagesFit);
    // shared memory map, offsets from a 1024-byte aligned base
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = QT * kTileBytes;
    // TF32 only: V^T of the current V tile, K-major (the TF32 B operand must be K-major):
    // 4 boxes of 32 keys (128 bytes) x D rows.
    static constexpr int kVtOff = kKVOff + kStages * kTileBytes;
    static constexpr int kVtBoxBytes = D * kBoxBytes;
    static constexpr int kVtBytes = kTF32 ? 4 * kVtBoxBytes : 0;
    static constexpr int kBarOff = kVtOff + kVtBytes;
    static constexpr int kNumBars = 9 + 2 * kStages;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    // tensor memory columns
    static constexpr uint32_t kTmemCols = QT == 2 ? 512 : 256;
    static constexpr uint32_t kOCol = 128 * QT;
    static constexpr uint32_t kFmt = kTF32 ? kFormatTF32 : kFormatBF16;
    static constexpr uint32_t kIdescQK = make_idesc(kFmt, 128, 128, false, false);
    static constexpr uint32_t kIdescPV = make_idesc(kFmt, 128, D, false, !kTF32);

    static_assert(kRowBytes % kBoxBytes == 0, "row must be whole 128-byte boxes");
    static_assert(kStages >= 2, "need at least two K/V stages");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(128 * QT + QT * D <= kTmemCols, "tensor memory budget");
    static_assert(!kTF32 || QT == 2, "the TF32 variant keeps two query tiles per CTA");
};

// barrier indices
template <int S> struct Bars {
    static constexpr int kQ = 0;
    static constexpr int kKVFull = 1;            // + stage
    static constexpr int kKVEmpty = 1 + S;       // + stage
    static constexpr int kSFull = 1 + 2 * S;     // + tile
    static constexpr int kPFull = 3 + 2 * S;     // + tile
    static constexpr int kODone = 5 + 2 * S;     // + tile
    static constexpr int kMmaDone = 7 + 2 * S;
    static constexpr int kVtFull = 8 + 2 * S;    // TF32: V^T of the current V tile written
};

// wait-site ids recorded in the device status word
enum : int {
    kSiteLoadEmpty = 11, kSiteMmaQ = 12, kSiteMmaKV = 13, kSiteMmaP = 14, kSiteSoftS = 15,
    kSiteSoftO = 16, kSiteEpiO = 17, kSiteDrain = 18, kSiteMmaDrain = 19
};

template <typename T, int D, int QT>
__global__ void __launch_bounds__(FwdCfg<T, D, QT>::kThreads, FwdCfg<T, D, QT>::kMinBlocks)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, T *__restrict__ out, float *__restrict__ lse,
           int N, int num_pairs, int group, float scale_log2, int causal, unsigned int *status) {
    using C = FwdCfg<T, D, QT>;
    constexpr int kMmaWarp = C::kMmaWarp;
    constexpr int kLoadWarp = C::kLoadWarp;
    using B = Bars<C::kStages>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kQOff;
    const uint32_t sKV = base + C::kKVOff;
    const uint32_t sBar = base + C::kBarOff;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kMiscOff);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kMiscOff + 4);
    const WaitCtx wc{abort_flag, status};
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int bh, rank;
    heavy_first_order(blockIdx.x, num_pairs, bh, rank);
    // grouped-query attention: `group` query heads share one key/value head
    const int bh_kv = bh / group;
    // rank 0 is the heaviest group of query tiles of a head when causal
    const int pair = causal ? (num_pairs - 1 - rank) : rank;
    const int nkv = (N + kTileRows - 1) / kTileRows;
    int ntile[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int qt = QT * pair + t;
        ntile[t] = (t >= QT || qt * kTileRows >= N) ? 0 : (causal ? min(qt + 1, nkv) : nkv);
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
        mbar_init(bar(B::kVtFull), 1);
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

    if (warp == kLoadWarp && C::kTF32) {
        // ------------------------------------------------------------ TMA producer, TF32
        // As below, and the whole warp transposes each landed V tile into V^T (K-major),
        // then signals kVtFull.  V tiles are every second fill, always stage 1.
        const uint32_t sVt = base + C::kVtOff;
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t) qbytes += ntile[t] > 0 ? C::kTileBytes : 0;
            mbar_arrive_expect_tx(bar(B::kQ), qbytes);
            for (int t = 0; t < 2; ++t) {
                if (ntile[t] == 0) continue;
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sQ + t * C::kTileBytes + b * C::kBoxTileBytes, &tm_q, bar(B::kQ),
                                b * C::kBoxCols, (QT * pair + t) * kTileRows, bh);
            }
        }
        int seq = 0;
        for (; seq < 2 * nmax; ++seq) {
            const int s = seq % C::kStages;
            const int use = seq / C::kStages;
            bool ok = true;
            if (lane == 0) {
                if (use > 0) ok = mbar_wait(bar(B::kKVEmpty + s), (use - 1) & 1, wc, kSiteLoadEmpty);
                if (ok) {
                    mbar_arrive_expect_tx(bar(B::kKVFull + s), C::kTileBytes);
                    const CUtensorMap *m = (seq & 1) ? &tm_v : &tm_k;
                    for (int b = 0; b < C::kBoxes; ++b)
                        tma_load_3d(sKV + s * C::kTileBytes + b * C::kBoxTileBytes, m, bar(B::kKVFull + s),
                                    b * C::kBoxCols, (seq >> 1) * kTileRows, bh_kv);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (seq & 1) {
                // V tile: wait for it, then write V^T.  Element (key k, column n) sits in box
                // n / 32 at row k, 16-byte chunk ((n % 32) / 4) ^ (k % 8); in V^T it goes to
                // box k / 32 at row n, chunk ((k % 32) / 4) ^ (n % 8).
                if (!__all_sync(0xffffffffu, mbar_wait(bar(B::kKVFull + s), use & 1, wc, kSiteLoadEmpty))) break;
                const uint8_t *vsrc = smem + C::kKVOff + s * C::kTileBytes;
                uint8_t *vdst = smem + C::kVtOff;
                for (int idx = lane; idx < kTileRows * D; idx += 32) {
                    const int k = idx / D, n = idx % D;
                    const int nb = n % 32, kb = k % 32;
                    const float val = *reinterpret_cast<const float *>(
                        vsrc + (n / 32) * C::kBoxTileBytes + k * kBoxBytes + ((((nb >> 2) ^ (k & 7)) << 4) | ((nb & 3) << 2)));
                    *reinterpret_cast<float *>(vdst + (k / 32) * C::kVtBoxBytes + n * kBoxBytes +
                                               ((((kb >> 2) ^ (n & 7)) << 4) | ((kb & 3) << 2))) = val;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B::kVtFull));
            }
        }
        (void)sVt;
        if (lane == 0) {
            mbar_wait_drain(bar(B::kQ), 0, wc, kSiteDrain);
            for (int s = 0; s < C::kStages && s < seq; ++s) {
                const int last = s + ((seq - 1 - s) / C::kStages) * C::kStages;
                mbar_wait_drain(bar(B::kKVFull + s), (last / C::kStages) & 1, wc, kSiteDrain);
            }
        }
    } else if (warp == kLoadWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            uint32_t qbytes = 0;
            for (int t = 0; t < 2; ++t) qbytes += ntile[t] > 0 ? C::kTileBytes : 0;
            mbar_arrive_expect_tx(bar(B::kQ), qbytes);
            for (int t = 0; t < 2; ++t) {
                if (ntile[t] == 0) continue;
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sQ + t * C::kTileBytes + b * C::kBoxTileBytes, &tm_q, bar(B::kQ),
                                b * C::kBoxCols, (QT * pair + t) * kTileRows, bh);
            }
            int seq = 0;
            for (; seq < 2 * nmax; ++seq) {
                const int s = seq % C::kStages;
                const int use = seq / C::kStages;
                if (use > 0 && !mbar_wait(bar(B::kKVEmpty + s), (use - 1) & 1, wc, kSiteLoadEmpty)) break;
                mbar_arrive_expect_tx(bar(B::kKVFull + s), C::kTileBytes);
                const CUtensorMap *m = (seq & 1) ? &tm_v : &tm_k;
                const int j = seq >> 1;
                for (int b = 0; b < C::kBoxes; ++b)
                    tma_load_3d(sKV + s * C::kTileBytes + b * C::kBoxTileBytes, m, bar(B::kKVFull + s),
                                b * C::kBoxCols, j * kTileRows, bh_kv);
            }
            // Every copy issued above must land before this CTA may exit.
            mbar_wait_drain(bar(B::kQ), 0, wc, kSiteDrain);
            for (int s = 0; s < C::kStages && s < seq; ++s) {
                const int last = s + ((seq - 1 - s) / C::kStages) * C::kStages;
                mbar_wait_drain(bar(B::kKVFull + s), (last / C::kStages) & 1, wc, kSiteDrain);
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs this loop (every wait is warp-uniform) and lane 0 issues.
        {
            auto mbar_wait_w = [&](uint32_t b, uint32_t parity, int site) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
            };
            const uint32_t tS[2] = {tmem, tmem + 128u};
            const uint32_t tO[2] = {tmem + C::kOCol, tmem + C::kOCol + D};
            auto wait_kv = [&](int seq) -> int {
                const int s = seq % C::kStages;
                if (!mbar_wait_w(bar(B::kKVFull + s), (seq / C::kStages) & 1, kSiteMmaKV)) return -1;
                tc_fence_after();
                return s;
            };
            auto issue_qk = [&](int t, int s) {
                if constexpr (!C::kTF32 && (C::kQKSteps == 4 || C::kQKSteps == 8)) {
                    // bf16: the whole product from one asm block
                    const uint64_t a0 = sdesc_sw128(sQ + t * C::kTileBytes, 16, 1024);
                    const uint64_t b0 = sdesc_sw128(sKV + s * C::kTileBytes, 16, 1024);
                    uint64_t a[C::kQKSteps], b[C::kQKSteps];
#pragma unroll
                    for (int kk = 0; kk < C::kQKSteps; ++kk) {
                        const uint32_t off = (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32;
                        a[kk] = sdesc_step(a0, off);
                        b[kk] = sdesc_step(b0, off);
                    }
                    if constexpr (C::kQKSteps == 8) umma_f16_ss_x8(tS[t], a, b, C::kIdescQK, 0u);
                    else umma_f16_ss_x4(tS[t], a, b, C::kIdescQK, 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::kQKSteps; ++kk) {
                        const uint32_t off = (kk >> 2) * C::kBoxTileBytes + (kk & 3) * 32;
                        const uint64_t a = sdesc_sw128(sQ + t * C::kTileBytes + off, 16, 1024);
                        const uint64_t b = sdesc_sw128(sKV + s * C::kTileBytes + off, 16, 1024);
                        umma_ss<C::kTF32>(tS[t], a, b, C::kIdescQK, kk > 0 ? 1u : 0u);
                    }
                }
            };
            auto issue_pv = [&](int t, int s, bool acc) {
                if constexpr (!C::kTF32 && C::kPVSteps == 8) {
                    // bf16: V as an MN-major B operand, 16 key rows (2 KB) per step
                    const uint64_t b0 = sdesc_sw128(sKV + s * C::kTileBytes, C::kBoxTileBytes, 1024);
                    uint64_t b[8];
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) b[kk] = sdesc_step(b0, kk * C::kKStep * kBoxBytes);
                    umma_f16_ts_x8(tO[t], tS[t], b, C::kIdescPV, acc ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < C::kPVSteps; ++kk) {
                        // TF32: V^T as a K-major B operand
                        const uint64_t b =
                            C::kTF32 ? sdesc_sw128(base + C::kVtOff + (kk >> 2) * C::kVtBoxBytes + (kk & 3) * 32, 16, 1024)
                                     : sdesc_sw128(sKV + s * C::kTileBytes + kk * C::kKStep * kBoxBytes,
                                                   C::kBoxTileBytes, 1024);
                        umma_ts<C::kTF32>(tO[t], tS[t] + kk * 8u, b, C::kIdescPV, (acc || kk > 0) ? 1u : 0u);
                    }
                }
            };
            bool ok = mbar_wait_w(bar(B::kQ), 0, kSiteMmaQ);
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
                int sv;
                if constexpr (C::kTF32) {
                    // V^T of V_j written by the producer warp (V tiles always use stage 1)
                    sv = mbar_wait_w(bar(B::kVtFull), j & 1, kSiteMmaKV) ? 1 : -1;
                    tc_fence_after();
                } else {
                    sv = wait_kv(2 * j + 1);
                }
                if (sv < 0) { ok = false; break; }
                int skn = -1;
                for (int t = 0; t < 2; ++t) {
                    if (j >= ntile[t]) continue;
                    if (!mbar_wait_w(bar(B::kPFull + t), j & 1, kSiteMmaP)) { ok = false; break; }
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
            // Drain the tensor pipe before tensor memory can be released.
            umma_commit(bar(B::kMmaDone));
            mbar_wait_drain(bar(B::kMmaDone), 0, wc, kSiteMmaDrain);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int row_g = (QT * pair + t) * kTileRows + row;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tSr = tmem + lane_off + 128u * t;
        const uint32_t tOr = tmem + lane_off + C::kOCol + D * t;
        float m_run = -INFINITY;  // running max, base-2 scaled units
        float l_run = 0.f;        // running sum of 2^(s*scale_log2 - m_run)
        bool ok = true;
        for (int j = 0; j < ntile[t]; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kSFull + t), j & 1, wc, kSiteSoftS));
            if (!ok) break;
            tc_fence_after();
            // mask: causal (key > query) and keys past N in the last tile
            const int kv0 = j * kTileRows;
            const int lim = min(causal ? row_g - kv0 : kTileRows - 1, N - 1 - kv0);
            // the whole row of S in registers, masked
            uint32_t sr[128];
            tmem_ld_x128(tSr, sr);
            if (lim < kTileRows - 1) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > lim) sr[c] = __float_as_uint(-INFINITY);
            }
            // Row max of the scaled scores (base-2 units): four chains of three-input max.
            auto row_max = [&]() -> float {
                float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 8) {
                    mx0 = max3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                    mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                    mx2 = max3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
                    mx3 = max3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
                }
                return fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
            };
            const float2 sl2 = make_float2(scale_log2, scale_log2);
            float alpha = 1.f;
            bool upd = false;
            float sum0, sum1;
            if constexpr (C::kTF32) {
                const float mx = row_max();
                upd = mx > m_run + kRescaleThreshold;
                if (upd) {
                    alpha = ex2(m_run - mx);
                    m_run = mx;
                }
                const float neg = (m_run == -INFINITY) ? 0.f : -m_run;
                const float2 ng2 = make_float2(neg, neg);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 128; c += 2) {
                    const float2 x = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2, ng2);
                    const float2 p = make_float2(ex2(x.x), ex2(x.y));
                    if ((c >> 1) & 1) acc1 = add2(acc1, p); else acc0 = add2(acc0, p);
                    sr[c] = __float_as_uint(p.x);
                    sr[c + 1] = __float_as_uint(p.y);
                }
                tmem_st_x128(tSr, sr);
                const float2 accs = add2(acc0, acc1);
                sum0 = accs.x;
                sum1 = accs.y;
            } else {
                // P = 2^(s * scale_log2 - m) as packed bf16, with paired FFMA and sums.
                uint32_t pk[64];
                auto exp_pass = [&](float m) -> float {
                    const float neg = (m == -INFINITY) ? 0.f : -m;
                    const float2 ng2 = make_float2(neg, neg);
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int u = 0; u < 64; ++u) {
                        const float2 x =
                            fma2(make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])), sl2, ng2);
                        const float2 p = make_float2(ex2(x.x), ex2(x.y));
                        if (u & 1) acc1 = add2(acc1, p); else acc0 = add2(acc0, p);
                        pk[u] = pack_bf16(p.x, p.y);
                    }
                    const float2 accs = add2(acc0, acc1);
                    return accs.x + accs.y;
                };
                // The row max first; the running max moves (and O is rescaled) only when the
                // row max exceeds it by more than the threshold (lazy rescale).
                const float mx = row_max();
                upd = mx > m_run + (m_run == -INFINITY ? 0.f : kRescaleThreshold);
                if (upd) {
                    alpha = ex2(m_run - mx);
                    m_run = mx;
                }
                const float blk = exp_pass(m_run);
                tmem_st_x64(tSr, pk);
                sum0 = blk;
                sum1 = 0.f;
            }
            l_run = l_run * alpha + (sum0 + sum1);
            if (j > 0 && __any_sync(0xffffffffu, upd)) {
                // O still holds sum_{j' < j} P V relative to the old max: rescale it once
                // the previous P V product has landed.
                ok = __all_sync(0xffffffffu, mbar_wait(bar(B::kODone + t), (j - 1) & 1, wc, kSiteSoftO));
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
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(B::kODone + t), (ntile[t] - 1) & 1, wc, kSiteEpiO));
            if (ok) {
                tc_fence_after();
                const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
                const bool valid = row_g < N;
                T *orow = out + (static_cast<int64_t>(bh) * N + (valid ? row_g : 0)) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld_x32(tOr + 32u * c, o);
                    if (valid) {
                        if constexpr (C::kTF32) {
                            float4 *dst = reinterpret_cast<float4 *>(orow + 32 * c);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l,
                                                     __uint_as_float(o[4 * i + 1]) * inv_l,
                                                     __uint_as_float(o[4 * i + 2]) * inv_l,
                                                     __uint_as_float(o[4 * i + 3]) * inv_l);
                        } else {
                            uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint4 w;
                                w.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l);
                                w.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l);
                                w.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l);
                                w.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l);
                                dst[i] = w;
                            }
                        }
                    }
                }
                if (valid)
                    lse[static_cast<int64_t>(bh) * N + row_g] =
                        l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
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

template <typename T, int D, int QT>
cudaError_t launch_fwd_t(const FwdArgs &a, cudaStream_t stream) {
    using C = FwdCfg<T, D, QT>;
    auto kern = fwd_kernel<T, D, QT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int group_rows = QT * kTileRows;
    const int num_groups = (a.N + group_rows - 1) / group_rows;
    const long long blocks = static_cast<long long>(a.BH) * num_groups;
    if (blocks <= 0 || blocks > INT_MAX) return cudaErrorInvalidValue;
    const float scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    kern<<<static_cast<unsigned>(blocks), C::kThreads, C::kSmemBytes, stream>>>(
        a.tm_q, a.tm_k, a.tm_v, static_cast<T *>(a.o), a.lse, a.N, num_groups, a.group, scale_log2,
        a.causal, a.status);
    return cudaGetLastError();
}

// bf16 tile policy (measured on GB300): two query tiles per CTA (for causal work the
// pair 2g, 2g+1 has nearly equal cost), except non-causal work at d = 64, where one tile
// per CTA and two CTAs per SM (each tile with its own MMA-issuing thread) is faster.
template <int D>
cudaError_t launch_fwd_bf16_d(const FwdArgs &a, cudaStream_t stream) {
    if constexpr (D == 64) {
        if (!a.causal) return launch_fwd_t<__nv_bfloat16, D, 1>(a, stream);
    }
    return launch_fwd_t<__nv_bfloat16, D, 2>(a, stream);
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdArgs &a, cudaStream_t stream) {
    if (a.d == 64) return launch_fwd_bf16_d<64>(a, stream);
    if (a.d == 128) return launch_fwd_bf16_d<128>(a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t stream) {
    if (a.d == 64) return launch_fwd_t<float, 64, 2>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
