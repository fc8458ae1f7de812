// fa_api.cu — the C ABI declared in include/fa.h: argument checks, tensor-map
// encoding, the device status word, and dispatch to the kernel launchers.
//
// Every check that needs no GPU runs first, so that argument errors are reported
// identically on a machine without one.  Nothing here allocates device memory
// or synchronises a stream (fa_get_device_status excepted, by contract).
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

// The device status word.  One copy per device (module-scope variable); kernels
// receive its address.
__device__ unsigned int g_status_word[2];

thread_local int t_last_cuda_error = 0;

// One warp waits on an mbarrier that nothing ever arrives at.  The bounded wait gives
// up after its time limit, raises the abort flag and records the timeout in the device
// status word; the kernel then returns normally, leaving the context usable.
__global__ void wait_selftest_kernel(unsigned int *status) {
    __shared__ __align__(8) unsigned long long barrier;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&barrier);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    const WaitCtx wc{&abort_flag, status};
    mbar_wait(bar, 0, wc, /*site=*/1);
}

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return FA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Shape checks shared by every entry point.  Products are formed in 64 bits.
int check_shape(int B, int H, int N, int d, int Hkv) {
    if (B < 1 || H < 1 || N < 1 || d < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > INT_MAX) return FA_ERR_INVALID_ARG;
    const long long elems = bh * N;
    if (elems > (1LL << 62) / d) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// ---- per-device state: the status word's address and the compute capability ----
constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned int *status = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        s.supported = (major == 10 && minor == 3);
        e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        if (s.supported) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_status_word);
            if (e != cudaSuccess) return cuda_fail(e);
            s.status = static_cast<unsigned int *>(p);
        }
        s.ready = true;
    }
    if (!s.supported) return FA_ERR_UNSUPPORTED;
    *out = &s;
    return FA_OK;
}

// ---- tensor maps ----
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiledFn *fn) {
    static EncodeTiledFn cached = nullptr;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q != cudaDriverEntryPointSuccess) err = cudaErrorSymbolNotFound;
        if (err == cudaSuccess) cached = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (cached == nullptr) return cuda_fail(err != cudaSuccess ? err : cudaErrorSymbolNotFound);
    *fn = cached;
    return FA_OK;
}

// [BH, N, d] viewed as 3-D: d innermost, then N, then BH.  One box is 128 bytes of a
// row by 128 rows, 128-byte swizzled (the layout the MMA descriptors expect).
int make_tmap(CUtensorMap *m, const void *ptr, CUtensorMapDataType dt, int eb, int d, int N, int BH,
              int rows = kTileRows) {
    EncodeTiledFn enc;
    int st = get_encoder(&enc);
    if (st != FA_OK) return st;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * eb, static_cast<cuuint64_t>(d) * eb * N};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kBoxBytes / eb), static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return FA_OK;
}

int fwd_common(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv,
               int N, int d, float scale, int causal, cudaStream_t stream, bool f32) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, N, d, Hkv);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (f32 && d != 64) return FA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
        return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    FwdArgs a;
    std::memset(&a, 0, sizeof(a));
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int eb = f32 ? 4 : 2;
    const int BH = B * H, BHkv = B * Hkv;
    if ((st = make_tmap(&a.tm_q, q, dt, eb, d, N, BH)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_k, k, dt, eb, d, N, BHkv)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_v, v, dt, eb, d, N, BHkv)) != FA_OK) return st;
    a.o = o;
    a.lse = lse;
    a.N = N;
    a.BH = BH;
    a.d = d;
    a.group = H / Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.status = ds->status;
    cudaError_t e = f32 ? launch_fwd_f32(a, stream) : launch_fwd_bf16(a, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

namespace fa {
int record_cuda_error(cudaError_t e) { return cuda_fail(e); }
}  // namespace fa

extern "C" int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N,
                      int d, float scale, int causal, fa_stream_t stream) {
    return fwd_common(q, k, v, o, lse, B, H, H, N, d, scale, causal, reinterpret_cast<cudaStream_t>(stream),
                      false);
}

extern "C" int fa_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                          int Hkv, int N, int d, float scale, int causal, fa_stream_t stream) {
    return fwd_common(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, reinterpret_cast<cudaStream_t>(stream),
                      false);
}

extern "C" int fa_fwd_f32(const float *q, const float *k, const float *v, float *o, float *lse, int B, int H,
                          int N, int d, float scale, int causal, fa_stream_t stream) {
    return fwd_common(q, k, v, o, lse, B, H, H, N, d, scale, causal, reinterpret_cast<cudaStream_t>(stream),
                      true);
}

extern "C" size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (check_shape(B, H, N, d, H) != FA_OK) return 0;
    const size_t bh = static_cast<size_t>(B) * H;
    const size_t npad = (static_cast<size_t>(N) + kTileRows - 1) / kTileRows * kTileRows;
    const size_t acc = bh * static_cast<size_t>(N) * d * sizeof(float);
    const size_t acc_aligned = (acc + 255) / 256 * 256;
    const size_t vec = (bh * npad * sizeof(float) + 255) / 256 * 256;
    return acc_aligned + 2 * vec;
}

extern "C" size_t fa_bwd_deterministic_workspace_size(int B, int H, int N, int d) {
    if (check_shape(B, H, N, d, H) != FA_OK) return 0;
    const size_t bh = static_cast<size_t>(B) * H;
    const size_t npad = (static_cast<size_t>(N) + kTileRows - 1) / kTileRows * kTileRows;
    const size_t vec = (bh * npad * sizeof(float) + 255) / 256 * 256;
    return 2 * vec;
}

namespace fa {
namespace {
int bwd_common(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
               void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes, int B, int H, int Hkv,
               int N, int d, float scale, int causal, bool deterministic, fa_stream_t stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, N, d, Hkv);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse) ||
        !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
        return FA_ERR_ALIGNMENT;
    const size_t need = deterministic ? fa_bwd_deterministic_workspace_size(B, H, N, d)
                                      : fa_bwd_workspace_size(B, H, N, d);
    if (workspace == nullptr || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    BwdArgs a;
    std::memset(&a, 0, sizeof(a));
    const int BH = B * H, BHkv = B * Hkv;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if ((st = make_tmap(&a.tm_q, q, dt, 2, d, N, BH)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_k, k, dt, 2, d, N, BHkv)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_v, v, dt, 2, d, N, BHkv)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_do, dout, dt, 2, d, N, BH)) != FA_OK) return st;
    const size_t npad = (static_cast<size_t>(N) + kTileRows - 1) / kTileRows * kTileRows;
    const size_t acc = static_cast<size_t>(BH) * N * d * sizeof(float);
    // the deterministic backward keeps no dQ accumulator: the workspace holds only D and L2
    const size_t acc_aligned = deterministic ? 0 : (acc + 255) / 256 * 256;
    const size_t vec = (static_cast<size_t>(BH) * npad * sizeof(float) + 255) / 256 * 256;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (!deterministic &&
        (st = make_tmap(&a.tm_dq, ws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, N, BH)) != FA_OK)
        return st;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dq_acc = deterministic ? nullptr : reinterpret_cast<float *>(ws);
    a.delta = reinterpret_cast<float *>(ws + acc_aligned);
    a.lse2 = reinterpret_cast<float *>(ws + acc_aligned + vec);
    a.N = N;
    a.Npad = static_cast<int>(npad);
    a.BH = BH;
    a.d = d;
    a.group = H / Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.deterministic = deterministic ? 1 : 0;
    a.status = ds->status;
    cudaError_t e = launch_bwd_bf16(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}
}  // namespace
}  // namespace fa

extern "C" int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                      const void *dout, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                      int B, int H, int N, int d, float scale, int causal, fa_stream_t stream) {
    return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, H, N, d, scale, causal,
                      false, stream);
}

extern "C" int fa_bwd_gqa(const void *q, const void *k, const void *v, const void *o, const float *lse,
                          const void *dout, void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                          int B, int H, int Hkv, int N, int d, float scale, int causal, fa_stream_t stream) {
    return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal,
                      false, stream);
}

extern "C" int fa_bwd_deterministic(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                    const void *dout, void *dq, void *dk, void *dv, void *workspace,
                                    size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
                                    int causal, fa_stream_t stream) {
    return bwd_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, scale, causal,
                      true, stream);
}

namespace fa {
namespace {
// Decoding: key chunks are whole 64-key stages; at most kDecodeMaxChunks per head.
constexpr int kDecodeChunkAlign = 64;

int decode_max_chunks(int Nk) {
    const int stages = (Nk + kDecodeChunkAlign - 1) / kDecodeChunkAlign;
    return stages < kDecodeMaxChunks ? stages : kDecodeMaxChunks;
}

int check_decode(int B, int H, int Hkv, int Nk, int d) {
    int st = check_shape(B, H, Nk, d, Hkv);
    if (st != FA_OK) return st;
    if (H / Hkv > kDecodeMaxGroup) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

size_t decode_workspace(int B, int H, int Nk, int d) {
    const size_t slots = static_cast<size_t>(B) * H * decode_max_chunks(Nk);
    const size_t vec = (slots * sizeof(float) + 255) / 256 * 256;
    return 2 * vec + slots * d * sizeof(float);
}
}  // namespace
}  // namespace fa

extern "C" size_t fa_decode_workspace_size(int B, int H, int Hkv, int Nk, int d) {
    if (check_decode(B, H, Hkv, Nk, d) != FA_OK) return 0;
    return decode_workspace(B, H, Nk, d);
}

extern "C" int fa_decode(const void *q, const void *k, const void *v, void *o, float *lse, void *workspace,
                         size_t workspace_bytes, int B, int H, int Hkv, int Nk, int d, float scale,
                         int num_chunks, fa_stream_t stream) {
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    int st = check_decode(B, H, Hkv, Nk, d);
    if (st != FA_OK) return st;
    if (!std::isfinite(scale) || num_chunks < 0) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned4(lse))
        return FA_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < decode_workspace(B, H, Nk, d)) return FA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    const int max_chunks = decode_max_chunks(Nk);
    const int BHkv = B * Hkv;
    const int stages = (Nk + kDecodeChunkAlign - 1) / kDecodeChunkAlign;
    int want = num_chunks;
    if (want == 0) {
        // Fill every CTA slot and keep the last wave full.  A CTA's time is about its
        // number of 64-key stages, so the kernel takes about waves x stages per chunk;
        // take the chunk count (up to 8 x the fewest that fill the slots) that
        // minimises it, the fewest chunks on a tie.
        int per_sm = 2;
        cudaError_t oe = decode_ctas_per_sm(d, H / Hkv, &per_sm);
        if (oe != cudaSuccess) return cuda_fail(oe);
        const long long slots = static_cast<long long>(per_sm > 0 ? per_sm : 1) * (ds->sm_count > 0 ? ds->sm_count : 1);
        const long long units = static_cast<long long>(BHkv) * (H / Hkv / decode_subgroup(H / Hkv));
        const long long w0 = std::min<long long>(std::max<long long>((slots + units - 1) / units, 1), max_chunks);
        long long best_cost = LLONG_MAX;
        for (long long w = w0; w <= std::min<long long>(8 * w0, max_chunks); ++w) {
            const long long cs = (stages + w - 1) / w;
            const long long n = (stages + cs - 1) / cs;
            const long long ctas = static_cast<long long>(BHkv) * (H / Hkv / decode_subgroup(H / Hkv)) * n;
            const long long waves = (ctas + slots - 1) / slots;
            const long long cost = waves * cs;
            if (cost < best_cost) {
                best_cost = cost;
                want = static_cast<int>(w);
            }
        }
    }
    if (want < 1) want = 1;
    if (want > max_chunks) want = max_chunks;
    const int chunk_stages = (stages + want - 1) / want;
    DecodeArgs a;
    std::memset(&a, 0, sizeof(a));
    if ((st = make_tmap(&a.tm_k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, Nk, BHkv, kDecodeBoxRows)) != FA_OK)
        return st;
    if ((st = make_tmap(&a.tm_v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, Nk, BHkv, kDecodeBoxRows)) != FA_OK)
        return st;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    const size_t slots = static_cast<size_t>(B) * H * max_chunks;
    const size_t vec = (slots * sizeof(float) + 255) / 256 * 256;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.part_m = reinterpret_cast<float *>(ws);
    a.part_l = reinterpret_cast<float *>(ws + vec);
    a.part_acc = reinterpret_cast<float *>(ws + 2 * vec);
    a.BHkv = BHkv;
    a.group = H / Hkv;
    a.Nk = Nk;
    a.d = d;
    a.chunk_keys = chunk_stages * kDecodeChunkAlign;
    a.num_chunks = (Nk + a.chunk_keys - 1) / a.chunk_keys;
    a.max_chunks = max_chunks;
    a.scale = scale;
    a.status = ds->status;
    cudaError_t e = launch_decode_bf16(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

// ---- FP8 forward and its quantization ----
namespace fa {
namespace {
size_t fp8_npad(int N) { return (static_cast<size_t>(N) + 15) / 16 * 16; }
}  // namespace
}  // namespace fa

extern "C" size_t fa_fp8_v_bytes(int B, int H, int N, int d) {
    if (check_shape(B, H, N, d, H) != FA_OK) return 0;
    return static_cast<size_t>(B) * H * d * fp8_npad(N);
}

extern "C" int fa_quantize_qk_fp8(const void *x, const float *signs, void *x8, float *descale, int B, int H, int N,
                                  int d, fa_stream_t stream) {
    if (!x || !x8 || !descale) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, N, d, H);
    if (st != FA_OK) return st;
    if (!aligned16(x) || !aligned16(x8) || !aligned4(descale) || (signs && !aligned4(signs))) return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    cudaError_t e = launch_quantize_qk_fp8(x, signs, x8, descale, B * H, N, d, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

extern "C" int fa_quantize_v_fp8(const void *v, void *vt8, float *descale, int B, int H, int N, int d,
                                 fa_stream_t stream) {
    if (!v || !vt8 || !descale) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, N, d, H);
    if (st != FA_OK) return st;
    if (!aligned16(v) || !aligned16(vt8) || !aligned4(descale)) return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    cudaError_t e = launch_quantize_v_fp8(v, vt8, descale, B * H, N, static_cast<int>(fp8_npad(N)), d,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

extern "C" int fa_fwd_fp8(const void *q8, const void *k8, const void *vt8, const float *descale_q,
                          const float *descale_k, const float *descale_v, void *o, float *lse, int B, int H, int Hkv,
                          int N, int d, float scale, int causal, fa_stream_t stream) {
    if (!q8 || !k8 || !vt8 || !descale_q || !descale_k || !descale_v || !o || !lse) return FA_ERR_INVALID_ARG;
    int st = check_shape(B, H, N, d, Hkv);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned4(lse) ||
        !aligned4(descale_q) || !aligned4(descale_k) || !aligned4(descale_v))
        return FA_ERR_ALIGNMENT;
    DeviceState *ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    Fp8FwdArgs a;
    std::memset(&a, 0, sizeof(a));
    const int BH = B * H, BHkv = B * Hkv;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if ((st = make_tmap(&a.tm_q, q8, u8, 1, d, N, BH)) != FA_OK) return st;
    if ((st = make_tmap(&a.tm_k, k8, u8, 1, d, N, BHkv)) != FA_OK) return st;
    // V codes [BHkv, d, Npad]: keys innermost, a box is 128 keys of 128 rows
    if ((st = make_tmap(&a.tm_vt, vt8, u8, 1, static_cast<int>(fp8_npad(N)), d, BHkv)) != FA_OK) return st;
    a.dsc_q = descale_q;
    a.dsc_k = descale_k;
    a.dsc_v = descale_v;
    a.o = o;
    a.lse = lse;
    a.N = N;
    a.BH = BH;
    a.d = d;
    a.group = H / Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.status = ds->status;
    cudaError_t e = launch_fwd_fp8(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

extern "C" int fa_get_device_status(fa_stream_t stream) {
    DeviceState *ds = nullptr;
    int st = device_state(&ds);
    if (st != FA_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int words[2] = {0, 0};
    e = cudaMemcpyFromSymbol(words, g_status_word, sizeof(words));
    if (e != cudaSuccess) return cuda_fail(e);
    if (words[0] != 0) {
        const unsigned int zero[2] = {0, 0};
        e = cudaMemcpyToSymbol(g_status_word, zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
        return FA_ERR_DEVICE_TIMEOUT;
    }
    return FA_OK;
}

extern "C" int fa_selftest_wait_timeout(fa_stream_t stream) {
    DeviceState *ds = nullptr;
    int st = device_state(&ds);
    if (st != FA_OK) return st;
    wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ds->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return FA_OK;
}

extern "C" const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument (null pointer, size < 1, size overflow or non-finite scale)";
        case FA_ERR_UNSUPPORTED: return "unsupported (head dim, dtype or device compute capability)";
        case FA_ERR_ALIGNMENT: return "pointer not aligned (16 bytes for tensors, 4 for lse, 256 for workspace)";
        case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_bwd_workspace_size()";
        case FA_ERR_CUDA: return "CUDA call failed (see fa_last_cuda_error)";
        case FA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out; outputs are undefined";
        default: return "unknown status";
    }
}

extern "C" int fa_last_cuda_error(void) { return t_last_cuda_error; }
