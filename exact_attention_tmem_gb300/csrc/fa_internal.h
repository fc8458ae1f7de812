// fa_internal.h — host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Per-launch description of one [BH, N, d] problem, filled by the ABI layer after
// argument checks.  Tensor maps view a [BH, N, d] tensor as 3-D (d innermost, then
// N, then BH) so that rows past N read as zeros and are never written.
struct FwdArgs {
    CUtensorMap tm_q, tm_k, tm_v;
    void *o;
    float *lse;
    int N, BH, d;
    int group;             // query heads per key/value head (1: plain multi-head attention)
    float scale;
    int causal;
    unsigned int *status;  // device status word
};

struct BwdArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    CUtensorMap tm_dq;  // the fp32 dQ accumulator, boxes of 32 columns x 128 rows
    const void *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    float *dq_acc;      // workspace: [BH, N, d] fp32 (null for the deterministic backward)
    float *delta;       // workspace: [BH, Npad] fp32, D = rowsum(dO o O)
    float *lse2;        // workspace: [BH, Npad] fp32, negated logsumexp in base 2 (-inf on padding rows)
    int N, Npad, BH, d;   // BH counts query heads
    int group;            // query heads per key/value head; B*H/group key/value heads
    float scale;
    int causal;
    int deterministic;    // 1: dQ from the query-block kernel (one writer per row), no accumulator
    unsigned int *status;
};

constexpr int kDecodeBoxRows = 64;    // keys per stage of the tensor-core decoding kernel
constexpr int kDecodeMmaMinGroup = 2; // query heads per key/value head from which decoding uses it
constexpr int kDecodeMaxGroup = 16;   // the tensor-core kernel's M dimension
constexpr int kDecodeMaxChunks = 256; // key chunks per head at most (the merge kernel's table)

// Decoding: one query row per head ([B*H, d]) against K, V [B*Hkv, Nk, d]; the keys of
// each key/value head are split into num_chunks chunks of chunk_keys keys (a multiple
// of 64), whose partial (m, l, acc) triples land in the workspace before the merge.
struct DecodeArgs {
    CUtensorMap tm_k, tm_v;   // [B*Hkv, Nk, d] with 64-row boxes (the tensor-core kernel)
    const void *q, *k, *v;
    void *o;
    float *lse;
    float *part_m, *part_l, *part_acc;   // workspace: [B*H, max_chunks] (+ [.., d] for acc)
    int BHkv, group, Nk, d;
    int chunk_keys, num_chunks, max_chunks;
    float scale;
    unsigned int *status;
};

// FP8 forward: Q and K codes [B*H|B*Hkv, N, d] e4m3, V codes transposed [B*Hkv, d, Npad],
// per-head descale factors; O bf16, L fp32.
struct Fp8FwdArgs {
    CUtensorMap tm_q, tm_k, tm_vt;
    const float *dsc_q, *dsc_k, *dsc_v;
    void *o;
    float *lse;
    int N, BH, d, group;
    float scale;
    int causal;
    unsigned int *status;
};

// Kernel launchers (fa_fwd.cu, fa_bwd.cu, fa_decode.cu, fa_fp8.cu).  They return the launch's cudaError_t.
cudaError_t launch_fwd_bf16(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_fwd_f32(const FwdArgs &a, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const BwdArgs &a, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t stream);
// Query heads per CTA of the decoding kernel for a group of `group` query heads per
// key/value head (groups above 4 are split when 4 or 3 divides them), and the CTAs of
// that kernel resident per SM (occupancy).
int decode_subgroup(int group);
cudaError_t decode_ctas_per_sm(int d, int group, int *out);
cudaError_t launch_fwd_fp8(const Fp8FwdArgs &a, cudaStream_t stream);
// descale doubles as the per-head amax scratch while the kernels run
cudaError_t launch_quantize_qk_fp8(const void *x, const float *signs, void *x8, float *descale, int BH, int N,
                                   int d, cudaStream_t stream);
cudaError_t launch_quantize_v_fp8(const void *v, void *vt8, float *descale, int BH, int N, int Npad, int d,
                                  cudaStream_t stream);

// Records a failed CUDA call for fa_last_cuda_error() (this thread) and returns FA_ERR_CUDA
// (fa_api.cu).
int record_cuda_error(cudaError_t e);

// Tile geometry shared by host and device code.
constexpr int kTileRows = 128;     // rows of Q, K, V per tile
constexpr int kBoxBytes = 128;     // inner extent of one TMA box (the 128-byte swizzle span)

}  // namespace fa
