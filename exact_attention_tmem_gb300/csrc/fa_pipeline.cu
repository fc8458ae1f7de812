// fa_pipeline.cu — fa_fwd_bwd_host: one training step of attention (forward, then
// backward) on inputs that live in host memory, with the host<->device copies
// overlapped with the kernels.
//
// Every (batch, head) pair is an independent problem ("FlashAttention" deep dive,
// section "How it works": Q, K, V of one head in, O and L of that head out, no state
// between calls), so the B*H heads are cut into chunks of consecutive heads and each
// chunk goes through three stages:
//   copy-in  stream: q, k, v, then dO of chunk c      host -> slot c % kSlots
//   compute  stream: fa_fwd once q, k, v have landed, fa_bwd once dO has; even chunks
//                    run on the caller's stream, odd ones on an internal stream
//   copy-out stream: o, lse of chunk c once its forward is done, then dq, dk, dv once
//                    its backward is                  slot -> host
// The copy-in of chunk c waits until the copy-out of chunk c - kSlots has drained the
// slot it reuses.  With three slots the copies of chunks c + 1 and c - 1 run while the
// kernels of chunk c do, and the kernels of two consecutive chunks may share the GPU
// where one leaves SMs idle (the tail of a launch).  Splitting each chunk's copies at
// the forward/backward boundary lets the forward start before dO has landed and o, L
// leave before the backward ends, which shortens the parts of the step (the first
// copy-in, the last copy-out) that nothing overlaps.  The device buffer (the slots)
// belongs to the caller; the internal streams and the events are created once per
// device and reused.
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kSlots = 3;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte layout of one slot for chunks of `hc` heads.
struct SlotLayout {
    size_t tensor = 0;   // one [hc, N, d] bf16 tensor
    size_t lse = 0;      // [hc, N] fp32
    size_t ws = 0;       // fa_bwd workspace of the chunk
    size_t bytes = 0;    // whole slot
    // offsets: q k v dO o dq dk dv (8 tensors), then lse, then workspace
    size_t tensor_off(int t) const { return static_cast<size_t>(t) * tensor; }
    size_t lse_off() const { return 8 * tensor; }
    size_t ws_off() const { return 8 * tensor + lse; }
};

bool slot_layout(int hc, int N, int d, SlotLayout *L) {
    const size_t ws = fa_bwd_workspace_size(1, hc, N, d);
    if (ws == 0) return false;
    L->tensor = round_up(static_cast<size_t>(hc) * N * d * 2);
    L->lse = round_up(static_cast<size_t>(hc) * N * 4);
    L->ws = round_up(ws);
    L->bytes = 8 * L->tensor + L->lse + L->ws;
    return true;
}

int resolve_chunk(int BH, int chunk_heads) {
    if (chunk_heads <= 0) chunk_heads = (BH + 15) / 16;   // about sixteen chunks
    return chunk_heads > BH ? BH : chunk_heads;
}

struct PipeState {
    bool ready = false;
    cudaStream_t copy_in = nullptr, copy_out = nullptr, compute = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    // per slot: q, k, v landed | dO landed | forward done | backward done | outputs copied
    cudaEvent_t h2d_fwd[kSlots] = {}, h2d_bwd[kSlots] = {}, fwd[kSlots] = {}, comp[kSlots] = {}, d2h[kSlots] = {};
};
PipeState g_pipe[kMaxDevices];
std::mutex g_pipe_mu;   // held for the whole enqueue: the events are shared per device

int pipe_state(PipeState **out, int *cuda_err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { *cuda_err = e; return FA_ERR_CUDA; }
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    PipeState &s = g_pipe[dev];
    if (!s.ready) {
        const unsigned ev_flags = cudaEventDisableTiming;
        e = cudaStreamCreateWithFlags(&s.copy_in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.copy_out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&s.compute, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.start, ev_flags);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.done, ev_flags);
        for (int i = 0; i < kSlots && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&s.h2d_fwd[i], ev_flags);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.h2d_bwd[i], ev_flags);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fwd[i], ev_flags);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.comp[i], ev_flags);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.d2h[i], ev_flags);
        }
        if (e != cudaSuccess) {   // release what was created; the next call starts over
            *cuda_err = e;
            for (int i = 0; i < kSlots; ++i) {
                for (cudaEvent_t ev : {s.h2d_fwd[i], s.h2d_bwd[i], s.fwd[i], s.comp[i], s.d2h[i]})
                    if (ev) cudaEventDestroy(ev);
            }
            if (s.start) cudaEventDestroy(s.start);
            if (s.done) cudaEventDestroy(s.done);
            if (s.copy_in) cudaStreamDestroy(s.copy_in);
            if (s.copy_out) cudaStreamDestroy(s.copy_out);
            if (s.compute) cudaStreamDestroy(s.compute);
            s = PipeState();
            return FA_ERR_CUDA;
        }
        s.ready = true;
    }
    *out = &s;
    return FA_OK;
}

}  // namespace

extern "C" size_t fa_fwd_bwd_host_buffer_size(int B, int H, int N, int d, int chunk_heads) {
    if (B < 1 || H < 1 || N < 1) return 0;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > INT_MAX) return 0;
    SlotLayout L;
    if (!slot_layout(resolve_chunk(static_cast<int>(bh), chunk_heads), N, d, &L)) return 0;
    return kSlots * L.bytes;
}

extern "C" int fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout, void *o, float *lse,
                               void *dq, void *dk, void *dv, void *dev_buf, size_t dev_buf_bytes, int B, int H,
                               int N, int d, float scale, int causal, int chunk_heads, fa_stream_t stream) {
    if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || static_cast<long long>(B) * H > INT_MAX) return FA_ERR_INVALID_ARG;
    const int BH = B * H;
    const int hc = resolve_chunk(BH, chunk_heads);
    SlotLayout L;
    if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (!slot_layout(hc, N, d, &L)) return (d == 64 || d == 128) ? FA_ERR_INVALID_ARG : FA_ERR_UNSUPPORTED;
    if (dev_buf == nullptr || dev_buf_bytes < kSlots * L.bytes) return FA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(dev_buf) & (kAlign - 1)) != 0) return FA_ERR_ALIGNMENT;

    std::lock_guard<std::mutex> lock(g_pipe_mu);
    PipeState *ps = nullptr;
    int cerr = 0;
    int st = pipe_state(&ps, &cerr);
    if (st == FA_ERR_CUDA) return fa::record_cuda_error(static_cast<cudaError_t>(cerr));
    if (st != FA_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    auto fail = [](cudaError_t e) { return fa::record_cuda_error(e); };
    cudaError_t e;
    // the copies may not start before earlier work on the caller's stream
    if ((e = cudaEventRecord(ps->start, cs)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(ps->copy_in, ps->start, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(ps->copy_out, ps->start, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(ps->compute, ps->start, 0)) != cudaSuccess) return fail(e);

    const size_t head_bytes = static_cast<size_t>(N) * d * 2;   // one head of a bf16 tensor
    const size_t head_lse = static_cast<size_t>(N) * 4;
    const void *in_host[4] = {q, k, v, dout};
    void *out_host[4] = {o, dq, dk, dv};
    const size_t ws_bytes = L.ws;
    uint8_t *base = static_cast<uint8_t *>(dev_buf);
    const int nchunks = (BH + hc - 1) / hc;
    for (int c = 0; c < nchunks; ++c) {
        const int s = c % kSlots;
        const int h0 = c * hc;
        const int n = BH - h0 < hc ? BH - h0 : hc;
        uint8_t *slot = base + static_cast<size_t>(s) * L.bytes;
        void *t[8];
        for (int i = 0; i < 8; ++i) t[i] = slot + L.tensor_off(i);   // q k v dO o dq dk dv
        float *lse_d = reinterpret_cast<float *>(slot + L.lse_off());
        void *ws = slot + L.ws_off();
        const size_t bytes = static_cast<size_t>(n) * head_bytes, off = static_cast<size_t>(h0) * head_bytes;
        // copy-in: the slot is free once the copy-out of chunk c - kSlots has read it;
        // q, k, v first (the forward's inputs), then dO (the backward's)
        if (c >= kSlots && (e = cudaStreamWaitEvent(ps->copy_in, ps->d2h[s], 0)) != cudaSuccess) return fail(e);
        for (int i = 0; i < 4; ++i) {
            e = cudaMemcpyAsync(t[i], static_cast<const uint8_t *>(in_host[i]) + off, bytes, cudaMemcpyHostToDevice,
                                ps->copy_in);
            if (e != cudaSuccess) return fail(e);
            if (i == 2 && (e = cudaEventRecord(ps->h2d_fwd[s], ps->copy_in)) != cudaSuccess) return fail(e);
        }
        if ((e = cudaEventRecord(ps->h2d_bwd[s], ps->copy_in)) != cudaSuccess) return fail(e);
        // kernels: even chunks on the caller's stream, odd chunks on the internal compute
        // stream, so that one chunk's kernels can fill the SMs the other's leave idle
        const cudaStream_t ks = (c & 1) ? ps->compute : cs;
        const fa_stream_t kss = reinterpret_cast<fa_stream_t>(ks);
        if ((e = cudaStreamWaitEvent(ks, ps->h2d_fwd[s], 0)) != cudaSuccess) return fail(e);
        st = fa_fwd(t[0], t[1], t[2], t[4], lse_d, 1, n, N, d, scale, causal, kss);
        if (st != FA_OK) return st;
        if ((e = cudaEventRecord(ps->fwd[s], ks)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(ks, ps->h2d_bwd[s], 0)) != cudaSuccess) return fail(e);
        st = fa_bwd(t[0], t[1], t[2], t[4], lse_d, t[3], t[5], t[6], t[7], ws, ws_bytes, 1, n, N, d, scale, causal,
                    kss);
        if (st != FA_OK) return st;
        if ((e = cudaEventRecord(ps->comp[s], ks)) != cudaSuccess) return fail(e);
        // copy-out: o and lse once the forward is done (the backward only reads o), then
        // dq, dk, dv
        if ((e = cudaStreamWaitEvent(ps->copy_out, ps->fwd[s], 0)) != cudaSuccess) return fail(e);
        e = cudaMemcpyAsync(static_cast<uint8_t *>(o) + off, t[4], bytes, cudaMemcpyDeviceToHost, ps->copy_out);
        if (e != cudaSuccess) return fail(e);
        e = cudaMemcpyAsync(reinterpret_cast<uint8_t *>(lse) + static_cast<size_t>(h0) * head_lse, lse_d, n * head_lse,
                            cudaMemcpyDeviceToHost, ps->copy_out);
        if (e != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(ps->copy_out, ps->comp[s], 0)) != cudaSuccess) return fail(e);
        for (int i = 5; i < 8; ++i) {   // dq dk dv
            e = cudaMemcpyAsync(static_cast<uint8_t *>(out_host[i - 4]) + off, t[i], bytes, cudaMemcpyDeviceToHost,
                                ps->copy_out);
            if (e != cudaSuccess) return fail(e);
        }
        if ((e = cudaEventRecord(ps->d2h[s], ps->copy_out)) != cudaSuccess) return fail(e);
    }
    // the caller's stream continues once every result is in host memory
    if ((e = cudaEventRecord(ps->done, ps->copy_out)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, ps->done, 0)) != cudaSuccess) return fail(e);
    return FA_OK;
}
