// Forward pass on host-resident tensors: the (batch, head) pairs are cut into
// chunks, and three internal activities run as a pipeline over a ring of
// device slots in the caller's workspace:
//
//   copy-in stream   : host -> device copy of chunk c + 1 (q, k, v rows of its
//                      heads, strided 2-D copies into a compact [N][heads][d] slot)
//   caller's stream  : the tensor-core kernel on chunk c (B = 1, H = its heads)
//   copy-out stream  : device -> host copy of chunk c - 1 (o rows, lse rows)
//
// Events order slot reuse: a slot is refilled only after its last copy-out
// has finished.  Each (batch, head) is computed exactly as in one call over
// the whole problem (heads are independent; the kernel's arithmetic does not
// depend on which other heads share the launch), so results are identical to
// attn_fwd / attn_fwd_fp8 on device copies of the same inputs.
//
// This is the runtime around the kernel for inputs that live in host memory
// (the pages' method is defined on device-resident Q, K, V; moving them is
// the caller's side of the "IO-aware" accounting on the "FlashAttention (HI)"
// page, section "Problems of standard attention": HBM traffic there, the
// host link here).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attn_gb300.h"
#include "attn_internal.h"

namespace {

constexpr int kSlots = 3;          // copy-in, compute and copy-out in flight at once
constexpr int kTargetChunks = 4;   // chunks per call when the heads allow it
constexpr int kMaxDevices = 64;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
    int hc = 0;            // heads per chunk (the last chunk of a batch row may have fewer)
    int groups = 0;        // chunks per batch row
    int n_chunks = 0;
    size_t q_bytes = 0, kv_bytes = 0, o_bytes = 0, lse_bytes = 0, ds_bytes = 0;
    size_t slot_bytes = 0;
    int slots = 0;
};

Plan make_plan(int B, int H, int N_q, int N_k, int d, int dtype) {
    Plan pl;
    const size_t e_in = dtype == attn::kE4M3 ? 1 : 2;
    const size_t per_head = ((size_t)N_q + 2 * (size_t)N_k) * d * e_in;
    const size_t total = (size_t)B * H * per_head;
    const size_t target = (total + kTargetChunks - 1) / kTargetChunks;
    size_t hc = per_head > 0 ? (target + per_head - 1) / per_head : (size_t)H;
    if (hc < 1) hc = 1;
    if (hc > (size_t)H) hc = H;
    pl.groups = (int)((H + hc - 1) / hc);
    pl.hc = (H + pl.groups - 1) / pl.groups;  // even the chunks out
    pl.n_chunks = B * pl.groups;
    pl.q_bytes = align256((size_t)N_q * pl.hc * d * e_in);
    pl.kv_bytes = align256((size_t)N_k * pl.hc * d * e_in);
    pl.o_bytes = align256((size_t)N_q * pl.hc * d * 2);
    pl.lse_bytes = align256((size_t)pl.hc * N_q * 4);
    pl.ds_bytes = dtype == attn::kE4M3 ? align256((size_t)3 * pl.hc * 4) : 0;
    pl.slot_bytes = pl.q_bytes + 2 * pl.kv_bytes + pl.o_bytes + pl.lse_bytes + pl.ds_bytes;
    pl.slots = pl.n_chunks < kSlots ? pl.n_chunks : kSlots;
    return pl;
}

// Internal streams and events, one set per device, made on first use and
// kept for the life of the process.  Enqueueing holds the set's mutex, so
// calls from several host threads on one device queue one after the other.
struct Pipes {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t filled[kSlots] = {}, computed[kSlots] = {}, drained[kSlots] = {};
    std::mutex mu;
};

Pipes g_pipes[kMaxDevices];

cudaError_t init_pipes(Pipes& p) {
    if (p.ready) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.end, cudaEventDisableTiming);
    for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&p.filled[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.computed[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.drained[s], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) p.ready = true;
    return e;
}

bool valid_dtype(int dtype) { return dtype == attn::kBF16 || dtype == attn::kFP16 || dtype == attn::kE4M3; }

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_bytes(int B, int H, int N_q, int N_k, int d, attn_dtype_t dtype) {
    if (B <= 0 || H <= 0 || N_q <= 0 || N_k < 0 || !valid_dtype((int)dtype)) return 0;
    if (d != 64 && d != 128 && d != 256) return 0;
    const Plan pl = make_plan(B, H, N_q, N_k, d, (int)dtype);
    return (size_t)pl.slots * pl.slot_bytes;
}

attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            const float* q_descale, const float* k_descale, const float* v_descale,
                            int B, int H, int N_q, int N_k, int d, float scale, int causal,
                            attn_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream) {
    const int dt = (int)dtype;
    if (B < 0 || H < 0 || N_q < 0 || N_k < 0 || !valid_dtype(dt)) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (N_q > ATTN_MAX_SEQ_LEN || N_k > ATTN_MAX_SEQ_LEN) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N_q == 0) return ATTN_OK;
    if (!q || !o || (N_k > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (dt == attn::kE4M3 && (!q_descale || !k_descale || !v_descale)) return ATTN_ERR_INVALID_ARG;
    const Plan pl = make_plan(B, H, N_q, N_k, d, dt);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0 ||
        workspace_bytes < (size_t)pl.slots * pl.slot_bytes)
        return ATTN_ERR_INVALID_ARG;

    int dev = 0;
    const cudaError_t eg = cudaGetDevice(&dev);
    if (eg != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        attn::note_cuda_error(eg != cudaSuccess ? eg : cudaErrorInvalidDevice);
        return ATTN_ERR_CUDA;
    }
    Pipes& P = g_pipes[dev];
    std::lock_guard<std::mutex> lock(P.mu);
    const cudaError_t ei = init_pipes(P);
    if (ei != cudaSuccess) {
        attn::note_cuda_error(ei);
        (void)cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    cudaStream_t us = static_cast<cudaStream_t>(stream);
    const size_t e_in = dt == attn::kE4M3 ? 1 : 2;
    const size_t row_in = (size_t)H * d * e_in;     // bytes of one token row (all heads), inputs
    const size_t row_out = (size_t)H * d * 2;       // the same for o
    const uint8_t* qh = static_cast<const uint8_t*>(q);
    const uint8_t* kh = static_cast<const uint8_t*>(k);
    const uint8_t* vh = static_cast<const uint8_t*>(v);
    uint8_t* oh = static_cast<uint8_t*>(o);
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    // everything starts after the work already queued on the caller's stream
    cudaError_t e = cudaEventRecord(P.start, us);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.in, P.start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.start, 0);
    attn_status_t st = ATTN_OK;
    for (int c = 0; c < pl.n_chunks && e == cudaSuccess && st == ATTN_OK; ++c) {
        const int b = c / pl.groups, h0 = (c % pl.groups) * pl.hc;
        const int nh = (H - h0) < pl.hc ? (H - h0) : pl.hc;
        const int slot = c % pl.slots;
        uint8_t* dq = ws + (size_t)slot * pl.slot_bytes;
        uint8_t* dk = dq + pl.q_bytes;
        uint8_t* dv = dk + pl.kv_bytes;
        uint8_t* dout = dv + pl.kv_bytes;
        float* dlse = reinterpret_cast<float*>(dout + pl.o_bytes);
        float* dds = reinterpret_cast<float*>(dout + pl.o_bytes + pl.lse_bytes);
        const size_t w_in = (size_t)nh * d * e_in, w_out = (size_t)nh * d * 2;
        // ---- copy in (after this slot's previous chunk has been copied out)
        if (c >= pl.slots) e = cudaStreamWaitEvent(P.in, P.drained[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dq, w_in, qh + ((size_t)b * N_q * H + h0) * d * e_in, row_in, w_in, N_q,
                                  cudaMemcpyHostToDevice, P.in);
        if (e == cudaSuccess && N_k > 0)
            e = cudaMemcpy2DAsync(dk, w_in, kh + ((size_t)b * N_k * H + h0) * d * e_in, row_in, w_in, N_k,
                                  cudaMemcpyHostToDevice, P.in);
        if (e == cudaSuccess && N_k > 0)
            e = cudaMemcpy2DAsync(dv, w_in, vh + ((size_t)b * N_k * H + h0) * d * e_in, row_in, w_in, N_k,
                                  cudaMemcpyHostToDevice, P.in);
        if (dt == attn::kE4M3) {
            const float* src[3] = {q_descale, k_descale, v_descale};
            for (int t = 0; t < 3 && e == cudaSuccess; ++t)
                e = cudaMemcpyAsync(dds + (size_t)t * pl.hc, src[t] + (size_t)b * H + h0, (size_t)nh * 4,
                                    cudaMemcpyHostToDevice, P.in);
        }
        if (e == cudaSuccess) e = cudaEventRecord(P.filled[slot], P.in);
        // ---- kernel on the caller's stream
        if (e == cudaSuccess) e = cudaStreamWaitEvent(us, P.filled[slot], 0);
        if (e != cudaSuccess) break;
        if (dt == attn::kE4M3)
            st = attn_fwd_fp8(dq, dk, dv, dout, dlse, dds, dds + pl.hc, dds + 2 * pl.hc, 1, nh, N_q, N_k, d, scale,
                              causal, us);
        else
            st = attn_fwd(dq, dk, dv, dout, dlse, 1, nh, N_q, N_k, d, scale, causal, dtype, us);
        if (st != ATTN_OK) break;
        e = cudaEventRecord(P.computed[slot], us);
        // ---- copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P.out, P.computed[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(oh + ((size_t)b * N_q * H + h0) * d * 2, row_out, dout, w_out, w_out, N_q,
                                  cudaMemcpyDeviceToHost, P.out);
        if (e == cudaSuccess && lse)
            e = cudaMemcpyAsync(lse + ((size_t)b * H + h0) * N_q, dlse, (size_t)nh * N_q * 4,
                                cudaMemcpyDeviceToHost, P.out);
        if (e == cudaSuccess) e = cudaEventRecord(P.drained[slot], P.out);
    }
    // Later work on the caller's stream waits for every copy this call
    // queued, in and out, also when the loop stopped early on an error (the
    // caller may free the buffers as soon as that work runs).  `start` has
    // been waited on already and is free to mark the copy-in tail.
    cudaError_t ej = cudaEventRecord(P.end, P.out);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(us, P.end, 0);
    if (ej == cudaSuccess) ej = cudaEventRecord(P.start, P.in);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(us, P.start, 0);
    if (e != cudaSuccess || ej != cudaSuccess) {
        attn::note_cuda_error(e != cudaSuccess ? e : ej);
        (void)cudaGetLastError();
        return ATTN_ERR_CUDA;
    }
    return st;
}

}  // extern "C"
