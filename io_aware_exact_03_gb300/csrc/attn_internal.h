// Internal interface between the C ABI (attn_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

enum Dtype : int { kBF16 = 0, kFP16 = 1, kE4M3 = 2, kFP32 = 3 };

// Device status bits, OR-ed into a per-kernel-file status word.
enum : unsigned { kStatusTimeout = 1u };

struct Problem {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;              // may be null
    const float* q_descale;  // [B*H] or null (unit) - e4m3 only
    const float* k_descale;
    const float* v_descale;
    int B, H, N_q, N_k, d;
    int H_kv;                // K/V heads (H for multi-head; H % H_kv == 0)
    float scale;
    int causal;
    int dtype;
    // Health check of the abort path only (attn_selftest_abort); 0 in normal
    // calls.  Every bounded wait then gives up after selftest_wait_ns, and the
    // K/V loader stops after selftest_items ring items.
    unsigned long long selftest_wait_ns = 0;
    int selftest_items = 0;
};

// Time limit of every bounded wait in a normal call; waits that only drain
// what a role already issued (on the abort path) always get at least this.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// CUDA-core kernel (attn_simt.cu).
cudaError_t launch_simt(const Problem& p, cudaStream_t stream);
cudaError_t simt_take_status(unsigned* out, cudaStream_t stream);

// Tensor-core kernel (attn_tc.cu).  Returns cudaErrorNotSupported for shapes
// it does not take.
cudaError_t launch_tc(const Problem& p, cudaStream_t stream);
cudaError_t tc_take_status(unsigned* out, cudaStream_t stream);

// Tensor-core kernel for head dimension 256 (attn_tc256.cu): one 128-row
// query tile per CTA.  n_splits > 1 writes fp32 partials as launch_tc_splitkv.
cudaError_t launch_tc256(const Problem& p, cudaStream_t stream, int n_splits, float* part_o,
                         float* part_lse);
cudaError_t tc256_take_status(unsigned* out, cudaStream_t stream);

// Backward pass (attn_bwd.cu): dq, dk, dv from q, k, v, o, lse, dO.
struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* o;
    const float* lse;
    const void* dO;
    void* dq;
    void* dk;
    void* dv;
    int B, H, N_q, N_k, d;
    int H_kv;         // K/V heads (H % H_kv == 0): dk, dv sum over the group's query heads
    float scale;
    int causal;
    int dtype;
    void* workspace;  // bwd_workspace_bytes(B, H, N_q), 16-byte aligned
};
size_t bwd_workspace_bytes(long long B, long long H, long long N_q);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream);
cudaError_t bwd_take_status(unsigned* out, cudaStream_t stream);

// Incoherent processing + per-head e4m3 quantisation (attn_quant.cu).
cudaError_t launch_quantize_e4m3(const void* x, int dtype, const float* signs, void* codes,
                                 float* descale, int B, int N, int H, int d, cudaStream_t stream);

// Bounded-wait health check (attn_tc.cu).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

// Remembers, per host thread, the CUDA error behind the last ATTN_ERR_CUDA
// (read back by attn_last_cuda_error).
void note_cuda_error(cudaError_t e);

// Split-KV on the tensor-core kernel plus the combine kernel (attn_tc.cu).
constexpr int kMaxSplits = 32;
// e4m3 forward whose V is first widened to fp16 in the caller's workspace
// (B * N_k * H_kv * d fp16 values; d = 64 or 128, else 0 bytes / unsupported).
size_t fp8_ws_workspace_bytes(long long B, long long H_kv, long long N_k, int d);
cudaError_t launch_tc_fp8_ws(const Problem& p, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream);
size_t splitkv_workspace_bytes(long long B, long long H, long long N_q, int d, int n_splits);
cudaError_t launch_tc_splitkv(const Problem& p, int n_splits, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

}  // namespace attn
