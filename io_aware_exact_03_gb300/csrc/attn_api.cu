// C ABI of the exact-attention forward pass (declared in include/attn_gb300.h).
// Validates arguments on the host, then enqueues one kernel on the caller's
// stream.  No device memory is allocated here.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_gb300.h"
#include "attn_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

attn_status_t validate(const attn::Problem& p) {
    if (p.B < 0 || p.H < 0 || p.N_q < 0 || p.N_k < 0) return ATTN_ERR_INVALID_ARG;
    if (!(p.scale > 0.f) || !isfinite(p.scale)) return ATTN_ERR_INVALID_ARG;
    if (p.dtype != attn::kBF16 && p.dtype != attn::kFP16 && p.dtype != attn::kE4M3)
        return ATTN_ERR_INVALID_ARG;
    if (p.d != 64 && p.d != 128 && p.d != 256) return ATTN_ERR_UNSUPPORTED;
    if (p.N_q > ATTN_MAX_SEQ_LEN || p.N_k > ATTN_MAX_SEQ_LEN) return ATTN_ERR_UNSUPPORTED;
    const bool empty = p.B == 0 || p.H == 0 || p.N_q == 0;
    if (empty) return ATTN_OK;
    if (!p.q || !p.o) return ATTN_ERR_INVALID_ARG;
    if (p.N_k > 0 && (!p.k || !p.v)) return ATTN_ERR_INVALID_ARG;
    if (!aligned(p.q, 16) || !aligned(p.o, 16) || (p.k && !aligned(p.k, 16)) ||
        (p.v && !aligned(p.v, 16)) || (p.lse && !aligned(p.lse, 4)))
        return ATTN_ERR_INVALID_ARG;
    if ((p.q_descale && !aligned(p.q_descale, 4)) || (p.k_descale && !aligned(p.k_descale, 4)) ||
        (p.v_descale && !aligned(p.v_descale, 4)))
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

attn_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return ATTN_OK;
    if (e == cudaErrorNotSupported) return ATTN_ERR_UNSUPPORTED;
    attn::note_cuda_error(e);
    return ATTN_ERR_CUDA;
}

attn::Problem make_problem(const void* q, const void* k, const void* v, void* o, float* lse,
                           const float* qd, const float* kd, const float* vd, int B, int H,
                           int N_q, int N_k, int d, float scale, int causal, int dtype) {
    attn::Problem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.q_descale = qd;
    p.k_descale = kd;
    p.v_descale = vd;
    p.B = B;
    p.H = H;
    p.H_kv = H;
    p.N_q = N_q;
    p.N_k = N_k;
    p.d = d;
    p.scale = scale;
    p.causal = causal ? 1 : 0;
    p.dtype = dtype;
    return p;
}

bool is_empty(const attn::Problem& p) { return p.B == 0 || p.H == 0 || p.N_q == 0; }

attn_status_t run_tc(const attn::Problem& p, cudaStream_t s) {
    attn_status_t st = validate(p);
    if (st != ATTN_OK || is_empty(p)) return st;
    cudaError_t e = attn::launch_tc(p, s);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

}  // namespace

namespace attn {
void note_cuda_error(cudaError_t e) { t_last_cuda_error = e; }
}  // namespace attn

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N_q, int N_k, int d, float scale, int causal,
                       attn_dtype_t dtype, void* stream) {
    attn::Problem p = make_problem(q, k, v, o, lse, nullptr, nullptr, nullptr, B, H, N_q, N_k, d,
                                   scale, causal, (int)dtype);
    return run_tc(p, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                           const float* q_descale, const float* k_descale,
                           const float* v_descale, int B, int H, int N_q, int N_k, int d,
                           float scale, int causal, void* stream) {
    if (!is_empty(make_problem(q, k, v, o, lse, nullptr, nullptr, nullptr, B, H, N_q, N_k, d,
                               scale, causal, attn::kE4M3)) &&
        (!q_descale || !k_descale || !v_descale))
        return ATTN_ERR_INVALID_ARG;
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, attn::kE4M3);
    return run_tc(p, static_cast<cudaStream_t>(stream));
}

size_t attn_fwd_fp8_workspace_bytes(int B, int H, int N_k, int d) {
    if (B < 0 || H < 0 || N_k < 0) return 0;
    return attn::fp8_ws_workspace_bytes(B, H, N_k, d);
}

attn_status_t attn_fwd_fp8_ws(const void* q, const void* k, const void* v, void* o, float* lse,
                              const float* q_descale, const float* k_descale,
                              const float* v_descale, int B, int H, int N_q, int N_k, int d,
                              float scale, int causal, void* workspace, size_t workspace_bytes,
                              void* stream) {
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, attn::kE4M3);
    attn_status_t st = validate(p);
    if (st != ATTN_OK || is_empty(p)) return st;
    if (!q_descale || !k_descale || !v_descale) return ATTN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (d == 256) return run_tc(p, s);  // widens V on chip; the workspace is not used
    const size_t need = attn::fp8_ws_workspace_bytes(B, H, N_k, d);
    if (need > 0 && (!workspace || !aligned(workspace, 16) || workspace_bytes < need))
        return ATTN_ERR_INVALID_ARG;
    cudaError_t e = attn::launch_tc_fp8_ws(p, workspace, workspace_bytes, s);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

attn_status_t attn_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                            const float* q_descale, const float* k_descale,
                            const float* v_descale, int B, int H, int N_q, int N_k, int d,
                            float scale, int causal, attn_dtype_t dtype, void* stream) {
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, (int)dtype);
    attn_status_t st = validate(p);
    if (st != ATTN_OK || is_empty(p)) return st;
    cudaError_t e = attn::launch_simt(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

size_t attn_splitkv_workspace_bytes(int B, int H, int N_q, int d, int num_splits) {
    if (B < 0 || H < 0 || N_q < 0 || (d != 64 && d != 128 && d != 256) || num_splits < 1 ||
        num_splits > attn::kMaxSplits)
        return 0;
    if (num_splits == 1) return 0;
    return attn::splitkv_workspace_bytes(B, H, N_q, d, num_splits);
}

int attn_splitkv_num_splits(int B, int H, int N_q, int N_k, int d, int num_sms) {
    if (B <= 0 || H <= 0 || N_q <= 0 || N_k <= 0 || num_sms <= 0) return 1;
    if (d != 64 && d != 128 && d != 256) return 1;
    // CTAs without splitting: one per (batch, head, query-tile pair), or per
    // query tile at d = 256; key tiles of 128 keys each CTA walks
    const long long rows_per_cta = d == 256 ? 128 : 256;
    const long long units = (long long)B * H * ((N_q + rows_per_cta - 1) / rows_per_cta);
    const long long tiles = (N_k + 127) / 128;
    // estimated time in key-tile steps: waves x (tiles per CTA + ~3 steps of
    // fixed cost per CTA), plus the combine pass (~1 step + s / 8)
    int best = 1;
    double best_cost = 0.0;
    for (int sp = 1; sp <= attn::kMaxSplits && sp <= tiles; ++sp) {
        const long long waves = (units * sp + num_sms - 1) / num_sms;
        const long long per = (tiles + sp - 1) / sp;
        const double cost = (double)waves * (double)(per + 3) + (sp > 1 ? 1.0 + sp / 8.0 : 0.0);
        if (sp == 1 || cost < best_cost) {
            best = sp;
            best_cost = cost;
        }
    }
    return best;
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               const float* q_descale, const float* k_descale,
                               const float* v_descale, int B, int H, int N_q, int N_k, int d,
                               float scale, int causal, attn_dtype_t dtype, int num_splits,
                               void* workspace, size_t workspace_bytes, void* stream) {
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, (int)dtype);
    attn_status_t st = validate(p);
    if (st != ATTN_OK) return st;
    if (num_splits < 1 || num_splits > attn::kMaxSplits) return ATTN_ERR_INVALID_ARG;
    if (is_empty(p)) return ATTN_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (num_splits == 1) {
        e = attn::launch_tc(p, s);
    } else {
        if (!workspace || !aligned(workspace, 16) ||
            workspace_bytes < attn::splitkv_workspace_bytes(B, H, N_q, d, num_splits))
            return ATTN_ERR_INVALID_ARG;
        e = attn::launch_tc_splitkv(p, num_splits, workspace, workspace_bytes, s);
    }
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           const float* q_descale, const float* k_descale,
                           const float* v_descale, int B, int H, int H_kv, int N_q, int N_k,
                           int d, float scale, int causal, attn_dtype_t dtype, void* stream) {
    if (H_kv < 1 || H < 0 || (H > 0 && H % H_kv != 0)) return ATTN_ERR_INVALID_ARG;
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, (int)dtype);
    p.H_kv = H_kv;
    return run_tc(p, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_quantize_e4m3(const void* x, attn_dtype_t x_dtype, void* codes,
                                 float* descale, int B, int N, int H, int d, const float* signs,
                                 void* stream) {
    if (B < 0 || N < 0 || H < 0) return ATTN_ERR_INVALID_ARG;
    if (x_dtype != ATTN_BF16 && x_dtype != ATTN_FP16 && x_dtype != ATTN_FP32)
        return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (N > ATTN_MAX_SEQ_LEN) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0) return ATTN_OK;
    if (!descale || !aligned(descale, 4)) return ATTN_ERR_INVALID_ARG;
    if (N > 0 && (!x || !codes || !aligned(codes, 16) || !aligned(x, 16)))
        return ATTN_ERR_INVALID_ARG;
    if (signs && !aligned(signs, 4)) return ATTN_ERR_INVALID_ARG;
    cudaError_t e = attn::launch_quantize_e4m3(x, (int)x_dtype, signs, codes, descale, B, N, H, d,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

size_t attn_bwd_workspace_bytes(int B, int H, int N_q) {
    if (B < 0 || H < 0 || N_q < 0) return 0;
    return attn::bwd_workspace_bytes(B, H, N_q);
}

attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv,
                           int B, int H, int H_kv, int N_q, int N_k, int d, float scale,
                           int causal, attn_dtype_t dtype, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (B < 0 || H < 0 || N_q < 0 || N_k < 0) return ATTN_ERR_INVALID_ARG;
    if (H_kv < 1 || (H > 0 && H % H_kv != 0)) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16) {
        if (dtype == ATTN_FP8_E4M3) return ATTN_ERR_UNSUPPORTED;
        return ATTN_ERR_INVALID_ARG;
    }
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (N_q > ATTN_MAX_SEQ_LEN || N_k > ATTN_MAX_SEQ_LEN) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || (N_q == 0 && N_k == 0)) return ATTN_OK;
    const void* need16[] = {q, k, v, o, dO, dq, dk, dv};
    const bool has_q = N_q > 0, has_k = N_k > 0;
    const bool present[] = {has_q, has_k, has_k, has_q, has_q, has_q, has_k, has_k};
    for (int i = 0; i < 8; ++i) {
        if (!present[i]) continue;
        if (!need16[i] || !aligned(need16[i], 16)) return ATTN_ERR_INVALID_ARG;
    }
    if (has_q && (!lse || !aligned(lse, 4))) return ATTN_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16) ||
        workspace_bytes < attn::bwd_workspace_bytes(B, H, N_q))
        return ATTN_ERR_INVALID_ARG;
    attn::BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.dO = dO;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.N_q = N_q;
    a.N_k = N_k;
    a.d = d;
    a.H_kv = H_kv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.dtype = (int)dtype;
    a.workspace = workspace;
    cudaError_t e = attn::launch_bwd(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                       int H, int N_q, int N_k, int d, float scale, int causal,
                       attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
    return attn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, H, H > 0 ? H : 1, N_q, N_k, d, scale,
                        causal, dtype, workspace, workspace_bytes, stream);
}

attn_status_t attn_selftest_wait(unsigned timeout_us, void* stream) {
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return ATTN_ERR_INVALID_ARG;
    cudaError_t e = attn::launch_wait_selftest(1000ull * timeout_us, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

attn_status_t attn_selftest_abort(const void* q, const void* k, const void* v, void* o,
                                  float* lse, const float* q_descale, const float* k_descale,
                                  const float* v_descale, int B, int H, int N_q, int N_k, int d,
                                  float scale, int causal, attn_dtype_t dtype, void* workspace,
                                  size_t workspace_bytes, unsigned timeout_us, void* stream) {
    if (timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return ATTN_ERR_INVALID_ARG;
    attn::Problem p = make_problem(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N_q,
                                   N_k, d, scale, causal, (int)dtype);
    attn_status_t st = validate(p);
    if (st != ATTN_OK) return st;
    // the check needs work to cut short: at least one query row and one key
    if (is_empty(p) || N_k == 0) return ATTN_ERR_INVALID_ARG;
    // with a workspace, e4m3 at d = 64 / 128 runs attn_fwd_fp8_ws's kernels
    const bool ws = workspace != nullptr && dtype == ATTN_FP8_E4M3 && (d == 64 || d == 128);
    if (workspace && !ws) return ATTN_ERR_INVALID_ARG;
    if (ws && (!aligned(workspace, 16) ||
               workspace_bytes < attn::fp8_ws_workspace_bytes(B, H, N_k, d)))
        return ATTN_ERR_INVALID_ARG;
    p.selftest_wait_ns = 1000ull * timeout_us;
    p.selftest_items = 1;  // the loader stops after the first K/V ring item
    cudaError_t e = ws ? attn::launch_tc_fp8_ws(p, workspace, workspace_bytes,
                                                static_cast<cudaStream_t>(stream))
                       : attn::launch_tc(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) (void)cudaGetLastError();
    return from_cuda(e);
}

attn_status_t attn_check_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    unsigned a = 0, b = 0, c = 0, g = 0;
    if (e == cudaSuccess) e = attn::tc_take_status(&a, s);
    if (e == cudaSuccess) e = attn::tc256_take_status(&c, s);
    if (e == cudaSuccess) e = attn::simt_take_status(&b, s);
    if (e == cudaSuccess) e = attn::bwd_take_status(&g, s);
    if (e != cudaSuccess) {
        attn::note_cuda_error(e);
        return ATTN_ERR_CUDA;
    }
    if ((a | b | c | g) & attn::kStatusTimeout) return ATTN_ERR_TIMEOUT;
    return ATTN_OK;
}

const char* attn_last_cuda_error(void) {
    const cudaError_t e = t_last_cuda_error;
    return e == cudaSuccess ? "none" : cudaGetErrorName(e);
}

const char* attn_status_string(attn_status_t s) {
    switch (s) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case ATTN_ERR_CUDA: return "CUDA error";
        case ATTN_ERR_TIMEOUT: return "bounded wait timed out inside a kernel";
        case ATTN_ERR_SCRATCH_LIMIT:
            return "problem needs more scratch than the library's fixed scratch array holds";
    }
    return "unknown status";
}

}  // extern "C"
