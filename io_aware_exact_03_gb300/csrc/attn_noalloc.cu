// Split-KV forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace buffer: for example a plugin
// running inside a host program that owns all device memory through its own
// pool and does not allow raw cudaMalloc, or a latency-critical loop where the
// device-wide synchronisation that cudaMalloc/cudaFree can cause is not
// acceptable.  attn_fwd_splitkv_static gives them the split-KV path with its
// scratch in a fixed array compiled into this library, so the call allocates
// nothing: not here, not in the kernels, not through any library routine.
//
// The array (ATTN_STATIC_SCRATCH_BYTES) is held by every GPU that loads the
// library until the process exits.  Host code cannot use the array's name as a
// device address (on the host it is only a stand-in symbol), so the address is
// looked up once per device with cudaGetSymbolAddress while that device is
// current, and passed to the kernels.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "attn_gb300.h"
#include "attn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_splitkv_scratch[ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_for_current_device() {
    int dev = -1;
    const cudaError_t eg = cudaGetDevice(&dev);
    if (eg != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        attn::note_cuda_error(eg != cudaSuccess ? eg : cudaErrorInvalidDevice);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t es = cudaGetSymbolAddress(&ptr, g_splitkv_scratch);
        if (es != cudaSuccess || !ptr) {
            attn::note_cuda_error(es != cudaSuccess ? es : cudaErrorInvalidSymbol);
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ATTN_API attn_status_t attn_fwd_splitkv_static(
    const void* q, const void* k, const void* v, void* o, float* lse, const float* q_descale,
    const float* k_descale, const float* v_descale, int B, int H, int N_q, int N_k, int d,
    float scale, int causal, attn_dtype_t dtype, int num_splits, void* stream) {
    // arguments: the same rules as attn_fwd_splitkv (checked before any CUDA call)
    if (B < 0 || H < 0 || N_q < 0 || N_k < 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_BF16 && dtype != ATTN_FP16 && dtype != ATTN_FP8_E4M3)
        return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (N_q > ATTN_MAX_SEQ_LEN || N_k > ATTN_MAX_SEQ_LEN) return ATTN_ERR_UNSUPPORTED;
    if (num_splits < 2 || num_splits > attn::kMaxSplits) return ATTN_ERR_INVALID_ARG;
    if (B == 0 || H == 0 || N_q == 0) return ATTN_OK;
    if (!q || !o || (N_k > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_descale) & 3u) || (reinterpret_cast<uintptr_t>(k_descale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_descale) & 3u))
        return ATTN_ERR_INVALID_ARG;
    // the fixed array must hold every split's partial outputs and lse
    const size_t need = attn::splitkv_workspace_bytes(B, H, N_q, d, num_splits);
    if (need > (size_t)ATTN_STATIC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH_LIMIT;

    void* scratch = scratch_for_current_device();
    if (!scratch) return ATTN_ERR_CUDA;

    attn::Problem p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.o = o;
    p.lse = lse;
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    p.B = B;
    p.H = H;
    p.H_kv = H;
    p.N_q = N_q;
    p.N_k = N_k;
    p.d = d;
    p.scale = scale;
    p.causal = causal ? 1 : 0;
    p.dtype = (int)dtype;
    // Every partial the combine reads is written first by the split kernel, so
    // the contents left by the previous call need no clearing.
    cudaError_t e = attn::launch_tc_splitkv(p, num_splits, scratch, (size_t)ATTN_STATIC_SCRATCH_BYTES,
                                            static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return ATTN_OK;
    (void)cudaGetLastError();
    return e == cudaErrorNotSupported ? ATTN_ERR_UNSUPPORTED : ATTN_ERR_CUDA;
}
