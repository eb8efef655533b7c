// Exact attention forward on the CUDA cores: a plain tiled kernel with an
// online softmax ("FlashAttention (HI)" page, sections "Tiling and block
// processing" and "Online softmax computation").  fp32 scores, fp32 exponentials, fp32 accumulation.  It is the
// second, independent GPU implementation that cross-checks the tensor-core
// kernel; it is not the timed path.
//
// One CTA = 64 query rows of one (b, h); 4 warps, 16 rows each.  K and V
// stream through shared memory in 64-key tiles (converted to fp32, V already
// multiplied by its descale).  For one row a warp scores two keys per lane,
// reduces the tile maximum and sum with shuffles, rescales its running output
// and adds the tile's P*V with each lane owning d/32 output columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "attn_internal.h"

namespace attn {
namespace {

__device__ unsigned g_simt_status = 0;

constexpr int kRows = 64;     // query rows per CTA
constexpr int kKeys = 64;     // keys per tile
constexpr int kThreads = 128;

__device__ __forceinline__ float load_elem(const void* base, int64_t idx, int dtype) {
    if (dtype == kBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    if (dtype == kFP16) return __half2float(reinterpret_cast<const __half*>(base)[idx]);
    __nv_fp8_e4m3 x;
    x.__x = reinterpret_cast<const __nv_fp8_storage_t*>(base)[idx];
    return float(x);
}

template <int D>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(Problem p) {
    constexpr int U = D / 32;     // output columns per lane
    extern __shared__ float smem[];
    float* Qs = smem;                          // [kRows][D]
    float* Ks = Qs + kRows * D;                // [kKeys][D+1]
    float* Vs = Ks + kKeys * (D + 1);          // [kKeys][D]

    const int b = blockIdx.z, h = blockIdx.y;
    const int row0 = blockIdx.x * kRows;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ldq = (int64_t)p.H * D;      // element stride between rows
    const int64_t q_base = ((int64_t)b * p.N_q * p.H + h) * D;
    const int h_kv = h / (p.H / p.H_kv);   // grouped-query attention: shared K/V head
    const int64_t ldk = (int64_t)p.H_kv * D;
    const int64_t k_base = ((int64_t)b * p.N_k * p.H_kv + h_kv) * D;
    const int bh = b * p.H + h;
    const int bh_kv = b * p.H_kv + h_kv;

    float dq = 1.f, dk = 1.f, dv = 1.f;
    if (p.dtype == kE4M3) {
        if (p.q_descale) dq = p.q_descale[bh];
        if (p.k_descale) dk = p.k_descale[bh_kv];
        if (p.v_descale) dv = p.v_descale[bh_kv];
    }
    // scores are kept in base 2: s2 = s * log2(e); the factor is folded into Q
    const float c = p.scale * dq * dk * 1.4426950408889634f;

    for (int e = tid; e < kRows * D; e += kThreads) {
        int r = e / D, t = e % D;
        int i = row0 + r;
        Qs[e] = (i < p.N_q) ? load_elem(p.q, q_base + (int64_t)i * ldq + t, p.dtype) * c : 0.f;
    }

    const int shift = p.N_k - p.N_q;
    const int last_row = min(row0 + kRows - 1, p.N_q - 1);
    int last_key = p.N_k - 1;
    if (p.causal) last_key = min(last_key, last_row + shift);
    const int n_tiles = last_key < 0 ? 0 : last_key / kKeys + 1;

    float m[16], l[16], o[16][U];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u) o[rr][u] = 0.f;
    }

    for (int kt = 0; kt < n_tiles; ++kt) {
        __syncthreads();
        for (int e = tid; e < kKeys * D; e += kThreads) {
            int r = e / D, t = e % D;
            int j = kt * kKeys + r;
            bool ok = j < p.N_k;
            int64_t gi = k_base + (int64_t)j * ldk + t;
            Ks[r * (D + 1) + t] = ok ? load_elem(p.k, gi, p.dtype) : 0.f;
            Vs[r * D + t] = ok ? load_elem(p.v, gi, p.dtype) * dv : 0.f;
        }
        __syncthreads();

#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            const int r = warp * 16 + rr;
            const int i = row0 + r;
            int lim = p.N_k - 1;
            if (p.causal) lim = min(lim, i + shift);
            const float* qr = Qs + r * D;
            float s0 = 0.f, s1 = 0.f;
            const float* k0 = Ks + lane * (D + 1);
            const float* k1 = Ks + (lane + 32) * (D + 1);
#pragma unroll 8
            for (int t = 0; t < D; ++t) {
                float qv = qr[t];
                s0 = fmaf(qv, k0[t], s0);
                s1 = fmaf(qv, k1[t], s1);
            }
            const int j0 = kt * kKeys + lane, j1 = j0 + 32;
            if (j0 > lim) s0 = -INFINITY;
            if (j1 > lim) s1 = -INFINITY;
            float mt = fmaxf(s0, s1);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m[rr], mt);
            if (m_new == -INFINITY) continue;          // nothing allowed yet (uniform per warp)
            const float alpha = exp2f(m[rr] - m_new);   // 0 when m = -inf
            const float p0 = exp2f(s0 - m_new), p1 = exp2f(s1 - m_new);
            float ps = p0 + p1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l[rr] = l[rr] * alpha + ps;
            m[rr] = m_new;
#pragma unroll
            for (int u = 0; u < U; ++u) o[rr][u] *= alpha;
#pragma unroll
            for (int jj = 0; jj < kKeys; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, jj < 32 ? p0 : p1, jj & 31);
                const float* vr = Vs + jj * D + lane;
#pragma unroll
                for (int u = 0; u < U; ++u) o[rr][u] = fmaf(pj, vr[32 * u], o[rr][u]);
            }
        }
    }

#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const int i = row0 + warp * 16 + rr;
        if (i >= p.N_q) continue;
        const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
        const int64_t ob = q_base + (int64_t)i * ldq;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float x = o[rr][u] * inv;
            if (p.dtype == kFP16)
                reinterpret_cast<__half*>(p.o)[ob + lane + 32 * u] = __float2half_rn(x);
            else
                reinterpret_cast<__nv_bfloat16*>(p.o)[ob + lane + 32 * u] = __float2bfloat16_rn(x);
        }
        if (lane == 0 && p.lse)
            p.lse[(int64_t)bh * p.N_q + i] =
                l[rr] > 0.f ? (m[rr] + log2f(l[rr])) * 0.69314718055994531f : -INFINITY;
    }
}

template <int D>
constexpr size_t simt_smem_bytes() {
    return sizeof(float) * (size_t)(kRows * D + kKeys * (D + 1) + kKeys * D);
}

template <int D>
cudaError_t launch_d(const Problem& p, cudaStream_t stream) {
    const size_t smem = simt_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.N_q + kRows - 1) / kRows, p.H, p.B);
    attn_simt_kernel<D><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const Problem& p, cudaStream_t stream) {
    if (p.H > 65535 || p.B > 65535) return cudaErrorNotSupported;
    if (p.d == 64) return launch_d<64>(p, stream);
    if (p.d == 128) return launch_d<128>(p, stream);
    if (p.d == 256) return launch_d<256>(p, stream);
    return cudaErrorNotSupported;
}

cudaError_t simt_take_status(unsigned* out, cudaStream_t stream) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_simt_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_simt_status, &zero, sizeof(unsigned), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace attn
