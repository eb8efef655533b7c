// Incoherent processing for FP8 attention ("FlashAttention-3 (BN)" page,
// section "Low precision (FP8) and reducing quantisation error"): multiply each
// query / key row by the random orthogonal matrix M = diag(signs) H_d / sqrt(d)
// (H_d the Sylvester Hadamard matrix, signs a caller-given +-1 vector), which
// spreads outlier values over all coordinates, then quantise to e4m3 with one
// fp32 scale per (batch, head): s = amax / 448, code = RNE(y / s) saturated.
// Q M (K M)^T = Q K^T, so attention on the rotated Q and K is unchanged up to
// the quantisation error, which the rotation reduces.  Without signs the same
// kernels quantise without rotation (as for V).
//
// One warp per row of d elements: each lane holds d/32 consecutive elements;
// the transform's butterflies run over the element index bits, the low bits
// inside a thread, the rest across lanes with shuffles.  Memory-bound: the
// input is read twice (amax pass, code pass) and the codes written once.
// The descale output doubles as the amax accumulator, so nothing is allocated.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kE4M3Max = 448.f;

template <int D>
__device__ __forceinline__ void load_row(const void* x, int dtype, size_t row, int lane,
                                         float (&v)[D / 32]) {
    constexpr int PER = D / 32;
    const size_t base = row * D + (size_t)lane * PER;
    if (dtype == kFP32) {
        const float* p = reinterpret_cast<const float*>(x) + base;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[e] = p[e];
    } else if (dtype == kFP16) {
        const __half* p = reinterpret_cast<const __half*>(x) + base;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[e] = __half2float(p[e]);
    } else {
        const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(x) + base;
#pragma unroll
        for (int e = 0; e < PER; ++e) v[e] = __bfloat162float(p[e]);
    }
}

// y = (x * signs) H_d / sqrt(d) for the row held by the warp.
template <int D>
__device__ __forceinline__ void rotate_row(float (&v)[D / 32], const float* signs, int lane) {
    constexpr int PER = D / 32;
#pragma unroll
    for (int e = 0; e < PER; ++e) v[e] *= signs[lane * PER + e];
    // element index = lane * PER + e: bits below log2(PER) are in-thread
#pragma unroll
    for (int h = 1; h < PER; h <<= 1) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            if ((e & h) == 0) {
                const float a = v[e], b = v[e + h];
                v[e] = a + b;
                v[e + h] = a - b;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const float other = __shfl_xor_sync(0xffffffffu, v[e], m);
            v[e] = upper ? (other - v[e]) : (v[e] + other);
        }
    }
    const float inv = 1.f / sqrtf((float)D);
#pragma unroll
    for (int e = 0; e < PER; ++e) v[e] *= inv;
}

// row = (b * N + n) * H + h  ->  b * H + h
__device__ __forceinline__ long long head_of(long long row, long long NH, int H) {
    return (row / NH) * H + row % H;
}

template <int D>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    quant_amax_kernel(const void* x, int dtype, const float* signs, unsigned* amax_bits,
                      long long rows, long long NH, int H) {
    const int lane = threadIdx.x & 31;
    for (long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); row < rows;
         row += (long long)gridDim.x * kWarpsPerBlock) {
        float v[D / 32];
        load_row<D>(x, dtype, (size_t)row, lane, v);
        if (signs) rotate_row<D>(v, signs, lane);
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < D / 32; ++e) m = fmaxf(m, fabsf(v[e]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        // non-negative floats order like their bit patterns
        if (lane == 0 && m > 0.f) atomicMax(amax_bits + head_of(row, NH, H), __float_as_uint(m));
    }
}

template <int D>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    quant_code_kernel(const void* x, int dtype, const float* signs, const unsigned* amax_bits,
                      uint8_t* codes, long long rows, long long NH, int H) {
    constexpr int PER = D / 32;
    const int lane = threadIdx.x & 31;
    for (long long row = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5); row < rows;
         row += (long long)gridDim.x * kWarpsPerBlock) {
        float v[PER];
        load_row<D>(x, dtype, (size_t)row, lane, v);
        if (signs) rotate_row<D>(v, signs, lane);
        const float amax = __uint_as_float(amax_bits[head_of(row, NH, H)]);
        const float s = amax > 0.f ? amax / kE4M3Max : 1.f;
        uint8_t* dst = codes + (size_t)row * D + (size_t)lane * PER;
#pragma unroll
        for (int e = 0; e < PER; e += 2) {
            const float a = fminf(fmaxf(v[e] / s, -kE4M3Max), kE4M3Max);
            const float b = fminf(fmaxf(v[e + 1] / s, -kE4M3Max), kE4M3Max);
            uint16_t pr;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pr) : "f"(b), "f"(a));
            *reinterpret_cast<uint16_t*>(dst + e) = pr;
        }
    }
}

__global__ void quant_finalize_kernel(float* descale, long long n) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float amax = __uint_as_float(reinterpret_cast<unsigned*>(descale)[i]);
    descale[i] = amax > 0.f ? amax / kE4M3Max : 1.f;
}

template <int D>
cudaError_t launch_quant(const void* x, int dtype, const float* signs, void* codes, float* descale,
                         long long B, long long N, int H, cudaStream_t stream) {
    const long long rows = B * N * H, NH = N * H, n_heads = B * H;
    cudaError_t e = cudaMemsetAsync(descale, 0, (size_t)n_heads * sizeof(float), stream);
    if (e != cudaSuccess) return e;
    if (rows > 0) {
        long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
        if (blocks > 65535LL * 16) blocks = 65535LL * 16;
        quant_amax_kernel<D><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, stream>>>(
            x, dtype, signs, reinterpret_cast<unsigned*>(descale), rows, NH, H);
        quant_code_kernel<D><<<(unsigned)blocks, 32 * kWarpsPerBlock, 0, stream>>>(
            x, dtype, signs, reinterpret_cast<const unsigned*>(descale),
            static_cast<uint8_t*>(codes), rows, NH, H);
    }
    quant_finalize_kernel<<<(unsigned)((n_heads + 255) / 256), 256, 0, stream>>>(descale, n_heads);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_e4m3(const void* x, int dtype, const float* signs, void* codes,
                                 float* descale, int B, int N, int H, int d, cudaStream_t stream) {
    if (d == 64) return launch_quant<64>(x, dtype, signs, codes, descale, B, N, H, stream);
    if (d == 128) return launch_quant<128>(x, dtype, signs, codes, descale, B, N, H, stream);
    if (d == 256) return launch_quant<256>(x, dtype, signs, codes, descale, B, N, H, stream);
    return cudaErrorNotSupported;
}

}  // namespace attn
