// Fused exact-attention forward on the fifth-generation tensor cores (sm_103a).
//
// The pages' method ("FlashAttention (HI)": "Tiling and block processing",
// "Online softmax computation", "Combining operations in one CUDA kernel";
// "FlashAttention-2 (BN)": "Improved parallelism"; "FlashAttention-3 (BN)":
// "Asynchronous execution and warp specialisation", "Reducing memory
// operations") mapped onto Blackwell:
//
//   * one CTA owns a 128-row query tile of one (batch, head); the grid spans
//     batch x heads x query tiles, so one head is spread over many SMs;
//   * warp 0 (producer) streams the Q tile once and then K_j / V_j tiles
//     through a ring of shared-memory slots with TMA, in the order the MMAs
//     consume them (K0, K1, V0, K2, V1, ...), guarded by mbarriers;
//   * warp 1 (one thread) issues tcgen05 MMAs: S_j = Q K_j^T into one of two
//     TMEM score buffers, and O += P_j V_j with P_j read from TMEM; it owns the
//     TMEM allocation;
//   * warps 2-5 (128 threads, one query row each) run the online softmax:
//     TMEM -> registers, causal / ragged mask on the tiles that need it, row
//     maximum, exp2, row sum, P back to TMEM as bf16 / fp16 / e4m3; they
//     rescale the running output in TMEM only when the row maximum grew (for
//     bf16 / fp16: by more than 2^8, so the P values stay <= 256), and write
//     O / lse at the end.
//   While the softmax works on S_j the tensor core already computes S_{j+1}
//   and finishes P_{j-1} V_{j-1}.
//
// Scores are kept in base 2: the logit scale folds in log2(e) (and, for e4m3,
// the q and k descales); lse is converted back to the natural log.
//
// Every mbarrier wait is bounded: after the time limit the waiting role sets
// the CTA abort flag and the device status word, drains what it issued, and
// the CTA exits normally (TMEM is always freed).  Nothing traps.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "attn_internal.h"
#include "tc_ptx.cuh"

namespace attn {
namespace {

using namespace ptx;

__device__ unsigned g_tc_status = 0;

constexpr int BM = 128;       // query rows per tile (MMA M)
constexpr int BN = 128;       // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 192; // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0;    // two score buffers: columns [0,128) and [128,256)
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;

template <int D, int KIND>
struct Cfg {
    static constexpr int E = (KIND == kE4M3) ? 1 : 2;     // bytes per element
    static constexpr int RB = D * E;                       // bytes per row
    static constexpr int CB = RB >= 128 ? 128 : RB;        // bytes per swizzle chunk
    static constexpr int NC = RB / CB;                     // chunks per row
    static constexpr int TILE = BM * RB;                   // bytes per 128-row tile
    static constexpr int CHUNK = BM * CB;                  // bytes per chunk of a tile
    static constexpr int SLOTS = (TILE >= 32768) ? 6 : 8;  // K/V ring depth
    static constexpr uint32_t LAYOUT = (CB == 128) ? 2u : 4u;  // 128B / 64B swizzle
    static constexpr int MMA_K = 32 / E;                   // K per MMA instruction
    static constexpr int NB = 1 + 2 * SLOTS + 2 + 2 + 1 + 1 + 1;  // mbarriers
    static constexpr size_t SMEM_USED = 1024 + (size_t)TILE * (1 + SLOTS) + NB * 8 + 16;
    // at least ~120 KB so two CTAs never share an SM (each takes all of TMEM)
    static constexpr size_t SMEM = SMEM_USED > 122880 ? SMEM_USED : 122880;
    static constexpr uint32_t FMT = (KIND == kBF16) ? 1u : 0u;  // bf16 = 1, f16 / e4m3 = 0
    static constexpr uint32_t IDESC_QK = instr_desc(FMT, FMT, 0, 0, BM, BN);
    static constexpr uint32_t IDESC_PV = instr_desc(FMT, FMT, 0, 1, BM, D);
    static constexpr uint32_t P_COLS = BN * E / 4;         // TMEM columns holding P
    // Rescale the running output only when the row maximum grew by more than
    // this (log2 units).  bf16/fp16 P tolerate values up to 2^8; an e4m3 P
    // must keep its largest weight exactly 1, so e4m3 rescales on every growth.
    static constexpr float RESCALE_THRESHOLD = (KIND == kE4M3) ? 0.0f : 8.0f;
};

struct TcParams {
    int B, H, N_q, N_k;
    int n_qt;
    int causal;
    float scale;
    void* o;
    float* lse;
    const float* q_descale;
    const float* k_descale;
    const float* v_descale;
    unsigned long long timeout_ns;
};

// Bounded wait on an mbarrier phase.  Returns false (after flagging) when the
// limit passes or another role already aborted.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       unsigned long long limit_ns) {
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(&g_tc_status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort_flag, limit_ns);
}

// Drain-only wait (used while aborting): bounded, never raises the flag.
__device__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ int kv_tiles_for(int q0, const TcParams& p) {
    const int last_row = min(q0 + BM - 1, p.N_q - 1);
    int last_key = p.N_k - 1;
    if (p.causal) last_key = min(last_key, last_row + (p.N_k - p.N_q));
    return last_key < 0 ? 0 : last_key / BN + 1;
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const TcParams p) {
    using C = Cfg<D, KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = smem + C::TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + (size_t)C::SLOTS * C::TILE);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const uint32_t b_q_full = smem_u32(bars);
    const uint32_t b_kv_full = smem_u32(bars + 1);                 // + 8 * slot
    const uint32_t b_kv_empty = smem_u32(bars + 1 + C::SLOTS);     // + 8 * slot
    const uint32_t b_s_full = smem_u32(bars + 1 + 2 * C::SLOTS);   // + 8 * buf
    const uint32_t b_s_free = smem_u32(bars + 3 + 2 * C::SLOTS);   // + 8 * buf
    const uint32_t b_p_full = smem_u32(bars + 5 + 2 * C::SLOTS);
    const uint32_t b_pv_done = smem_u32(bars + 6 + 2 * C::SLOTS);
    const uint32_t b_drain = smem_u32(bars + 7 + 2 * C::SLOTS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int qt = p.causal ? (p.n_qt - 1 - (int)blockIdx.y) : (int)blockIdx.y;
    const int q0 = qt * BM;
    const int n_kv = kv_tiles_for(q0, p);
    const unsigned long long lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        for (int s = 0; s < C::SLOTS; ++s) {
            mbar_init(b_kv_full + 8 * s, 1);
            mbar_init(b_kv_empty + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_s_full + 8 * i, 1);
            mbar_init(b_s_free + 8 * i, 128);
        }
        mbar_init(b_p_full, 128);
        mbar_init(b_pv_done, 1);
        mbar_init(b_drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && n_kv > 0) {
            mbar_arrive_expect_tx(b_q_full, C::TILE);
            for (int c = 0; c < C::NC; ++c)
                tma_load_4d(smem_u32(sQ + c * C::CHUNK), &tmQ, b_q_full, c * (C::CB / C::E), h, q0,
                            b);
            int it = 0;
            bool ok = true;
            // consumption order: K0, then per j: K_{j+1} (if any), V_j
            const int n_items = 2 * n_kv;
            for (int item = 0; item < n_items && ok; ++item) {
                int tile;
                const CUtensorMap* tm;
                if (item == 0) {
                    tile = 0;
                    tm = &tmK;
                } else {
                    const int j = (item - 1) >> 1;
                    const bool is_k = ((item - 1) & 1) == 0 && (j + 1 < n_kv);
                    if (j + 1 < n_kv) {
                        tile = is_k ? j + 1 : j;
                        tm = is_k ? &tmK : &tmV;
                    } else {
                        // last tile: only V_{n-1} remains (item == 2 n - 1)
                        tile = n_kv - 1;
                        tm = &tmV;
                    }
                }
                const int slot = it % C::SLOTS;
                const uint32_t ph = (uint32_t)(it / C::SLOTS) & 1u;
                if (!wait_bar(b_kv_empty + 8 * slot, ph ^ 1u, abort_flag, lim)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(b_kv_full + 8 * slot, C::TILE);
                uint8_t* dst = sKV + (size_t)slot * C::TILE;
                for (int c = 0; c < C::NC; ++c)
                    tma_load_4d(smem_u32(dst + c * C::CHUNK), tm, b_kv_full + 8 * slot,
                                c * (C::CB / C::E), h, tile * BN, b);
                ++it;
            }
            if (!ok) {
                // let every load already issued land before the CTA can exit
                wait_drain(b_q_full, 0, lim);
                for (int k = (it > C::SLOTS ? it - C::SLOTS : 0); k < it; ++k)
                    wait_drain(b_kv_full + 8 * (k % C::SLOTS), (uint32_t)(k / C::SLOTS) & 1u, lim);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        if (lane == 0 && n_kv > 0) {
            bool ok = wait_bar(b_q_full, 0, abort_flag, lim);
            int it = 0;
            const uint32_t q_base = smem_u32(sQ);
            auto issue_qk = [&](int buf, int slot) {
                const uint32_t k_base = smem_u32(sKV + (size_t)slot * C::TILE);
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t off = c * C::CHUNK + ks * 32;
                        const uint64_t da = smem_desc(q_base + off, 16, 8 * C::CB, C::LAYOUT);
                        const uint64_t db = smem_desc(k_base + off, 16, 8 * C::CB, C::LAYOUT);
                        const uint32_t acc = (c | ks) != 0;
                        if constexpr (KIND == kE4M3)
                            mma_f8_ss(tmem + kColS0 + 128u * buf, da, db, C::IDESC_QK, acc);
                        else
                            mma_f16_ss(tmem + kColS0 + 128u * buf, da, db, C::IDESC_QK, acc);
                    }
                }
            };
            auto issue_pv = [&](int slot, bool first) {
                const uint32_t v_base = smem_u32(sKV + (size_t)slot * C::TILE);
#pragma unroll
                for (int ks = 0; ks < BN / C::MMA_K; ++ks) {
                    // V is MN-major: 8-key groups 8*CB apart, d-chunks CHUNK apart
                    const uint64_t db = smem_desc(v_base + ks * C::MMA_K * C::CB, C::CHUNK,
                                                  8 * C::CB, C::LAYOUT);
                    const uint32_t a_tmem = tmem + kColP + ks * (C::MMA_K * C::E / 4);
                    const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
                    if constexpr (KIND == kE4M3)
                        mma_f8_ts(tmem + kColO, a_tmem, db, C::IDESC_PV, acc);
                    else
                        mma_f16_ts(tmem + kColO, a_tmem, db, C::IDESC_PV, acc);
                }
            };
            if (ok) {
                // S_0 = Q K_0^T
                ok = wait_bar(b_kv_full, 0, abort_flag, lim);
                if (ok) {
                    tc_fence_after();
                    issue_qk(0, 0);
                    mma_commit(b_kv_empty);
                    mma_commit(b_s_full);
                    it = 1;
                }
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                if (j + 1 < n_kv) {
                    const int slot = it % C::SLOTS;
                    const int jj = j + 1, buf = jj & 1;
                    ok = wait_bar(b_kv_full + 8 * slot, (uint32_t)(it / C::SLOTS) & 1u, abort_flag,
                                  lim);
                    if (ok && jj >= 2)
                        ok = wait_bar(b_s_free + 8 * buf, (uint32_t)((jj >> 1) - 1) & 1u,
                                      abort_flag, lim);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(buf, slot);
                    mma_commit(b_kv_empty + 8 * slot);
                    mma_commit(b_s_full + 8 * buf);
                    ++it;
                }
                ok = wait_bar(b_p_full, (uint32_t)j & 1u, abort_flag, lim);
                if (!ok) break;
                const int slot = it % C::SLOTS;
                ok = wait_bar(b_kv_full + 8 * slot, (uint32_t)(it / C::SLOTS) & 1u, abort_flag, lim);
                if (!ok) break;
                tc_fence_after();
                issue_pv(slot, j == 0);
                if (j + 1 < n_kv) mma_commit(b_kv_empty + 8 * slot);
                mma_commit(b_pv_done);
                ++it;
            }
            if (!ok) {
                // make sure no MMA is still reading or writing when TMEM is freed
                mma_commit(b_drain);
                wait_drain(b_drain, 0, lim);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax + epilogue (128 thr)
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int row_g = q0 + r;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const int shift = p.N_k - p.N_q;
        int row_lim = p.N_k - 1;  // last allowed key of this row
        if (p.causal) row_lim = min(row_lim, row_g + shift);
        const int tile_lim = p.causal ? min(p.N_k - 1, q0 + shift) : p.N_k - 1;  // row 0's
        float dq = 1.f, dk = 1.f, dv = 1.f;
        if (KIND == kE4M3) {
            if (p.q_descale) dq = p.q_descale[bh];
            if (p.k_descale) dk = p.k_descale[bh];
            if (p.v_descale) dv = p.v_descale[bh];
        }
        const float c = p.scale * dq * dk * 1.4426950408889634f;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            if (!__all_sync(0xffffffffu,
                            wait_bar(b_s_full + 8 * buf, (uint32_t)(j >> 1) & 1u, abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[BN];
            {
                uint32_t rr[32];
#pragma unroll
                for (int u = 0; u < BN / 32; ++u) {
                    tmem_ld32(t_row + kColS0 + 128u * buf + 32 * u, rr);
                    tmem_ld_wait();
                    reg_fence32(rr);
#pragma unroll
                    for (int x = 0; x < 32; ++x) s[32 * u + x] = __uint_as_float(rr[x]);
                }
            }
            tc_fence_before();
            mbar_arrive(b_s_free + 8 * buf);

            const int kbase = j * BN;
            if (kbase + BN - 1 > tile_lim) {
                const int cl = row_lim - kbase;  // columns > cl are masked
#pragma unroll
                for (int x = 0; x < BN; ++x)
                    if (x > cl) s[x] = -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int x = 1; x < BN; ++x) mx = fmaxf(mx, s[x]);
            const float m_new = mx * c;
            const bool need = m_new > m_used + C::RESCALE_THRESHOLD;
            const bool any = __any_sync(0xffffffffu, need);
            float alpha = 1.f;
            if (any) {
                const float mu = fmaxf(m_used, m_new);
                alpha = (mu == m_used) ? 1.f : ex2(m_used - mu);
                m_used = mu;
            }
            const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
            uint32_t pk[C::P_COLS];
            float sum = 0.f;
            if constexpr (KIND == kE4M3) {
#pragma unroll
                for (int x = 0; x < BN; x += 4) {
                    const float p0 = ex2(fmaf(s[x], c, -m_ref));
                    const float p1 = ex2(fmaf(s[x + 1], c, -m_ref));
                    const float p2 = ex2(fmaf(s[x + 2], c, -m_ref));
                    const float p3 = ex2(fmaf(s[x + 3], c, -m_ref));
                    sum += (p0 + p1) + (p2 + p3);
                    pk[x / 4] = pack_e4m3(p0, p1, p2, p3);
                }
            } else {
#pragma unroll
                for (int x = 0; x < BN; x += 2) {
                    const float p0 = ex2(fmaf(s[x], c, -m_ref));
                    const float p1 = ex2(fmaf(s[x + 1], c, -m_ref));
                    sum += p0 + p1;
                    pk[x / 2] = (KIND == kBF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
                }
            }
            l = l * alpha + sum;

            if (j > 0) {
                if (!__all_sync(0xffffffffu,
                                wait_bar(b_pv_done, (uint32_t)(j - 1) & 1u, abort_flag, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (any) {
                    uint32_t oo[32];
#pragma unroll
                    for (int u = 0; u < D / 32; ++u) {
                        tmem_ld32(t_row + kColO + 32 * u, oo);
                        tmem_ld_wait();
                        reg_fence32(oo);
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            oo[x] = __float_as_uint(__uint_as_float(oo[x]) * alpha);
                        tmem_st32(t_row + kColO + 32 * u, oo);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < (int)C::P_COLS / 32; ++u) {
                uint32_t pp[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) pp[x] = pk[32 * u + x];
                tmem_st32(t_row + kColP + 32 * u, pp);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(b_p_full);
        }

        if (ok && n_kv > 0)
            ok = __all_sync(0xffffffffu,
                            wait_bar(b_pv_done, (uint32_t)(n_kv - 1) & 1u, abort_flag, lim));
        if (ok) {
            tc_fence_after();
            const bool valid = row_g < p.N_q;
            const bool has = l > 0.f;
            const float inv = has ? dv / l : 0.f;
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                             (((size_t)b * p.N_q + (valid ? row_g : 0)) * p.H + h) * D;
#pragma unroll
            for (int u = 0; u < D / 32; ++u) {
                uint32_t oo[32];
                if (n_kv > 0) {
                    tmem_ld32(t_row + kColO + 32 * u, oo);
                    tmem_ld_wait();
                    reg_fence32(oo);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) oo[x] = 0u;
                }
                uint32_t packed[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float a0 = __uint_as_float(oo[2 * x]) * inv;
                    const float a1 = __uint_as_float(oo[2 * x + 1]) * inv;
                    packed[x] = (KIND == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                }
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * u);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        dst[x] = make_uint4(packed[4 * x], packed[4 * x + 1], packed[4 * x + 2],
                                            packed[4 * x + 3]);
                }
            }
            if (valid && p.lse)
                p.lse[(size_t)bh * p.N_q + row_g] =
                    has ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// [B, N, H, d] tensor seen as a 4-D map {d, H, N, B}; box = one swizzle chunk
// of d x 1 head x 128 rows x 1 batch.
bool encode_map(CUtensorMap* m, const void* base, int dtype, int B, int N, int H, int d,
                int chunk_elems) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const int E = dtype == kE4M3 ? 1 : 2;
    const CUtensorMapDataType dt = dtype == kBF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == kFP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(N > 0 ? N : 1),
                                (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * E, (cuuint64_t)H * d * E,
                                   (cuuint64_t)(N > 0 ? N : 1) * H * d * E};
    const cuuint32_t box[4] = {(cuuint32_t)chunk_elems, 1, (cuuint32_t)BM, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw =
        chunk_elems * E == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int KIND>
cudaError_t launch_t(const Problem& pr, cudaStream_t stream) {
    using C = Cfg<D, KIND>;
    CUtensorMap mq, mk, mv;
    const int ce = C::CB / C::E;
    if (!encode_map(&mq, pr.q, KIND, pr.B, pr.N_q, pr.H, D, ce) ||
        !encode_map(&mk, pr.N_k > 0 ? pr.k : pr.q, KIND, pr.B, pr.N_k, pr.H, D, ce) ||
        !encode_map(&mv, pr.N_k > 0 ? pr.v : pr.q, KIND, pr.B, pr.N_k, pr.H, D, ce))
        return cudaErrorInvalidValue;
    TcParams p;
    p.B = pr.B;
    p.H = pr.H;
    p.N_q = pr.N_q;
    p.N_k = pr.N_k;
    p.n_qt = (pr.N_q + BM - 1) / BM;
    p.causal = pr.causal;
    p.scale = pr.scale;
    p.o = pr.o;
    p.lse = pr.lse;
    p.q_descale = pr.q_descale;
    p.k_descale = pr.k_descale;
    p.v_descale = pr.v_descale;
    p.timeout_ns = 2000000000ull;
    if (p.n_qt > 65535) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(pr.B * pr.H), (unsigned)p.n_qt);
    attn_tc_kernel<D, KIND><<<grid, kThreads, C::SMEM, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc(const Problem& p, cudaStream_t stream) {
    if ((long long)p.B * p.H > 0x7fffffffLL) return cudaErrorNotSupported;
    switch (p.dtype) {
        case kBF16:
            if (p.d == 64) return launch_t<64, kBF16>(p, stream);
            if (p.d == 128) return launch_t<128, kBF16>(p, stream);
            break;
        case kFP16:
            if (p.d == 64) return launch_t<64, kFP16>(p, stream);
            if (p.d == 128) return launch_t<128, kFP16>(p, stream);
            break;
        case kE4M3:
            if (p.d == 64) return launch_t<64, kE4M3>(p, stream);
            if (p.d == 128) return launch_t<128, kE4M3>(p, stream);
            break;
    }
    return cudaErrorNotSupported;
}

cudaError_t tc_take_status(unsigned* out, cudaStream_t stream) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_tc_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace attn
