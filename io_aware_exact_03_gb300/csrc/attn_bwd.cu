// Backward pass of exact attention on the fifth-generation tensor cores
// (sm_103a): dQ, dK, dV from Q, K, V, the forward's O and lse, and the upstream
// gradient dO.
//
// The pages motivate the backward pass only through training speedups
// ("FlashAttention (HI)" page, section "Empirical results"); the arithmetic is
// the derivative of the forward definition (same page, section "Problems of
// standard attention"), organised like the forward: tiles in shared memory,
// the scores recomputed on chip from Q, K and the forward's lse, nothing
// N x N in HBM (same page, sections "Tiling and block processing" and
// "Combining operations in one CUDA kernel"):
//
//   P_ij = exp(scale q_i.k_j - lse_i)            (lse from the forward)
//   D_i  = sum_t dO_it O_it
//   dV   = P^T dO,   dP = dO V^T,   dS = P (dP - D)
//   dQ   = scale dS K,   dK = scale dS^T Q
//
// Three kernels, each using only MMA forms of the forward kernel:
//   * bwd_prep: D_i and lse_i in base 2 into a padded workspace (D / 8 lanes per
//     row; rows with no key get lse2 = +inf so their P is exactly 0);
//   * bwd_dkdv: one CTA per 128-key tile.  Per query tile: S^T = K Q^T and
//     dP^T = V dO^T into TMEM (both K-major from shared memory, the forward's
//     score form), one thread per key row turns them into P^T and dS^T (bf16 /
//     fp16, over the same TMEM columns), then dV += P^T dO and dK += dS^T Q
//     (A from TMEM, B MN-major from shared memory: the forward's P V form).
//     The per-query vectors lse2 and D ride with each Q / dO tile;
//   * bwd_dq: one CTA per 128-row query tile.  Per key tile: S = Q K^T and
//     dP = dO V^T, one thread per query row forms dS, then dQ += dS K.
// Every output element is written by one CTA: no atomics, deterministic.
// Warps: 0 TMA producer, 1 MMA issuer (TMEM owner), 2-5 elementwise (bwd_dkdv:
// 2-5 and 6-9, one group per half of each query tile's queries).  Every
// mbarrier wait is bounded; on expiry the CTA drains, frees TMEM and exits
// with the status word set.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "attn_internal.h"
#include "bounded_wait.cuh"
#include "tc_ptx.cuh"
#include "tma_map.cuh"

namespace attn {
namespace {

using namespace ptx;

__device__ unsigned g_bwd_status = 0;

constexpr int BM = 128;        // query rows per tile
constexpr int BN = 128;        // keys per tile
constexpr int kThreads = 192;    // bwd_dq: producer, MMA issuer, 4 elementwise warps
constexpr int kThreadsKV = 320;  // bwd_dkdv: producer, MMA issuer, 2 x 4 elementwise warps
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 232448;

template <int D, int KIND>
struct BCfg {
    static constexpr int E = 2;                       // bytes per element (bf16 / fp16)
    static constexpr int CB = 128;                    // bytes per swizzle chunk row
    static constexpr int CE = CB / E;                 // 64 elements per chunk
    static constexpr int NC = D * E / CB;             // chunks per row: 1 (d 64), 2 (d 128)
    static constexpr int TILE = 128 * D * E;          // one 128-row tile
    static constexpr int CHUNK = 128 * CB;            // one d-chunk of a tile
    static constexpr int MMA_K = 16;
    static constexpr uint32_t FMT = (KIND == kBF16) ? 1u : 0u;
    // scores-like: A and B K-major, N = 128;  accumulate: A from TMEM, B MN-major, N = D
    static constexpr uint32_t IDESC_S = instr_desc(FMT, FMT, 0, 0, 128, 128);
    static constexpr uint32_t IDESC_ACC = instr_desc(FMT, FMT, 0, 1, 128, D);
    // bwd_dkdv ring item: Q tile, dO tile, lse2[128], D[128]
    static constexpr int ITEM_KV = 2 * TILE + 1024;
    static constexpr int SLOTS_KV_FIT = (kSmemLimit - 1024 - 2 * TILE - 512) / ITEM_KV;
    static constexpr int SLOTS_KV = SLOTS_KV_FIT > 6 ? 6 : SLOTS_KV_FIT;
    static constexpr size_t SMEM_KV = 1024 + 2 * (size_t)TILE + (size_t)SLOTS_KV * ITEM_KV + 512;
    // bwd_dq: separate K and V rings (V_j is free once dP_j is issued, K_j only
    // after dQ_j): two V slots, the rest of shared memory (up to four) for K
    static constexpr int V_SLOTS_Q = 2;
    static constexpr int TILES_Q_FIT = (kSmemLimit - 1024 - 2 * TILE - 512) / TILE;
    static constexpr int K_SLOTS_Q = (TILES_Q_FIT - V_SLOTS_Q) > 4 ? 4 : (TILES_Q_FIT - V_SLOTS_Q);
    static constexpr size_t SMEM_Q =
        1024 + 2 * (size_t)TILE + (size_t)(K_SLOTS_Q + V_SLOTS_Q) * TILE + 512;
    static_assert(SLOTS_KV >= 2 && K_SLOTS_Q >= 3, "ring depth");
    static_assert(SMEM_KV <= (size_t)kSmemLimit && SMEM_Q <= (size_t)kSmemLimit, "smem");
};

// TMEM columns (both kernels): S or S^T [0,128), dP or dP^T [128,256),
// accumulators from 256 (dV then dK, or dQ); bwd_dq keeps a second S buffer
// in [384, 512) (its accumulator takes at most 128 columns).
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256, kColS1 = 384;

struct BwdParams {
    int B, H, N_q, N_k, N_pad;
    int H_kv;             // K/V heads; query head h uses K/V head h / group
    int group;            // H / H_kv
    int n_units_tiles;    // key tiles (dkdv) or query tiles (dq)
    int heads_per_group;
    int causal;
    float scale;
    const float* lse2;    // [B*H][N_pad]: lse * log2(e), +inf for padding / no key
    const float* Dvec;    // [B*H][N_pad]
    void* out_a;          // dkdv: dV; dq: dQ    [B, N, H, D]
    void* out_b;          // dkdv: dK
    unsigned long long timeout_ns;
};

// Bounded waits (shared implementation) reporting to this file's status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long limit_ns) {
    return bounded_wait(bar, parity, abort_flag, limit_ns, &g_bwd_status);
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    bounded_drain(bar, parity, limit_ns);
}

// unit L -> (b, head, tile rank) over n_heads heads per batch, in groups of
// heads_per_group heads, the tile rank the slow coordinate inside a group
__device__ __forceinline__ void decode(long long L, const BwdParams& p, int n_heads, int* b, int* h,
                                       int* rank) {
    const long long n_bh = (long long)p.B * n_heads;
    const long long G = p.heads_per_group;
    const long long per_group = (long long)p.n_units_tiles * G;
    const long long n_full = n_bh / G;
    long long g, rem, Gg;
    if (L < n_full * per_group) {
        g = L / per_group;
        rem = L % per_group;
        Gg = G;
    } else {
        g = n_full;
        rem = L - n_full * per_group;
        Gg = n_bh - n_full * G;
    }
    *rank = (int)(rem / Gg);
    const int bh = (int)(g * G + rem % Gg);
    *b = bh / n_heads;
    *h = bh % n_heads;
}

// ---------------------------------------------------------------- prep
// Memory-bound (reads o and dO once).  Each lane loads 16 bytes (8 values) of
// o and of dO per row, D / 8 lanes covering a row; a warp takes 4 rows, so
// every lane has 4 loads of 16 bytes in flight (d = 64: 2) before its first
// use.  Measured on B2 H16 N4096 d128 (whole backward call): 4 rows per warp
// 0.4456 ms, 8 rows 0.4504, 16 rows 0.4545 (more registers, fewer resident
// blocks).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const void* o, const void* dO, const float* lse,
                                                       float* lse2, float* Dvec, int B, int H, int N_q,
                                                       int N_pad, int fp16) {
    constexpr int LPR = D / 8;      // lanes per row: 16 (d 128) or 8 (d 64)
    constexpr int RPI = 32 / LPR;   // rows per warp load: 2 or 4
    constexpr int RPW = 4;          // rows per warp
    constexpr int NI = RPW / RPI;   // load rounds: 2 or 1
    static_assert(NI >= 1 && RPW % RPI == 0, "whole load rounds");
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR, cl = lane % LPR;
    const long long total = (long long)B * H * N_pad;
    const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
    uint4 ov[NI], gv[NI];
    bool live[NI];
#pragma unroll
    for (int k = 0; k < NI; ++k) {
        const long long row = row0 + k * RPI + sub;
        const long long bh = row / N_pad;
        const int i = (int)(row % N_pad);
        live[k] = row < total && i < N_q;
        ov[k] = make_uint4(0u, 0u, 0u, 0u);
        gv[k] = ov[k];
        if (live[k]) {
            const int b = (int)(bh / H), h = (int)(bh % H);
            const size_t base = (((size_t)b * N_q + i) * H + h) * D + (size_t)cl * 8;
            ov[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(o) + base);
            gv[k] = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(dO) + base);
        }
    }
#pragma unroll
    for (int k = 0; k < NI; ++k) {
        const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
        const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
        float dsum = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            float2 af, gf;
            if (fp16) {
                af = __half22float2(*reinterpret_cast<const __half2*>(&ow[w]));
                gf = __half22float2(*reinterpret_cast<const __half2*>(&gw[w]));
            } else {
                af = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[w]));
                gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[w]));
            }
            dsum = fmaf(af.x, gf.x, fmaf(af.y, gf.y, dsum));
        }
        // sum over the LPR lanes of this row (an aligned group of lanes)
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, off);
        const long long row = row0 + k * RPI + sub;
        if (cl == 0 && row < total) {
            const long long bh = row / N_pad;
            const int i = (int)(row % N_pad);
            float l2 = INFINITY;  // padding rows and rows with no key: P is exactly 0
            if (i < N_q) {
                const float ls = lse[bh * N_q + i];
                l2 = ls == -INFINITY ? INFINITY : ls * 1.4426950408889634f;
            }
            Dvec[row] = live[k] ? dsum : 0.f;
            lse2[row] = l2;
        }
    }
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreadsKV, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const BwdParams p) {
    using C = BCfg<D, KIND>;
    constexpr int SLOTS = C::SLOTS_KV;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by offsetting the shared array itself, so that every
    // pointer derived from it stays in the shared address space (plain loads
    // through it compile to shared-memory loads, not generic ones)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sK = smem;
    uint8_t* sV = smem + C::TILE;
    uint8_t* sRing = smem + 2 * C::TILE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRing + (size_t)SLOTS * C::ITEM_KV);
    constexpr int NB = 6 + 2 * SLOTS;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t b_kv_full = smem_u32(bars);
    const uint32_t b_s_full = smem_u32(bars + 1);
    // P^T / dS^T of queries [0, 64) and [64, 128): the accumulating MMAs of
    // the first half run while the elementwise warps form the second
    const uint32_t b_p_half0 = smem_u32(bars + 2), b_p_half1 = smem_u32(bars + 5);
    const uint32_t b_acc_done = smem_u32(bars + 3);
    const uint32_t b_drain = smem_u32(bars + 4);
    const uint32_t b_item_full = smem_u32(bars + 6);           // + 8 * slot
    const uint32_t b_item_empty = smem_u32(bars + 6 + SLOTS);  // + 8 * slot

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int b, hk, kt;
    decode(blockIdx.x, p, p.H_kv, &b, &hk, &kt);  // key tiles: first (heaviest under causal) first
    const int key0 = kt * BN;
    const int shift = p.N_k - p.N_q;
    // query tiles that see any key of this tile: rows qi >= key0 - shift
    const int n_qt = (p.N_q + BM - 1) / BM;
    int i_lo = 0;
    if (p.causal) {
        const int first_row = key0 - shift;
        i_lo = first_row <= 0 ? 0 : first_row / BM;
    }
    // per query head of the K/V head's group: query tiles i_lo .. n_qt - 1
    const int per_head = (key0 < p.N_k && i_lo < n_qt) ? n_qt - i_lo : 0;
    const int n_steps = per_head * p.group;
    const unsigned long long lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_kv_full, 1);
        mbar_init(b_s_full, 1);
        mbar_init(b_p_half0, 128);
        mbar_init(b_p_half1, 128);
        mbar_init(b_acc_done, 1);
        mbar_init(b_drain, 1);
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(b_item_full + 8 * s, 1);
            mbar_init(b_item_empty + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
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
        if (lane == 0 && n_steps > 0) {
            mbar_arrive_expect_tx(b_kv_full, 2u * C::TILE);
            for (int c = 0; c < C::NC; ++c) {
                tma_load_4d(smem_u32(sK + c * C::CHUNK), &tmK, b_kv_full, c * C::CE, hk, key0, b);
                tma_load_4d(smem_u32(sV + c * C::CHUNK), &tmV, b_kv_full, c * C::CE, hk, key0, b);
            }
            bool ok = true;
            int s = 0;
            for (; s < n_steps; ++s) {
                const int slot = s % SLOTS;
                if (!wait_bar(b_item_empty + 8 * slot, ((uint32_t)(s / SLOTS) & 1u) ^ 1u, abort_flag, lim)) {
                    ok = false;
                    break;
                }
                const int h = hk * p.group + s / per_head;  // query head of this step
                const int q0 = (i_lo + s % per_head) * BM;
                uint8_t* dst = sRing + (size_t)slot * C::ITEM_KV;
                mbar_arrive_expect_tx(b_item_full + 8 * slot, (uint32_t)C::ITEM_KV);
                for (int c = 0; c < C::NC; ++c) {
                    tma_load_4d(smem_u32(dst + c * C::CHUNK), &tmQ, b_item_full + 8 * slot, c * C::CE, h, q0, b);
                    tma_load_4d(smem_u32(dst + C::TILE + c * C::CHUNK), &tmG, b_item_full + 8 * slot,
                                c * C::CE, h, q0, b);
                }
                const size_t vo = ((size_t)b * p.H + h) * p.N_pad + q0;
                bulk_load(smem_u32(dst + 2 * C::TILE), p.lse2 + vo, 512, b_item_full + 8 * slot);
                bulk_load(smem_u32(dst + 2 * C::TILE + 512), p.Dvec + vo, 512, b_item_full + 8 * slot);
            }
            if (!ok) {
                wait_drain(b_kv_full, 0, kWaitLimitNs);
                for (int k = (s > SLOTS ? s - SLOTS : 0); k < s; ++k)
                    wait_drain(b_item_full + 8 * (k % SLOTS), (uint32_t)(k / SLOTS) & 1u, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // The whole warp runs the issue loop (warp-uniform operands); one
        // elected lane issues each MMA and commit.
        auto wb = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
        };
        if (n_steps > 0) {
            const uint64_t kd = smem_desc(smem_u32(sK), 16, 8 * C::CB, 2u);
            const uint64_t vd = smem_desc(smem_u32(sV), 16, 8 * C::CB, 2u);
            bool ok = wb(b_kv_full, 0);
            for (int s = 0; s < n_steps && ok; ++s) {
                const int slot = s % SLOTS;
                ok = wb(b_item_full + 8 * slot, (uint32_t)(s / SLOTS) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint32_t qa = smem_u32(sRing + (size_t)slot * C::ITEM_KV);
                const uint32_t ga = qa + C::TILE;
                const uint64_t qd = smem_desc(qa, 16, 8 * C::CB, 2u);
                const uint64_t gd = smem_desc(ga, 16, 8 * C::CB, 2u);
                // S^T = K Q^T and dP^T = V dO^T (K-major operands, N = 128 queries)
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t o16 = (uint32_t)(c * C::CHUNK + ks * 32) >> 4;
                        const uint32_t acc = (c | ks) != 0;
                        mma_f16_ss_1(tmem + kColS, kd + o16, qd + o16, C::IDESC_S, acc);
                        mma_f16_ss_1(tmem + kColDP, vd + o16, gd + o16, C::IDESC_S, acc);
                    }
                }
                mma_commit_1(b_s_full);
                // dV += P^T dO, dK += dS^T Q: A from TMEM (K = 128 queries, in two
                // halves as the elementwise warps finish them), B MN-major
                const uint64_t gmn = smem_desc(ga, C::CHUNK, 8 * C::CB, 2u);
                const uint64_t qmn = smem_desc(qa, C::CHUNK, 8 * C::CB, 2u);
                for (int half = 0; half < 2 && ok; ++half) {
                    ok = wb(half ? b_p_half1 : b_p_half0, (uint32_t)s & 1u);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kh = 0; kh < BM / C::MMA_K / 2; ++kh) {
                        const int ks = half * (BM / C::MMA_K / 2) + kh;
                        const uint32_t o16 = (uint32_t)(ks * C::MMA_K * C::CB) >> 4;
                        const uint32_t acc = (s > 0 || ks > 0) ? 1u : 0u;
                        // P^T / dS^T of query half h: the first 32 of its own 64 columns
                        const uint32_t pcol = 64u * half + kh * (C::MMA_K / 2);
                        mma_f16_ts_1(tmem + kColAcc, tmem + kColS + pcol, gmn + o16, C::IDESC_ACC, acc);
                        mma_f16_ts_1(tmem + kColAcc + D, tmem + kColDP + pcol, qmn + o16, C::IDESC_ACC,
                                     acc);
                    }
                }
                if (!ok) break;
                mma_commit_1(b_item_empty + 8 * slot);
            }
            if (ok) {
                mma_commit_1(b_acc_done);
            } else {
                mma_commit_1(b_drain);
                wait_drain(b_drain, 0, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ------------------------ elementwise: one key row per thread, two groups
        // Warps 2-5 take the step's queries [0, 64), warps 6-9 queries [64,
        // 128), side by side (two warps per sub-partition hide each other's
        // TMEM and exp latencies); each writes its P^T / dS^T over the first 32
        // of its own 64 columns, which only it has read.
        const int quad = warp & 3;
        const int hq = (warp - 2) >> 2;  // query half of this warp group
        const int r = quad * 32 + lane;
        const int kk = key0 + r;                 // this thread's key
        const bool key_ok = kk < p.N_k;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const float cl = p.scale * 1.4426950408889634f;
        bool ok = true;
        for (int s = 0; s < n_steps; ++s) {
            if (!__all_sync(0xffffffffu, wait_bar(b_s_full, (uint32_t)s & 1u, abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int q0 = (i_lo + s % per_head) * BM;
            const float* vl = reinterpret_cast<const float*>(sRing + (size_t)(s % SLOTS) * C::ITEM_KV + 2 * C::TILE);
            const float* vD = vl + 128;
            // query column c is allowed for this key iff kk <= q0 + c + shift,
            // i.e. c > kk - shift - q0 - 1
            const int c_min = p.causal ? kk - shift - q0 - 1 : -1;
            {
                const int v = hq;
                uint32_t sr[64], dr[64];
                tmem_ld32(t_row + kColS + 64 * v, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_ld32(t_row + kColS + 64 * v + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                tmem_ld32(t_row + kColDP + 64 * v, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
                tmem_ld32(t_row + kColDP + 64 * v + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
                tmem_ld_wait();
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
                uint32_t pk[32], dk[32];
                // every column of this step allowed for every key of the warp:
                // no per-element mask, packed f32x2 arithmetic
                if (__all_sync(0xffffffffu, key_ok && c_min < 64 * v)) {
#pragma unroll
                    for (int x = 0; x < 64; x += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(vl + 64 * v + x);
                        const float4 d4 = *reinterpret_cast<const float4*>(vD + 64 * v + x);
                        float pv[4], dsv[4], a[4], tt[4];
                        ffma2(a[0], a[1], __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), cl, cl,
                              -l4.x, -l4.y);
                        ffma2(a[2], a[3], __uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3]), cl,
                              cl, -l4.z, -l4.w);
#pragma unroll
                        for (int e = 0; e < 4; ++e) pv[e] = ex2(a[e]);
                        fadd2(tt[0], tt[1], __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]),
                              -d4.x, -d4.y);
                        fadd2(tt[2], tt[3], __uint_as_float(dr[x + 2]), __uint_as_float(dr[x + 3]),
                              -d4.z, -d4.w);
                        ffma2(dsv[0], dsv[1], pv[0], pv[1], tt[0], tt[1], 0.f, 0.f);
                        ffma2(dsv[2], dsv[3], pv[2], pv[3], tt[2], tt[3], 0.f, 0.f);
                        if constexpr (KIND == kBF16) {
                            pk[x / 2] = pack_bf16(pv[0], pv[1]);
                            pk[x / 2 + 1] = pack_bf16(pv[2], pv[3]);
                            dk[x / 2] = pack_bf16(dsv[0], dsv[1]);
                            dk[x / 2 + 1] = pack_bf16(dsv[2], dsv[3]);
                        } else {
                            pk[x / 2] = pack_f16(pv[0], pv[1]);
                            pk[x / 2 + 1] = pack_f16(pv[2], pv[3]);
                            dk[x / 2] = pack_f16(dsv[0], dsv[1]);
                            dk[x / 2 + 1] = pack_f16(dsv[2], dsv[3]);
                        }
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 64; x += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(vl + 64 * v + x);
                        const float4 d4 = *reinterpret_cast<const float4*>(vD + 64 * v + x);
                        float pv[4], dsv[4];
                        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = 64 * v + x + e;
                            const bool allowed = key_ok && col > c_min;
                            const float pe = allowed ? ex2(fmaf(__uint_as_float(sr[x + e]), cl, -lv[e])) : 0.f;
                            pv[e] = pe;
                            dsv[e] = pe * (__uint_as_float(dr[x + e]) - dv[e]);
                        }
                        if constexpr (KIND == kBF16) {
                            pk[x / 2] = pack_bf16(pv[0], pv[1]);
                            pk[x / 2 + 1] = pack_bf16(pv[2], pv[3]);
                            dk[x / 2] = pack_bf16(dsv[0], dsv[1]);
                            dk[x / 2 + 1] = pack_bf16(dsv[2], dsv[3]);
                        } else {
                            pk[x / 2] = pack_f16(pv[0], pv[1]);
                            pk[x / 2 + 1] = pack_f16(pv[2], pv[3]);
                            dk[x / 2] = pack_f16(dsv[0], dsv[1]);
                            dk[x / 2 + 1] = pack_f16(dsv[2], dsv[3]);
                        }
                    }
                }
                // 64 queries of P^T / dS^T = 32 columns, over columns this
                // thread has already read; then this half may be consumed
                tmem_st32(t_row + kColS + 64 * v, pk);
                tmem_st32(t_row + kColDP + 64 * v, dk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(v ? b_p_half1 : b_p_half0);
            }
        }
        // ---- epilogue: dV (warps 2-5) and scale * dK (warps 6-9) for this key row
        if (ok && n_steps > 0)
            ok = __all_sync(0xffffffffu, wait_bar(b_acc_done, 0u, abort_flag, lim));
        if (ok) {
            tc_fence_after();
            {
                const int which = hq;
                uint16_t* dst = reinterpret_cast<uint16_t*>(which == 0 ? p.out_a : p.out_b) +
                                (((size_t)b * p.N_k + (key_ok ? kk : 0)) * p.H_kv + hk) * D;
                const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll 1
                for (int u = 0; u < D / 32; ++u) {
                    uint32_t oo[32];
                    if (n_steps > 0) {
                        tmem_ld32(t_row + kColAcc + which * D + 32 * u, oo);
                        tmem_ld_wait();
                        reg_fence32(oo);
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) oo[x] = 0u;
                    }
                    if (!key_ok) continue;
                    uint32_t packed[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float a0 = __uint_as_float(oo[2 * x]) * mul;
                        const float a1 = __uint_as_float(oo[2 * x + 1]) * mul;
                        packed[x] = (KIND == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                    }
                    uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * u);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        d4[x] = make_uint4(packed[4 * x], packed[4 * x + 1], packed[4 * x + 2], packed[4 * x + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- dQ
template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                  const BwdParams p) {
    using C = BCfg<D, KIND>;
    constexpr int KS = C::K_SLOTS_Q, VS = C::V_SLOTS_Q;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by offsetting the shared array itself, so that every
    // pointer derived from it stays in the shared address space (plain loads
    // through it compile to shared-memory loads, not generic ones)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* sQ = smem;
    uint8_t* sG = smem + C::TILE;
    uint8_t* sK = smem + 2 * C::TILE;   // KS K tiles
    uint8_t* sV = sK + (size_t)KS * C::TILE;  // VS V tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(sV + (size_t)VS * C::TILE);
    constexpr int NB = 7 + 2 * (KS + VS);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t b_q_full = smem_u32(bars);
    const uint32_t b_s_full = smem_u32(bars + 1);
    // dS of keys [0, 64) and [64, 128): the dQ MMAs of the first half run while
    // the elementwise warps form the second
    const uint32_t b_p_half0 = smem_u32(bars + 2), b_p_half1 = smem_u32(bars + 5);
    const uint32_t b_acc_done = smem_u32(bars + 3);
    const uint32_t b_drain = smem_u32(bars + 4);
    // dP_j has been read into registers: dP_{j+1} may overwrite it
    const uint32_t b_dp_free = smem_u32(bars + 6);
    const uint32_t b_k_full = smem_u32(bars + 7);                 // + 8 * K slot
    const uint32_t b_k_empty = smem_u32(bars + 7 + KS);           // + 8 * K slot
    const uint32_t b_v_full = smem_u32(bars + 7 + 2 * KS);        // + 8 * V slot
    const uint32_t b_v_empty = smem_u32(bars + 7 + 2 * KS + VS);  // + 8 * V slot

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int b, h, rank;
    decode(blockIdx.x, p, p.H, &b, &h, &rank);
    const int hk = h / p.group;  // K/V head
    const int qt = p.causal ? (p.n_units_tiles - 1 - rank) : rank;  // heaviest first
    const int bh = b * p.H + h;
    const int q0 = qt * BM;
    const int shift = p.N_k - p.N_q;
    int n = 0;  // key tiles this query tile needs
    if (q0 < p.N_q) {
        const int last_row = min(q0 + BM - 1, p.N_q - 1);
        int last_key = p.N_k - 1;
        if (p.causal) last_key = min(last_key, last_row + shift);
        n = last_key < 0 ? 0 : last_key / BN + 1;
    }
    const unsigned long long lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        mbar_init(b_s_full, 1);
        mbar_init(b_p_half0, 128);
        mbar_init(b_p_half1, 128);
        mbar_init(b_acc_done, 1);
        mbar_init(b_drain, 1);
        mbar_init(b_dp_free, 128);
        for (int s = 0; s < KS; ++s) {
            mbar_init(b_k_full + 8 * s, 1);
            mbar_init(b_k_empty + 8 * s, 1);
        }
        for (int s = 0; s < VS; ++s) {
            mbar_init(b_v_full + 8 * s, 1);
            mbar_init(b_v_empty + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
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
        if (lane == 0 && n > 0) {
            mbar_arrive_expect_tx(b_q_full, 2u * C::TILE);
            for (int c = 0; c < C::NC; ++c) {
                tma_load_4d(smem_u32(sQ + c * C::CHUNK), &tmQ, b_q_full, c * C::CE, h, q0, b);
                tma_load_4d(smem_u32(sG + c * C::CHUNK), &tmG, b_q_full, c * C::CE, h, q0, b);
            }
            // K_j then V_j, each into its own ring
            bool ok = true;
            int nk = 0, nv = 0;  // tiles issued into each ring
            for (int j = 0; j < n && ok; ++j) {
                const int ks = j % KS, vs = j % VS;
                ok = wait_bar(b_k_empty + 8 * ks, ((uint32_t)(j / KS) & 1u) ^ 1u, abort_flag, lim);
                if (!ok) break;
                mbar_arrive_expect_tx(b_k_full + 8 * ks, (uint32_t)C::TILE);
                for (int c = 0; c < C::NC; ++c)
                    tma_load_4d(smem_u32(sK + (size_t)ks * C::TILE + c * C::CHUNK), &tmK, b_k_full + 8 * ks,
                                c * C::CE, hk, j * BN, b);
                ++nk;
                ok = wait_bar(b_v_empty + 8 * vs, ((uint32_t)(j / VS) & 1u) ^ 1u, abort_flag, lim);
                if (!ok) break;
                mbar_arrive_expect_tx(b_v_full + 8 * vs, (uint32_t)C::TILE);
                for (int c = 0; c < C::NC; ++c)
                    tma_load_4d(smem_u32(sV + (size_t)vs * C::TILE + c * C::CHUNK), &tmV, b_v_full + 8 * vs,
                                c * C::CE, hk, j * BN, b);
                ++nv;
            }
            if (!ok) {
                wait_drain(b_q_full, 0, kWaitLimitNs);
                for (int k = (nk > KS ? nk - KS : 0); k < nk; ++k)
                    wait_drain(b_k_full + 8 * (k % KS), (uint32_t)(k / KS) & 1u, kWaitLimitNs);
                for (int k = (nv > VS ? nv - VS : 0); k < nv; ++k)
                    wait_drain(b_v_full + 8 * (k % VS), (uint32_t)(k / VS) & 1u, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // The whole warp runs the issue loop (warp-uniform operands); one
        // elected lane issues each MMA and commit.
        auto wb = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
        };
        if (n > 0) {
            const uint64_t qd = smem_desc(smem_u32(sQ), 16, 8 * C::CB, 2u);
            const uint64_t gd = smem_desc(smem_u32(sG), 16, 8 * C::CB, 2u);
            // S_j goes to S buffer j % 2 and dS_j over it, so the scores of key
            // tile j + 1 run while the elementwise warps work on tile j: S_{j+1}
            // at once (its buffer was last read by dQ_{j-1}, issued before), dP_{j+1}
            // once dP_j has been read (dp_free); then dQ_j from dS_j.
            auto sbuf = [](int j) { return (j & 1) ? kColS1 : kColS; };
            auto k_addr = [&](int j) { return smem_u32(sK + (size_t)(j % KS) * C::TILE); };
            auto v_desc = [&](int j) {
                return smem_desc(smem_u32(sV + (size_t)(j % VS) * C::TILE), 16, 8 * C::CB, 2u);
            };
            auto wait_k = [&](int j) { return wb(b_k_full + 8 * (j % KS), (uint32_t)(j / KS) & 1u); };
            auto wait_v = [&](int j) { return wb(b_v_full + 8 * (j % VS), (uint32_t)(j / VS) & 1u); };
            auto issue_s = [&](int j, uint64_t kd) {  // S_j = Q K_j^T
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t o16 = (uint32_t)(c * C::CHUNK + ks * 32) >> 4;
                        mma_f16_ss_1(tmem + sbuf(j), qd + o16, kd + o16, C::IDESC_S, (c | ks) != 0);
                    }
                }
            };
            auto issue_dp = [&](uint64_t vd) {  // dP_j = dO V_j^T
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t o16 = (uint32_t)(c * C::CHUNK + ks * 32) >> 4;
                        mma_f16_ss_1(tmem + kColDP, gd + o16, vd + o16, C::IDESC_S, (c | ks) != 0);
                    }
                }
            };
            bool ok = wb(b_q_full, 0);
            if (ok) ok = wait_k(0);
            if (ok) ok = wait_v(0);
            if (ok) {
                tc_fence_after();
                issue_s(0, smem_desc(k_addr(0), 16, 8 * C::CB, 2u));
                issue_dp(v_desc(0));
                mma_commit_1(b_s_full);
                mma_commit_1(b_v_empty);  // V_0 is read by dP_0 only
            }
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n) {
                    ok = wait_k(j + 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j + 1, smem_desc(k_addr(j + 1), 16, 8 * C::CB, 2u));
                    ok = wait_v(j + 1);
                    if (ok) ok = wb(b_dp_free, (uint32_t)j & 1u);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dp(v_desc(j + 1));
                    mma_commit_1(b_s_full);
                    mma_commit_1(b_v_empty + 8 * ((j + 1) % VS));
                }
                // dQ += dS K: A = dS_j from S buffer j % 2 (K = 128 keys, in two
                // halves), B = K_j MN-major
                const uint64_t kmn = smem_desc(k_addr(j), C::CHUNK, 8 * C::CB, 2u);
                for (int half = 0; half < 2 && ok; ++half) {
                    ok = wb(half ? b_p_half1 : b_p_half0, (uint32_t)j & 1u);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kh = 0; kh < BN / C::MMA_K / 2; ++kh) {
                        const int ks = half * (BN / C::MMA_K / 2) + kh;
                        const uint32_t o16 = (uint32_t)(ks * C::MMA_K * C::CB) >> 4;
                        const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
                        mma_f16_ts_1(tmem + kColAcc, tmem + sbuf(j) + ks * (C::MMA_K / 2), kmn + o16,
                                     C::IDESC_ACC, acc);
                    }
                }
                if (!ok) break;
                mma_commit_1(b_k_empty + 8 * (j % KS));  // K_j is read by S_j and dQ_j
            }
            if (ok) {
                mma_commit_1(b_acc_done);
            } else {
                mma_commit_1(b_drain);
                wait_drain(b_drain, 0, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------- elementwise: one query row per thread
        const int quad = warp & 3;
        const int r = quad * 32 + lane;
        const int qi = q0 + r;
        const bool row_ok = qi < p.N_q;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const float cl = p.scale * 1.4426950408889634f;
        const size_t vo = (size_t)bh * p.N_pad + (row_ok ? qi : 0);
        const float l2 = row_ok ? p.lse2[vo] : INFINITY;
        const float Dr = row_ok ? p.Dvec[vo] : 0.f;
        int row_lim = p.N_k - 1;  // last allowed key of this row
        if (p.causal) row_lim = min(row_lim, qi + shift);
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (!__all_sync(0xffffffffu, wait_bar(b_s_full, (uint32_t)j & 1u, abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sb = (j & 1) ? kColS1 : kColS;  // S buffer of this key tile
            const int cl_max = row_lim - j * BN;  // columns > cl_max are masked
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                uint32_t sr[64], dr[64];
                tmem_ld32(t_row + sb + 64 * v, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                tmem_ld32(t_row + sb + 64 * v + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                tmem_ld32(t_row + kColDP + 64 * v, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
                tmem_ld32(t_row + kColDP + 64 * v + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
                tmem_ld_wait();
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
                if (v == 1) {
                    // all of dP_j is in registers: the next tile's dP may overwrite it
                    tc_fence_before();
                    mbar_arrive(b_dp_free);
                }
                uint32_t dk[32];
                // every key of this step allowed for every row of the warp: no
                // per-element mask, packed f32x2 arithmetic
                if (__all_sync(0xffffffffu, row_ok && cl_max >= BN - 1)) {
#pragma unroll
                    for (int x = 0; x < 64; x += 2) {
                        float a0, a1, t0, t1, d0, d1;
                        ffma2(a0, a1, __uint_as_float(sr[x]), __uint_as_float(sr[x + 1]), cl, cl,
                              -l2, -l2);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        fadd2(t0, t1, __uint_as_float(dr[x]), __uint_as_float(dr[x + 1]), -Dr, -Dr);
                        ffma2(d0, d1, p0, p1, t0, t1, 0.f, 0.f);
                        dk[x / 2] = (KIND == kBF16) ? pack_bf16(d0, d1) : pack_f16(d0, d1);
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < 64; x += 2) {
                        float ds[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int col = 64 * v + x + e;
                            const float pe = (row_ok && col <= cl_max)
                                                 ? ex2(fmaf(__uint_as_float(sr[x + e]), cl, -l2))
                                                 : 0.f;
                            ds[e] = pe * (__uint_as_float(dr[x + e]) - Dr);
                        }
                        dk[x / 2] = (KIND == kBF16) ? pack_bf16(ds[0], ds[1]) : pack_f16(ds[0], ds[1]);
                    }
                }
                // dS of these 64 keys = 32 columns, over S columns read above
                tmem_st32(t_row + sb + 32 * v, dk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(v ? b_p_half1 : b_p_half0);
            }
        }
        if (ok && n > 0) ok = __all_sync(0xffffffffu, wait_bar(b_acc_done, 0u, abort_flag, lim));
        if (ok) {
            tc_fence_after();
            uint16_t* dst = reinterpret_cast<uint16_t*>(p.out_a) +
                            (((size_t)b * p.N_q + (row_ok ? qi : 0)) * p.H + h) * D;
#pragma unroll 1
            for (int u = 0; u < D / 32; ++u) {
                uint32_t oo[32];
                if (n > 0) {
                    tmem_ld32(t_row + kColAcc + 32 * u, oo);
                    tmem_ld_wait();
                    reg_fence32(oo);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) oo[x] = 0u;
                }
                if (!row_ok) continue;
                uint32_t packed[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const float a0 = __uint_as_float(oo[2 * x]) * p.scale;
                    const float a1 = __uint_as_float(oo[2 * x + 1]) * p.scale;
                    packed[x] = (KIND == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                }
                uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * u);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    d4[x] = make_uint4(packed[4 * x], packed[4 * x + 1], packed[4 * x + 2], packed[4 * x + 3]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// heads scheduled together so the tiles they stream (2 N d E bytes per head)
// fill ~48 MiB of L2, group sizes evened out
int heads_per_group(long long n_bh, long long stream_bytes_per_head) {
    long long G = (48LL << 20) / (stream_bytes_per_head > 0 ? stream_bytes_per_head : 1);
    if (G < 1) G = 1;
    if (G > n_bh) G = n_bh;
    const long long n_groups = (n_bh + G - 1) / G;
    return (int)((n_bh + n_groups - 1) / n_groups);
}

template <int D, int KIND>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream) {
    using C = BCfg<D, KIND>;
    if (a.N_q == 0) {
        // no query rows: every key and value gradient is zero
        const size_t bytes = (size_t)a.B * a.N_k * a.H_kv * D * 2;
        cudaError_t e0 = cudaMemsetAsync(a.dk, 0, bytes, stream);
        if (e0 != cudaSuccess) return e0;
        return cudaMemsetAsync(a.dv, 0, bytes, stream);
    }
    const int N_pad = (a.N_q + BM - 1) / BM * BM;
    float* lse2 = static_cast<float*>(a.workspace);
    float* Dvec = lse2 + (size_t)a.B * a.H * N_pad;
    const long long rows = (long long)a.B * a.H * N_pad;
    bwd_prep_kernel<D><<<(unsigned)((rows + 31) / 32), 256, 0, stream>>>(a.o, a.dO, a.lse, lse2, Dvec, a.B,
                                                                      a.H, a.N_q, N_pad, KIND == kFP16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap mq, mk, mv, mg;
    if (!tma::encode_map(&mq, a.q, KIND, a.B, a.N_q, a.H, D, C::CE, BM) ||
        !tma::encode_map(&mk, a.N_k > 0 ? a.k : a.q, KIND, a.B, a.N_k, a.H_kv, D, C::CE, BN) ||
        !tma::encode_map(&mv, a.N_k > 0 ? a.v : a.q, KIND, a.B, a.N_k, a.H_kv, D, C::CE, BN) ||
        !tma::encode_map(&mg, a.dO, KIND, a.B, a.N_q, a.H, D, C::CE, BM))
        return cudaErrorInvalidValue;
    BwdParams p;
    p.B = a.B;
    p.H = a.H;
    p.H_kv = a.H_kv;
    p.group = a.H / a.H_kv;
    p.N_q = a.N_q;
    p.N_k = a.N_k;
    p.N_pad = N_pad;
    p.causal = a.causal;
    p.scale = a.scale;
    p.lse2 = lse2;
    p.Dvec = Dvec;
    p.timeout_ns = kWaitLimitNs;
    const long long n_bh = (long long)a.B * a.H;
    // dK, dV: one CTA per (K/V head, key tile); the query side streams Q and
    // dO of the group's query heads
    const long long n_bhk = (long long)a.B * a.H_kv;
    const int n_kt = (a.N_k + BN - 1) / BN;
    if (n_kt > 0) {
        p.n_units_tiles = n_kt;
        p.heads_per_group = heads_per_group(n_bhk, 2LL * a.N_q * D * 2 * p.group);
        p.out_a = a.dv;
        p.out_b = a.dk;
        const long long n_cta = (long long)n_kt * n_bhk;
        if (n_cta > 0x7fffffffLL) return cudaErrorNotSupported;
        e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::SMEM_KV);
        if (e != cudaSuccess) return e;
        bwd_dkdv_kernel<D, KIND><<<(unsigned)n_cta, kThreadsKV, C::SMEM_KV, stream>>>(mq, mk, mv, mg, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // dQ: one CTA per query tile; the key side streams K and V
    const int n_qt = (a.N_q + BM - 1) / BM;
    p.n_units_tiles = n_qt;
    p.heads_per_group = heads_per_group(n_bh, 2LL * (a.N_k > 0 ? a.N_k : 1) * D * 2 / p.group);
    p.out_a = a.dq;
    p.out_b = nullptr;
    const long long n_cta = (long long)n_qt * n_bh;
    if (n_cta > 0x7fffffffLL) return cudaErrorNotSupported;
    e = cudaFuncSetAttribute(bwd_dq_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM_Q);
    if (e != cudaSuccess) return e;
    bwd_dq_kernel<D, KIND><<<(unsigned)n_cta, kThreads, C::SMEM_Q, stream>>>(mq, mk, mv, mg, p);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(long long B, long long H, long long N_q) {
    const long long N_pad = (N_q + BM - 1) / BM * BM;
    return (size_t)(2 * B * H * N_pad) * sizeof(float);
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream) {
    if (a.dtype == kBF16) {
        if (a.d == 64) return launch_bwd_t<64, kBF16>(a, stream);
        if (a.d == 128) return launch_bwd_t<128, kBF16>(a, stream);
    } else if (a.dtype == kFP16) {
        if (a.d == 64) return launch_bwd_t<64, kFP16>(a, stream);
        if (a.d == 128) return launch_bwd_t<128, kFP16>(a, stream);
    }
    return cudaErrorNotSupported;
}

cudaError_t bwd_take_status(unsigned* out, cudaStream_t stream) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_bwd_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace attn
