// Fused exact-attention forward for head dimension 256 on the fifth-generation
// tensor cores (sm_103a).
//
// The same method as the d = 64 / 128 kernel ("FlashAttention (HI)": "Tiling
// and block processing", "Online softmax computation", "Combining operations
// in one CUDA kernel", and "Development and further research", which names
// head size 256 among FlashAttention-2's extensions; "FlashAttention-2 (BN)":
// "Improved parallelism"; "FlashAttention-3 (BN)": "Asynchronous execution and
// warp specialisation"), laid out for a 256-column output accumulator:
//
//   * one CTA owns one 128-row query tile of one (batch, head): a fp32 O of
//     128 x 256 takes half of TMEM, so two tiles per CTA do not fit;
//   * TMEM = two score buffers S_0, S_1 (128 columns each) + O (256 columns).
//     The scores of key tile j go to S_{j mod 2}; P_j overwrites the start of
//     that buffer, and the scores of key tile j + 2 are issued right behind
//     P_j V_j into the same columns (one thread's MMAs execute in issue order).
//     While the softmax works on S_j, the tensor core runs P_{j-1} V_{j-1} and
//     S_{j+1} (2048 cycles of bf16 MMA per 128-key tile against ~1250 cycles
//     of softmax), so one query tile keeps the tensor pipe busy by itself;
//   * a K or V tile is 64 KB (bf16), so the ring moves half tiles: K split by
//     d (each score MMA reads one 128-key d-chunk), V split by keys (each P V
//     MMA reads 16 keys of all 256 d-columns).  Items are loaded in the order
//     the MMAs first use them: K_0, K_1, V_0, K_2, V_1, K_3, ...;
//   * warp 0 produces (TMA), warp 1 issues MMAs and owns TMEM, warps 2-5 run
//     the softmax, one query row per thread.
//
// Scores are kept in base 2 (the logit scale folds in log2(e) and, for e4m3,
// the q and k descales).  Every mbarrier wait is bounded; on expiry the CTA
// drains what it issued, frees TMEM and exits with the status word set.
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

__device__ unsigned g_tc256_status = 0;

constexpr int D = 256;
constexpr int BM = 128;        // query rows per tile (MMA M)
constexpr int BN = 128;        // keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 232448;

template <int KIND>
struct Cfg256 {
    static constexpr int E = (KIND == kE4M3) ? 1 : 2;   // bytes per element
    // e4m3 inputs: P goes to the P V product as fp16 (as in the d <= 128
    // kernel: an e4m3 P keeps 3 mantissa bits, too few for a weight that is a
    // sizeable share of its row), and V is widened from e4m3 to fp16 in
    // shared memory by a converter warp (exact), whole key tiles, double
    // buffered.
    static constexpr bool F16P = (KIND == kE4M3);
    // producer, MMA issuer, 4 softmax warps (+ 2 V converters for F16P; with
    // eight warps every warp may hold up to 255 registers)
    static constexpr int CONV_WARP0 = 6;
    static constexpr int CONV_WARPS = F16P ? 2 : 0;
    static constexpr int THREADS = 32 * (6 + CONV_WARPS);
    static constexpr int CB = 128;                       // bytes per swizzle chunk row
    static constexpr int CE = CB / E;                    // elements per chunk
    static constexpr int NC = D * E / CB;                // chunks per row: 4 (16-bit), 2 (e4m3)
    static constexpr int QTILE = BM * D * E;             // Q tile bytes
    static constexpr int ITEM = QTILE / 2;               // ring item: half a K or V tile
    static constexpr int KCH = NC / 2;                   // d-chunks per K item
    static constexpr int KCHUNK = BN * CB;               // one K d-chunk: 128 keys x 128 B
    static constexpr int VCHUNK = (BN / 2) * CB;         // one V d-chunk: 64 keys x 128 B
    // fp16 copy of one V half (64 keys x 256 values): four 64-value chunks of
    // 64 keys x 128 B, the layout of a 16-bit V item; one key tile = 2 halves
    static constexpr int V16_HALF = (BN / 2) * D * 2;
    static constexpr int V16_VCHUNK = (BN / 2) * 128;
    static constexpr int V16T = F16P ? 2 * V16_HALF : 0;
    // q_full, s_full x2, p_full x2, pv_done, drain, o_done, v16_full x2, v16_empty x2
    static constexpr int NB_FIXED = 1 + 2 + 2 + 1 + 1 + 1 + 4;
    static constexpr int SLOTS_FIT = (kSmemLimit - 1024 - QTILE - 2 * V16T - 512) / ITEM;
    static constexpr int SLOTS = SLOTS_FIT > 12 ? 12 : SLOTS_FIT;
    static constexpr int NB = NB_FIXED + 2 * SLOTS;
    static constexpr size_t SMEM =
        1024 + (size_t)QTILE + 2 * (size_t)V16T + (size_t)SLOTS * ITEM + NB * 8 + 16;
    static constexpr int MMA_K = 32 / E;                 // K per Q K^T MMA instruction
    static constexpr int PV_K = F16P ? 16 : MMA_K;       // keys per P V MMA instruction
    static constexpr int PE = F16P ? 2 : E;              // bytes per P element
    static constexpr uint32_t FMT = (KIND == kBF16) ? 1u : 0u;
    static constexpr uint32_t IDESC_QK = instr_desc(FMT, FMT, 0, 0, BM, BN);
    static constexpr uint32_t IDESC_PV =
        instr_desc(F16P ? 0u : FMT, F16P ? 0u : FMT, 0, 1, BM, D);
    static constexpr uint32_t P_COLS = BN * PE / 4;      // TMEM columns holding P
    // Rescale rule as in the d = 64 / 128 kernel: the running output is
    // rescaled when the row maximum grew by more than 2^8 (P stays <= 256).
    static constexpr float RESCALE_THRESHOLD = 8.0f;
    static_assert(SLOTS >= 4, "ring depth");
    static_assert(!F16P || SLOTS % 4 == 0, "F16P: K and V items keep to their own slots");
    static_assert(SMEM <= (size_t)kSmemLimit, "shared memory budget");
};

// TMEM columns: S_0 [0,128), S_1 [128,256) (P_j overwrites the start of
// S_{j mod 2}), O [256, 512).
constexpr uint32_t kColO = 256;

struct Tc256Params {
    int B, H, N_q, N_k;
    int H_kv;
    int n_tiles;          // ceil(N_q / 128)
    int heads_per_group;
    int causal;
    float scale;
    void* o;
    float* lse;
    const float* q_descale;
    const float* k_descale;
    const float* v_descale;
    unsigned long long timeout_ns;  // limit of every bounded wait
    unsigned long long drain_ns;    // limit of the abort path's drains (>= 2 s)
    int items_limit;                // K/V ring items the loader issues (abort-path check)
    int n_splits;
    float* part_o;    // [n_splits][B*H][N_q][256]
    float* part_lse;  // [n_splits][B*H][N_q]
};

// Bounded waits (shared implementation) reporting to this file's status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long limit_ns) {
    return bounded_wait(bar, parity, abort_flag, limit_ns, &g_tc256_status);
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    bounded_drain(bar, parity, limit_ns);
}

__device__ __forceinline__ int kv_tiles_for(int q0, const Tc256Params& p) {
    if (q0 >= p.N_q) return 0;
    const int last_row = min(q0 + BM - 1, p.N_q - 1);
    int last_key = p.N_k - 1;
    if (p.causal) last_key = min(last_key, last_row + (p.N_k - p.N_q));
    return last_key < 0 ? 0 : last_key / BN + 1;
}

// Ring items in load order, each group two items (halves); returns false past
// the end, *is_v and *tile say what group g is.
//  16-bit kinds: K_0, K_1 (if any), then for j = 0..n-1: V_j, K_{j+2} (if any):
//   the MMA thread consumes every item, so slots may alternate freely between
//   K and V.
//  F16P (ALT): K_0, V_0, K_1, V_1, ...: with the ring a multiple of four items
//   a slot only ever holds K (read by the MMA thread) or only V (read by the
//   converter), so each slot's barriers have one waiter that sees every phase
//   (a parity wait is only sound for a waiter at most one phase behind).
template <bool ALT>
__device__ __forceinline__ bool group_of(int g, int n, bool* is_v, int* tile) {
    if (n <= 0) return false;
    if (ALT) {
        if (g >= 2 * n) return false;
        *is_v = (g & 1) != 0;
        *tile = g >> 1;
        return true;
    }
    const int nk0 = n > 1 ? 2 : 1;  // leading K groups
    if (g < nk0) {
        *is_v = false;
        *tile = g;
        return true;
    }
    int r = g - nk0;  // pairs (V_j, K_{j+2}) while j + 2 < n, then V_j alone
    const int paired = n > 2 ? n - 2 : 0;
    if (r < 2 * paired) {
        *is_v = (r & 1) == 0;
        *tile = *is_v ? (r >> 1) : (r >> 1) + 2;
        return true;
    }
    r -= 2 * paired;
    const int j = paired + r;
    if (j >= n) return false;
    *is_v = true;
    *tile = j;
    return true;
}

template <int KIND>
__global__ void __launch_bounds__(Cfg256<KIND>::THREADS, 1)
    attn_tc256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const Tc256Params p) {
    using C = Cfg256<KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;
    uint8_t* sV16 = smem + C::QTILE;          // two fp16 V tiles (F16P only)
    uint8_t* sKV = sV16 + 2 * C::V16T;        // SLOTS items
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + (size_t)C::SLOTS * C::ITEM);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    // Phases: an mbarrier parity wait is unambiguous only while the barrier is
    // at most one phase away from the awaited one.  The softmax can run two key
    // tiles ahead of the MMA thread's P wait (S_{j+1} was issued before P_j V_j),
    // so P has one barrier per score buffer; and the epilogue waits on o_done,
    // committed once after the last P V, because pv_done may then be two phases
    // behind.
    const uint32_t b_q_full = smem_u32(bars);
    const uint32_t b_s_full = smem_u32(bars + 1);  // + 8 * buffer
    const uint32_t b_p_full = smem_u32(bars + 3);  // + 8 * buffer
    const uint32_t b_pv_done = smem_u32(bars + 5);
    const uint32_t b_drain = smem_u32(bars + 6);
    const uint32_t b_o_done = smem_u32(bars + 7);
    const uint32_t b_v16_full = smem_u32(bars + 8);   // + 8 * buffer (F16P)
    const uint32_t b_v16_empty = smem_u32(bars + 10); // + 8 * buffer (F16P)
    const uint32_t b_kv_full = smem_u32(bars + C::NB_FIXED);               // + 8 * slot
    const uint32_t b_kv_empty = smem_u32(bars + C::NB_FIXED + C::SLOTS);   // + 8 * slot

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- schedule: groups of heads whose K/V fit in L2; inside a group the
    // query tile is the slow coordinate (heaviest causal tile first).
    const long long n_bh = (long long)p.B * p.H;
    const long long G = p.heads_per_group;
    const long long per_group = (long long)p.n_tiles * G;
    const long long n_full = n_bh / G;
    const long long L = blockIdx.x;
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
    const int rank = (int)(rem / Gg);
    const int bh = (int)(g * G + rem % Gg);
    const int b = bh / p.H, h = bh % p.H;
    const int h_kv = h / (p.H / p.H_kv);
    const int tile = p.causal ? (p.n_tiles - 1 - rank) : rank;
    const int q0 = tile * BM;
    int n = kv_tiles_for(q0, p);
    int j0 = 0;
    if (p.n_splits > 1) {
        const int per = (n + p.n_splits - 1) / p.n_splits;
        j0 = min(n, (int)blockIdx.y * per);
        n = max(0, min(n, j0 + per) - j0);
    }
    const unsigned long long lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        mbar_init(b_s_full, 1);
        mbar_init(b_s_full + 8, 1);
        mbar_init(b_p_full, 128);
        mbar_init(b_p_full + 8, 128);
        mbar_init(b_pv_done, 1);
        mbar_init(b_drain, 1);
        mbar_init(b_o_done, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(b_v16_full + 8 * t, 2);    // the two converter warps
            mbar_init(b_v16_empty + 8 * t, 1);   // the P V MMAs of the tile
        }
        for (int s = 0; s < C::SLOTS; ++s) {
            mbar_init(b_kv_full + 8 * s, 1);
            mbar_init(b_kv_empty + 8 * s, 1);
        }
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
    auto slot_of = [](int it) { return it % C::SLOTS; };
    auto par_of = [](int it) { return (uint32_t)(it / C::SLOTS) & 1u; };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && n > 0) {
            mbar_arrive_expect_tx(b_q_full, (uint32_t)C::QTILE);
            for (int c = 0; c < C::NC; ++c)
                tma_load_4d(smem_u32(sQ + c * C::KCHUNK), &tmQ, b_q_full, c * C::CE, h, q0, b);
            int it = 0;
            bool ok = true;
            bool is_v;
            int t_kv;
            for (int grp = 0; ok && group_of<C::F16P>(grp, n, &is_v, &t_kv); ++grp) {
                const int key0 = (j0 + t_kv) * BN;
                for (int half = 0; half < 2; ++half, ++it) {
                    if (it >= p.items_limit) {
                        ok = false;  // stop loading; nothing issued needs a drain beyond the usual
                        break;
                    }
                    const int slot = slot_of(it);
                    if (!wait_bar(b_kv_empty + 8 * slot, par_of(it) ^ 1u, abort_flag, lim)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_kv_full + 8 * slot, C::ITEM);
                    uint8_t* dst = sKV + (size_t)slot * C::ITEM;
                    if (is_v) {
                        // keys [key0 + 64 half, +64), every d-chunk
                        for (int c = 0; c < C::NC; ++c)
                            tma_load_4d(smem_u32(dst + c * C::VCHUNK), &tmV, b_kv_full + 8 * slot,
                                        c * C::CE, h_kv, key0 + half * (BN / 2), b);
                    } else {
                        // d-chunks [half KCH, +KCH) of all 128 keys
                        for (int c = 0; c < C::KCH; ++c)
                            tma_load_4d(smem_u32(dst + c * C::KCHUNK), &tmK, b_kv_full + 8 * slot,
                                        (half * C::KCH + c) * C::CE, h_kv, key0, b);
                    }
                }
            }
            if (!ok) {
                wait_drain(b_q_full, 0, p.drain_ns);
                for (int k = (it > C::SLOTS ? it - C::SLOTS : 0); k < it; ++k)
                    wait_drain(b_kv_full + 8 * slot_of(k), par_of(k), p.drain_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        // The whole warp runs the issue loop (warp-uniform operands); one
        // elected lane issues each MMA and commit.
        auto wb = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
        };
        if (n > 0) {
            // S_{buf} = Q K^T from the two K items at ring positions it, it + 1
            auto issue_qk = [&](int buf, int it) {
                const uint64_t qd = smem_desc(smem_u32(sQ), 16, 8 * C::CB, 2u);
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
                    const int item = it + c / C::KCH;
                    const uint64_t kd = smem_desc(
                        smem_u32(sKV + (size_t)slot_of(item) * C::ITEM + (c % C::KCH) * C::KCHUNK), 16,
                        8 * C::CB, 2u);
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t a16 = (uint32_t)(c * C::KCHUNK + ks * 32) >> 4;
                        const uint32_t b16 = (uint32_t)(ks * 32) >> 4;
                        const uint32_t acc = (c | ks) != 0;
                        if constexpr (KIND == kE4M3)
                            mma_f8_ss_1(tmem + 128u * buf, qd + a16, kd + b16, C::IDESC_QK, acc);
                        else
                            mma_f16_ss_1(tmem + 128u * buf, qd + a16, kd + b16, C::IDESC_QK, acc);
                    }
                }
            };
            // O += P_{buf} V from the two V items at ring positions it, it + 1
            auto issue_pv = [&](int buf, int it, bool first) {
                if constexpr (C::F16P) {
                    // B = the fp16 copy of V_j in buffer `it` (here the buffer index)
#pragma unroll
                    for (int ks = 0; ks < BN / C::PV_K; ++ks) {
                        const int key = ks * C::PV_K;
                        const uint64_t vd = smem_desc(
                            smem_u32(sV16 + (size_t)it * C::V16T + (key / (BN / 2)) * C::V16_HALF +
                                     (key % (BN / 2)) * 128),
                            C::V16_VCHUNK, 8 * 128, 2u);
                        const uint32_t a_tmem = tmem + 128u * buf + ks * (C::PV_K * 2 / 4);
                        const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
                        mma_f16_ts_1(tmem + kColO, a_tmem, vd, C::IDESC_PV, acc);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < BN / C::MMA_K; ++ks) {
                        const int key = ks * C::MMA_K;
                        const int item = it + key / (BN / 2);
                        // V is MN-major: 8-key groups 8*CB apart, d-chunks VCHUNK apart
                        const uint64_t vd = smem_desc(
                            smem_u32(sKV + (size_t)slot_of(item) * C::ITEM + (key % (BN / 2)) * C::CB),
                            C::VCHUNK, 8 * C::CB, 2u);
                        const uint32_t a_tmem = tmem + 128u * buf + ks * (C::MMA_K * C::E / 4);
                        const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
                        if constexpr (KIND == kE4M3)
                            mma_f8_ts_1(tmem + kColO, a_tmem, vd, C::IDESC_PV, acc);
                        else
                            mma_f16_ts_1(tmem + kColO, a_tmem, vd, C::IDESC_PV, acc);
                    }
                }
            };
            auto wait_items = [&](int it) {
                return wb(b_kv_full + 8 * slot_of(it), par_of(it)) &&
                       wb(b_kv_full + 8 * slot_of(it + 1), par_of(it + 1));
            };
            auto release_items = [&](int it) {
                mma_commit_1(b_kv_empty + 8 * slot_of(it));
                mma_commit_1(b_kv_empty + 8 * slot_of(it + 1));
            };

            // ring position of the next group (16-bit kinds); F16P: K_t sits at
            // positions 4t, 4t + 1
            int it = 0;
            bool ok = wb(b_q_full, 0);
            // scores of K_0 and K_1 into S_0 and S_1
            for (int t = 0; t < 2 && t < n && ok; ++t) {
                const int pos = C::F16P ? 4 * t : it;
                ok = wait_items(pos);
                if (!ok) break;
                tc_fence_after();
                issue_qk(t, pos);
                mma_commit_1(b_s_full + 8 * t);
                release_items(pos);
                it += 2;
            }
            // per key tile j: O += P_j V_j, then the scores of K_{j+2} into the
            // buffer P_j was read from (the same thread's MMAs run in order)
            for (int j = 0; j < n && ok; ++j) {
                const int buf = j & 1;
                // F16P: the V items go to the converter; P V reads its fp16 copy
                ok = C::F16P ? wb(b_v16_full + 8 * (j & 1), (uint32_t)(j >> 1) & 1u) : wait_items(it);
                if (ok) ok = wb(b_p_full + 8 * buf, (uint32_t)(j >> 1) & 1u);
                if (!ok) break;
                tc_fence_after();
                issue_pv(buf, C::F16P ? (j & 1) : it, j == 0);
                mma_commit_1(b_pv_done);
                if (j + 1 == n) mma_commit_1(b_o_done);
                if constexpr (C::F16P)
                    mma_commit_1(b_v16_empty + 8 * (j & 1));
                else
                    release_items(it);
                it += 2;
                if (j + 2 < n) {
                    const int pos = C::F16P ? 4 * (j + 2) : it;
                    ok = wait_items(pos);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(buf, pos);
                    mma_commit_1(b_s_full + 8 * buf);
                    release_items(pos);
                    it += 2;
                }
            }
            if (!ok) {
                mma_commit_1(b_drain);
                wait_drain(b_drain, 0, p.drain_ns);
            }
        }
        __syncwarp();
    } else if (C::F16P && warp >= C::CONV_WARP0) {
        // ------------------------------------------ V converters (F16P only)
        // Two warps widen each V tile (ring positions 4j + 2, 4j + 3: two
        // half items) into fp16 buffer j % 2, laid out like a 16-bit V item.
        // Warp c takes half item c (64 keys x 256 values): it loads its 16 KB
        // into registers, frees the ring slot at once (so the next V tile's
        // load overlaps this conversion), then waits for the fp16 buffer and
        // writes it.
        // Lane-to-unit mapping: the eight lanes of a quarter-warp take two
        // adjacent rows whose units go to different fp16 chunks, so both the
        // e4m3 loads and the fp16 stores hit eight different bank groups.
        const int hh = warp - C::CONV_WARP0;
        constexpr int PER = (BN / 2) * (D / 16) / 32;  // 16-byte units per lane: 32
        for (int jv = 0; jv < n; ++jv) {
            const int it = 4 * jv + 2 + hh;
            bool ok = __all_sync(0xffffffffu, wait_bar(b_kv_full + 8 * slot_of(it), par_of(it), abort_flag, lim));
            if (!ok) break;
            const uint32_t src = smem_u32(sKV + (size_t)slot_of(it) * C::ITEM);
            uint32_t x[PER][4];
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                // unit lane + 32 k: e4m3 d-chunk k / 16 (values 128 (k / 16) .. +127)
                const int cc = k >> 4, i2 = (lane + 32 * k) & 511;
                const int w_lo = i2 & 3, half = (i2 >> 2) & 1, sel = (i2 >> 3) & 1;
                const int rr = 2 * (i2 >> 4) + half, w = 4 * (half ^ sel) + w_lo;
                ld_shared_v4(src + (uint32_t)(cc * C::VCHUNK + rr * 128 + ((w ^ (rr & 7)) << 4)), x[k]);
            }
            // the loads are complete once their values are used; the release
            // below orders them before the producer's next TMA into the slot
            uint32_t keep = 0;
#pragma unroll
            for (int k = 0; k < PER; ++k) keep |= x[k][0] | x[k][1] | x[k][2] | x[k][3];
            asm volatile("" ::"r"(keep));
            __syncwarp();
            mbar_arrive_1(b_kv_empty + 8 * slot_of(it));
            ok = __all_sync(0xffffffffu, wait_bar(b_v16_empty + 8 * (jv & 1),
                                                  ((uint32_t)(jv >> 1) & 1u) ^ 1u, abort_flag, lim));
            if (!ok) break;
            const uint32_t dst = smem_u32(sV16 + (size_t)(jv & 1) * C::V16T + hh * C::V16_HALF);
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                const int cc = k >> 4, i2 = (lane + 32 * k) & 511;
                const int w_lo = i2 & 3, half = (i2 >> 2) & 1, sel = (i2 >> 3) & 1;
                const int rr = 2 * (i2 >> 4) + half, w = 4 * (half ^ sel) + w_lo;
                uint32_t hv[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    hv[2 * e] = e4m3x2_to_f16x2((uint16_t)(x[k][e] & 0xffffu));
                    hv[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(x[k][e] >> 16));
                }
                // values d = 128 cc + 16 w .. +15: fp16 chunk 2 cc + w / 4, units 2 (w % 4), +1
                const uint32_t row = dst + (uint32_t)((2 * cc + (w >> 2)) * C::V16_VCHUNK + rr * 128);
                const int u0 = 2 * (w & 3);
                st_shared_v4(row + (uint32_t)((u0 ^ (rr & 7)) << 4), hv[0], hv[1], hv[2], hv[3]);
                st_shared_v4(row + (uint32_t)(((u0 + 1) ^ (rr & 7)) << 4), hv[4], hv[5], hv[6], hv[7]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            mbar_arrive_1(b_v16_full + 8 * (jv & 1));
        }
    } else {
        // --------------------------------------- softmax + epilogue (128 thr)
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;
        const int row_g = q0 + r;
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const int shift = p.N_k - p.N_q;
        int row_lim = p.N_k - 1;
        if (p.causal) row_lim = min(row_lim, row_g + shift);
        const int tile_lim = p.causal ? min(p.N_k - 1, q0 + shift) : p.N_k - 1;
        float dq = 1.f, dk = 1.f, dv = 1.f;
        if (KIND == kE4M3) {
            if (p.q_descale) dq = p.q_descale[bh];
            if (p.k_descale) dk = p.k_descale[b * p.H_kv + h_kv];
            if (p.v_descale) dv = p.v_descale[b * p.H_kv + h_kv];
        }
        const float c = p.scale * dq * dk * 1.4426950408889634f;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;

        for (int j = 0; j < n; ++j) {
            const int buf = j & 1;
            if (!__all_sync(0xffffffffu, wait_bar(b_s_full + 8 * buf, (uint32_t)(j >> 1) & 1u,
                                                  abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[BN];
            float rmx;  // the row's maximum, from the load itself
            tmem_ld128_max(t_row + 128u * buf, sr, rmx);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < BN / 32; ++u)
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * u]));
            reg_fence_f(rmx);
            float s[BN];
#pragma unroll
            for (int x = 0; x < BN; ++x) s[x] = __uint_as_float(sr[x]);

            const int kbase = (j0 + j) * BN;
            float mx;
            if (kbase + BN - 1 > tile_lim) {
                const int cl = row_lim - kbase;
#pragma unroll
                for (int x = 0; x < BN; ++x)
                    if (x > cl) s[x] = -INFINITY;
                // row maximum of the masked row (the load's maximum includes
                // the masked columns)
                float mc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mc[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
                for (int x = 16; x < BN; x += 16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) mc[k] = max3(mc[k], s[x + k], s[x + k + 8]);
                }
                mx = max3(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7]));
            } else {
                mx = rmx;
            }
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
            float sc[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) sc[k] = 0.f;
            constexpr int PER_CHUNK = 32 * 4 / C::PE;  // score columns per 32 TMEM columns
#pragma unroll
            for (int u = 0; u < (int)C::P_COLS / 32; ++u) {
                uint32_t pk[32];
#pragma unroll
                for (int x = 0; x < PER_CHUNK; x += 2) {
                    const int y = u * PER_CHUNK + x;
                    float a0, a1;
                    ffma2(a0, a1, s[y], s[y + 1], c, c, -m_ref, -m_ref);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    const int k = ((x / 2) & 3) * 2;
                    fadd2(sc[k], sc[k + 1], sc[k], sc[k + 1], p0, p1);
                    pk[x / 2] = (KIND == kBF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
                }
                tmem_st32(t_row + 128u * buf + 32 * u, pk);
            }
            const float sum =
                ((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7]));
            l = l * alpha + sum;

            if (any && j > 0) {
                // O is stable once P_{j-1} V_{j-1} has completed.  S_j exists,
                // so P_{j-2} V_{j-2} has completed (the score MMA ran after it)
                // and P_j V_j is not issued yet: pv_done is in phase j-1 or j.
                if (!__all_sync(0xffffffffu,
                                wait_bar(b_pv_done, (uint32_t)(j - 1) & 1u, abort_flag, lim))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int u = 0; u < D / 64; ++u) {
                    uint32_t oo[64];
                    const uint32_t ta = t_row + kColO + 64 * u;
                    tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(&oo[0]));
                    tmem_ld32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(&oo[32]));
                    tmem_ld_wait();
                    reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&oo[0]));
                    reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&oo[32]));
#pragma unroll
                    for (int x = 0; x < 64; x += 2) {
                        float a0 = __uint_as_float(oo[x]), a1 = __uint_as_float(oo[x + 1]);
                        ffma2(a0, a1, a0, a1, alpha, alpha, 0.f, 0.f);
                        oo[x] = __float_as_uint(a0);
                        oo[x + 1] = __float_as_uint(a1);
                    }
                    tmem_st32(ta, *reinterpret_cast<const uint32_t(*)[32]>(&oo[0]));
                    tmem_st32(ta + 32, *reinterpret_cast<const uint32_t(*)[32]>(&oo[32]));
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(b_p_full + 8 * buf);
        }

        if (ok && n > 0)
            ok = __all_sync(0xffffffffu, wait_bar(b_o_done, 0u, abort_flag, lim));
        if (ok) {
            tc_fence_after();
            const bool valid = row_g < p.N_q;
            const bool has = l > 0.f;
            const float inv = has ? dv / l : 0.f;
            const bool split = p.n_splits > 1;
            const size_t prow_idx =
                ((size_t)blockIdx.y * ((size_t)p.B * p.H) + bh) * p.N_q + (valid ? row_g : 0);
            uint16_t* orow = reinterpret_cast<uint16_t*>(p.o) +
                             (((size_t)b * p.N_q + (valid ? row_g : 0)) * p.H + h) * D;
            float* prow = split ? p.part_o + prow_idx * D : nullptr;
#pragma unroll 1
            for (int u = 0; u < D / 32; ++u) {
                uint32_t oo[32];
                if (n > 0) {
                    tmem_ld32(t_row + kColO + 32 * u, oo);
                    tmem_ld_wait();
                    reg_fence32(oo);
                } else {
#pragma unroll
                    for (int x = 0; x < 32; ++x) oo[x] = 0u;
                }
                if (!valid) continue;
                if (split) {
                    float4* dst = reinterpret_cast<float4*>(prow + 32 * u);
#pragma unroll
                    for (int x = 0; x < 8; ++x)
                        dst[x] = make_float4(__uint_as_float(oo[4 * x]) * inv,
                                             __uint_as_float(oo[4 * x + 1]) * inv,
                                             __uint_as_float(oo[4 * x + 2]) * inv,
                                             __uint_as_float(oo[4 * x + 3]) * inv);
                } else {
                    uint32_t packed[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float a0 = __uint_as_float(oo[2 * x]) * inv;
                        const float a1 = __uint_as_float(oo[2 * x + 1]) * inv;
                        packed[x] = (KIND == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                    }
                    uint4* dst = reinterpret_cast<uint4*>(orow + 32 * u);
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        dst[x] = make_uint4(packed[4 * x], packed[4 * x + 1], packed[4 * x + 2],
                                            packed[4 * x + 3]);
                }
            }
            const float lse_row = has ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            if (valid && split)
                p.part_lse[prow_idx] = lse_row;
            else if (valid && p.lse)
                p.lse[(size_t)bh * p.N_q + row_g] = lse_row;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int KIND>
cudaError_t launch_k(const Problem& pr, cudaStream_t stream, int n_splits, float* part_o,
                     float* part_lse) {
    using C = Cfg256<KIND>;
    CUtensorMap mq, mk, mv;
    if (!tma::encode_map(&mq, pr.q, KIND, pr.B, pr.N_q, pr.H, D, C::CE, BM) ||
        !tma::encode_map(&mk, pr.N_k > 0 ? pr.k : pr.q, KIND, pr.B, pr.N_k, pr.H_kv, D, C::CE, BN) ||
        !tma::encode_map(&mv, pr.N_k > 0 ? pr.v : pr.q, KIND, pr.B, pr.N_k, pr.H_kv, D, C::CE, BN / 2))
        return cudaErrorInvalidValue;
    Tc256Params p;
    p.B = pr.B;
    p.H = pr.H;
    p.H_kv = pr.H_kv;
    p.N_q = pr.N_q;
    p.N_k = pr.N_k;
    p.n_tiles = (pr.N_q + BM - 1) / BM;
    p.causal = pr.causal;
    p.scale = pr.scale;
    p.o = pr.o;
    p.lse = pr.lse;
    p.q_descale = pr.q_descale;
    p.k_descale = pr.k_descale;
    p.v_descale = pr.v_descale;
    p.timeout_ns = pr.selftest_wait_ns ? pr.selftest_wait_ns : kWaitLimitNs;
    p.drain_ns = kWaitLimitNs;
    p.items_limit = pr.selftest_items > 0 ? pr.selftest_items : 0x7fffffff;
    p.n_splits = n_splits;
    p.part_o = part_o;
    p.part_lse = part_lse;
    const long long n_bh = (long long)pr.B * pr.H;
    // Heads scheduled together: their K/V (2 N_k d E bytes per K/V head, a K/V
    // head shared by H / H_kv query heads) fill ~48 MiB of L2, groups evened out.
    const long long kv_head_bytes = 2LL * (pr.N_k > 0 ? pr.N_k : 1) * D * C::E;
    long long G = (48LL << 20) * (pr.H / pr.H_kv) / kv_head_bytes;
    if (G < 1) G = 1;
    if (G > n_bh) G = n_bh;
    const long long n_groups = (n_bh + G - 1) / G;
    G = (n_bh + n_groups - 1) / n_groups;
    p.heads_per_group = (int)G;
    const long long n_cta = (long long)p.n_tiles * n_bh;
    if (n_cta > 0x7fffffffLL) return cudaErrorNotSupported;
    if (n_splits < 1 || n_splits > 65535) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(attn_tc256_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)n_cta, (unsigned)n_splits);
    attn_tc256_kernel<KIND><<<grid, C::THREADS, C::SMEM, stream>>>(mq, mk, mv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc256(const Problem& p, cudaStream_t stream, int n_splits, float* part_o,
                         float* part_lse) {
    if (p.d != D) return cudaErrorNotSupported;
    switch (p.dtype) {
        case kBF16: return launch_k<kBF16>(p, stream, n_splits, part_o, part_lse);
        case kFP16: return launch_k<kFP16>(p, stream, n_splits, part_o, part_lse);
        case kE4M3: return launch_k<kE4M3>(p, stream, n_splits, part_o, part_lse);
    }
    return cudaErrorNotSupported;
}

cudaError_t tc256_take_status(unsigned* out, cudaStream_t stream) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_tc256_status, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyToSymbolAsync(g_tc256_status, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace attn
