// Fused exact-attention forward on the fifth-generation tensor cores (sm_103a).
//
// The pages' method ("FlashAttention (HI)": "Tiling and block processing",
// "Online softmax computation", "Combining operations in one CUDA kernel";
// "FlashAttention-2 (BN)": "Improved parallelism"; "FlashAttention-3 (BN)":
// "Asynchronous execution and warp specialisation", "Reducing memory
// operations") mapped onto Blackwell:
//
//   * one CTA owns two adjacent 128-row query tiles (A, B) of one (batch,
//     head), so every K/V tile brought on chip serves 256 query rows; the
//     grid spans batch x heads x tile pairs (one head over many SMs), a few
//     heads at a time so their K/V stay in L2, heaviest causal pairs first;
//   * warp 0 (producer) streams Q_A, Q_B once and then K_0, V_0, K_1, V_1, ...
//     through a ring of shared-memory slots with TMA, guarded by mbarriers;
//   * warps 1 and 2 issue the tcgen05 MMAs, one warp per tile (the whole warp
//     runs the issue loop on warp-uniform operands, one elected lane issues;
//     warp 1 owns TMEM): S_t = Q_t K_j^T into one TMEM score buffer that the
//     two tiles take in turns (A_0, B_0, A_1, ...), and O_t += P_t V_j with
//     P_t read from a TMEM buffer of its own;
//   * warps 3-6 (tile A) and 7-10 (tile B), one query row per thread, run the
//     online softmax: TMEM -> registers (after which the score buffer is free
//     for the other tile's next Q K^T), causal / ragged mask on the tiles that
//     need it, row maximum, exp2, row sum, P to its TMEM buffer as bf16 /
//     fp16 (fp16 for e4m3 inputs); they rescale the running output in TMEM
//     only when the row maximum grew by more than 2^8 (P stays <= 256), and
//     write O / lse at the end;
//   * e4m3 inputs: V is widened to fp16 on chip by a converter warp (warp 11)
//     with shares taken by the producer and the issuers, or, with a caller
//     workspace, once per call by widen_e4m3_kernel before this kernel.
//   The two softmax groups interleave with each other's MMAs: while group A
//   turns S_A into P_A the tensor core runs P_B V_j and the next S_B, and the
//   other way round (the pages' ping-pong between two warp groups).
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
#include "bounded_wait.cuh"
#include "tc_ptx.cuh"
#include "tma_map.cuh"

namespace attn {
namespace {

using namespace ptx;

__device__ unsigned g_tc_status = 0;

// Kernel kinds: the input dtype (kBF16, kFP16, kE4M3), plus the flag kV16
// for e4m3 inputs whose V arrives already widened to fp16 (the host runs
// widen_e4m3_kernel into the caller's workspace first): Q and K are e4m3, V
// tiles come into the ring by TMA as fp16.
constexpr int kV16 = 16;
constexpr int kE4M3_V16 = kE4M3 | kV16;

// a compile-time int passed as a value (picks a generic lambda's instance)
template <int N>
struct IntC {
    static constexpr int value = N;
};

constexpr int BM = 128;        // query rows per tile (MMA M)
constexpr int BN = 128;        // keys per tile (MMA N of Q K^T, K of P V)
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 232448;  // max dynamic shared memory per CTA

template <int D, int KIND>
struct Cfg {
    static constexpr int BASE = KIND & 15;                 // input dtype
    static constexpr bool E4 = (BASE == kE4M3);            // e4m3 Q and K
    static constexpr int E = E4 ? 1 : 2;                   // bytes per element of Q, K
    static constexpr int RB = D * E;                       // bytes per row
    static constexpr int CB = RB >= 128 ? 128 : RB;        // bytes per swizzle chunk
    static constexpr int NC = RB / CB;                     // chunks per row
    static constexpr int TILE = BM * RB;                   // bytes per 128-row tile
    static constexpr int CHUNK = BM * CB;                  // bytes per chunk of a tile
    // TMEM: one score buffer S that the two tiles take in turns (each tile's
    // softmax frees it as soon as it has loaded its scores), P_A and P_B (64
    // columns each: 128 16-bit values per row) and O_A, O_B.  With P in
    // buffers of its own, a tile's next Q K^T waits only for the other
    // tile's softmax to load its scores, not for the tile's own P V (as it
    // would with P written over S); measured against P over S (bf16, d =
    // 128, causal, B1 H16 N16384): 0.650 -> 0.645 ms, (B2 H16 N4096): 0.108
    // -> 0.103 ms; against P in shared memory (bf16, d = 64, B4 H16 N1024):
    // 0.032 -> 0.0285 ms.
    // e4m3 inputs: P goes to the P V product as fp16, not e4m3.  An e4m3 P
    // keeps 3 mantissa bits, so a weight that is a sizeable share of its row
    // but not the row maximum is off by up to 2^-4 of itself, and with V
    // values of a few tens (the 0.1 % x10 outliers) that is an O error of
    // several 1e-2 to a few 1e-1 on rare rows; fp16 P (10 bits) keeps every
    // row within about 1e-3 of exact.  The P V MMA is then kind::f16 with
    // A = P in TMEM and B = V in fp16 (every e4m3 value is exact in fp16),
    // widened either on chip, a tile ahead of its use, or once per call into
    // a workspace (kV16).
    static constexpr bool V16G = (KIND & kV16) != 0;
    // e4m3 V widened on chip (converter warp, two fp16 V buffers); otherwise
    // P V reads the 16-bit V tile straight from its ring slot
    static constexpr bool CONV = E4 && !V16G;
    // Warps: 0 producer; 1 and 2 MMA issuers, one per tile, each answering
    // only its own tile's barriers; then 2 x 4 softmax warps; on-chip
    // widening adds a V converter warp last.
    static constexpr int ISSUERS = 2;
    // 16-bit inputs: the O tile (bf16 / fp16) is exactly a Q tile, so the
    // epilogue stages O in the tile's own Q buffer (free once its last P V is
    // done) and writes it with one TMA store.
    static constexpr bool TMA_O = !E4;
    static constexpr int SOFTMAX_WARP0 = 1 + ISSUERS;
    static constexpr int CONVERTER_WARP = SOFTMAX_WARP0 + 8;
    static constexpr int THREADS = 32 * (SOFTMAX_WARP0 + 8 + (CONV ? 1 : 0));
    // a 16-bit V tile (a ring tile for 16-bit inputs, the fp16 copy for
    // e4m3): 128 keys x D, 128-byte swizzled chunks of 64 values
    static constexpr int V16_CB = 2 * D >= 128 ? 128 : 2 * D;
    static constexpr int V16_CHUNK = BN * V16_CB;
    static constexpr int V16T = BN * 2 * D;
    static constexpr int V16_NC = 2 * D / V16_CB;          // 128-byte chunks per 16-bit V row
    // the two fp16 V buffers widened on chip (kE4M3 only)
    static constexpr int V16BUF = CONV ? V16T : 0;
    // bytes per ring slot: a K or V tile of the input type, or (V16G) the
    // larger of an e4m3 K tile and an fp16 V tile
    static constexpr int SLOT = (V16G && V16T > TILE) ? V16T : TILE;
    // q_full, s_full x2, p_full x2, pv_done x2, drain, s_free x2, drain of
    // issuer B, v16_full x2, v16_empty x2
    static constexpr int NB_FIXED = 1 + 2 + 2 + 2 + 1 + 2 + 1 + 4;
    static constexpr int SLOTS_FIT = (kSmemLimit - 1024 - 2 * TILE - 2 * V16BUF - 512) / SLOT;
    // K/V ring depth; on-chip widening needs it even (K items in even slots,
    // V in odd: the two kinds of slot are released by different warps)
    static constexpr int SLOTS = (SLOTS_FIT > 8 ? 8 : SLOTS_FIT) & (CONV ? ~1 : ~0);
    static constexpr uint32_t LAYOUT = (CB == 128) ? 2u : 4u;  // 128B / 64B swizzle
    static constexpr int NB = NB_FIXED + 2 * SLOTS;        // mbarriers
    static constexpr size_t SMEM_USED =
        1024 + (size_t)TILE * 2 + (size_t)SLOT * SLOTS + 2 * (size_t)V16BUF + NB * 8 + 16;
    // at least ~120 KB so two CTAs never share an SM (each takes all of TMEM)
    static constexpr size_t SMEM = SMEM_USED > 122880 ? SMEM_USED : 122880;
    static constexpr uint32_t FMT = (BASE == kBF16) ? 1u : 0u;  // bf16 = 1, f16 / e4m3 = 0
    static_assert(!V16G || (E4 && D <= 128), "fp16 V from global memory: e4m3, d = 64 or 128");
    static constexpr uint32_t IDESC_QK = instr_desc(FMT, FMT, 0, 0, BM, BN);
    // P V: 16-bit operands (e4m3 inputs: fp16 P and fp16 V)
    static constexpr uint32_t IDESC_PV = instr_desc(E4 ? 0u : FMT, E4 ? 0u : FMT, 0, 1, BM, D);
    static constexpr int PV_K = 16;                        // keys per P V MMA instruction
    static constexpr uint32_t P_COLS = BN * 2 / 4;         // TMEM columns holding P (16-bit)
    // Rescale the running output only when the row maximum grew by more than
    // this (log2 units): P values then stay <= 2^8, inside every P type's range.
    static constexpr float RESCALE_THRESHOLD = 8.0f;
    static_assert(SLOTS >= 2, "K/V ring depth");
    static_assert(SMEM_USED <= (size_t)kSmemLimit, "shared memory budget");
};

// TMEM columns: one S [0,128) for both tiles, P_A [128,192), P_B [192,256),
// O_A [256, 256+D), O_B [256+D, 256+2D).
constexpr uint32_t kColS = 0;
__device__ __forceinline__ uint32_t col_p(int t) { return 128u + 64u * (uint32_t)t; }
template <int D>
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + (uint32_t)(D * t); }

struct TcParams {
    int B, H, N_q, N_k;
    int H_kv;          // K/V heads: query head h reads K/V head h / (H / H_kv)
    int n_pairs;       // ceil(N_q / 256)
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
    // split-KV: grid.y = n_splits CTAs share one query-tile pair's K/V range;
    // each writes its partial (O normalised within the split, fp32) and lse
    int n_splits;
    float* part_o;    // [n_splits][B*H][N_q][D]
    float* part_lse;  // [n_splits][B*H][N_q]
};

// Bounded waits (shared implementation) reporting to this file's status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned long long limit_ns) {
    return bounded_wait(bar, parity, abort_flag, limit_ns, &g_tc_status);
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    bounded_drain(bar, parity, limit_ns);
}

// Number of K/V tiles the query tile starting at row q0 needs (0 if the tile
// is past N_q or every row in it is fully masked).
__device__ __forceinline__ int kv_tiles_for(int q0, const TcParams& p) {
    if (q0 >= p.N_q) return 0;
    const int last_row = min(q0 + BM - 1, p.N_q - 1);
    int last_key = p.N_k - 1;
    if (p.causal) last_key = min(last_key, last_row + (p.N_k - p.N_q));
    return last_key < 0 ? 0 : last_key / BN + 1;
}

template <int D, int KIND>
__global__ void __launch_bounds__(Cfg<D, KIND>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const TcParams p) {
    using C = Cfg<D, KIND>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                      // two tiles: A then B
    uint8_t* sV16 = smem + 2 * C::TILE;      // two fp16 V tiles (on-chip widening only)
    uint8_t* sKV = sV16 + 2 * C::V16BUF;     // SLOTS slots of C::SLOT bytes
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + (size_t)C::SLOTS * C::SLOT);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const uint32_t b_q_full = smem_u32(bars);
    const uint32_t b_s_full = smem_u32(bars + 1);     // + 8 * tile
    const uint32_t b_p_full = smem_u32(bars + 3);     // + 8 * tile
    const uint32_t b_pv_done = smem_u32(bars + 5);    // + 8 * tile
    const uint32_t b_drain = smem_u32(bars + 7);
    const uint32_t b_s_free = smem_u32(bars + 8);     // + 8 * tile
    const uint32_t b_drain_b = smem_u32(bars + 10);
    const uint32_t b_v16_full = smem_u32(bars + 11);  // + 8 * buffer (on-chip widening)
    const uint32_t b_v16_empty = smem_u32(bars + 13); // + 8 * buffer (on-chip widening)
    const uint32_t b_kv_full = smem_u32(bars + 15);               // + 8 * slot
    const uint32_t b_kv_empty = smem_u32(bars + 15 + C::SLOTS);   // + 8 * slot

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- schedule: groups of heads_per_group heads; inside a group the pair
    // index is the slow coordinate (heaviest causal pair first) and the head
    // the fast one, so CTAs running together share a few heads' K/V.
    const long long n_bh = (long long)p.B * p.H;
    const long long G = p.heads_per_group;
    const long long per_group = (long long)p.n_pairs * G;
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
    const int h_kv = h / (p.H / p.H_kv);  // grouped-query attention: shared K/V head
    const int pair = p.causal ? (p.n_pairs - 1 - rank) : rank;
    int q0[2], n_kv[2];
    q0[0] = pair * 2 * BM;
    q0[1] = q0[0] + BM;
    n_kv[0] = kv_tiles_for(q0[0], p);
    n_kv[1] = kv_tiles_for(q0[1], p);
    // Split-KV: this CTA takes K/V tiles [j0, j1) of the pair's range; the loops
    // below count tiles from 0 and only the tile coordinates add j0.
    int j0 = 0;
    if (p.n_splits > 1) {
        const int n_all = max(n_kv[0], n_kv[1]);
        const int per = (n_all + p.n_splits - 1) / p.n_splits;
        j0 = min(n_all, (int)blockIdx.y * per);
        const int j1 = min(n_all, j0 + per);
        n_kv[0] = max(0, min(j1, n_kv[0]) - j0);
        n_kv[1] = max(0, min(j1, n_kv[1]) - j0);
    }
    const int n_max = max(n_kv[0], n_kv[1]);
    const unsigned long long lim = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(b_q_full, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(b_s_full + 8 * t, 1);
            mbar_init(b_p_full + 8 * t, 4);    // one arrival per softmax warp
            mbar_init(b_pv_done + 8 * t, 1);
            mbar_init(b_s_free + 8 * t, 4);    // one arrival per softmax warp
        }
        mbar_init(b_drain, 1);
        mbar_init(b_drain_b, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(b_v16_full + 8 * t, 4);    // converter, producer and both issuers
            mbar_init(b_v16_empty + 8 * t, 2);   // one release per tile's issuer
        }
        for (int s = 0; s < C::SLOTS; ++s) {
            mbar_init(b_kv_full + 8 * s, 1);
            // one release per issuer (both read every K and V item); with
            // on-chip widening the V items (odd slots) are released instead by
            // the four warps that widen them
            mbar_init(b_kv_empty + 8 * s, (C::CONV && (s & 1)) ? 4 : C::ISSUERS);
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

    // On-chip widening: V_j's e4m3 tile (ring item 2j + 1) widened into fp16
    // buffer j % 2, laid out as a 16-bit V tile loaded by TMA would be (128-byte rows of 64
    // values, 128-byte swizzle; every e4m3 value is exact in fp16).  The work
    // is shared out by 16-byte units between the converter warp, the producer
    // warp and each MMA issuer (right after issuing its P V of the step
    // before), so that the fp16 stores are spread over the four SM
    // sub-partitions instead of loading one: from one warp they went through
    // its sub-partition's shared-memory / special-function issue path beside
    // two softmax warps and cost ~17 % of the time on e4m3 B2 H16 N8192 d128.
    constexpr int V_UNITS = C::CB / 16;       // 16-byte units per e4m3 row
    constexpr int V_PER = BN * V_UNITS / 32;  // units per lane, whole tile
    // shares, in units per lane: converter warp [0, V_CONV), producer warp
    // [V_PROD0, +V_PROD), issuer t [V_ISS0 + t V_ISS, +V_ISS).  Measured on
    // e4m3 B2 H16 N8192 d128 (ms per call; shares in 32nds of a tile per
    // warp): all on the converter 0.635; converter 16, issuers 8 each 0.605;
    // 8 each on all four warps 0.616; issuers 16 each 0.734; converter 16,
    // producer 8, issuers 4 each 0.572-0.581; converter 20, producer 8,
    // issuers 2 each 0.567-0.571 (kept: the issuers' MMA issue tolerates
    // little extra work); converter 24, producer 4, issuers 2 each 0.595;
    // one-unit issuer shares 0.59-0.60.
    constexpr int V_CONV = 5 * V_PER / 8, V_ISS = V_PER / 16, V_PROD = V_PER - V_CONV - 2 * V_ISS;
    constexpr int V_PROD0 = V_CONV, V_ISS0 = V_CONV + V_PROD;
    static_assert(V_CONV + V_PROD + 2 * V_ISS == V_PER, "the shares cover every unit");
    // Unit idx of the tile -> (row rr, 16-byte unit w of the e4m3 row),
    // chosen so that the eight lanes of each quarter-warp hit eight different
    // 16-byte bank groups both when they load (e4m3 swizzle) and when they
    // store (fp16 swizzle, the two 64-value chunks 16 KB apart).  d = 128: a
    // quarter takes two adjacent rows, one row's units in fp16 chunk 0 and the
    // other's in chunk 1.  d = 64: a quarter takes two adjacent rows, four
    // units each.
    auto unit_of = [&](int idx, int& rr, int& w) {
        if constexpr (V_UNITS == 8) {
            const int w_lo = idx & 3, half = (idx >> 2) & 1, sel = (idx >> 3) & 1;
            rr = 2 * (idx >> 4) + half;
            w = 4 * (half ^ sel) + w_lo;
        } else {
            rr = idx / V_UNITS;
            w = idx % V_UNITS;
        }
    };
    // one share (this lane's units [k_begin, k_end)) of V_j: wait for the tile
    // and for the buffer (released by both tiles' P V MMAs two tiles
    // earlier), widen with loads batched so their latency overlaps, then hand
    // the share over (every lane's writes fenced for the async proxy, one
    // arrival per warp on v16_full and on the ring slot's release)
    auto widen_share = [&](int j, int k_begin, int k_end) -> bool {
        const int itV = 2 * j + 1;
        const int slot = itV % C::SLOTS;
        bool ok = __all_sync(0xffffffffu, wait_bar(b_kv_full + 8 * slot, (uint32_t)(itV / C::SLOTS) & 1u,
                                                   abort_flag, lim));
        if (ok)
            ok = __all_sync(0xffffffffu, wait_bar(b_v16_empty + 8 * (j & 1), ((uint32_t)(j >> 1) & 1u) ^ 1u,
                                                  abort_flag, lim));
        if (!ok) return false;
        const uint32_t src = smem_u32(sKV + (size_t)slot * C::SLOT);
        const uint32_t dst = smem_u32(sV16 + (size_t)(j & 1) * C::V16BUF);
        // Units in batches of NU: the batch's loads all go out before its first
        // conversion.  Batches of 8, or of 4, 2 or 1 where the share is not a
        // multiple of 8.
        auto widen_units = [&](auto nu) {
            constexpr int NU = decltype(nu)::value;
#pragma unroll 1
            for (int k0 = k_begin; k0 < k_end; k0 += NU) {
                uint32_t x[NU][4];
#pragma unroll
                for (int k = 0; k < NU; ++k) {
                    int rr, w;
                    unit_of(lane + 32 * (k0 + k), rr, w);
                    // e4m3 row rr: 128-byte swizzle (w ^ rr%8) or 64-byte (w ^ (rr/2)%4)
                    const int wp = (C::CB == 128) ? (w ^ (rr & 7)) : (w ^ ((rr >> 1) & 3));
                    ld_shared_v4(src + (uint32_t)(rr * C::CB + wp * 16), x[k]);
                }
#pragma unroll
                for (int k = 0; k < NU; ++k) {
                    int rr, w;
                    unit_of(lane + 32 * (k0 + k), rr, w);
                    uint32_t hv[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hv[2 * e] = e4m3x2_to_f16x2((uint16_t)(x[k][e] & 0xffffu));
                        hv[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(x[k][e] >> 16));
                    }
                    // values d = 16 w .. 16 w + 15: fp16 chunk w / 4, units 2 (w % 4), +1
                    const uint32_t row = dst + (uint32_t)((w >> 2) * C::V16_CHUNK + rr * C::V16_CB);
                    const int u0 = 2 * (w & 3);
                    st_shared_v4(row + (uint32_t)((u0 ^ (rr & 7)) << 4), hv[0], hv[1], hv[2], hv[3]);
                    st_shared_v4(row + (uint32_t)(((u0 + 1) ^ (rr & 7)) << 4), hv[4], hv[5], hv[6], hv[7]);
                }
            }
        };
        const int n_units = k_end - k_begin;
        if (n_units % 8 == 0)
            widen_units(IntC<8>{});
        else if (n_units % 4 == 0)
            widen_units(IntC<4>{});
        else if (n_units % 2 == 0)
            widen_units(IntC<2>{});
        else
            widen_units(IntC<1>{});
        fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive_1(b_v16_full + 8 * (j & 1));
        mbar_arrive_1(b_kv_empty + 8 * slot);
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        // Q_A and Q_B (a tile with no key tile to read is not loaded), once
        auto load_q = [&] {
            const int nq = (n_kv[0] > 0) + (n_kv[1] > 0);
            mbar_arrive_expect_tx(b_q_full, (uint32_t)(nq * C::TILE));
            for (int t = 0; t < 2; ++t) {
                if (n_kv[t] == 0) continue;
                for (int c = 0; c < C::NC; ++c)
                    tma_load_4d(smem_u32(sQ + t * C::TILE + c * C::CHUNK), &tmQ, b_q_full,
                                c * (C::CB / C::E), h, q0[t], b);
            }
        };
        if constexpr (C::CONV) {
            // The whole warp runs the loop (lane 0 issues the copies) and also
            // widens its share of every V tile: its share of V_c right after
            // V_{c+LAG}'s load has gone out.  LAG must stay below the ring's
            // depth in tiles (V_{c+SLOTS/2} reuses V_c's slot, which only the
            // complete widening of V_c frees); 3 measured best on e4m3 B2
            // H16 N8192 d128 (0.576 ms per call against 0.581 for 1 or 2).
            constexpr int LAG = 3;
            static_assert(!C::CONV || LAG < C::SLOTS / 2, "the producer's share must come before its slot is needed");
            if (n_max > 0) {
                if (lane == 0) load_q();
                __syncwarp();
                // item 2j = K_j, item 2j+1 = V_j (the order the MMAs first use them)
                int it = 0, next_share = 0;
                bool ok = true;
                for (; it < 2 * n_max && it < p.items_limit && ok; ++it) {
                    const int slot = it % C::SLOTS;
                    const uint32_t ph = (uint32_t)(it / C::SLOTS) & 1u;
                    ok = __all_sync(0xffffffffu, wait_bar(b_kv_empty + 8 * slot, ph ^ 1u, abort_flag, lim));
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(b_kv_full + 8 * slot, C::TILE);
                        const CUtensorMap* tm = (it & 1) ? &tmV : &tmK;
                        uint8_t* dst = sKV + (size_t)slot * C::SLOT;
                        for (int c = 0; c < C::NC; ++c)
                            tma_load_4d(smem_u32(dst + c * C::CHUNK), tm, b_kv_full + 8 * slot,
                                        c * (C::CB / C::E), h_kv, (j0 + (it >> 1)) * BN, b);
                    }
                    __syncwarp();
                    if ((it & 1) && (it >> 1) >= LAG) ok = widen_share(next_share++, V_PROD0, V_PROD0 + V_PROD);
                }
                // the last tiles' shares
                for (; ok && next_share < n_max; ++next_share) ok = widen_share(next_share, V_PROD0, V_PROD0 + V_PROD);
                if (!ok && lane == 0) {
                    // let every load already issued land before the CTA can exit
                    wait_drain(b_q_full, 0, p.drain_ns);
                    for (int k = (it > C::SLOTS ? it - C::SLOTS : 0); k < it; ++k)
                        wait_drain(b_kv_full + 8 * (k % C::SLOTS), (uint32_t)(k / C::SLOTS) & 1u, p.drain_ns);
                }
            }
        } else {
            if (lane == 0 && n_max > 0) {
                load_q();
                // item 2j = K_j, item 2j+1 = V_j (the order the MMAs first use them)
                int it = 0;
                bool ok = true;
                for (; it < 2 * n_max && it < p.items_limit; ++it) {
                    const int slot = it % C::SLOTS;
                    const uint32_t ph = (uint32_t)(it / C::SLOTS) & 1u;
                    if (!wait_bar(b_kv_empty + 8 * slot, ph ^ 1u, abort_flag, lim)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = sKV + (size_t)slot * C::SLOT;
                    if (C::V16G && (it & 1)) {
                        // fp16 V tile: V16_NC chunks of 64 values
                        mbar_arrive_expect_tx(b_kv_full + 8 * slot, C::V16T);
                        for (int c = 0; c < C::V16_NC; ++c)
                            tma_load_4d(smem_u32(dst + c * C::V16_CHUNK), &tmV, b_kv_full + 8 * slot,
                                        c * (C::V16_CB / 2), h_kv, (j0 + (it >> 1)) * BN, b);
                    } else {
                        mbar_arrive_expect_tx(b_kv_full + 8 * slot, C::TILE);
                        const CUtensorMap* tm = (it & 1) ? &tmV : &tmK;
                        for (int c = 0; c < C::NC; ++c)
                            tma_load_4d(smem_u32(dst + c * C::CHUNK), tm, b_kv_full + 8 * slot,
                                        c * (C::CB / C::E), h_kv, (j0 + (it >> 1)) * BN, b);
                    }
                }
                if (!ok) {
                    // let every load already issued land before the CTA can exit
                    wait_drain(b_q_full, 0, p.drain_ns);
                    for (int k = (it > C::SLOTS ? it - C::SLOTS : 0); k < it; ++k)
                        wait_drain(b_kv_full + 8 * (k % C::SLOTS), (uint32_t)(k / C::SLOTS) & 1u, p.drain_ns);
                }
            }
        }
        __syncwarp();
    } else if (warp < C::SOFTMAX_WARP0) {
        // ----------------------------------------------------- MMA issuer(s)
        // The whole warp runs the issue loop (warp-uniform operands); one
        // elected lane issues each MMA, commit and arrive.
        auto wb = [&](uint32_t bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_bar(bar, par, abort_flag, lim));
        };
        if (n_max > 0) {
            auto issue_qk = [&](int t, int slot) {
                // descriptors of the tile bases; each MMA adds its byte offset / 16
                const uint64_t qd = smem_desc(smem_u32(sQ + t * C::TILE), 16, 8 * C::CB, C::LAYOUT);
                const uint64_t kd =
                    smem_desc(smem_u32(sKV + (size_t)slot * C::SLOT), 16, 8 * C::CB, C::LAYOUT);
#pragma unroll
                for (int c = 0; c < C::NC; ++c) {
#pragma unroll
                    for (int ks = 0; ks < C::CB / 32; ++ks) {
                        const uint32_t off16 = (uint32_t)(c * C::CHUNK + ks * 32) >> 4;
                        const uint64_t da = qd + off16;
                        const uint64_t db = kd + off16;
                        const uint32_t acc = (c | ks) != 0;
                        if constexpr (C::E4)
                            mma_f8_ss_1(tmem + kColS, da, db, C::IDESC_QK, acc);
                        else
                            mma_f16_ss_1(tmem + kColS, da, db, C::IDESC_QK, acc);
                    }
                }
            };
            auto issue_pv = [&](int t, int slot, bool first) {
                // A = 16-bit P_t in TMEM (8 columns per 16 keys); B = the 16-bit
                // V tile in ring slot `slot` (on-chip widening: in fp16 buffer
                // `slot`), MN-major: 8-key groups 8*128 bytes apart, 64-value
                // d-chunks V16_CHUNK apart
                const uint8_t* vt = C::CONV ? sV16 + (size_t)slot * C::V16BUF
                                            : sKV + (size_t)slot * C::SLOT;
                const uint64_t vd = smem_desc(smem_u32(vt), C::V16_CHUNK, 8 * C::V16_CB, 2u);
#pragma unroll
                for (int ks = 0; ks < BN / C::PV_K; ++ks) {
                    const uint64_t db = vd + ((uint32_t)(ks * C::PV_K * C::V16_CB) >> 4);
                    const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
                    mma_f16_ts_1(tmem + col_o<D>(t), tmem + col_p(t) + ks * (C::PV_K * 2 / 4),
                                 db, C::IDESC_PV, acc);
                }
            };
            auto slot_of = [](int it) { return it % C::SLOTS; };
            auto par_of = [](int it) { return (uint32_t)(it / C::SLOTS) & 1u; };

            bool ok = true;
            // One issuer per tile; the two share one TMEM score buffer S.
            // The score MMAs into S run in the order A_0 B_0 A_1 B_1 ...
            // (a tile past its own key range drops out), and each waits
            // until the softmax of the one before it has loaded its scores
            // (s_free).  P_t V_j reads fp16 P_t from TMEM and the fp16 copy
            // of V_j in buffer j % 2 (widened by the converter warp and both
            // issuers); the buffer is released when the MMA has read it.
            // V16G: the fp16 V_j is ring item 2j + 1 itself, released to the
            // producer by both issuers' P V commits, like K_j.
            // Key tiles this tile never reads release their K slot and V
            // buffer once filled (and still get this issuer's share of V).
            const int t = __shfl_sync(0xffffffffu, warp, 0) - 1;
            const int nt = n_kv[t], nt_o = n_kv[1 - t];
            const uint32_t drain_t = t == 0 ? b_drain : b_drain_b;
            auto s_ready = [&](int j) -> bool {
                int pt = -1, pj = 0;  // the score MMA before tile t's j-th
                if (t == 0) {
                    if (j >= 1) {
                        pt = (j - 1 < nt_o) ? 1 : 0;
                        pj = j - 1;
                    }
                } else if (j < nt_o) {
                    pt = 0;
                    pj = j;
                } else if (j >= 1) {
                    pt = 1;
                    pj = j - 1;
                }
                return pt < 0 || wb(b_s_free + 8 * pt, (uint32_t)pj & 1u);
            };
            // this issuer's quarter of every V tile's units
            const int vk0 = V_ISS0 + t * V_ISS, vk1 = vk0 + V_ISS;
            ok = wb(b_q_full, 0);
            if (ok && nt > 0) {
                ok = wb(b_kv_full + 8 * slot_of(0), par_of(0));
                if (ok) ok = s_ready(0);
                if (ok) {
                    tc_fence_after();
                    issue_qk(t, slot_of(0));
                    mma_commit_1(b_s_full + 8 * t);
                    mma_commit_1(b_kv_empty + 8 * slot_of(0));
                }
            }
            if constexpr (C::CONV)
                if (ok && n_max > 0) ok = widen_share(0, vk0, vk1);
            for (int j = 0; j < nt && ok; ++j) {
                const int itK = 2 * j + 2;
                if (j + 1 < nt) {
                    ok = wb(b_kv_full + 8 * slot_of(itK), par_of(itK));
                    if (ok) ok = s_ready(j + 1);
                    if (!ok) break;
                    tc_fence_after();
                    issue_qk(t, slot_of(itK));
                    mma_commit_1(b_s_full + 8 * t);
                    mma_commit_1(b_kv_empty + 8 * slot_of(itK));
                }
                const int itV = 2 * j + 1;
                if constexpr (!C::CONV)
                    ok = wb(b_kv_full + 8 * slot_of(itV), par_of(itV));
                else
                    ok = wb(b_v16_full + 8 * (j & 1), (uint32_t)(j >> 1) & 1u);
                if (ok) ok = wb(b_p_full + 8 * t, (uint32_t)j & 1u);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, C::CONV ? (j & 1) : slot_of(itV), j == 0);
                mma_commit_1(b_pv_done + 8 * t);
                if constexpr (!C::CONV) {
                    mma_commit_1(b_kv_empty + 8 * slot_of(itV));
                } else {
                    mma_commit_1(b_v16_empty + 8 * (j & 1));
                    // the MMAs run on their own: widen this issuer's share of the next V
                    if (j + 1 < n_max) ok = widen_share(j + 1, vk0, vk1);
                }
            }
            for (int j = nt; j < n_max && ok; ++j) {
                ok = wb(b_kv_full + 8 * slot_of(2 * j), par_of(2 * j));
                if (ok) mbar_arrive_1(b_kv_empty + 8 * slot_of(2 * j));
                if constexpr (!C::CONV) {
                    if (ok) ok = wb(b_kv_full + 8 * slot_of(2 * j + 1), par_of(2 * j + 1));
                    if (ok) mbar_arrive_1(b_kv_empty + 8 * slot_of(2 * j + 1));
                } else {
                    if (ok) ok = wb(b_v16_full + 8 * (j & 1), (uint32_t)(j >> 1) & 1u);
                    if (ok) mbar_arrive_1(b_v16_empty + 8 * (j & 1));
                    if (ok && j + 1 < n_max) ok = widen_share(j + 1, vk0, vk1);
                }
            }
            if (!ok) {
                // make sure none of this issuer's MMAs still runs when TMEM is freed
                mma_commit_1(drain_t);
                wait_drain(drain_t, 0, p.drain_ns);
            }
        }
        __syncwarp();
    } else if (C::CONV && warp == C::CONVERTER_WARP) {
        // --------------------------------------- V converter (on-chip widening)
        // Its share of every V tile's units (producer and issuers take the rest).
        for (int j = 0; j < n_max; ++j)
            if (!widen_share(j, 0, V_CONV)) break;
    } else {
        // --------------------------------------- softmax + epilogue (2 x 128 thr)
        const int t = (warp - C::SOFTMAX_WARP0) >> 2;  // tile of this warp group
        const int quad = warp & 3;           // TMEM lane quadrant this warp may access
        const int r = quad * 32 + lane;
        const int row_g = q0[t] + r;
        const int nt = n_kv[t];
        const uint32_t t_row = tmem + ((uint32_t)(quad * 32) << 16);
        const uint32_t s_full = b_s_full + 8 * t, p_full = b_p_full + 8 * t;
        const uint32_t pv_done = b_pv_done + 8 * t;
        const int shift = p.N_k - p.N_q;
        int row_lim = p.N_k - 1;  // last allowed key of this row
        if (p.causal) row_lim = min(row_lim, row_g + shift);
        // tiles with any column beyond the tile's first row's limit need a mask
        const int tile_lim = p.causal ? min(p.N_k - 1, q0[t] + shift) : p.N_k - 1;
        float dq = 1.f, dk = 1.f, dv = 1.f;
        if (C::E4) {
            if (p.q_descale) dq = p.q_descale[bh];
            if (p.k_descale) dk = p.k_descale[b * p.H_kv + h_kv];
            if (p.v_descale) dv = p.v_descale[b * p.H_kv + h_kv];
        }
        const float c = p.scale * dq * dk * 1.4426950408889634f;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;

        // The scores of the next step and the release of the P buffer are
        // tested early (mbar_test) and the results used later, so the barrier
        // round trips overlap the softmax; a failed test falls back to the
        // bounded wait.
        uint32_t s_pre = 0, pv_pre = 0;
        for (int j = 0; j < nt && ok; ++j) {
            if (!__all_sync(0xffffffffu, s_pre != 0u) &&
                !__all_sync(0xffffffffu, wait_bar(s_full, (uint32_t)j & 1u, abort_flag, lim))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // one 128-column load, which also returns the row's maximum
            uint32_t sr[BN];
            float rmx;  // the row's maximum, from the load itself
            tmem_ld128_max(t_row + kColS, sr, rmx);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < BN / 32; ++u)
                reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * u]));
            reg_fence_f(rmx);
            // the scores are in registers: the next score MMA may overwrite them
            tc_fence_before();
            __syncwarp();
            mbar_arrive_1(b_s_free + 8 * t);
            if (j > 0) pv_pre = mbar_test(pv_done, (uint32_t)(j - 1) & 1u);
            float s[BN];
#pragma unroll
            for (int x = 0; x < BN; ++x) s[x] = __uint_as_float(sr[x]);

            const int kbase = (j0 + j) * BN;
            float mx;
            if (kbase + BN - 1 > tile_lim) {
                const int cl = row_lim - kbase;  // columns > cl are masked
#pragma unroll
                for (int x = 0; x < BN; ++x)
                    if (x > cl) s[x] = -INFINITY;
                // row maximum of the masked row (the load's maximum includes
                // the masked columns): 8 independent 3-input-max chains, then
                // a small tree
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
            float sc[8];  // independent partial row sums (four packed pairs)
#pragma unroll
            for (int k = 0; k < 8; ++k) sc[k] = 0.f;
            // P_t as bf16 / fp16 (e4m3 inputs: fp16), 32 TMEM columns (64
            // scores) at a time so only one chunk of packed P is live.  P_t's
            // buffer is free once P_{j-1} V_{j-1} has completed.  The
            // scale-and-subtract and the sums use packed f32x2 instructions.
            constexpr int PER_CHUNK = 32 * 4 / 2;  // 16-bit scores per 32 TMEM columns
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
                    pk[x / 2] = (C::BASE == kBF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
                }
                if (u == 0 && j > 0 && !__all_sync(0xffffffffu, pv_pre != 0u) &&
                    !__all_sync(0xffffffffu, wait_bar(pv_done, (uint32_t)(j - 1) & 1u,
                                                      abort_flag, lim))) {
                    ok = false;
                    break;
                }
                if (u == 0 && j > 0) tc_fence_after();  // P V_{j-1} has read P_t
                tmem_st32(t_row + col_p(t) + 32 * u, pk);
            }
            if (!ok) break;
            s_pre = (j + 1 < nt) ? mbar_test(s_full, (uint32_t)(j + 1) & 1u) : 0u;
            const float sum =
                ((sc[0] + sc[1]) + (sc[2] + sc[3])) + ((sc[4] + sc[5]) + (sc[6] + sc[7]));
            l = l * alpha + sum;

            if (any && j > 0) {
                // O_t is touched only to rescale it; it is stable once
                // P_{j-1} V_{j-1} has completed (confirmed before the first P
                // store above)
                tc_fence_after();
                // 64 columns per load round: two loads in flight per wait
#pragma unroll
                for (int u = 0; u < D / 64; ++u) {
                    uint32_t oo[64];
                    const uint32_t ta = t_row + col_o<D>(t) + 64 * u;
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
            __syncwarp();
            mbar_arrive_1(p_full);
        }

        if (ok && nt > 0)
            ok = __all_sync(0xffffffffu, wait_bar(pv_done, (uint32_t)(nt - 1) & 1u, abort_flag, lim));
        // e4m3, d = 128: O (bf16) is staged in Q_t's buffer, which holds one
        // 64-column chunk of it (16 KB), and written by two TMA stores, so the
        // rows leave as whole 128-byte lines (stored from registers, each warp
        // store instruction touched 32 rows 4 KB apart).  Q_t is no longer
        // read: this issuer's pv_done covers its last score MMA.
        constexpr bool STAGE_O8 = (C::E4 && D == 128);
        if (STAGE_O8 && p.n_splits == 1) {
            const bool valid = row_g < p.N_q;
            const float inv = l > 0.f ? dv / l : 0.f;
            if (ok) tc_fence_after();
            const uint32_t row_base =
                smem_u32(sQ + t * C::TILE) + (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
            for (int c = 0; c < D / 64; ++c) {
                if (ok) {
#pragma unroll
                    for (int uu = 0; uu < 2; ++uu) {
                        uint32_t oo[32];
                        if (nt > 0) {
                            tmem_ld32(t_row + col_o<D>(t) + 32 * (2 * c + uu), oo);
                            tmem_ld_wait();
                            reg_fence32(oo);
                        } else {
#pragma unroll
                            for (int x = 0; x < 32; ++x) oo[x] = 0u;
                        }
                        uint32_t packed[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x)
                            packed[x] = pack_bf16(__uint_as_float(oo[2 * x]) * inv,
                                                  __uint_as_float(oo[2 * x + 1]) * inv);
                        // row r of the 128-byte-swizzled chunk: unit w at w ^ (r % 8)
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int w = uu * 4 + x;
                            st_shared_v4(row_base + ((uint32_t)(w ^ (r & 7)) << 4), packed[4 * x],
                                         packed[4 * x + 1], packed[4 * x + 2], packed[4 * x + 3]);
                        }
                    }
                }
                // every thread of the tile reaches both barriers, whether or not
                // its waits succeeded; one thread stores the chunk (rows past
                // N_q are not written) and waits until it has been read
                fence_proxy_async_smem();
                named_barrier(1 + t, 128);
                if (r == 0 && ok && !*abort_flag && q0[t] < p.N_q) {
                    tma_store_4d(&tmO, smem_u32(sQ + t * C::TILE), c * 64, h, q0[t], b);
                    bulk_commit_group();
                    bulk_wait_group_read0();
                }
                named_barrier(1 + t, 128);
            }
            if (ok && valid && p.lse)
                p.lse[(size_t)bh * p.N_q + row_g] =
                    l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
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
#pragma unroll
                for (int u = 0; u < D / 32; ++u) {
                    uint32_t oo[32];
                    if (nt > 0) {
                        tmem_ld32(t_row + col_o<D>(t) + 32 * u, oo);
                        tmem_ld_wait();
                        reg_fence32(oo);
                    } else {
#pragma unroll
                        for (int x = 0; x < 32; ++x) oo[x] = 0u;
                    }
                    if (C::TMA_O && !split) {
                        // row r of the 128-byte-swizzled tile in Q_t's buffer: 16-byte
                        // unit w of d-chunk c sits at unit w ^ (r % 8)
                        uint32_t packed[16];
#pragma unroll
                        for (int x = 0; x < 16; ++x) {
                            const float a0 = __uint_as_float(oo[2 * x]) * inv;
                            const float a1 = __uint_as_float(oo[2 * x + 1]) * inv;
                            packed[x] = (C::BASE == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                        }
                        const uint32_t row_base = smem_u32(sQ + t * C::TILE + (u / 2) * C::CHUNK) +
                                                  (uint32_t)(r >> 3) * 1024u + (uint32_t)(r & 7) * 128u;
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const int w = (u % 2) * 4 + x;
                            st_shared_v4(row_base + ((uint32_t)(w ^ (r & 7)) << 4), packed[4 * x],
                                         packed[4 * x + 1], packed[4 * x + 2], packed[4 * x + 3]);
                        }
                        continue;
                    }
                    if (split) {
                        // partial of this split, normalised by its own row sum
                        if (valid) {
                            float4* dst = reinterpret_cast<float4*>(prow + 32 * u);
#pragma unroll
                            for (int x = 0; x < 8; ++x)
                                dst[x] = make_float4(__uint_as_float(oo[4 * x]) * inv,
                                                     __uint_as_float(oo[4 * x + 1]) * inv,
                                                     __uint_as_float(oo[4 * x + 2]) * inv,
                                                     __uint_as_float(oo[4 * x + 3]) * inv);
                        }
                        continue;
                    }
                    uint32_t packed[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const float a0 = __uint_as_float(oo[2 * x]) * inv;
                        const float a1 = __uint_as_float(oo[2 * x + 1]) * inv;
                        packed[x] = (C::BASE == kFP16) ? pack_f16(a0, a1) : pack_bf16(a0, a1);
                    }
                    if (valid) {
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
            if (C::TMA_O && p.n_splits == 1) {
                // Every thread of the tile reaches this barrier, whether or not its
                // waits succeeded (a barrier that an aborted warp skipped would
                // never open).  Then one thread stores the tile from Q_t's buffer
                // (rows past N_q are not written) and waits until the store has
                // read shared memory.
                fence_proxy_async_smem();
                named_barrier(1 + t, 128);
                if (r == 0 && ok && !*abort_flag && q0[t] < p.N_q) {
                    for (int c = 0; c < C::NC; ++c)
                        tma_store_4d(&tmO, smem_u32(sQ + t * C::TILE + c * C::CHUNK), c * (C::CB / C::E),
                                     h, q0[t], b);
                    bulk_commit_group();
                    bulk_wait_group_read0();
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

// Health check of the bounded-wait path: one thread waits on an mbarrier that
// nothing arrives at, with the same wait the attention kernel uses, and must
// come back with the timeout flagged instead of hanging.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    (void)wait_bar(smem_u32(&bar), 0, &abort_flag, limit_ns);
}

// Split-KV combine: one warp per query row.  Exact merge of the splits'
// softmaxes: lse = log sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s.
template <int D>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ part_o,
                                                              const float* __restrict__ part_lse,
                                                              void* o, float* lse, int n_splits,
                                                              int H, int N_q, long long rows,
                                                              int out_fp16) {
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long long bh = row / N_q;
    const int i = (int)(row % N_q);
    const size_t stride = (size_t)rows;  // one split's [B*H][N_q] block
    const float ls = lane < n_splits ? part_lse[(size_t)lane * stride + row] : -INFINITY;
    float mx = ls;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float w = (mx == -INFINITY) ? 0.f : __expf(ls - mx);
    float tot = w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int x = 0; x < PER; ++x) acc[x] = 0.f;
    for (int sidx = 0; sidx < n_splits; ++sidx) {
        const float ws = __shfl_sync(0xffffffffu, w, sidx);
        if (ws == 0.f) continue;
        const float* src = part_o + ((size_t)sidx * stride + row) * D;
#pragma unroll
        for (int x = 0; x < PER; ++x) acc[x] = fmaf(ws, src[lane + 32 * x], acc[x]);
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    const int b = (int)(bh / H), h = (int)(bh % H);
    const size_t ob = (((size_t)b * N_q + i) * H + h) * D;
#pragma unroll
    for (int x = 0; x < PER; ++x) {
        const float val = acc[x] * inv;
        if (out_fp16)
            reinterpret_cast<__half*>(o)[ob + lane + 32 * x] = __float2half_rn(val);
        else
            reinterpret_cast<__nv_bfloat16*>(o)[ob + lane + 32 * x] = __float2bfloat16_rn(val);
    }
    if (lane == 0 && lse) lse[(size_t)bh * N_q + i] = tot > 0.f ? mx + __logf(tot) : -INFINITY;
}

// V for kE4M3_V16: e4m3 codes -> fp16 values (exact: every e4m3 value is an
// fp16 value).  Each thread takes units of 8 codes (8 bytes in, 16 bytes
// out), so one warp instruction loads 256 and stores 512 contiguous bytes;
// four independent loads per thread are in flight before the first
// conversion.  n8 = element count / 8.
__device__ __forceinline__ uint4 widen8(const uint2 x) {
    return make_uint4(e4m3x2_to_f16x2((uint16_t)(x.x & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.x >> 16)),
                      e4m3x2_to_f16x2((uint16_t)(x.y & 0xffffu)), e4m3x2_to_f16x2((uint16_t)(x.y >> 16)));
}

__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint2* __restrict__ v,
                                                         uint4* __restrict__ v16, long long n8) {
    const long long stride = (long long)gridDim.x * 256;
    long long i = (long long)blockIdx.x * 256 + threadIdx.x;
    for (; i + 3 * stride < n8; i += 4 * stride) {
        uint2 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = __ldg(v + i + u * stride);
#pragma unroll
        for (int u = 0; u < 4; ++u) v16[i + u * stride] = widen8(x[u]);
    }
    for (; i < n8; i += stride) v16[i] = widen8(__ldg(v + i));
}

// ------------------------------------------------------------------- host side
template <int D, int KIND>
cudaError_t launch_t(const Problem& pr, cudaStream_t stream, int n_splits = 1,
                     float* part_o = nullptr, float* part_lse = nullptr,
                     const void* v16 = nullptr) {
    using C = Cfg<D, KIND>;
    CUtensorMap mq, mk, mv, mo;
    const int ce = C::CB / C::E;
    const int dt = C::BASE;  // element type of Q and K (and V, O for 16-bit inputs)
    // O has the layout of Q; for 16-bit inputs also its element size
    // e4m3 at d = 128: O is bf16, 64-column chunks staged in the Q buffer
    const bool o8 = C::E4 && D == 128 && n_splits == 1;
    if (C::TMA_O && n_splits == 1) {
        if (!tma::encode_map(&mo, pr.o, dt, pr.B, pr.N_q, pr.H, D, ce, BM))
            return cudaErrorInvalidValue;
    } else if (o8) {
        if (!tma::encode_map(&mo, pr.o, kBF16, pr.B, pr.N_q, pr.H, D, 64, BM))
            return cudaErrorInvalidValue;
    }
    if (C::V16G && pr.N_k > 0 && !v16) return cudaErrorInvalidValue;
    const void* vsrc = pr.N_k == 0 ? pr.q : (C::V16G ? v16 : pr.v);
    if (!tma::encode_map(&mq, pr.q, dt, pr.B, pr.N_q, pr.H, D, ce, BM) ||
        !tma::encode_map(&mk, pr.N_k > 0 ? pr.k : pr.q, dt, pr.B, pr.N_k, pr.H_kv, D, ce, BN) ||
        !(C::V16G ? tma::encode_map(&mv, vsrc, kFP16, pr.B, pr.N_k, pr.H_kv, D, C::V16_CB / 2, BN)
                  : tma::encode_map(&mv, vsrc, dt, pr.B, pr.N_k, pr.H_kv, D, ce, BN)))
        return cudaErrorInvalidValue;
    TcParams p;
    p.B = pr.B;
    p.H = pr.H;
    p.H_kv = pr.H_kv;
    p.N_q = pr.N_q;
    p.N_k = pr.N_k;
    p.n_pairs = (pr.N_q + 2 * BM - 1) / (2 * BM);
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
    // Heads scheduled together: their K/V (2 N_k d E bytes per K/V head, or
    // 3 N_k d with e4m3 K and fp16 V; a K/V head is shared by H / H_kv query
    // heads) fill ~48 MiB of L2.  The groups are then evened out so the last
    // one is not a lone small group that would run by itself at the end.
    const long long kv_head_bytes =
        (long long)(pr.N_k > 0 ? pr.N_k : 1) * D * (C::V16G ? 3 : 2 * C::E);
    long long G = (48LL << 20) * (pr.H / pr.H_kv) / kv_head_bytes;
    if (G < 1) G = 1;
    if (G > n_bh) G = n_bh;
    const long long n_groups = (n_bh + G - 1) / G;
    G = (n_bh + n_groups - 1) / n_groups;
    p.heads_per_group = (int)G;
    const long long n_cta = (long long)p.n_pairs * n_bh;
    if (n_cta > 0x7fffffffLL) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D, KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    if (n_splits < 1 || n_splits > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)n_cta, (unsigned)n_splits);
    if (!(C::TMA_O && n_splits == 1) && !o8) mo = mq;  // not read
    attn_tc_kernel<D, KIND><<<grid, C::THREADS, C::SMEM, stream>>>(mq, mk, mv, mo, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc(const Problem& p, cudaStream_t stream) {
    if (p.d == 256) return launch_tc256(p, stream, 1, nullptr, nullptr);
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

size_t fp8_ws_workspace_bytes(long long B, long long H_kv, long long N_k, int d) {
    if (d != 64 && d != 128) return 0;
    return (size_t)(B * N_k * H_kv) * (size_t)d * 2;
}

cudaError_t launch_tc_fp8_ws(const Problem& p, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    if (p.dtype != kE4M3 || (p.d != 64 && p.d != 128)) return cudaErrorNotSupported;
    if (workspace_bytes < fp8_ws_workspace_bytes(p.B, p.H_kv, p.N_k, p.d))
        return cudaErrorInvalidValue;
    const long long n8 = (long long)p.B * p.N_k * p.H_kv * p.d / 8;
    if (n8 > 0) {
        // four 8-code units per thread (one batch of loads), up to 2^20 blocks
        const long long want = (n8 + 1023) / 1024;
        const unsigned blocks = (unsigned)(want < (1LL << 20) ? want : (1LL << 20));
        widen_e4m3_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint2*>(p.v),
                                                     static_cast<uint4*>(workspace), n8);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.d == 64) return launch_t<64, kE4M3_V16>(p, stream, 1, nullptr, nullptr, workspace);
    return launch_t<128, kE4M3_V16>(p, stream, 1, nullptr, nullptr, workspace);
}

size_t splitkv_workspace_bytes(long long B, long long H, long long N_q, int d, int n_splits) {
    return (size_t)n_splits * (size_t)(B * H * N_q) * (size_t)(d + 1) * sizeof(float);
}

cudaError_t launch_tc_splitkv(const Problem& p, int n_splits, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    if (n_splits < 2 || n_splits > kMaxSplits) return cudaErrorInvalidValue;
    const long long rows = (long long)p.B * p.H * p.N_q;
    if (workspace_bytes < splitkv_workspace_bytes(p.B, p.H, p.N_q, p.d, n_splits))
        return cudaErrorInvalidValue;
    float* part_o = static_cast<float*>(workspace);
    float* part_lse = part_o + (size_t)n_splits * rows * p.d;
    cudaError_t e = cudaErrorNotSupported;
    if (p.d == 256) e = launch_tc256(p, stream, n_splits, part_o, part_lse);
    switch (p.d == 256 ? -1 : p.dtype) {
        case kBF16:
            if (p.d == 64) e = launch_t<64, kBF16>(p, stream, n_splits, part_o, part_lse);
            if (p.d == 128) e = launch_t<128, kBF16>(p, stream, n_splits, part_o, part_lse);
            break;
        case kFP16:
            if (p.d == 64) e = launch_t<64, kFP16>(p, stream, n_splits, part_o, part_lse);
            if (p.d == 128) e = launch_t<128, kFP16>(p, stream, n_splits, part_o, part_lse);
            break;
        case kE4M3:
            if (p.d == 64) e = launch_t<64, kE4M3>(p, stream, n_splits, part_o, part_lse);
            if (p.d == 128) e = launch_t<128, kE4M3>(p, stream, n_splits, part_o, part_lse);
            break;
    }
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    if (p.d == 64)
        splitkv_combine_kernel<64><<<blocks, 256, 0, stream>>>(part_o, part_lse, p.o, p.lse,
                                                              n_splits, p.H, p.N_q, rows,
                                                              p.dtype == kFP16);
    else if (p.d == 256)
        splitkv_combine_kernel<256><<<blocks, 256, 0, stream>>>(part_o, part_lse, p.o, p.lse,
                                                               n_splits, p.H, p.N_q, rows,
                                                               p.dtype == kFP16);
    else
        splitkv_combine_kernel<128><<<blocks, 256, 0, stream>>>(part_o, part_lse, p.o, p.lse,
                                                               n_splits, p.H, p.N_q, rows,
                                                               p.dtype == kFP16);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
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
