// fa_fwd_kernel.cuh - fused attention forward for sm_103a (GB300).
//
// What it computes is the online-softmax form of attention described in
// "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (sections "第四步" and
// "第五步", Table 2: per query row the raw-score maximum m, the weight sum l
// and the unnormalised numerator U; "最后": O = U / l, LSE = s m + ln l) with
// the FlashAttention-2 loop order of "CUDA 算子工程" ch. 14, section 14.5
// (outer loop over query tiles; inner loop over key/value tiles).
//
// How it maps onto the GB300 SM (the pages' SM80 cp.async / mma.sync design is
// prior art only):
//   * a persistent grid (one CTA per SM) walks units: a unit is a pair of
//     128-row query tiles (A, B) of one (batch, head), and with split-KV one
//     key range of it; both tiles share every K/V tile that lands in shared
//     memory.  Rings, barrier phases and TMEM run on from one unit to the
//     next, so the next unit's Q and first products overlap this unit's
//     last tiles and epilogue.  10 warps:
//       warps 0-3  softmax + epilogue of tile A, warps 4-7 the same for B:
//                  thread t owns query row t of its tile (= TMEM lane t), so
//                  the row max and row sums need no shuffles;
//       warp 8     loader: TMA (cp.async.bulk.tensor) of both Q tiles of a
//                  unit, then K tiles running ahead of V tiles through two
//                  rings;
//       warp 9     tensor-core issuer: warp-uniform loop, elect.sync lane
//                  issues tcgen05.mma.
//   * TMEM (512 columns): S_A at 0, S_B at 128 (128 fp32 columns each; the
//     16-bit weights P overwrite the first 64 columns of their tile's S),
//     U_A at 256, U_B at 384 (d fp32 columns each).
//   * tensor-core order per key tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1).
//     While the softmax warps of tile A turn S_A(j+1) into weights, the tensor
//     core works on tile B (and vice versa), so the two softmax groups and the
//     tensor core overlap.  Each PV_X(j) runs in two halves of 64 keys: the
//     softmax warps hand over the weights of keys 0-63 before computing those
//     of keys 64-127, so the first half of the product runs meanwhile and
//     only the second half and S_X(j+1) remain between the end of one
//     softmax and the start of the next.  Because S_X(j+1) is issued after
//     PV_X(j), its completion also means U_X holds P_X(j) V_j: the softmax
//     warps may rescale U_X right away, without another wait.
//   * weights are computed against the running reference maximum m of the
//     previous tiles, without taking the new tile's maximum first; their fp32
//     sum bounds every weight (all are >= 0), so while it stays below a bound
//     that keeps each weight inside the 16-bit type, l, U and the weights keep
//     the old reference, which is exact because l, U and LSE all refer to the
//     same m.  Only the first tile of a row, or a tile whose first half would
//     pass the bound, takes the tile maximum, moves m, rescales U in TMEM and
//     recomputes the weights from the scores still in TMEM.  A second half
//     that would pass it moves m to that half's maximum once U has absorbed
//     the first half (which carries the old reference like the rest of U).
//   * O is normalised by the sum of the 16-bit weights actually fed to P.V,
//     so it is an exact convex combination of those weights; LSE uses the sum
//     of the fp32 weights.
//   * key tiles wholly in the future are skipped and the diagonal tile is
//     masked element-wise ("causal 模式在哪一步生效"); keys >= N (zero-filled by
//     TMA) are masked; query rows >= N are clipped by the TMA store, which
//     each softmax warp issues for its 32 rows from its own staging box.
//   * every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT
//     in a device status word, drains its in-flight copies and MMAs, frees
//     its TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kTileM = 128;           // rows per query tile (= TMEM lanes = MMA M)
constexpr int kBlockM = 2 * kTileM;   // rows per unit of work (tiles A and B)
constexpr int kBlockN = 128;          // keys per tile (= MMA N of S = Q K^T)
constexpr int kThreads = 320;         // 8 softmax warps + loader warp + MMA warp
constexpr int kLoaderWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSubBytes = 128 * 128;  // one 128-row x 64-column 16-bit swizzle sub-tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemU = 256;      // U_A at 256, U_B at 384

// Device status word (FA_OK / FA_ERR_TIMEOUT); read and cleared by the host.
__device__ unsigned int g_fa_status;

struct FwdParams {
    int num_units;            // query blocks x heads x key ranges
    float* lse;               // LSE of (b, h, row) at lse + b lse_sb + h lse_sh + row
    long long lse_sb, lse_sh;
    int Nq, Nk;               // query rows and keys per (b, h)
    int H;                    // heads (bh = b H + h)
    int mask_offset;          // causal: key j visible to row i iff j <= i + mask_offset
    int num_q_blocks;  // ceil(Nq / 256)
    // split-KV only: key tiles of each query block are divided into
    // num_splits contiguous ranges; each CTA writes a partial result
    int num_splits;
    int BH;
    float* o_part;    // [num_splits][BH][Nq][d] fp32, O of the range (normalised by its lhat)
    float* lse_part;  // [2][num_splits][BH][Nq] fp32: LSE of the range, and its log-sum of
                      // the rounded weights (the weight of its O in the merge)
    float scale;       // s
    float scale_log2;  // s * log2(e): exp(s x) = 2^(x * scale_log2)
    unsigned long long timeout_ns;
    int fault_mode;
};

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kSub = D / 64;                  // 64-column swizzle sub-tiles per row
    static constexpr int kTileBytes = kTileM * D * 2;    // one Q, K or V tile
    static constexpr int kKStages = D == 128 ? 2 : 4;    // K ring depth
    static constexpr int kVStages = D == 128 ? 2 : 4;    // V ring depth
    static constexpr int kOffQ = 0;                      // Q_A, Q_B
    static constexpr int kOffK = 2 * kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    // O staging: one 32-row x 64-column swizzled box per softmax warp
    static constexpr int kOffStage = kOffV + kVStages * kTileBytes;
    static constexpr int kStageBytes = 32 * 128;
    // d = 64: P.V also multiplies the weights by a column of ones (16 of them,
    // N = 80), so U carries the sum of the 16-bit weights in column 64.  The
    // ones live in one 128-row x 64-column tile that every V slot's
    // descriptor reaches as its second 64-column group.
    static constexpr bool kOnes = D == 64;
    static constexpr int kUCols = kOnes ? D + 16 : D;    // columns of U written by P.V
    static constexpr int kOffOnes = kOffStage + 8 * kStageBytes;
    static constexpr int kOnesBytes = kOnes ? kTileM * 128 : 0;
    static constexpr int kOffCtl = kOffOnes + kOnesBytes;
    static constexpr int kSmemBytes = kOffCtl + 512 + 1024;  // control block + alignment slack
};

template <int NK, int NV>
struct alignas(8) Ctl {
    uint64_t q_full;
    uint64_t q_empty;     // the S products of a unit are done: Q_A, Q_B may be reloaded
    uint64_t k_full[NK];
    uint64_t k_empty[NK];
    uint64_t v_full[NV];
    uint64_t v_empty[NV];
    uint64_t s_full[2];   // per query tile: S_X(j) is in TMEM
    uint64_t p_half[2];   // per query tile: the weights of keys 0-63 of tile j are in TMEM
    uint64_t p_full[2];   // per query tile: all of P_X(j) is in TMEM (and U_X rescaled)
    uint64_t o_half[2];   // per query tile: U_X has absorbed keys 0-63 of P_X(j) V_j
    uint64_t o_ready[2];  // per query tile: U_X has absorbed P_X(j) V_j
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
};

// Shared-memory matrix descriptor for tcgen05.mma: 128-byte swizzle,
// start address, leading/stride byte offsets (16-byte units), version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t instr_desc(bool bf16, int m, int n, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | ((static_cast<uint32_t>(n) >> 3) << 17) |
           ((static_cast<uint32_t>(m) >> 4) << 24);
}

// Bounded wait on an mbarrier phase.  The waiting thread sleeps in the
// barrier unit (woken when the phase completes) instead of spinning, so it
// takes no issue slots from the warps that share its sub-partition.  Returns
// false when the CTA is aborting (another role gave up) or when this wait ran
// past the limit (then it sets the abort flag and the device status).
constexpr uint32_t kSleepHintNs = 200000;

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                       unsigned long long timeout_ns, bool abortable) {
    const uint64_t t0 = ptx::globaltimer();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (abortable && *abort) return false;
        if (ptx::globaltimer() - t0 > timeout_ns) {
            *abort = 1u;
            atomicCAS(&g_fa_status, 0u, 5u /* FA_ERR_TIMEOUT */);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         unsigned long long timeout_ns, bool abortable = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort, timeout_ns, abortable);
}

// Warp-uniform wait: every lane waits on the same phase; the verdict is made
// uniform (a lane that gave up makes the warp give up).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                          unsigned long long timeout_ns, bool abortable = true) {
    const bool ok = wait_bar(bar, parity, abort, timeout_ns, abortable);
    return __all_sync(0xffffffffu, ok);
}

// Round two fp32 values to the 16-bit type (nearest even) and pack them,
// `lo` in the low half: the order tcgen05 reads K-adjacent elements from TMEM.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Exact fp32 values of a packed 16-bit pair.
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
    } else {
        __half2 h;
        *reinterpret_cast<uint32_t*>(&h) = v;
        return __half22float2(h);
    }
}

// acc.x += lo, acc.y += hi of a packed 16-bit pair: each half is widened
// exactly and added in fp32 (round to nearest) by one mixed-precision add.
template <bool BF16>
__device__ __forceinline__ void add_packed(float2& acc, uint32_t v) {
    if constexpr (BF16)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc.x), "+f"(acc.y)
            : "r"(v));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
            : "+f"(acc.x), "+f"(acc.y)
            : "r"(v));
}

// Weights are first computed against the current reference maximum; the tile
// maximum is only taken when their fp32 sum exceeds this bound, which keeps
// every weight finite and exact-range in the 16-bit type (all weights are
// >= 0, so each is at most the sum).
template <bool BF16>
__host__ __device__ constexpr float weight_sum_limit() { return BF16 ? 4294967296.0f : 32768.0f; }

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using C = Cfg<D>;
    constexpr int NK = C::kKStages;
    constexpr int NV = C::kVStages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled tiles need 1024-byte-aligned shared addresses
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    Ctl<NK, NV>* ctl = reinterpret_cast<Ctl<NK, NV>*>(smem + C::kOffCtl);
    volatile uint32_t* abort = &ctl->abort;
    const unsigned long long tmo = p.timeout_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkv = (p.Nk + kBlockN - 1) / kBlockN;

    // ---- work units.  A unit is one query block (two 128-row tiles) of one
    // (batch, head), and with split-KV one range of its key tiles.  The grid
    // is persistent: CTA c takes units c, then 2G - 1 - c, 2G + c, ... (G
    // CTAs; the direction alternates by round, so that with the causal mask,
    // where units are ordered longest first, every CTA gets a similar share).
    // Without the mask consecutive units share a head, so its K/V stay in L2.
    struct Unit {
        int bh, qb, split, k0, nA, nB;
    };
    const int S = SPLIT ? p.num_splits : 1;
    auto unit_id = [&](int r) {
        const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
        return r * G + ((r & 1) ? G - 1 - c : c);
    };
    auto unit_of = [&](int u) {
        Unit w;
        if (CAUSAL) {
            const int per_qb = p.BH * S;
            w.qb = p.num_q_blocks - 1 - u / per_qb;
            w.bh = (u % per_qb) / S;
            w.split = u % S;
        } else {
            w.bh = u / (p.num_q_blocks * S);
            w.qb = (u / S) % p.num_q_blocks;
            w.split = u % S;
        }
        // key tiles visible to query tile A (rows qb*256 + [0,128)) and B
        // ([128,256)): with the causal mask, up to the tile holding key
        // (last row + offset)
        auto visible_tiles = [&](int x) {
            if (!CAUSAL) return nkv;
            const int last = min(w.qb * kBlockM + x * kTileM + kTileM - 1, p.Nq - 1) + p.mask_offset;
            return last < 0 ? 0 : min(last / kBlockN + 1, nkv);
        };
        // the unit visits key tiles k0 .. k0 + n_x - 1 for tile x (all of them
        // unless split-KV divides the range of the block into num_splits parts)
        const int T_A = visible_tiles(0), T_B = visible_tiles(1);
        w.k0 = 0;
        w.nA = T_A;
        w.nB = T_B;
        if constexpr (SPLIT) {
            const int chunk = (T_B + S - 1) / S;
            w.k0 = w.split * chunk;
            const int k1 = min(w.k0 + chunk, T_B);
            w.nB = max(0, k1 - w.k0);
            w.nA = max(0, min(k1, T_A) - w.k0);
        }
        return w;
    };

    const uint32_t bar_q = ptx::smem_addr(&ctl->q_full);
    const uint32_t bar_qe = ptx::smem_addr(&ctl->q_empty);
    auto bar_kf = [&](int s) { return ptx::smem_addr(&ctl->k_full[s]); };
    auto bar_ke = [&](int s) { return ptx::smem_addr(&ctl->k_empty[s]); };
    auto bar_vf = [&](int s) { return ptx::smem_addr(&ctl->v_full[s]); };
    auto bar_ve = [&](int s) { return ptx::smem_addr(&ctl->v_empty[s]); };
    auto bar_sf = [&](int x) { return ptx::smem_addr(&ctl->s_full[x]); };
    auto bar_ph = [&](int x) { return ptx::smem_addr(&ctl->p_half[x]); };
    auto bar_pf = [&](int x) { return ptx::smem_addr(&ctl->p_full[x]); };
    auto bar_oh = [&](int x) { return ptx::smem_addr(&ctl->o_half[x]); };
    auto bar_o = [&](int x) { return ptx::smem_addr(&ctl->o_ready[x]); };
    const uint32_t bar_drain = ptx::smem_addr(&ctl->drain);
    auto sQ = [&](int x) { return sbase + C::kOffQ + x * C::kTileBytes; };
    auto sK = [&](int s) { return sbase + C::kOffK + s * C::kTileBytes; };
    auto sV = [&](int s) { return sbase + C::kOffV + s * C::kTileBytes; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_q, 1);
        ptx::mbar_init(bar_qe, 1);
        for (int s = 0; s < NK; ++s) {
            ptx::mbar_init(bar_kf(s), 1);
            ptx::mbar_init(bar_ke(s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            ptx::mbar_init(bar_vf(s), 1);
            ptx::mbar_init(bar_ve(s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            ptx::mbar_init(bar_sf(x), 1);
            ptx::mbar_init(bar_ph(x), kTileM);
            ptx::mbar_init(bar_pf(x), kTileM);
            ptx::mbar_init(bar_oh(x), 1);
            ptx::mbar_init(bar_o(x), 1);
        }
        ptx::mbar_init(bar_drain, 1);
        ctl->abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kLoaderWarp && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    if constexpr (C::kOnes) {
        // the ones tile (every 16-bit element 1.0, so any swizzle of it is the
        // same), written once and made visible to the tensor core's reads
        constexpr uint32_t kOne2 = BF16 ? 0x3F803F80u : 0x3C003C00u;
        uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::kOffOnes);
        for (int i = threadIdx.x; i < C::kOnesBytes / 4; i += kThreads) ones[i] = kOne2;
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kLoaderWarp) {
        // =============================================================== loader
        // Per unit: Q_A, Q_B once the previous unit's S products are done
        // (q_empty), then K_0, K_1, V_0, K_2, V_1, ...: a K tile is only gated
        // by the S = Q K^T products that free its slot, never by the slower
        // P.V.  The rings run on across units, so the first tiles of a unit
        // load while the previous one finishes.
        int issued_k[NK], issued_v[NV];
#pragma unroll
        for (int s = 0; s < NK; ++s) issued_k[s] = 0;
#pragma unroll
        for (int s = 0; s < NV; ++s) issued_v[s] = 0;
        uint32_t kc = 0, vc = 0;  // K and V tiles loaded so far
        int nq = 0;               // units whose Q was loaded
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            if (w.nB == 0) continue;
            const int b_idx = w.bh / p.H, h_idx = w.bh % p.H;
            if (nq > 0 && !(ok = wait_warp(bar_qe, (nq - 1) & 1, abort, tmo))) break;
            if (lane == 0) {
                if constexpr (SPLIT) {
                    // (the other key ranges of the block read the same Q)
                    ptx::mbar_arrive_expect_tx(bar_q, 2 * C::kTileBytes);
#pragma unroll
                    for (int x = 0; x < 2; ++x)
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d(sQ(x) + c * kSubBytes, &tm_q, bar_q, 64 * c,
                                             w.qb * kBlockM + x * kTileM, h_idx, b_idx);
                } else {
                    // Q is read by this unit only: evicted first from L2, ahead of
                    // the K and V lines the other query blocks of its head read
                    const uint64_t pol_q = ptx::l2_policy_evict_first();
                    ptx::mbar_arrive_expect_tx(bar_q, 2 * C::kTileBytes);
#pragma unroll
                    for (int x = 0; x < 2; ++x)
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d_hint(sQ(x) + c * kSubBytes, &tm_q, bar_q, 64 * c,
                                                  w.qb * kBlockM + x * kTileM, h_idx, b_idx, pol_q);
                }
            }
            ++nq;
            for (int j = 0; j <= w.nB; ++j) {
                if (j < w.nB) {
                    const int s = kc % NK;
                    if (kc >= NK && !(ok = wait_warp(bar_ke(s), ((kc / NK) - 1) & 1, abort, tmo))) break;
                    const bool skip = (p.fault_mode == 1 && kc == 0);
                    if (lane == 0 && !skip) {
                        ptx::mbar_arrive_expect_tx(bar_kf(s), C::kTileBytes);
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d(sK(s) + c * kSubBytes, &tm_k, bar_kf(s), 64 * c,
                                             (w.k0 + j) * kBlockN, h_idx, b_idx);
                    }
                    if (!skip) ++issued_k[s];
                    ++kc;
                }
                if (j >= 1) {
                    const int s = vc % NV;
                    if (vc >= NV && !(ok = wait_warp(bar_ve(s), ((vc / NV) - 1) & 1, abort, tmo))) break;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar_vf(s), C::kTileBytes);
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d(sV(s) + c * kSubBytes, &tm_v, bar_vf(s), 64 * c,
                                             (w.k0 + j - 1) * kBlockN, h_idx, b_idx);
                    }
                    ++issued_v[s];
                    ++vc;
                }
            }
        }
        // Never leave the CTA with copies still landing in its shared memory.
        if (nq > 0) wait_warp(bar_q, (nq - 1) & 1, abort, tmo, false);
        for (int s = 0; s < NK; ++s)
            if (issued_k[s] > 0) wait_warp(bar_kf(s), (issued_k[s] - 1) & 1, abort, tmo, false);
        for (int s = 0; s < NV; ++s)
            if (issued_v[s] > 0) wait_warp(bar_vf(s), (issued_v[s] - 1) & 1, abort, tmo, false);
    } else if (warp == kMmaWarp) {
        // ====================================================== tensor-core issuer
        constexpr uint32_t idesc_s = instr_desc(BF16, kTileM, kBlockN, false);
        constexpr uint32_t idesc_pv = instr_desc(BF16, kTileM, C::kUCols, true);
        // stage s of a ring (and tile x of Q) is kTileBytes further on: its
        // descriptor is the first one plus that offset in 16-byte units; the
        // steps along K inside a group are built into the mma_*_k* helpers
        constexpr uint64_t kTileStep = C::kTileBytes / 16;
        const uint64_t q_desc0 = smem_desc(sQ(0), 16, 1024);
        const uint64_t k_desc0 = smem_desc(sK(0), 16, 1024);
        // V (MN-major): the next 64 columns of d are one sub-tile further on;
        // with the ones column, the ones tile (slot s: its start field is 1024 s
        // further on, its group stride 1024 s shorter)
        const uint64_t v_desc0 =
            C::kOnes ? smem_desc(sV(0), C::kOffOnes - C::kOffV, 1024) : smem_desc(sV(0), kSubBytes, 1024);
        // S_x = Q_x K_s^T into TMEM columns [128 x, 128 x + 128)
        auto issue_s = [&](int x, int s) {
            const uint64_t qd = q_desc0 + x * kTileStep, kd = k_desc0 + s * kTileStep;
            if constexpr (D == 128)
                ptx::mma_ss_k128(tmem + x * 128, qd, kd, idesc_s, 0u);
            else
                ptx::mma_ss_k64(tmem + x * 128, qd, kd, idesc_s, 0u);
        };
        // U_x (+)= P_x V_s, P_x read from TMEM, in two halves of 64 keys (4
        // K-steps of 16 each): the first half runs while the softmax warps
        // still compute the weights of the second
        // both halves of P_x V_s for the n-th key tile of query tile x, each
        // issued once the softmax warps have written its weights; o_half /
        // o_ready signal that U_x absorbed them.  Everything but the products
        // is computed before the waits: the issuer shares its sub-partition
        // with two softmax warps, so each instruction between a barrier and
        // the product it releases delays the tensor core.
        auto pv_tile = [&](int x, int s, uint32_t n, bool acc) {
            const uint64_t vd = C::kOnes ? v_desc0 + s * kTileStep - ((s * kTileStep) << 16)
                                         : v_desc0 + s * kTileStep;
            const uint32_t d_u = tmem + kTmemU + x * 128, a_p = tmem + x * 128;
            const uint32_t b_ph = bar_ph(x), b_pf = bar_pf(x), b_oh = bar_oh(x), b_o = bar_o(x);
            const uint32_t par = n & 1, acc0 = acc ? 1u : 0u;
            if (!wait_warp(b_ph, par, abort, tmo)) return false;
            ptx::tc_fence_after_sync();
            ptx::mma_ts_k64(d_u, a_p, vd, idesc_pv, acc0);
            ptx::tc_commit_elect(b_oh);
            if (!wait_warp(b_pf, par, abort, tmo)) return false;
            ptx::tc_fence_after_sync();
            ptx::mma_ts_k64(d_u, a_p + 32, vd + 512, idesc_pv, 1u);
            ptx::tc_commit_elect(b_o);
            return true;
        };
        uint32_t kc = 0, vc = 0;    // K and V tiles consumed so far (same order as loaded)
        uint32_t na = 0, nb = 0;    // key tiles of query tile A and B so far
        uint32_t nq = 0;            // units so far (q_full phase)
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            if (w.nB == 0) continue;
            if (!(ok = wait_warp(bar_q, nq & 1, abort, tmo))) break;
            ++nq;
            {
                const int s0 = kc % NK;
                if (!(ok = wait_warp(bar_kf(s0), (kc / NK) & 1, abort, tmo))) break;
                ptx::tc_fence_after_sync();
                // S_x(0) overwrites columns the softmax warps finished with
                // when they signalled the last P of the previous unit
                if (w.nA > 0) {
                    issue_s(0, s0);
                    ptx::tc_commit_elect(bar_sf(0));
                }
                issue_s(1, s0);
                ptx::tc_commit_elect(bar_sf(1));
                ptx::tc_commit_elect(bar_ke(s0));
                if (w.nB == 1) ptx::tc_commit_elect(bar_qe);  // Q_A, Q_B read for the last time
                ++kc;
                __syncwarp();
            }
            for (int j = 0; j < w.nB; ++j) {
                const int sv = vc % NV;
                const int sk = kc % NK;
                // V_j, and with a ring of four K tiles K_{j+1} for the next S
                // products: it was loaded long before, and waiting for it here
                // keeps the wait off the path from a softmax signal to the
                // product it releases.  With two K tiles it may still be on its
                // way, and is only waited for just before the first S needs it.
                constexpr bool kEarlyK = NK >= 4;
                bool k_ready = false;
                if (!(ok = wait_warp(bar_vf(sv), (vc / NV) & 1, abort, tmo))) break;
                if (kEarlyK && j + 1 < w.nB) {
                    if (!(ok = wait_warp(bar_kf(sk), (kc / NK) & 1, abort, tmo))) break;
                    k_ready = true;
                }
                if (j < w.nA) {
                    // the first product of a unit overwrites U_x; the softmax
                    // warps read the previous unit's U_x before they signal P
                    if (!(ok = pv_tile(0, sv, na, j > 0))) break;
                    ++na;
                    if (j + 1 < w.nA) {
                        if (!k_ready && !(ok = wait_warp(bar_kf(sk), (kc / NK) & 1, abort, tmo))) break;
                        k_ready = true;
                        ptx::tc_fence_after_sync();
                        issue_s(0, sk);
                        ptx::tc_commit_elect(bar_sf(0));
                    }
                    __syncwarp();
                }
                if (!(ok = pv_tile(1, sv, nb, j > 0))) break;
                ++nb;
                if (j + 1 < w.nB) {
                    if (!k_ready && !(ok = wait_warp(bar_kf(sk), (kc / NK) & 1, abort, tmo))) break;
                    ptx::tc_fence_after_sync();
                    issue_s(1, sk);
                    ptx::tc_commit_elect(bar_sf(1));
                    ptx::tc_commit_elect(bar_ke(sk));
                    if (j + 2 == w.nB) ptx::tc_commit_elect(bar_qe);
                    ++kc;
                }
                ptx::tc_commit_elect(bar_ve(sv));
                ++vc;
                __syncwarp();
            }
        }
        // Drain: nothing of ours may still run on the tensor core at teardown.
        ptx::tc_commit_elect(bar_drain);
        __syncwarp();
        wait_warp(bar_drain, 0, abort, tmo, false);
    } else {
        // ======================================== softmax + epilogue of tile x
        const int x = warp >> 2;                          // 0: tile A, 1: tile B
        const int t = threadIdx.x & 127;                  // row in the tile = TMEM lane
        // of the current unit: this thread's query index in the head, the
        // tile's first one, the first key tile and how many are visited
        int row = 0, first_row = 0, k0 = 0, T = 0;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + x * 128;
        const uint32_t u_addr = tmem + lane_off + kTmemU + x * 128;
        const float c2 = p.scale_log2;
        const float2 c2v = make_float2(c2, c2);
        // whether key tile j (local index) holds a key some row of this tile
        // may not see: keys >= Nk, or keys past the causal limit of the tile's
        // first row (with a bottom-right offset that can be two tiles)
        auto tile_masked = [&](int j) {
            const int kend = (k0 + j + 1) * kBlockN;
            return kend > p.Nk || (CAUSAL && kend - 1 > first_row + p.mask_offset);
        };
        // key limit (exclusive) of this row relative to `kbase`
        auto key_limit = [&](int kbase) {
            int limit = p.Nk - kbase;
            if (CAUSAL) limit = min(limit, row + p.mask_offset - kbase + 1);
            return limit;
        };
        // this row's 128 scores of the current tile, with the keys it may not
        // see (>= Nk, or past the causal limit) masked to -inf
        auto load_scores = [&](uint32_t(&sv)[kBlockN], int j) {
#pragma unroll
            for (int c = 0; c < kBlockN / 64; ++c)
                ptx::tmem_ld_32x32b_x64(s_addr + c * 64,
                                        *reinterpret_cast<uint32_t(*)[64]>(&sv[c * 64]));
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) ptx::reg_fence(sv[c]);
            if (tile_masked(j)) {
                const int limit = key_limit((k0 + j) * kBlockN);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= limit) sv[c] = __float_as_uint(-INFINITY);
            }
        };
        // weights 2^(x c2 + neg_ref) of 2n scores, packed to 16 bits; the fp32
        // weights are added to rs and the rounded ones (those fed to P.V) to rh
        auto weights = [&](const uint32_t* sv, int n, float neg_ref, uint32_t* pk, float2 (&rs)[2],
                           float2 (&rh)[2]) {
            const float2 nrv = make_float2(neg_ref, neg_ref);
#pragma unroll
            for (int c = 0; c < n; ++c) {
                const float2 e = __ffma2_rn(
                    make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2v, nrv);
                const float2 pw = make_float2(ptx::ex2_approx(e.x), ptx::ex2_approx(e.y));
                rs[c & 1] = __fadd2_rn(rs[c & 1], pw);
                pk[c] = pack2<BF16>(pw.x, pw.y);
                if constexpr (!C::kOnes) add_packed<BF16>(rh[c & 1], pk[c]);  // else P.V sums them
            }
        };
        // scores [32 c, 32 c + 32) of this row, masked like load_scores
        auto load_chunk = [&](uint32_t(&sv)[32], int c, int j) {
            ptx::tmem_ld_32x32b_x32(s_addr + c * 32, sv);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) ptx::reg_fence(sv[u]);
            if (tile_masked(j)) {
                const int limit = key_limit((k0 + j) * kBlockN + c * 32);
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    if (u >= limit) sv[u] = __float_as_uint(-INFINITY);
            }
        };
        uint32_t n = 0;  // key tiles of this query tile so far, over all units (barrier phases)
        bool aborted = false;
        for (int r = 0; !aborted; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            const int b_idx = w.bh / p.H, h_idx = w.bh % p.H;
            first_row = w.qb * kBlockM + x * kTileM;
            row = first_row + t;
            k0 = w.k0;
            T = x == 0 ? w.nA : w.nB;
            if (SPLIT && w.nB == 0) {  // empty key range: its partials carry no weight
                if (row < p.Nq) {
                    const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + row;
                    const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                    p.lse_part[i] = -INFINITY;
                    p.lse_part[plane + i] = -INFINITY;
                }
                continue;
            }
            float m_ref = -INFINITY;              // reference maximum of the raw scores
            float2 lsum = make_float2(0.f, 0.f);  // sum of the fp32 weights (for LSE) in .x
            float2 lhat = make_float2(0.f, 0.f);  // sum of the 16-bit weights fed to P.V (for O) in .x

            for (int j = 0; j < T; ++j, ++n) {
                if (!wait_warp(bar_sf(x), n & 1, abort, tmo)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                // keys 0-63 of the previous key tile are in U_x (S_x(j) was issued
                // after them); taking that phase here keeps a later wait on this
                // tile's phase unambiguous
                if (j > 0 && !wait_warp(bar_oh(x), (n - 1) & 1, abort, tmo)) {
                    aborted = true;
                    break;
                }
                // common case: weights against the current reference, checked by
                // their sum before they are written, one 64-key half at a time: the
                // first half goes to the tensor core while the second is computed.
                // The first tile (no reference yet) or a first half above the bound
                // takes the tile maximum and recomputes all weights from the scores
                // still in TMEM; a second half above the bound moves the reference
                // for that half only (all branches warp-uniform).
                uint32_t pk[kBlockN / 2];
                float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // keys 64-127 (or all)
                float2 rh[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                float r1 = 0.f, h1 = 0.f;  // sums of keys 0-63 when they were sent on the old reference
                // (tcgen05.ld is warp-collective: every branch around it is uniform)
                bool redo = (m_ref == -INFINITY);
                bool half_sent = false;
                float alpha = 1.f;
                float m_new = m_ref;
                if (!__any_sync(0xffffffffu, redo)) {
                    uint32_t sv[kBlockN];
                    load_scores(sv, j);
                    float2 s1[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    float2 t1[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                    weights(sv, kBlockN / 4, -m_ref * c2, pk, s1, t1);
                    r1 = s1[0].x + s1[0].y + s1[1].x + s1[1].y;
                    redo = r1 > weight_sum_limit<BF16>();
                    if (!__any_sync(0xffffffffu, redo)) {
                        ptx::tmem_st_32x32b_x32(s_addr, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before_sync();
                        ptx::mbar_arrive(bar_ph(x));
                        half_sent = true;
                        const float2 h = __fadd2_rn(t1[0], t1[1]);
                        h1 = h.x + h.y;
                        weights(sv + kBlockN / 2, kBlockN / 4, -m_ref * c2, pk + kBlockN / 4, rs, rh);
                        const bool redo2 =
                            rs[0].x + rs[0].y + rs[1].x + rs[1].y > weight_sum_limit<BF16>();
                        if (__any_sync(0xffffffffu, redo2)) {
                            float mt = -INFINITY;
#pragma unroll 1
                            for (int c = 2; c < kBlockN / 32; ++c) {
                                uint32_t sc[32];
                                load_chunk(sc, c, j);
#pragma unroll
                                for (int u = 0; u < 32; u += 2)
                                    mt = ptx::fmax3(mt, __uint_as_float(sc[u]), __uint_as_float(sc[u + 1]));
                            }
                            if (redo2) {
                                m_new = fmaxf(mt, m_ref);
                                alpha = ptx::ex2_approx((m_ref - m_new) * c2);
                            }
                            rs[0] = rs[1] = rh[0] = rh[1] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int c = 2; c < kBlockN / 32; ++c) {
                                uint32_t sc[32];
                                load_chunk(sc, c, j);
                                weights(sc, 16, -m_new * c2, &pk[16 * c], rs, rh);
                            }
                        }
                    } else {
                        r1 = 0.f;
                    }
                }
                if (!half_sent) {
                    float mt = -INFINITY;
#pragma unroll 1
                    for (int c = 0; c < kBlockN / 32; ++c) {
                        uint32_t sv[32];
                        load_chunk(sv, c, j);
                        float mx[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) mx[u] = __uint_as_float(sv[u]);
#pragma unroll
                        for (int u = 4; u + 8 <= 32; u += 8)
#pragma unroll
                            for (int w = 0; w < 4; ++w)
                                mx[w] = ptx::fmax3(mx[w], __uint_as_float(sv[u + w]),
                                                   __uint_as_float(sv[u + 4 + w]));
#pragma unroll
                        for (int w = 0; w < 4; ++w) mx[w] = fmaxf(mx[w], __uint_as_float(sv[28 + w]));
                        mt = ptx::fmax3(mt, fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                    }
                    // every lane takes the tile maximum: a lane whose first half
                    // was in range may still overflow in its second half, which
                    // was never checked (alpha is exactly 1 where m does not move)
                    m_new = fmaxf(mt, m_ref);
                    if (m_ref != -INFINITY) alpha = ptx::ex2_approx((m_ref - m_new) * c2);
                    // a row with no valid key so far keeps all weights at zero
                    const float neg_ref = (m_new == -INFINITY) ? 0.f : -m_new * c2;
#pragma unroll
                    for (int c = 0; c < kBlockN / 32; ++c) {
                        uint32_t sv[32];
                        load_chunk(sv, c, j);
                        weights(sv, 16, neg_ref, &pk[16 * c], rs, rh);
                    }
                    ptx::tmem_st_32x32b_x32(s_addr, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
                }
                // l = alpha (l + keys sent on the old reference) + the rest
                const float2 r = __fadd2_rn(rs[0], rs[1]), hh = __fadd2_rn(rh[0], rh[1]);
                lsum.x = fmaf(lsum.x + r1, alpha, r.x + r.y);
                lhat.x = fmaf(lhat.x + h1, alpha, hh.x + hh.y);
                ptx::tmem_st_32x32b_x32(s_addr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
                // U_x holds P(j-1) V, since S_x(j) was issued after that product.
                // Rescale it by alpha when the reference maximum moved (warp-uniform);
                // if keys 0-63 of this tile were already sent, U_x must absorb them
                // first: they carry the old reference too.
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    if (half_sent) {
                        if (!wait_warp(bar_oh(x), n & 1, abort, tmo)) {
                            aborted = true;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                    }
                    const float2 av = make_float2(alpha, alpha);
#pragma unroll 1
                    for (int c = 0; c < C::kUCols / 16; ++c) {  // with the sum column, if any
                        uint32_t ov[16];
                        ptx::tmem_ld_32x32b_x16(u_addr + c * 16, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 16; u += 2) {
                            ptx::reg_fence(ov[u]);
                            ptx::reg_fence(ov[u + 1]);
                            const float2 r = __fmul2_rn(
                                make_float2(__uint_as_float(ov[u]), __uint_as_float(ov[u + 1])), av);
                            ov[u] = __float_as_uint(r.x);
                            ov[u + 1] = __float_as_uint(r.y);
                        }
                        ptx::tmem_st_32x32b_x16(u_addr + c * 16, ov);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                if (!half_sent) ptx::mbar_arrive(bar_ph(x));
                ptx::mbar_arrive(bar_pf(x));
                m_ref = m_new;
            }

            // ---- epilogue: O = U / lhat -> 16-bit (each thread its own row),
            // through the warp's staging box and TMA stores; Q's shared memory
            // is free for the next unit as soon as its last S product is done
            if (!aborted && T > 0) aborted = !wait_warp(bar_o(x), (n - 1) & 1, abort, tmo);
            if (aborted) break;
            const float l_all = lsum.x + lsum.y;
            float lhat_all = lhat.x + lhat.y;
            if constexpr (C::kOnes) {
                // the sum of the 16-bit weights is U's column 64 (warp-uniform
                // branch around the collective load)
                lhat_all = 0.f;
                if (T > 0) {
                    ptx::tc_fence_after_sync();
                    uint32_t lv = ptx::tmem_ld_32x32b_x1(u_addr + D);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence(lv);
                    lhat_all = __uint_as_float(lv);
                }
            }
            if constexpr (SPLIT) {
                // partial result of this key range: O normalised by its own lhat
                // (fp32) and the two log-sums that weight it in the merge
                // (warp-uniform branches around the collective tcgen05.ld)
                const bool mine = row < p.Nq && !*abort;
                const bool any = T > 0 && l_all > 0.f;
                const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + (mine ? row : 0);
                const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                if (mine) {
                    p.lse_part[i] = any ? m_ref * p.scale + logf(l_all) : -INFINITY;
                    p.lse_part[plane + i] = any ? m_ref * p.scale + logf(lhat_all) : -INFINITY;
                }
                if (T > 0) {
                    // through the warp's staging box, 32 fp32 columns at a
                    // time (tm_o maps the partials here; rows >= Nq clipped)
                    ptx::tc_fence_after_sync();
                    const float inv = any ? 1.f / lhat_all : 0.f;
                    const uint32_t stage = sbase + C::kOffStage + warp * C::kStageBytes;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        ptx::tmem_ld_32x32b_x32(u_addr + c * 32, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ptx::reg_fence(ov[e]);
                        // the previous store from this box has read it
                        if (lane == 0) ptx::bulk_wait_group_read0();
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t dst = stage + lane * 128 + ((q ^ (lane & 7)) << 4);
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                                         "f"(__uint_as_float(ov[4 * q]) * inv),
                                         "f"(__uint_as_float(ov[4 * q + 1]) * inv),
                                         "f"(__uint_as_float(ov[4 * q + 2]) * inv),
                                         "f"(__uint_as_float(ov[4 * q + 3]) * inv)
                                         : "memory");
                        }
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && !*abort) {
                            ptx::tma_store_4d(&tm_o, stage, 32 * c, first_row + 32 * (warp & 3), w.bh,
                                              w.split);
                            ptx::bulk_commit_group();
                        }
                    }
                }
            } else {
                // each warp stores its 32 rows, 64 columns at a time, through
                // its own staging box (the 128-byte-swizzled layout the TMA
                // store expects); rows >= Nq and columns >= d are clipped
                ptx::tc_fence_after_sync();
                const bool mine = row < p.Nq && !*abort;
                const float inv = lhat_all > 0.f ? 1.f / lhat_all : 0.f;
                const float2 iv = make_float2(inv, inv);
                const uint32_t stage = sbase + C::kOffStage + warp * C::kStageBytes;
#pragma unroll
                for (int h = 0; h < C::kSub; ++h) {
                    // the previous store from this box has read it
                    if (lane == 0) ptx::bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        if (T > 0) {
                            ptx::tmem_ld_32x32b_x32(u_addr + (2 * h + cc) * 32, ov);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) ptx::reg_fence(ov[e]);
                        } else {  // no key visible to this tile: O = 0 (U was not written)
#pragma unroll
                            for (int e = 0; e < 32; ++e) ov[e] = 0u;
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t wv[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c8 = q4 * 8 + 2 * e;
                                const float2 o2 = __fmul2_rn(
                                    make_float2(__uint_as_float(ov[c8]), __uint_as_float(ov[c8 + 1])), iv);
                                wv[e] = pack2<BF16>(o2.x, o2.y);
                            }
                            const uint32_t dst = stage + lane * 128 + (((cc * 4 + q4) ^ (lane & 7)) << 4);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(wv[0]),
                                         "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                                         : "memory");
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && !*abort) {
                        // O is written once: its lines leave L2 first
                        ptx::tma_store_4d_hint(&tm_o, stage, 64 * h, first_row + 32 * (warp & 3), h_idx,
                                               b_idx, ptx::l2_policy_evict_first());
                        ptx::bulk_commit_group();
                    }
                }
                if (mine) {
                    const float lse = (l_all > 0.f) ? m_ref * p.scale + logf(l_all) : -INFINITY;
                    p.lse[b_idx * p.lse_sb + h_idx * p.lse_sh + row] = lse;
                }
            }
        }  // units
        // the CTA's shared memory must outlive the stores that read it
        if (lane == 0) ptx::bulk_wait_group0();
    }

    // ---- teardown: every tcgen05 op of this CTA has completed
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == kMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---- split-KV merge ("CUDA 算子工程" 14.7.1: every split writes a partial O
// and LSE, merged afterwards).  Per query row: LSE = ln sum_s e^{LSE_s}, and
// O = sum_s w_s O_s / sum_s w_s with w_s = e^{LSEhat_s - max}: O_s is
// normalised by the sum of its rounded weights, so w_s is that sum on the
// common scale, which keeps O an exact convex combination of every weight
// fed to P.V.  A warp per row; each lane owns D/32 consecutive columns of the
// kernel's width D, of which the first d_out are written.  The merge is bound
// by memory latency, not bandwidth, so a row's loads are issued before any is
// used: lane s reads range s's two log-sums while the partial O rows of up to
// eight ranges are read, all in one round trip.
struct MergeParams {
    const float* o_part;
    const float* lse_part;
    void* o;                            // row (b, h, i) at o + b o_sb + h o_sh + i o_sn
    long long o_sb, o_sh, o_sn;
    float* lse;                         // at lse + b lse_sb + h lse_sh + i
    long long lse_sb, lse_sh;
    int num_splits, H, Nq;              // num_splits <= 32 (one lane per range)
    int d_out;                          // columns of O written (<= D, a multiple of 8)
    long long rows;                     // B H Nq
};

// Maximum and sum over lanes [0, n) of a warp (n <= 32; the other lanes of
// each aligned group of the next power of two >= n hold the identity), given
// to every lane: butterfly steps below that power of two, then lane 0's value.
__device__ __forceinline__ float lanes_max(float v, int n) {
    for (int o = 1; o < n; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return __shfl_sync(0xffffffffu, v, 0);
}

__device__ __forceinline__ float lanes_sum(float v, int n) {
    for (int o = 1; o < n; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return __shfl_sync(0xffffffffu, v, 0);
}

template <int D, bool BF16, int kBatch>
__global__ void __launch_bounds__(256) fa_split_merge_kernel(const MergeParams mp) {
    // kBatch: ranges whose partial rows are in flight together (2, 4 or 8: the
    // range count rounded up, so that few ranges keep few registers and many
    // resident warps, which the larger partials of few ranges need)
    constexpr int kPer = D / 32;
    // launched as a programmatic dependent of the attention kernel: wait until
    // that grid has finished and its partials are visible (no-op otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const long long rows = mp.rows;
    const int num_splits = mp.num_splits;
    if (r >= rows) return;  // whole warps: the shuffles below see all 32 lanes
    // (b, h, i) of the row, in 32-bit arithmetic where it fits (a 64-bit
    // division costs about as many instructions as the rest of the row)
    long long bh, i;
    if (rows <= 0x7fffffffll) {
        const unsigned ru = static_cast<unsigned>(r), nq = static_cast<unsigned>(mp.Nq);
        const unsigned qu = ru / nq;
        bh = qu;
        i = ru - qu * nq;
    } else {
        bh = r / mp.Nq;
        i = r - bh * mp.Nq;
    }
    const unsigned hu = static_cast<unsigned>(mp.H), bu = static_cast<unsigned>(bh) / hu;  // BH < 2^31
    const long long b = bu, h = static_cast<unsigned>(bh) - bu * hu;
    const size_t plane = static_cast<size_t>(num_splits) * rows;
    const float* src = mp.o_part + r * D + lane * kPer;
    // the partial rows of up to kBatch ranges, loaded whatever their weight
    // (they do not depend on it): with the log-sums below, one round trip to
    // memory for the row.  A range with no weight wrote no row; its stale
    // values are dropped by selection, never multiplied by zero.
    auto load_batch = [&](int s0, float (&v)[kBatch][kPer]) {
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
#pragma unroll
            for (int e = 0; e < kPer; ++e) v[j][e] = 0.f;
            if (s0 + j < num_splits) {
                const float* row_s = src + static_cast<size_t>(s0 + j) * rows * D;
                if constexpr (kPer % 4 == 0) {
#pragma unroll
                    for (int e = 0; e < kPer; e += 4) {
                        const float4 x = *reinterpret_cast<const float4*>(row_s + e);
                        v[j][e] = x.x; v[j][e + 1] = x.y; v[j][e + 2] = x.z; v[j][e + 3] = x.w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < kPer; e += 2) {
                        const float2 x = *reinterpret_cast<const float2*>(row_s + e);
                        v[j][e] = x.x; v[j][e + 1] = x.y;
                    }
                }
            }
        }
    };
    float v[kBatch][kPer];
    load_batch(0, v);
    const float ls = lane < num_splits ? mp.lse_part[lane * rows + r] : -INFINITY;
    const float lh = lane < num_splits ? mp.lse_part[plane + lane * rows + r] : -INFINITY;
    const float ml = lanes_max(ls, num_splits), mh = lanes_max(lh, num_splits);
    // an empty range (-inf) has no weight and wrote no O row
    const float lsum = lanes_sum(ls == -INFINITY ? 0.f : __expf(ls - ml), num_splits);
    const float w = lh == -INFINITY ? 0.f : __expf(lh - mh);
    const float wsum = lanes_sum(w, num_splits);
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
    for (int s0 = 0; s0 < num_splits; s0 += kBatch) {
        if (s0 > 0) load_batch(s0, v);
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, (s0 + j) & 31);
            const bool use = s0 + j < num_splits && wj > 0.f;
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] = use ? fmaf(wj, v[j][e], acc[e]) : acc[e];
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint32_t packed[kPer / 2];
#pragma unroll
    for (int e = 0; e < kPer; e += 2) packed[e / 2] = pack2<BF16>(acc[e] * inv, acc[e + 1] * inv);
    uint32_t* dst = reinterpret_cast<uint32_t*>(
        static_cast<uint16_t*>(mp.o) + b * mp.o_sb + h * mp.o_sh + i * mp.o_sn + lane * kPer);
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e)
        if (lane * kPer + 2 * e < mp.d_out) dst[e] = packed[e];
    if (lane == 0)
        mp.lse[b * mp.lse_sb + h * mp.lse_sh + i] = (ml == -INFINITY) ? -INFINITY : ml + logf(lsum);
}

}  // namespace fa
