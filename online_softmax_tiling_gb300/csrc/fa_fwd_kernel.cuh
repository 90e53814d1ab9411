// fa_fwd_kernel.cuh - fused attention forward for sm_103a (GB300).
//
// What it computes is the online-softmax form of attention described in
// "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (sections "第四步" and
// "第五步", Table 2: per query row the raw-score maximum m, the weight sum l
// and the unnormalised numerator U; "最后": O = U / l, LSE = s m + ln l) with
// the FlashAttention-2 loop order of "CUDA 算子工程" ch. 14, section 14.5
// (outer loop over query tiles, one per CTA; inner loop over key/value tiles).
//
// How it maps onto the GB300 SM (the pages' SM80 cp.async / mma.sync design is
// prior art only):
//   * one CTA per 128-row query tile, 6 warps with fixed roles:
//       warps 0-3  softmax + epilogue: thread t owns query row t, which is
//                  TMEM lane t, so the row max and row sums need no shuffles;
//       warp 4     loader: TMA (cp.async.bulk.tensor) of Q once and of the
//                  K, V tiles into an NS-stage shared-memory ring;
//       warp 5     tensor-core issuer: tcgen05.mma S = Q K^T into one of two
//                  TMEM score buffers, then O += P V with P read from TMEM.
//   * TMEM (512 columns): score buffers S0, S1 (128 fp32 columns each; the
//     16-bit weights P overwrite the first 64 columns of their own buffer) and
//     the fp32 accumulator U (d columns).  Two score buffers let the tensor
//     core compute S_{j+1} while the softmax warps work on S_j.
//   * the running maximum is only moved when it grows by more than 2^8 in
//     weight units; until then the weights stay <= 256 and l, U keep using the
//     old reference, which is exact because l, U and LSE all refer to the
//     same m.  U is therefore rescaled in TMEM only on those rare steps.
//   * key tiles wholly in the future are skipped and the diagonal tile is
//     masked element-wise ("causal 模式在哪一步生效"); keys >= N (zero-filled by
//     TMA) are masked; query rows >= N are clipped by the TMA store.
//   * every mbarrier wait is bounded; on expiry the CTA records FA_ERR_TIMEOUT
//     in a device status word, drains its in-flight copies and MMAs, frees
//     its TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;          // query rows per CTA (= TMEM lanes = MMA M)
constexpr int kBlockN = 128;          // keys per tile (= MMA N of S = Q K^T)
constexpr int kThreads = 192;         // 4 softmax warps + loader warp + MMA warp
constexpr int kSubBytes = 128 * 128;  // one 128-row x 64-column 16-bit swizzle sub-tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;      // first column of the U accumulator
constexpr float kRescaleLog2 = 8.0f;  // move m only when weights would exceed 2^8

// Device status word (FA_OK / FA_ERR_TIMEOUT); read and cleared by the host.
__device__ unsigned int g_fa_status;

struct FwdParams {
    float* lse;
    int N;
    int num_q_tiles;
    float scale;       // s
    float scale_log2;  // s * log2(e): exp(s x) = 2^(x * scale_log2)
    unsigned long long timeout_ns;
    int fault_mode;
};

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kSub = D / 64;                  // 64-column swizzle sub-tiles per row
    static constexpr int kTileBytes = kBlockM * D * 2;   // one Q, K or V tile
    static constexpr int kStages = D == 128 ? 2 : 4;     // K/V ring depth
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffV = kTileBytes * (1 + kStages);
    static constexpr int kOffCtl = kTileBytes * (1 + 2 * kStages);
    static constexpr int kSmemBytes = kOffCtl + 512 + 1024;  // control block + alignment slack
};

template <int NS>
struct alignas(8) Ctl {
    uint64_t q_full;
    uint64_t k_full[NS];
    uint64_t k_empty[NS];
    uint64_t v_full[NS];
    uint64_t v_empty[NS];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_ready[2];  // o_ready[j & 1] completes when P_j V_j has been accumulated
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

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (another role gave up) or when this wait ran past the limit (then it sets
// the abort flag and the device status).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                       unsigned long long timeout_ns, bool abortable) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (abortable && *abort) return false;
            if (ptx::globaltimer() - t0 > timeout_ns) {
                *abort = 1u;
                atomicCAS(&g_fa_status, 0u, 5u /* FA_ERR_TIMEOUT */);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         unsigned long long timeout_ns, bool abortable = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, abort, timeout_ns, abortable);
}

// Warp-uniform wait: lane 0 waits, the verdict is broadcast.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                          unsigned long long timeout_ns, bool abortable = true) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort, timeout_ns, abortable);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using C = Cfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled tiles need 1024-byte-aligned shared addresses
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    Ctl<NS>* ctl = reinterpret_cast<Ctl<NS>*>(smem + C::kOffCtl);
    volatile uint32_t* abort = &ctl->abort;
    const unsigned long long tmo = p.timeout_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- which tile: consecutive CTAs share a head, so its K/V stay in L2;
    // with the causal mask the longest query tiles of each head start first.
    const int bh = blockIdx.x / p.num_q_tiles;
    int qt = blockIdx.x % p.num_q_tiles;
    if (CAUSAL) qt = p.num_q_tiles - 1 - qt;
    const int nkv = (p.N + kBlockN - 1) / kBlockN;
    const int T = CAUSAL ? min(qt + 1, nkv) : nkv;  // key/value tiles to visit

    const uint32_t bar_q = ptx::smem_addr(&ctl->q_full);
    auto bar_kf = [&](int s) { return ptx::smem_addr(&ctl->k_full[s]); };
    auto bar_ke = [&](int s) { return ptx::smem_addr(&ctl->k_empty[s]); };
    auto bar_vf = [&](int s) { return ptx::smem_addr(&ctl->v_full[s]); };
    auto bar_ve = [&](int s) { return ptx::smem_addr(&ctl->v_empty[s]); };
    auto bar_sf = [&](int b) { return ptx::smem_addr(&ctl->s_full[b]); };
    auto bar_pf = [&](int b) { return ptx::smem_addr(&ctl->p_full[b]); };
    // Two alternating barriers for the P.V completions keep every parity wait
    // on them unambiguous even though the softmax warps skip most of them.
    auto bar_o = [&](int b) { return ptx::smem_addr(&ctl->o_ready[b]); };
    const uint32_t bar_drain = ptx::smem_addr(&ctl->drain);
    const uint32_t sQ = sbase + C::kOffQ;
    auto sK = [&](int s) { return sbase + C::kOffK + s * C::kTileBytes; };
    auto sV = [&](int s) { return sbase + C::kOffV + s * C::kTileBytes; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_q, 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar_kf(s), 1);
            ptx::mbar_init(bar_ke(s), 1);
            ptx::mbar_init(bar_vf(s), 1);
            ptx::mbar_init(bar_ve(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_sf(b), 1);
            ptx::mbar_init(bar_pf(b), 128);
        }
        ptx::mbar_init(bar_o(0), 1);
        ptx::mbar_init(bar_o(1), 1);
        ptx::mbar_init(bar_drain, 1);
        ctl->abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 4 && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 4) {
        // =============================================================== loader
        int issued_k[NS], issued_v[NS];
#pragma unroll
        for (int s = 0; s < NS; ++s) issued_k[s] = issued_v[s] = 0;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar_q, C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kSub; ++c)
                ptx::tma_load_3d(sQ + c * kSubBytes, &tm_q, bar_q, 64 * c, qt * kBlockM, bh);
        }
        for (int j = 0; j < T; ++j) {
            const int s = j % NS;
            const uint32_t par = static_cast<uint32_t>((j / NS) - 1) & 1u;
            if (j >= NS && !wait_warp(bar_ke(s), par, abort, tmo)) break;
            const bool skip = (p.fault_mode == 1 && j == 0);
            if (lane == 0 && !skip) {
                ptx::mbar_arrive_expect_tx(bar_kf(s), C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kSub; ++c)
                    ptx::tma_load_3d(sK(s) + c * kSubBytes, &tm_k, bar_kf(s), 64 * c, j * kBlockN, bh);
            }
            if (!skip) ++issued_k[s];
            if (j >= NS && !wait_warp(bar_ve(s), par, abort, tmo)) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar_vf(s), C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kSub; ++c)
                    ptx::tma_load_3d(sV(s) + c * kSubBytes, &tm_v, bar_vf(s), 64 * c, j * kBlockN, bh);
            }
            ++issued_v[s];
        }
        // Never leave the CTA with copies still landing in its shared memory.
        wait_warp(bar_q, 0, abort, tmo, false);
        for (int s = 0; s < NS; ++s) {
            if (issued_k[s] > 0) wait_warp(bar_kf(s), (issued_k[s] - 1) & 1, abort, tmo, false);
            if (issued_v[s] > 0) wait_warp(bar_vf(s), (issued_v[s] - 1) & 1, abort, tmo, false);
        }
    } else if (warp == 5) {
        // ====================================================== tensor-core issuer
        constexpr uint32_t idesc_s = instr_desc(BF16, kBlockM, kBlockN, false);
        constexpr uint32_t idesc_pv = instr_desc(BF16, kBlockM, D, true);
        auto issue_s = [&](int buf, int s) {
            const uint32_t d_tmem = tmem + buf * kBlockN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kSubBytes + (kk & 3) * 32;
                ptx::mma_ss(d_tmem, smem_desc(sQ + off, 16, 1024), smem_desc(sK(s) + off, 16, 1024),
                            idesc_s, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int buf, int s, bool acc) {
            const uint32_t a_tmem = tmem + buf * kBlockN;
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
                ptx::mma_ts(tmem + kTmemO, a_tmem + kk * 8,
                            smem_desc(sV(s) + kk * 2048, kSubBytes, 1024), idesc_pv,
                            (acc || kk > 0) ? 1u : 0u);
            }
        };
        bool ok = wait_warp(bar_q, 0, abort, tmo) && wait_warp(bar_kf(0), 0, abort, tmo);
        if (ok) {
            ptx::tc_fence_after_sync();
            if (lane == 0) {
                issue_s(0, 0);
                ptx::tc_commit(bar_sf(0));
                ptx::tc_commit(bar_ke(0));
            }
            __syncwarp();
        }
        for (int j = 0; ok && j < T; ++j) {
            if (j + 1 < T) {
                const int s = (j + 1) % NS;
                if (!(ok = wait_warp(bar_kf(s), ((j + 1) / NS) & 1, abort, tmo))) break;
                ptx::tc_fence_after_sync();
                if (lane == 0) {
                    issue_s((j + 1) & 1, s);
                    ptx::tc_commit(bar_sf((j + 1) & 1));
                    ptx::tc_commit(bar_ke(s));
                }
                __syncwarp();
            }
            if (!(ok = wait_warp(bar_pf(j & 1), (j >> 1) & 1, abort, tmo))) break;
            if (!(ok = wait_warp(bar_vf(j % NS), (j / NS) & 1, abort, tmo))) break;
            ptx::tc_fence_after_sync();
            if (lane == 0) {
                issue_pv(j & 1, j % NS, j > 0);
                ptx::tc_commit(bar_o(j & 1));
                ptx::tc_commit(bar_ve(j % NS));
            }
            __syncwarp();
        }
        // Drain: nothing of ours may still run on the tensor core at teardown.
        if (lane == 0) ptx::tc_commit(bar_drain);
        __syncwarp();
        wait_warp(bar_drain, 0, abort, tmo, false);
    } else {
        // ============================================ softmax + epilogue (rows)
        const int t = threadIdx.x;             // row within the tile = TMEM lane
        const int row = qt * kBlockM + t;      // query index within the head
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const float c2 = p.scale_log2;
        float m_ref = -INFINITY;  // reference maximum of the raw scores
        float l = 0.f;            // sum of fp32 weights (for LSE)
        float l_hat = 0.f;        // sum of the 16-bit weights fed to P.V (for O)
        bool aborted = false;

        for (int j = 0; j < T; ++j) {
            const int b = j & 1;
            if (!wait_warp(bar_sf(b), (j >> 1) & 1, abort, tmo)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            const uint32_t s_addr = tmem + lane_off + b * kBlockN;
            uint32_t sv[kBlockN];
#pragma unroll
            for (int c = 0; c < kBlockN / 32; ++c)
                ptx::tmem_ld_32x32b_x32(s_addr + c * 32,
                                        *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
            ptx::tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) ptx::reg_fence(sv[c]);

            // mask keys >= N and, on the diagonal tile, keys in the future
            if (j == T - 1) {
                const int kbase = j * kBlockN;
                int limit = p.N - kbase;
                if (CAUSAL) limit = min(limit, row - kbase + 1);
#pragma unroll
                for (int c = 0; c < kBlockN; ++c)
                    if (c >= limit) sv[c] = __float_as_uint(-INFINITY);
            }
            // tile maximum of the raw scores
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(sv[u]);
#pragma unroll
            for (int c = 8; c < kBlockN; ++c) mx[c & 7] = fmaxf(mx[c & 7], __uint_as_float(sv[c]));
            const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            float alpha = 1.f;
            const bool first = (m_ref == -INFINITY);
            float m_new = m_ref;
            if (first) {
                m_new = mt;
            } else if ((mt - m_ref) * c2 > kRescaleLog2) {
                m_new = mt;
                alpha = ptx::ex2_approx((m_ref - mt) * c2);
            }
            // a row with no valid key so far keeps all weights at zero
            const float neg_ref = (m_new == -INFINITY) ? 0.f : -m_new * c2;
            // weights, their sums, and the packed 16-bit copy for P.V
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
            float rh[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kBlockN / 2];
#pragma unroll
            for (int c = 0; c < kBlockN / 2; ++c) {
                const float p0 = ptx::ex2_approx(fmaf(__uint_as_float(sv[2 * c]), c2, neg_ref));
                const float p1 = ptx::ex2_approx(fmaf(__uint_as_float(sv[2 * c + 1]), c2, neg_ref));
                rs[c & 3] += p0 + p1;
                pk[c] = pack2<BF16>(p0, p1);
                if constexpr (BF16)
                    rh[c & 3] += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xFFFF0000u);
            }
            l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
            if constexpr (BF16) l_hat = l_hat * alpha + ((rh[0] + rh[1]) + (rh[2] + rh[3]));
#pragma unroll
            for (int c = 0; c < kBlockN / 64; ++c)
                ptx::tmem_st_32x32b_x32(s_addr + c * 32,
                                        *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
            // rescale U by alpha when the reference maximum moved (warp-uniform)
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
                if (!wait_warp(bar_o((j - 1) & 1), ((j - 1) >> 1) & 1, abort, tmo)) {
                    ptx::tmem_wait_st();
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t o_addr = tmem + lane_off + kTmemO;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    ptx::tmem_ld_32x32b_x32(o_addr + c * 32, ov);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        ptx::reg_fence(ov[u]);
                        ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
                    }
                    ptx::tmem_st_32x32b_x32(o_addr + c * 32, ov);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar_pf(b));
            m_ref = m_new;
        }

        // ---- epilogue: O = U / l_hat -> 16-bit -> swizzled smem -> TMA store
        if (!aborted) aborted = !wait_warp(bar_o((T - 1) & 1), ((T - 1) >> 1) & 1, abort, tmo);
        if (!aborted) {
            ptx::tc_fence_after_sync();
            const float l_norm = BF16 ? l_hat : l;
            const float inv = l_norm > 0.f ? 1.f / l_norm : 0.f;
            const uint32_t o_addr = tmem + lane_off + kTmemO;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                ptx::tmem_ld_32x32b_x32(o_addr + c * 32, ov);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 32; ++u) ptx::reg_fence(ov[u]);
                // 32 outputs = four 16-byte chunks of this row; the Q tile's
                // shared memory is free now and becomes the staging buffer,
                // in the same 128-byte-swizzled layout the TMA store expects.
                const uint32_t sub = sQ + (c >> 1) * kSubBytes + t * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int chunk = (c & 1) * 4 + q4;
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack2<BF16>(__uint_as_float(ov[q4 * 8 + 2 * e]) * inv,
                                           __uint_as_float(ov[q4 * 8 + 2 * e + 1]) * inv);
                    const uint32_t dst = sub + ((chunk ^ (t & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w[0]),
                                 "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            ptx::fence_proxy_async_smem();
        }
        ptx::named_barrier_sync(1, 128);
        if (t == 0 && !*abort) {
#pragma unroll
            for (int c = 0; c < C::kSub; ++c)
                ptx::tma_store_3d(&tm_o, sQ + c * kSubBytes, 64 * c, qt * kBlockM, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();
        }
        if (!aborted && row < p.N) {
            const float lse = (l > 0.f) ? m_ref * p.scale + logf(l) : -INFINITY;
            p.lse[static_cast<size_t>(bh) * p.N + row] = lse;
        }
    }

    // ---- teardown: every tcgen05 op of this CTA has completed
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 5) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
