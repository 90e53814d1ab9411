// naive_attention.cuh - attention computed step by step, with the N x N
// matrices S and P stored in HBM: the "standard attention" whose HBM traffic
// "CUDA 算子工程" ch. 14, section 14.2 counts (S = Q K^T written, a softmax that
// reads S three times and writes P, then O = P V), kept here as the
// comparison the fused kernel is measured against.  Nothing on the fused path
// calls it.
//
// Element sizes follow that count: S and P are 16-bit (the input type), so
// for one (b, h) with N = 4096, d = 64 the traffic is 194 MiB.
//   1. fa_naive_scores_kernel: one CTA per 128 x 128 tile of S = s Q K^T
//      (TMA loads of the Q and K tiles, tcgen05.mma into TMEM, scale, round,
//      TMA store);
//   2. fa_naive_softmax_kernel: one CTA per row, three passes over the row of
//      S in global memory (maximum, sum of exponentials, normalised weights
//      written as P), and LSE = m + ln l;
//   3. fa_naive_pv_kernel: one CTA per 128-row tile of O = P V (TMA ring of P
//      and V tiles, tcgen05.mma accumulating in TMEM).
// Masked keys (causal, or >= N) get weight 0 in the softmax; S is computed in
// full, as a plain implementation would.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kNaiveThreads = 128;  // scores and softmax-free parts: 4 warps
constexpr int kNaiveSoftmaxThreads = 256;
constexpr int kNaivePvThreads = 192;  // 4 epilogue warps + loader warp + MMA warp

template <int D>
struct NaiveScoresCfg {
    static constexpr int kTileBytes = kTileM * D * 2;  // Q or K tile, 128 rows x D
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffS = 2 * kTileBytes;         // staging of the S tile, 128 x 128
    static constexpr int kOffCtl = kOffS + kTileM * 128 * 2;
    static constexpr int kSmemBytes = kOffCtl + 64 + 1024;
};

// ---- step 1: S = s Q K^T, one 128 x 128 tile per CTA
template <int D, bool BF16>
__global__ void __launch_bounds__(kNaiveThreads)
    fa_naive_scores_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_s, int H, float scale,
                           unsigned long long timeout_ns) {
    using C = NaiveScoresCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffCtl);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffCtl + 16);
    volatile uint32_t* abort = reinterpret_cast<uint32_t*>(smem + C::kOffCtl + 20);
    const uint32_t bar_ld = ptx::smem_addr(&bars[0]);
    const uint32_t bar_mma = ptx::smem_addr(&bars[1]);
    const int warp = threadIdx.x >> 5, t = threadIdx.x;
    const int kt = blockIdx.x, qt = blockIdx.y, bh = blockIdx.z;
    const int b_idx = bh / H, h_idx = bh % H;

    if (t == 0) {
        ptx::mbar_init(bar_ld, 1);
        ptx::mbar_init(bar_mma, 1);
        *abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), 128);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (t == 0) {
        ptx::mbar_arrive_expect_tx(bar_ld, 2 * C::kTileBytes);
        for (int c = 0; c < D / 64; ++c) {
            ptx::tma_load_4d(sbase + C::kOffQ + c * kSubBytes, &tm_q, bar_ld, 64 * c, qt * kTileM,
                             h_idx, b_idx);
            ptx::tma_load_4d(sbase + C::kOffK + c * kSubBytes, &tm_k, bar_ld, 64 * c, kt * kTileM,
                             h_idx, b_idx);
        }
    }
    bool ok = true;
    if (warp == 0) {
        ok = wait_warp(bar_ld, 0, abort, timeout_ns);
        if (ok) {
            ptx::tc_fence_after_sync();
            constexpr uint32_t idesc = instr_desc(BF16, kTileM, 128, false);
            const uint64_t qd = smem_desc(sbase + C::kOffQ, 16, 1024);
            const uint64_t kd = smem_desc(sbase + C::kOffK, 16, 1024);
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint64_t off = (k >> 2) * (kSubBytes / 16) + (k & 3) * 2;
                    ptx::mma_ss(tmem, qd + off, kd + off, idesc, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
            ptx::tc_commit_elect(bar_mma);
            __syncwarp();
        }
    }
    ok = wait_warp(bar_mma, 0, abort, timeout_ns) && ok;
    if (ok) {
        ptx::tc_fence_after_sync();
        const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t sv[32];
            ptx::tmem_ld_32x32b_x32(row_addr + c * 32, sv);
            ptx::tmem_wait_ld();
            const uint32_t sub = sbase + C::kOffS + (c >> 1) * kSubBytes + t * 128;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int u = q4 * 8 + 2 * e;
                    w[e] = pack2<BF16>(__uint_as_float(sv[u]) * scale, __uint_as_float(sv[u + 1]) * scale);
                }
                const int chunk = (c & 1) * 4 + q4;
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 sub + ((chunk ^ (t & 7)) << 4)),
                             "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                             : "memory");
            }
        }
        ptx::fence_proxy_async_smem();
    }
    __syncthreads();
    if (t == 0 && !*abort) {
        for (int c = 0; c < 2; ++c)
            ptx::tma_store_4d(&tm_s, sbase + C::kOffS + c * kSubBytes, kt * 128 + 64 * c,
                              qt * kTileM, bh, 0);
        ptx::bulk_commit_group();
        ptx::bulk_wait_group_read0();
    }
    if (t == 0 && *abort) {
        // the loads may still land: wait for them (bounded) before leaving
        wait_bar(bar_ld, 0, abort, timeout_ns, false);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 0) ptx::tmem_dealloc(tmem, 128);
}

// ---- step 2: P = softmax(S) row by row, three passes over the row in HBM
// (the row is re-read with L2-only loads each pass, as three separate reads).
// key j of row i is visible iff j < N and (no mask, or j <= i + mask_offset).
template <bool BF16>
__device__ __forceinline__ float2 unpack_any(uint32_t v) { return unpack2<BF16>(v); }

template <bool BF16>
__global__ void __launch_bounds__(kNaiveSoftmaxThreads)
    fa_naive_softmax_kernel(const uint16_t* __restrict__ S, uint16_t* __restrict__ P,
                            float* __restrict__ lse, int N, int causal, int mask_offset) {
    __shared__ float red[kNaiveSoftmaxThreads / 32];
    __shared__ float bcast;
    const long long r = blockIdx.x;  // row index bh * N + i
    const int i = static_cast<int>(r % N);
    const int limit = causal ? min(N, max(0, i + mask_offset + 1)) : N;  // visible keys [0, limit)
    const uint4* srow = reinterpret_cast<const uint4*>(S + r * N);
    uint4* prow = reinterpret_cast<uint4*>(P + r * N);
    const int nvec = N / 8;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    constexpr float kLog2e = 1.4426950408889634f;

    auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float u = __shfl_xor_sync(0xffffffffu, v, o);
            v = is_max ? fmaxf(v, u) : v + u;
        }
        if (lane == 0) red[warp] = v;
        __syncthreads();
        if (t == 0) {
            float a = red[0];
            for (int w = 1; w < kNaiveSoftmaxThreads / 32; ++w) a = is_max ? fmaxf(a, red[w]) : a + red[w];
            bcast = a;
        }
        __syncthreads();
        const float res = bcast;
        __syncthreads();
        return res;
    };

    // pass 1: maximum
    float m = -INFINITY;
    for (int vi = t; vi < nvec; vi += kNaiveSoftmaxThreads) {
        const uint4 x = __ldcg(srow + vi);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_any<BF16>(w[e]);
            const int j = vi * 8 + 2 * e;
            if (j < limit) m = fmaxf(m, f.x);
            if (j + 1 < limit) m = fmaxf(m, f.y);
        }
    }
    m = block_reduce(m, true);
    const float mm = (m == -INFINITY) ? 0.f : m * kLog2e;
    // pass 2: sum of exponentials
    float l = 0.f;
    for (int vi = t; vi < nvec; vi += kNaiveSoftmaxThreads) {
        const uint4 x = __ldcg(srow + vi);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_any<BF16>(w[e]);
            const int j = vi * 8 + 2 * e;
            if (j < limit) l += ptx::ex2_approx(fmaf(f.x, kLog2e, -mm));
            if (j + 1 < limit) l += ptx::ex2_approx(fmaf(f.y, kLog2e, -mm));
        }
    }
    l = block_reduce(l, false);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    // pass 3: normalised weights, written as P
    for (int vi = t; vi < nvec; vi += kNaiveSoftmaxThreads) {
        const uint4 x = __ldcg(srow + vi);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_any<BF16>(w[e]);
            const int j = vi * 8 + 2 * e;
            const float p0 = j < limit ? ptx::ex2_approx(fmaf(f.x, kLog2e, -mm)) * inv : 0.f;
            const float p1 = j + 1 < limit ? ptx::ex2_approx(fmaf(f.y, kLog2e, -mm)) * inv : 0.f;
            o[e] = pack2<BF16>(p0, p1);
        }
        prow[vi] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (t == 0) lse[r] = l > 0.f ? m + logf(l) : -INFINITY;
}

// ---- step 3: O = P V, one 128-row tile per CTA, P and V tiles through a
// two-stage TMA ring, U accumulated in TMEM
template <int D>
struct NaivePvCfg {
    static constexpr int kPBytes = kTileM * 128 * 2;   // P tile 128 rows x 128 keys
    static constexpr int kVBytes = 128 * D * 2;        // V tile 128 keys x D
    static constexpr int kStages = 2;
    static constexpr int kOffP = 0;
    static constexpr int kOffV = kStages * kPBytes;
    static constexpr int kOffO = kOffV + kStages * kVBytes;  // staging of the O tile
    static constexpr int kOffCtl = kOffO + kTileM * D * 2;
    static constexpr int kSmemBytes = kOffCtl + 128 + 1024;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kNaivePvThreads)
    fa_naive_pv_kernel(const __grid_constant__ CUtensorMap tm_p,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, int H, int N,
                       unsigned long long timeout_ns) {
    using C = NaivePvCfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffCtl);  // full[2], empty[2], done, drain
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffCtl + 64);
    volatile uint32_t* abort = reinterpret_cast<uint32_t*>(smem + C::kOffCtl + 68);
    auto bar_full = [&](int s) { return ptx::smem_addr(&bars[s]); };
    auto bar_empty = [&](int s) { return ptx::smem_addr(&bars[2 + s]); };
    const uint32_t bar_done = ptx::smem_addr(&bars[4]);
    const uint32_t bar_drain = ptx::smem_addr(&bars[5]);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, bh = blockIdx.y;
    const int b_idx = bh / H, h_idx = bh % H;
    const int nk = (N + 127) / 128;
    constexpr uint32_t kCols = D < 32 ? 32 : D;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_empty(s), 1);
        }
        ptx::mbar_init(bar_done, 1);
        ptx::mbar_init(bar_drain, 1);
        *abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), kCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;

    if (warp == 4) {
        // loader: P tile j (two 64-key sub-tiles) and V tile j (D/64 sub-tiles)
        int issued[NS] = {};
        for (int j = 0; j < nk; ++j) {
            const int s = j % NS;
            if (j >= NS && !wait_warp(bar_empty(s), ((j / NS) - 1) & 1, abort, timeout_ns)) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar_full(s), C::kPBytes + C::kVBytes);
                for (int c = 0; c < 2; ++c)
                    ptx::tma_load_4d(sbase + C::kOffP + s * C::kPBytes + c * kSubBytes, &tm_p,
                                     bar_full(s), j * 128 + 64 * c, qt * kTileM, bh, 0);
                for (int c = 0; c < D / 64; ++c)
                    ptx::tma_load_4d(sbase + C::kOffV + s * C::kVBytes + c * kSubBytes, &tm_v,
                                     bar_full(s), 64 * c, j * 128, h_idx, b_idx);
            }
            ++issued[s];
        }
        for (int s = 0; s < NS; ++s)
            if (issued[s] > 0) wait_warp(bar_full(s), (issued[s] - 1) & 1, abort, timeout_ns, false);
    } else if (warp == 5) {
        constexpr uint32_t idesc = instr_desc(BF16, kTileM, D, true);
        bool ok = true;
        for (int j = 0; ok && j < nk; ++j) {
            const int s = j % NS;
            if (!(ok = wait_warp(bar_full(s), (j / NS) & 1, abort, timeout_ns))) break;
            ptx::tc_fence_after_sync();
            const uint64_t pd = smem_desc(sbase + C::kOffP + s * C::kPBytes, 16, 1024);
            const uint64_t vd = smem_desc(sbase + C::kOffV + s * C::kVBytes, kSubBytes, 1024);
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t po = (k >> 2) * (kSubBytes / 16) + (k & 3) * 2;
                    ptx::mma_ss(tmem, pd + po, vd + k * 128, idesc, (j > 0 || k > 0) ? 1u : 0u);
                }
            }
            __syncwarp();
            ptx::tc_commit_elect(bar_empty(s));
            __syncwarp();
        }
        if (ok) ptx::tc_commit_elect(bar_done);
        __syncwarp();
        ptx::tc_commit_elect(bar_drain);
        __syncwarp();
        wait_warp(bar_drain, 0, abort, timeout_ns, false);
    } else {
        // epilogue warps 0-3: O (already normalised: P rows sum to 1) -> 16-bit
        const int t = threadIdx.x;
        const bool ok = wait_warp(bar_done, 0, abort, timeout_ns);
        if (ok) {
            ptx::tc_fence_after_sync();
            const uint32_t row_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t ov[32];
                ptx::tmem_ld_32x32b_x32(row_addr + c * 32, ov);
                ptx::tmem_wait_ld();
                const uint32_t sub = sbase + C::kOffO + (c >> 1) * kSubBytes + t * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int u = q4 * 8 + 2 * e;
                        w[e] = pack2<BF16>(__uint_as_float(ov[u]), __uint_as_float(ov[u + 1]));
                    }
                    const int chunk = (c & 1) * 4 + q4;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                     sub + ((chunk ^ (t & 7)) << 4)),
                                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
            }
            ptx::fence_proxy_async_smem();
        }
        ptx::named_barrier_sync(1, 128);
        if (t == 0 && !*abort) {
            for (int c = 0; c < D / 64; ++c)
                ptx::tma_store_4d(&tm_o, sbase + C::kOffO + c * kSubBytes, 64 * c, qt * kTileM,
                                  h_idx, b_idx);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();
        }
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == 5) ptx::tmem_dealloc(tmem, kCols);
}

}  // namespace fa
