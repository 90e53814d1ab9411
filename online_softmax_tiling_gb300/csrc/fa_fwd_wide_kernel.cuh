// fa_fwd_wide_kernel.cuh - the same fused attention forward for head
// dimensions 192 and 256 on sm_103a.
//
// It computes exactly what fa_fwd_kernel computes (the online softmax of
// "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程", sections "第四步",
// "第五步" and "最后", in the FlashAttention-2 loop order of "CUDA 算子工程"
// ch. 14, section 14.5), with the same reference-first weights, the same two
// weight sums, masks, split-KV partials and bounded waits.  What changes is
// the tiling, because a wide head does not fit the two-query-tile layout:
// two tiles would need 2 x (128 + d) TMEM columns, more than the 512 an SM has.
//
//   * a persistent grid: each CTA walks units of one 128-row query tile of
//     one (batch, head) (and with split-KV one key range of it), in the
//     order of fa_fwd_kernel (longest first with the causal mask, the
//     direction alternating by round); 6 warps: warps 0-3 softmax +
//     epilogue (thread t owns row t = TMEM lane t), warp 4 the TMA loader,
//     warp 5 the tensor-core issuer;
//   * key tiles of 128 keys, so that S = Q K^T runs as M128 N128 products
//     (an N64 product takes 48 cycles for 32 cycles of work); K and V tiles
//     of 128 x d fit once each in shared memory next to Q for d = 256 (K
//     twice for d = 192), so each tile loads while the product before its
//     first use runs;
//   * TMEM: two score buffers S0 at column 0 and S1 at 128 (128 fp32
//     columns; the weights P overwrite the first 64), U at column 256 (d
//     columns).  Key tiles are counted over all units of the CTA; tile g
//     uses buffer g & 1, so the buffers, rings and barrier phases run on
//     from one unit to the next;
//   * tensor-core order per unit: S(0), S(1), then per key tile j: PV(j),
//     S(j+2).  The softmax of tile j+1 runs while the tensor core computes
//     PV(j) and S(j+2) - with d = 256 each is 1024 cycles, so the softmax of
//     128 keys (about 1200 cycles) stays off the critical path.  The next
//     unit's Q is loaded once this unit's last S product is done, and its
//     first two S products follow this unit's last PV;
//   * S(j+1) is issued before PV(j), so U may still be absorbing P(j-1) V
//     when the softmax of tile j wants to rescale it: that (rare) rescale
//     first waits for PV(j-1).  Each score buffer has its own "weights
//     written" barrier, because the softmax can run one tile ahead of the
//     issuer's wait; and "U has absorbed P(g) V" alternates between two
//     barriers by the parity of g: when a softmax warp finishes tile g,
//     PV(g-2) is certain to be complete but PV(g-1) is not, so a single
//     barrier could be two phases behind the one awaited, and a parity wait
//     cannot tell two phases apart;
//   * O leaves through two 4 KB staging boxes per softmax warp (32 rows x 64
//     columns, 128-byte swizzle) and TMA stores, never through Q's shared
//     memory, which the next unit's Q may already occupy.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kWideBlockN = 128;     // keys per tile
constexpr int kWideThreads = 192;    // 4 softmax warps + loader warp + MMA warp
constexpr int kWideLoaderWarp = 4;
constexpr int kWideMmaWarp = 5;
constexpr uint32_t kWideTmemU = 256;  // S0 at 0, S1 at 128, U at 256

template <int D>
struct WideCfg {
    static_assert(D == 192 || D == 256, "wide head dim");
    static constexpr int kSub = D / 64;                      // 64-column swizzle sub-tiles
    static constexpr int kQSubBytes = kTileM * 128;          // 128 rows x 128 bytes
    static constexpr int kKVSubBytes = kWideBlockN * 128;    // 128 rows x 128 bytes
    static constexpr int kQBytes = kSub * kQSubBytes;
    static constexpr int kKVBytes = kSub * kKVSubBytes;
    // one K and one V slot for d = 256; for d = 192 the second slot goes to V,
    // whose slot frees only when P.V is done (K's when the shorter S is)
    static constexpr int kKStages = 1;
    static constexpr int kVStages = D == 256 ? 1 : 2;
    // With one V slot (d = 256) each V tile travels as two 64-key parts with
    // their own barriers: P.V runs part by part, and the next tile's first
    // part loads while this tile's second part is in use.
    static constexpr int kVParts = D == 256 ? 2 : 1;
    static constexpr int kVPartRows = kWideBlockN / kVParts;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kQBytes;
    static constexpr int kOffV = kOffK + kKStages * kKVBytes;
    // O staging: two 32-row x 64-column swizzled boxes per softmax warp
    static constexpr int kOffStage = kOffV + kVStages * kKVBytes;
    static constexpr int kStageBytes = 32 * 128;
    static constexpr int kOffCtl = kOffStage + 4 * 2 * kStageBytes;
    static constexpr int kSmemBytes = kOffCtl + 512 + 1024;  // control block + alignment slack
};

template <int NK, int NV>  // barrier pairs: NK for K (slots x parts), NV for V
struct alignas(8) WideCtl {
    uint64_t q_full;
    uint64_t q_empty;    // the S products of a unit are done: Q may be reloaded
    uint64_t k_full[NK];
    uint64_t k_empty[NK];
    uint64_t v_full[NV];
    uint64_t v_empty[NV];
    uint64_t s_full[2];  // per score buffer: S(j) is in TMEM
    uint64_t p_full[2];  // per score buffer: P(j) is in TMEM (and U rescaled)
    uint64_t o_ready[2];  // by the parity of g: U has absorbed P(g) V_g
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
};

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(kWideThreads, 1)
    fa_fwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
    using C = WideCfg<D>;
    constexpr int NK = C::kKStages;
    constexpr int NV = C::kVStages;
    constexpr int BN = kWideBlockN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    constexpr int VP = C::kVParts;
    // K tiles travel as their 64-column sub-tiles, each with its own barriers:
    // S = Q K^T reads them in that order (four K16 steps each), so S can start
    // on the first while the rest land, and each frees as soon as S is past it
    constexpr int KP = C::kSub;
    WideCtl<NK * KP, NV * VP>* ctl = reinterpret_cast<WideCtl<NK * KP, NV * VP>*>(smem + C::kOffCtl);
    volatile uint32_t* abort = &ctl->abort;
    const unsigned long long tmo = p.timeout_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int nkv = (p.Nk + BN - 1) / BN;
    // ---- work units (as in fa_fwd_kernel): CTA c takes units c, 2G - 1 - c,
    // 2G + c, ...; with the causal mask the longest query tiles come first
    struct Unit {
        int bh, qb, split, k0, n;
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
        int T = nkv;  // key tiles visible to the tile
        if (CAUSAL) {
            const int last = min(w.qb * kTileM + kTileM - 1, p.Nq - 1) + p.mask_offset;
            T = last < 0 ? 0 : min(last / BN + 1, nkv);
        }
        w.k0 = 0;
        w.n = T;  // the unit visits key tiles k0 .. k0 + n - 1
        if constexpr (SPLIT) {
            const int chunk = (T + S - 1) / S;
            w.k0 = w.split * chunk;
            w.n = max(0, min(w.k0 + chunk, T) - w.k0);
        }
        return w;
    };

    const uint32_t bar_q = ptx::smem_addr(&ctl->q_full);
    const uint32_t bar_qe = ptx::smem_addr(&ctl->q_empty);
    auto bar_kf = [&](int s) { return ptx::smem_addr(&ctl->k_full[s]); };
    auto bar_ke = [&](int s) { return ptx::smem_addr(&ctl->k_empty[s]); };
    auto bar_vf = [&](int s) { return ptx::smem_addr(&ctl->v_full[s]); };
    auto bar_ve = [&](int s) { return ptx::smem_addr(&ctl->v_empty[s]); };
    auto bar_sf = [&](int b) { return ptx::smem_addr(&ctl->s_full[b]); };
    auto bar_pf = [&](int b) { return ptx::smem_addr(&ctl->p_full[b]); };
    auto bar_o = [&](uint32_t g) { return ptx::smem_addr(&ctl->o_ready[g & 1]); };
    const uint32_t bar_drain = ptx::smem_addr(&ctl->drain);
    const uint32_t sQ = sbase + C::kOffQ;
    auto sK = [&](int s) { return sbase + C::kOffK + s * C::kKVBytes; };
    auto sV = [&](int s) { return sbase + C::kOffV + s * C::kKVBytes; };

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_q, 1);
        ptx::mbar_init(bar_qe, 1);
        for (int s = 0; s < NK * KP; ++s) {
            ptx::mbar_init(bar_kf(s), 1);
            ptx::mbar_init(bar_ke(s), 1);
        }
        for (int s = 0; s < NV * VP; ++s) {
            ptx::mbar_init(bar_vf(s), 1);
            ptx::mbar_init(bar_ve(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_sf(b), 1);
            ptx::mbar_init(bar_pf(b), kTileM);
        }
        ptx::mbar_init(bar_o(0), 1);
        ptx::mbar_init(bar_o(1), 1);
        ptx::mbar_init(bar_drain, 1);
        ctl->abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kWideLoaderWarp && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == kWideMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kWideLoaderWarp) {
        // =============================================================== loader
        // Per unit: Q once the previous unit's S products are done, then
        // K_0, K_1, V_0, K_2, V_1, ...: K runs one tile ahead of V.  The
        // rings run on across units.
        int issued_k[NK * KP], issued_v[NV * VP];
#pragma unroll
        for (int s = 0; s < NK * KP; ++s) issued_k[s] = 0;
#pragma unroll
        for (int s = 0; s < NV * VP; ++s) issued_v[s] = 0;
        uint32_t kc = 0, vc = 0;  // K and V tiles loaded so far
        int nq = 0;               // units whose Q was loaded
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            if (w.n == 0) continue;
            const int b_idx = w.bh / p.H, h_idx = w.bh % p.H;
            if (nq > 0 && !(ok = wait_warp(bar_qe, (nq - 1) & 1, abort, tmo))) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar_q, C::kQBytes);
#pragma unroll
                for (int c = 0; c < C::kSub; ++c)
                    ptx::tma_load_4d(sQ + c * C::kQSubBytes, &tm_q, bar_q, 64 * c, w.qb * kTileM, h_idx,
                                     b_idx);
            }
            ++nq;
            // K tile j and V tile j - 1; with more V slots than K slots the V
            // tile goes first, since the K slot frees only when S(j - 1) is done
            auto load_k = [&](int j) {
                const int s = kc % NK;
                const bool skip = (p.fault_mode == 1 && kc == 0);
#pragma unroll
                for (int c = 0; c < KP; ++c) {
                    const int bi = s * KP + c;
                    if (kc >= NK && !wait_warp(bar_ke(bi), ((kc / NK) - 1) & 1, abort, tmo)) return false;
                    if (lane == 0 && !skip) {
                        ptx::mbar_arrive_expect_tx(bar_kf(bi), C::kKVSubBytes);
                        ptx::tma_load_4d(sK(s) + c * C::kKVSubBytes, &tm_k, bar_kf(bi), 64 * c,
                                         (w.k0 + j) * BN, h_idx, b_idx);
                    }
                    if (!skip) ++issued_k[bi];
                }
                ++kc;
                return true;
            };
            auto load_v = [&](int j) {
                const int s = vc % NV;
#pragma unroll
                for (int h = 0; h < VP; ++h) {
                    const int bi = s * VP + h;
                    if (vc >= NV && !wait_warp(bar_ve(bi), ((vc / NV) - 1) & 1, abort, tmo)) return false;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(bar_vf(bi), C::kKVBytes / VP);
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d(sV(s) + c * C::kKVSubBytes + h * C::kVPartRows * 128, &tm_v,
                                             bar_vf(bi), 64 * c, (w.k0 + j) * BN + h * C::kVPartRows,
                                             h_idx, b_idx);
                    }
                    ++issued_v[bi];
                }
                ++vc;
                return true;
            };
            for (int j = 0; j <= w.n; ++j) {
                if constexpr (NV > NK) {
                    if (j >= 1 && !(ok = load_v(j - 1))) break;
                    if (j < w.n && !(ok = load_k(j))) break;
                } else {
                    if (j < w.n && !(ok = load_k(j))) break;
                    if (j >= 1 && !(ok = load_v(j - 1))) break;
                }
            }
        }
        // Never leave the CTA with copies still landing in its shared memory.
        if (nq > 0) wait_warp(bar_q, (nq - 1) & 1, abort, tmo, false);
        for (int s = 0; s < NK * KP; ++s)
            if (issued_k[s] > 0) wait_warp(bar_kf(s), (issued_k[s] - 1) & 1, abort, tmo, false);
        for (int s = 0; s < NV * VP; ++s)
            if (issued_v[s] > 0) wait_warp(bar_vf(s), (issued_v[s] - 1) & 1, abort, tmo, false);
    } else if (warp == kWideMmaWarp) {
        // ====================================================== tensor-core issuer
        constexpr uint32_t idesc_s = instr_desc(BF16, kTileM, BN, false);
        constexpr uint32_t idesc_pv = instr_desc(BF16, kTileM, D, true);
        const uint64_t q_desc = smem_desc(sQ, 16, 1024);
        const uint64_t k_desc0 = smem_desc(sK(0), 16, 1024);
        // V is MN-major: the next 64 columns of d are one sub-tile further on
        const uint64_t v_desc0 = smem_desc(sV(0), C::kKVSubBytes, 1024);
        constexpr uint64_t kStageStep = C::kKVBytes / 16;
        // S_b = Q K_s^T over the 64-column sub-tile c of d: four K16 steps,
        // +32 bytes per step inside a 128-byte swizzle row
        auto issue_s = [&](int b, int s, int c) {
            if (ptx::elect_one()) {
                const uint64_t kd = k_desc0 + s * kStageStep;
#pragma unroll
                for (int k = 4 * c; k < 4 * c + 4; ++k) {
                    const uint64_t ao = (k >> 2) * (C::kQSubBytes / 16) + (k & 3) * 2;
                    const uint64_t bo = (k >> 2) * (C::kKVSubBytes / 16) + (k & 3) * 2;
                    ptx::mma_ss(tmem + b * BN, q_desc + ao, kd + bo, idesc_s, k > 0 ? 1u : 0u);
                }
            }
            __syncwarp();
        };
        // steps [k_begin, k_end) of U (+)= P_b V_s: 128 keys = 8 steps of K16;
        // P advances 8 TMEM columns (16 packed 16-bit weights), V 16 rows =
        // 2048 bytes per step
        auto issue_pv = [&](int b, int s, bool acc, int k_begin, int k_end) {
            if (ptx::elect_one()) {
                const uint64_t vd = v_desc0 + s * kStageStep;
#pragma unroll
                for (int k = k_begin; k < k_end; ++k)
                    ptx::mma_ts(tmem + kWideTmemU, tmem + b * BN + k * 8, vd + k * 128, idesc_pv,
                                (acc || k > 0) ? 1u : 0u);
            }
            __syncwarp();
        };
        // S of the key tile counted g over all units, from K slot kc % NK;
        // the last S of a unit also releases its Q
        uint32_t kc = 0, vc = 0;  // K and V tiles consumed so far (same order as loaded)
        uint32_t g = 0;           // key tiles of all previous units
        uint32_t nq = 0;          // units so far (q_full phase)
        bool ok = true;
        auto s_tile = [&](uint32_t gg, bool last) {
            const int s = kc % NK;
#pragma unroll
            for (int c = 0; c < KP; ++c) {
                if (!wait_warp(bar_kf(s * KP + c), (kc / NK) & 1, abort, tmo)) return false;
                ptx::tc_fence_after_sync();
                issue_s(gg & 1, s, c);  // into the buffer PV(gg - 2) has read (issued in order)
                ptx::tc_commit_elect(bar_ke(s * KP + c));
            }
            ptx::tc_commit_elect(bar_sf(gg & 1));
            if (last) ptx::tc_commit_elect(bar_qe);
            ++kc;
            __syncwarp();
            return true;
        };
        for (int r = 0; ok; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            if (w.n == 0) continue;
            if (!(ok = wait_warp(bar_q, nq & 1, abort, tmo))) break;
            ++nq;
            for (int j = 0; ok && j < 2 && j < w.n; ++j) ok = s_tile(g + j, j == w.n - 1);
            for (int j = 0; ok && j < w.n; ++j) {
                const uint32_t gg = g + j;
                const int b = gg & 1;
                const int sv = vc % NV;
                if (!(ok = wait_warp(bar_pf(b), (gg >> 1) & 1, abort, tmo))) break;
                // part by part as V arrives; each part's slot is released
                // once the product that read it is done
#pragma unroll
                for (int h = 0; h < VP; ++h) {
                    if (!(ok = wait_warp(bar_vf(sv * VP + h), (vc / NV) & 1, abort, tmo))) break;
                    ptx::tc_fence_after_sync();
                    // the first product of a unit overwrites U
                    issue_pv(b, sv, j > 0, h * (BN / 16) / VP, (h + 1) * (BN / 16) / VP);
                    ptx::tc_commit_elect(bar_ve(sv * VP + h));
                }
                if (!ok) break;
                ptx::tc_commit_elect(bar_o(gg));
                ++vc;
                __syncwarp();
                if (j + 2 < w.n) ok = s_tile(gg + 2, j + 3 == w.n);
            }
            g += w.n;
        }
        // Drain: nothing of ours may still run on the tensor core at teardown.
        ptx::tc_commit_elect(bar_drain);
        __syncwarp();
        wait_warp(bar_drain, 0, abort, tmo, false);
    } else {
        // ======================================== softmax + epilogue (warps 0-3)
        const int t = threadIdx.x;                    // row in the tile = TMEM lane
        // of the current unit: the tile's first query index, this thread's,
        // and the first key tile visited
        int first_row = 0, row = 0, k0 = 0;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t u_addr = tmem + lane_off + kWideTmemU;
        const float c2 = p.scale_log2;
        const float2 c2v = make_float2(c2, c2);
        auto tile_masked = [&](int j) {
            const int kend = (k0 + j + 1) * BN;
            return kend > p.Nk || (CAUSAL && kend - 1 > first_row + p.mask_offset);
        };
        auto key_limit = [&](int kbase) {
            int limit = p.Nk - kbase;
            if (CAUSAL) limit = min(limit, row + p.mask_offset - kbase + 1);
            return limit;
        };
        // scores [32 c, 32 c + 32) of tile j (buffer at s_addr), masked to -inf
        // where this row may not see the key
        auto load_chunk = [&](uint32_t s_addr, uint32_t(&sv)[32], int c, int j) {
            ptx::tmem_ld_32x32b_x32(s_addr + c * 32, sv);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) ptx::reg_fence(sv[u]);
            if (tile_masked(j)) {
                const int limit = key_limit((k0 + j) * BN + c * 32);
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    if (u >= limit) sv[u] = __float_as_uint(-INFINITY);
            }
        };
        auto weights = [&](const uint32_t* sv, int npairs, float neg_ref, uint32_t* pk,
                           float2 (&rs)[2], float2 (&rh)[2]) {
            const float2 nrv = make_float2(neg_ref, neg_ref);
#pragma unroll
            for (int c = 0; c < npairs; ++c) {
                const float2 e = __ffma2_rn(
                    make_float2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), c2v, nrv);
                const float2 pw = make_float2(ptx::ex2_approx(e.x), ptx::ex2_approx(e.y));
                rs[c & 1] = __fadd2_rn(rs[c & 1], pw);
                pk[c] = pack2<BF16>(pw.x, pw.y);
                add_packed<BF16>(rh[c & 1], pk[c]);
            }
        };
        uint32_t g = 0;  // key tiles of all previous units (buffers and barrier phases)
        bool aborted = false;
        for (int r = 0; !aborted; ++r) {
            const int u = unit_id(r);
            if (u >= p.num_units) break;
            const Unit w = unit_of(u);
            const int b_idx = w.bh / p.H, h_idx = w.bh % p.H;
            first_row = w.qb * kTileM;
            row = first_row + t;
            k0 = w.k0;
            const int n = w.n;
            if (SPLIT && n == 0) {  // empty key range: its partials carry no weight
                if (row < p.Nq) {
                    const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + row;
                    const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                    p.lse_part[i] = -INFINITY;
                    p.lse_part[plane + i] = -INFINITY;
                }
                continue;
            }
            float m_ref = -INFINITY;
            float2 lsum = make_float2(0.f, 0.f);
            float2 lhat = make_float2(0.f, 0.f);

            for (int j = 0; j < n; ++j) {
                const uint32_t gg = g + j;
                const int b = gg & 1;
                if (!wait_warp(bar_sf(b), (gg >> 1) & 1, abort, tmo)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t s_addr = tmem + lane_off + b * BN;
                uint32_t pk[BN / 2];
                float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                float2 rh[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                // (tcgen05.ld is warp-collective: every branch around it is uniform)
                bool redo = (m_ref == -INFINITY);
                if (!__any_sync(0xffffffffu, redo)) {
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t sv[32];
                        load_chunk(s_addr, sv, c, j);
                        weights(sv, 16, -m_ref * c2, &pk[16 * c], rs, rh);
                    }
                    redo = rs[0].x + rs[0].y + rs[1].x + rs[1].y > weight_sum_limit<BF16>();
                }
                float alpha = 1.f;
                float m_new = m_ref;
                if (__any_sync(0xffffffffu, redo)) {
                    float mt = -INFINITY;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t sv[32];
                        load_chunk(s_addr, sv, c, j);
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
                    if (redo) {
                        m_new = fmaxf(mt, m_ref);
                        if (m_ref != -INFINITY) alpha = ptx::ex2_approx((m_ref - m_new) * c2);
                    }
                    const float neg_ref = (m_new == -INFINITY) ? 0.f : -m_new * c2;
                    rs[0] = rs[1] = rh[0] = rh[1] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t sv[32];
                        load_chunk(s_addr, sv, c, j);
                        weights(sv, 16, neg_ref, &pk[16 * c], rs, rh);
                    }
                }
                const float2 av = make_float2(alpha, alpha);
                const float2 r = __fadd2_rn(rs[0], rs[1]), hh = __fadd2_rn(rh[0], rh[1]);
                lsum.x = fmaf(lsum.x, alpha, r.x + r.y);
                lhat.x = fmaf(lhat.x, alpha, hh.x + hh.y);
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                    ptx::tmem_st_32x32b_x32(s_addr + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c * 32]));
                // U may still be absorbing P(j-1) V (issued after S(j)): a rescale
                // waits for that product first (warp-uniform)
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    if (j > 0 && !wait_warp(bar_o(gg - 1), ((gg - 1) >> 1) & 1, abort, tmo)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t ov[16];
                        ptx::tmem_ld_32x32b_x16(u_addr + c * 16, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 16; u += 2) {
                            ptx::reg_fence(ov[u]);
                            ptx::reg_fence(ov[u + 1]);
                            const float2 rr = __fmul2_rn(
                                make_float2(__uint_as_float(ov[u]), __uint_as_float(ov[u + 1])), av);
                            ov[u] = __float_as_uint(rr.x);
                            ov[u + 1] = __float_as_uint(rr.y);
                        }
                        ptx::tmem_st_32x32b_x16(u_addr + c * 16, ov);
                    }
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                ptx::mbar_arrive(bar_pf(b));
                m_ref = m_new;
            }

            // ---- epilogue: O = U / lhat -> 16-bit -> per-warp staging boxes -> TMA
            if (!aborted && n > 0) aborted = !wait_warp(bar_o(g + n - 1), ((g + n - 1) >> 1) & 1, abort, tmo);
            g += n;
            if (aborted) break;
            const float l_all = lsum.x + lsum.y;
            const float lhat_all = lhat.x + lhat.y;
            if constexpr (SPLIT) {
                const bool mine = row < p.Nq && !*abort;
                const bool any = l_all > 0.f;
                const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + (mine ? row : 0);
                const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                if (mine) {
                    p.lse_part[i] = any ? m_ref * p.scale + logf(l_all) : -INFINITY;
                    p.lse_part[plane + i] = any ? m_ref * p.scale + logf(lhat_all) : -INFINITY;
                }
                // O through the warp's two staging boxes in turn, 32 fp32
                // columns at a time (tm_o maps the partials here; rows >= Nq
                // clipped)
                ptx::tc_fence_after_sync();
                const float inv = any ? 1.f / lhat_all : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    const uint32_t stage = sbase + C::kOffStage + (warp * 2 + (c & 1)) * C::kStageBytes;
                    uint32_t ov[32];
                    ptx::tmem_ld_32x32b_x32(u_addr + c * 32, ov);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) ptx::reg_fence(ov[e]);
                    // the store that last used this box (two stores back) has read it
                    if (lane == 0) ptx::bulk_wait_group_read1();
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
                        ptx::tma_store_4d(&tm_o, stage, 32 * c, first_row + 32 * warp, w.bh, w.split);
                        ptx::bulk_commit_group();
                    }
                }
            } else {
                // each warp stores its 32 rows, 64 columns at a time, through two
                // staging boxes used in turn (128-byte swizzle, as the TMA store
                // expects); rows >= Nq and columns >= d are clipped
                ptx::tc_fence_after_sync();
                const bool mine = row < p.Nq && !*abort;
                const float inv = lhat_all > 0.f ? 1.f / lhat_all : 0.f;
                const float2 iv = make_float2(inv, inv);
#pragma unroll 1
                for (int h = 0; h < C::kSub; ++h) {
                    const uint32_t stage = sbase + C::kOffStage + (warp * 2 + (h & 1)) * C::kStageBytes;
                    // the store that last used this box (two stores back) has read it
                    if (lane == 0) ptx::bulk_wait_group_read1();
                    __syncwarp();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        if (n > 0) {
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
                        ptx::tma_store_4d(&tm_o, stage, 64 * h, first_row + 32 * warp, h_idx, b_idx);
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
    if (warp == kWideMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
