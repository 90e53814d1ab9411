// fa_fwd_qtile_kernel.cuh - fused attention forward for head dimensions 64
// and 128 on sm_103a: one query tile per unit, two softmax warps per row.
//
// It computes exactly what fa_fwd_kernel computes (the online softmax of
// "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程", sections "第四步",
// "第五步" and "最后", in the FlashAttention-2 loop order of "CUDA 算子工程"
// ch. 14, section 14.5), with the same reference-first weights, the same two
// weight sums, masks, split-KV partials and bounded waits.  What changes is
// who computes the weights of a key tile, and when.
//
// A key tile's softmax (128 weights per row) is the longest link of the
// chain S -> weights -> P.V -> next S.  Here every row has two softmax
// warps, one per 64-key half of each tile, so each warp holds 64 scores and
// the link is about half as long; and the scores are double-buffered in
// TMEM, so the tensor core always has the next S to compute while a tile's
// weights are made:
//   * a persistent grid: each CTA walks units of one 128-row query tile of
//     one (batch, head) (with split-KV, one key range of it), in the order
//     of fa_fwd_kernel (longest first with the causal mask, the direction
//     alternating by round).  10 warps: warps 0-3 take keys 0-63 of every
//     tile, warps 4-7 keys 64-127; warps w and w + 4 share TMEM lane group
//     w (rows 32 w .. 32 w + 31, thread = row), so both run on the same SM
//     sub-partition; warp 8 is the TMA loader, warp 9 the tensor-core issuer;
//   * TMEM: scores S0 at column 0 and S1 at 128 (128 fp32 columns each), U at
//     256 (d columns).  The 16-bit weights of keys 0-63 overwrite columns
//     0-31 of their buffer, those of keys 64-127 columns 64-95: each warp
//     writes only over scores it has already read;
//   * tensor-core order per unit: S(0), S(1), then per key tile j: PV(j) in
//     two halves of 64 keys (each as soon as its warps have written its
//     weights), S(j + 2) into the buffer PV(j) has just read (the products run
//     in issue order).  The next unit's Q loads once this unit's last S is
//     done;
//   * the two warps of a row agree on the reference maximum through a small
//     exchange in shared memory guarded by an mbarrier (bounded waits, like
//     every other wait): each tile they swap whether any weight sum passed
//     the bound; on a row's first tile or a pass they swap their halves'
//     maxima and both recompute their weights against the common new
//     reference.  Each keeps its own weight sums; the two are added at the
//     end of the unit.  A rescale of U (rare) is split by columns, waits for
//     the previous P.V, and both warps finish it before either hands over
//     its weights;
//   * O: each warp normalises its half of U's columns (d = 128; for d = 64
//     the first warp stores all 64) through its own 4 KB staging box and a
//     TMA store; the first warp writes LSE.
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kQtThreads = 320;   // 8 softmax warps + loader warp + MMA warp
constexpr int kQtLoaderWarp = 8;
constexpr int kQtMmaWarp = 9;
constexpr int kQtBlockN = 128;    // keys per tile
constexpr uint32_t kQtTmemU = 256;  // S0 at 0, S1 at 128, U at 256

template <int D>
struct QtCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kSub = D / 64;                    // 64-column swizzle sub-tiles
    static constexpr int kTileBytes = kTileM * D * 2;      // one Q, K or V tile
    static constexpr int kKStages = D == 128 ? 2 : 4;
    static constexpr int kVStages = D == 128 ? 2 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kTileBytes;
    static constexpr int kOffV = kOffK + kKStages * kTileBytes;
    static constexpr int kOffStage = kOffV + kVStages * kTileBytes;
    static constexpr int kStageBytes = 32 * 128;           // one 32-row box per softmax warp
    static constexpr int kOffXch = kOffStage + 8 * kStageBytes;
    static constexpr int kXchBytes = 4 * 2 * 2 * 32 * 8;   // [lane group][slot][half][lane] float2
    static constexpr int kOffCtl = kOffXch + kXchBytes;
    static constexpr int kSmemBytes = kOffCtl + 512 + 1024;  // control block + alignment slack
};

template <int NK, int NV>
struct alignas(8) QtCtl {
    uint64_t q_full;
    uint64_t q_empty;      // the S products of a unit are done: Q may be reloaded
    uint64_t k_full[NK];
    uint64_t k_empty[NK];
    uint64_t v_full[NV];
    uint64_t v_empty[NV];
    uint64_t s_full[2];    // per score buffer: S(j) is in TMEM
    uint64_t p_half[2][2];  // per score buffer and key half: its weights are in TMEM
    uint64_t o_ready[2];   // by the parity of g: U has absorbed P(g) V_g
    uint64_t xch[4][2];    // per lane group and exchange slot: both warps wrote it
    uint64_t drain;
    uint32_t tmem_base;
    uint32_t abort;
};

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(kQtThreads, 1)
    fa_fwd_qtile_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
    using C = QtCfg<D>;
    constexpr int NK = C::kKStages;
    constexpr int NV = C::kVStages;
    constexpr int BN = kQtBlockN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = ptx::smem_addr(smem);
    QtCtl<NK, NV>* ctl = reinterpret_cast<QtCtl<NK, NV>*>(smem + C::kOffCtl);
    volatile uint32_t* abort = &ctl->abort;
    const unsigned long long tmo = p.timeout_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nkv = (p.Nk + BN - 1) / BN;

    // ---- work units: CTA c takes units c, 2G - 1 - c, 2G + c, ...; with the
    // causal mask the longest query tiles come first
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
    auto bar_ph = [&](int b, int h) { return ptx::smem_addr(&ctl->p_half[b][h]); };
    auto bar_o = [&](uint32_t g) { return ptx::smem_addr(&ctl->o_ready[g & 1]); };
    auto bar_x = [&](int lg, int slot) { return ptx::smem_addr(&ctl->xch[lg][slot]); };
    const uint32_t bar_drain = ptx::smem_addr(&ctl->drain);
    const uint32_t sQ = sbase + C::kOffQ;
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
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_sf(b), 1);
            ptx::mbar_init(bar_ph(b, 0), kTileM);
            ptx::mbar_init(bar_ph(b, 1), kTileM);
        }
        ptx::mbar_init(bar_o(0), 1);
        ptx::mbar_init(bar_o(1), 1);
        for (int lg = 0; lg < 4; ++lg) {
            ptx::mbar_init(bar_x(lg, 0), 64);
            ptx::mbar_init(bar_x(lg, 1), 64);
        }
        ptx::mbar_init(bar_drain, 1);
        ctl->abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == kQtLoaderWarp && lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::prefetch_tensormap(&tm_o);
    }
    if (warp == kQtMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == kQtLoaderWarp) {
        // =============================================================== loader
        // Per unit: Q once the previous unit's S products are done, then K_0,
        // K_1, V_0, K_2, V_1, ...: a K tile is only gated by the S products
        // that free its slot.  The rings run on across units.
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
            if (w.n == 0) continue;
            const int b_idx = w.bh / p.H, h_idx = w.bh % p.H;
            if (nq > 0 && !(ok = wait_warp(bar_qe, (nq - 1) & 1, abort, tmo))) break;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(bar_q, C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kSub; ++c)
                    ptx::tma_load_4d(sQ + c * kSubBytes, &tm_q, bar_q, 64 * c, w.qb * kTileM, h_idx,
                                     b_idx);
            }
            ++nq;
            for (int j = 0; j <= w.n; ++j) {
                if (j < w.n) {
                    const int s = kc % NK;
                    if (kc >= NK && !(ok = wait_warp(bar_ke(s), ((kc / NK) - 1) & 1, abort, tmo))) break;
                    const bool skip = (p.fault_mode == 1 && kc == 0);
                    if (lane == 0 && !skip) {
                        ptx::mbar_arrive_expect_tx(bar_kf(s), C::kTileBytes);
#pragma unroll
                        for (int c = 0; c < C::kSub; ++c)
                            ptx::tma_load_4d(sK(s) + c * kSubBytes, &tm_k, bar_kf(s), 64 * c,
                                             (w.k0 + j) * BN, h_idx, b_idx);
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
                                             (w.k0 + j - 1) * BN, h_idx, b_idx);
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
    } else if (warp == kQtMmaWarp) {
        // ====================================================== tensor-core issuer
        constexpr uint32_t idesc_s = instr_desc(BF16, kTileM, BN, false);
        constexpr uint32_t idesc_pv = instr_desc(BF16, kTileM, D, true);
        constexpr uint64_t kTileStep = C::kTileBytes / 16;
        const uint64_t q_desc = smem_desc(sQ, 16, 1024);
        const uint64_t k_desc0 = smem_desc(sK(0), 16, 1024);
        const uint64_t v_desc0 = smem_desc(sV(0), kSubBytes, 1024);
        // U (+)= P_h V over the keys of half h: the weights of keys 0-63 are
        // at columns 0-31 of the buffer, those of keys 64-127 at 64-95; V
        // rows 64 h .. 64 h + 63 start 8192 bytes (512 descriptor units) on
        auto issue_pv = [&](int b, int s, int h, bool acc) {
            ptx::mma_ts_k64(tmem + kQtTmemU, tmem + b * BN + h * 64, v_desc0 + s * kTileStep + h * 512,
                            idesc_pv, acc ? 1u : 0u);
        };
        uint32_t kc = 0, vc = 0;  // K and V tiles consumed so far (same order as loaded)
        uint32_t g = 0;           // key tiles of all previous units
        uint32_t nq = 0;          // units so far (q_full phase)
        bool ok = true;
        // S of the key tile counted gg over all units into buffer gg & 1 (the
        // one PV(gg - 2) read: issued after it, so in order); the last S of a
        // unit also releases its Q
        auto s_tile = [&](uint32_t gg, bool last) {
            const int s = kc % NK;
            if (!wait_warp(bar_kf(s), (kc / NK) & 1, abort, tmo)) return false;
            ptx::tc_fence_after_sync();
            const uint64_t kd = k_desc0 + s * kTileStep;
            if constexpr (D == 128)
                ptx::mma_ss_k128(tmem + (gg & 1) * BN, q_desc, kd, idesc_s, 0u);
            else
                ptx::mma_ss_k64(tmem + (gg & 1) * BN, q_desc, kd, idesc_s, 0u);
            ptx::tc_commit_elect(bar_ke(s));
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
                const uint32_t ph = (gg >> 1) & 1;
                const int sv = vc % NV;
                if (!(ok = wait_warp(bar_vf(sv), (vc / NV) & 1, abort, tmo))) break;
                // the first product of a unit overwrites all of U: both warps
                // of every row must be done with the previous unit's U first
                if (j == 0 && !(ok = wait_warp(bar_ph(b, 1), ph, abort, tmo))) break;
                if (!(ok = wait_warp(bar_ph(b, 0), ph, abort, tmo))) break;
                ptx::tc_fence_after_sync();
                issue_pv(b, sv, 0, j > 0);
                if (j > 0 && !(ok = wait_warp(bar_ph(b, 1), ph, abort, tmo))) break;
                ptx::tc_fence_after_sync();
                issue_pv(b, sv, 1, true);
                ptx::tc_commit_elect(bar_ve(sv));
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
        // ============================== softmax + epilogue: key half h, lane group lg
        const int h = warp >> 2;
        const int lg = warp & 3;
        const int t = lg * 32 + lane;                     // row in the tile = TMEM lane
        int first_row = 0, row = 0, k0 = 0;
        const uint32_t lane_off = static_cast<uint32_t>(lg * 32) << 16;
        const uint32_t u_addr = tmem + lane_off + kQtTmemU;
        const float c2 = p.scale_log2;
        const float2 c2v = make_float2(c2, c2);
        float2* xch = reinterpret_cast<float2*>(smem + C::kOffXch);
        uint32_t xc = 0;  // exchanges with the partner warp so far (slot and phase)
        // swap one float2 per row with the other warp of this lane group;
        // false if the CTA is aborting (the partner may never arrive)
        auto exchange = [&](float2 mine, float2& other) {
            const int slot = xc & 1;
            float2* base = xch + ((lg * 2 + slot) * 2) * 32;
            base[h * 32 + lane] = mine;
            ptx::mbar_arrive(bar_x(lg, slot));
            const bool ok = wait_warp(bar_x(lg, slot), (xc >> 1) & 1, abort, tmo);
            other = base[(h ^ 1) * 32 + lane];
            ++xc;
            return ok;
        };
        // whether this warp's 64 keys of tile j hold a key some of its rows
        // may not see: keys >= Nk, or past the causal limit of its first row
        auto half_masked = [&](int j) {
            const int kend = (k0 + j) * BN + h * 64 + 64;
            return kend > p.Nk || (CAUSAL && kend - 1 > first_row + lg * 32 + p.mask_offset);
        };
        auto key_limit = [&](int kbase) {
            int limit = p.Nk - kbase;
            if (CAUSAL) limit = min(limit, row + p.mask_offset - kbase + 1);
            return limit;
        };
        // weights 2^(x c2 + neg_ref) of this warp's 64 scores, packed to 16
        // bits; the fp32 weights are added to rs, the rounded ones to rh
        auto weights = [&](const uint32_t(&sv)[64], float neg_ref, uint32_t(&pk)[32], float2(&rs)[2],
                           float2(&rh)[2]) {
            const float2 nrv = make_float2(neg_ref, neg_ref);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
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
                if (h == 0 && row < p.Nq) {
                    const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + row;
                    const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                    p.lse_part[i] = -INFINITY;
                    p.lse_part[plane + i] = -INFINITY;
                }
                continue;
            }
            float m_ref = -INFINITY;              // reference maximum of the row's raw scores
            float2 lsum = make_float2(0.f, 0.f);  // this half's fp32 weights (for LSE), in .x
            float2 lhat = make_float2(0.f, 0.f);  // this half's 16-bit weights (for O), in .x

            for (int j = 0; j < n; ++j) {
                const uint32_t gg = g + j;
                const int b = gg & 1;
                if (!wait_warp(bar_sf(b), (gg >> 1) & 1, abort, tmo)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t s_addr = tmem + lane_off + b * BN + h * 64;
                uint32_t sv[64];
                ptx::tmem_ld_32x32b_x64(s_addr, sv);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 64; ++c) ptx::reg_fence(sv[c]);
                if (half_masked(j)) {
                    const int limit = key_limit((k0 + j) * BN + h * 64);
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (c >= limit) sv[c] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[32];
                float2 rs[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                float2 rh[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                // (the pair takes every branch below together: m_ref is the same
                // in both warps of a row, and each swap gives both the same facts)
                bool redo = __any_sync(0xffffffffu, m_ref == -INFINITY);
                if (!redo) {
                    // common case: weights against the current reference; the
                    // pair swaps whether either half's sum passed the bound
                    weights(sv, -m_ref * c2, pk, rs, rh);
                    const bool over = rs[0].x + rs[0].y + rs[1].x + rs[1].y > weight_sum_limit<BF16>();
                    float2 other;
                    if (!exchange(make_float2(over ? 1.f : 0.f, 0.f), other)) {
                        aborted = true;
                        break;
                    }
                    redo = __any_sync(0xffffffffu, over || other.x != 0.f);
                }
                float alpha = 1.f;
                float m_new = m_ref;
                if (redo) {
                    // the row's first tile, or a sum past the bound: the tile's
                    // maximum over both halves becomes the reference
                    float mx[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) mx[q] = __uint_as_float(sv[q]);
#pragma unroll
                    for (int c = 4; c + 8 <= 64; c += 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            mx[q] = ptx::fmax3(mx[q], __uint_as_float(sv[c + q]), __uint_as_float(sv[c + 4 + q]));
#pragma unroll
                    for (int q = 0; q < 4; ++q) mx[q] = fmaxf(mx[q], __uint_as_float(sv[60 + q]));
                    const float mt = ptx::fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
                    float2 other;
                    if (!exchange(make_float2(mt, 0.f), other)) {
                        aborted = true;
                        break;
                    }
                    m_new = ptx::fmax3(m_ref, mt, other.x);
                    if (m_ref != -INFINITY) alpha = ptx::ex2_approx((m_ref - m_new) * c2);
                    // a row with no valid key so far keeps all weights at zero
                    const float neg_ref = (m_new == -INFINITY) ? 0.f : -m_new * c2;
                    rs[0] = rs[1] = rh[0] = rh[1] = make_float2(0.f, 0.f);
                    weights(sv, neg_ref, pk, rs, rh);
                }
                const float2 rr = __fadd2_rn(rs[0], rs[1]), hh = __fadd2_rn(rh[0], rh[1]);
                lsum.x = fmaf(lsum.x, alpha, rr.x + rr.y);
                lhat.x = fmaf(lhat.x, alpha, hh.x + hh.y);
                ptx::tmem_st_32x32b_x32(s_addr, pk);
                // U holds P(j-1) V once PV(j-1) is done (it was issued after
                // S(j)): a rescale waits for it, each warp takes half of U's
                // columns, and neither hands over its weights before both are
                // done (the next product accumulates into all columns)
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
                    if (j > 0 && !wait_warp(bar_o(gg - 1), ((gg - 1) >> 1) & 1, abort, tmo)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const float2 av = make_float2(alpha, alpha);
#pragma unroll 1
                    for (int c = h * D / 32; c < (h + 1) * D / 32; ++c) {
                        uint32_t ov[16];
                        ptx::tmem_ld_32x32b_x16(u_addr + c * 16, ov);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; e += 2) {
                            ptx::reg_fence(ov[e]);
                            ptx::reg_fence(ov[e + 1]);
                            const float2 sc = __fmul2_rn(
                                make_float2(__uint_as_float(ov[e]), __uint_as_float(ov[e + 1])), av);
                            ov[e] = __float_as_uint(sc.x);
                            ov[e + 1] = __float_as_uint(sc.y);
                        }
                        ptx::tmem_st_32x32b_x16(u_addr + c * 16, ov);
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before_sync();
                    float2 other;
                    if (!exchange(make_float2(0.f, 0.f), other)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                ptx::mbar_arrive(bar_ph(b, h));
                m_ref = m_new;
            }

            // ---- epilogue: the pair adds its weight sums; O = U / lhat -> 16-bit
            // through each warp's staging box and TMA; LSE from the first warp
            if (!aborted && n > 0) aborted = !wait_warp(bar_o(g + n - 1), ((g + n - 1) >> 1) & 1, abort, tmo);
            g += n;
            if (aborted) break;
            float2 other;
            if (!exchange(make_float2(lsum.x, lhat.x), other)) break;
            const float l_all = lsum.x + other.x;
            const float lhat_all = lhat.x + other.y;
            ptx::tc_fence_after_sync();
            const uint32_t stage = sbase + C::kOffStage + warp * C::kStageBytes;
            const int out_row = first_row + 32 * lg;
            if constexpr (SPLIT) {
                // partial result of this key range: O normalised by its own
                // lhat (fp32, 32-column boxes: columns [32 c, 32 c + 32) for c
                // in this warp's half of d) and, from the first warp, the two
                // log-sums that weight it in the merge
                const bool mine = row < p.Nq && !*abort;
                const bool any = n > 0 && l_all > 0.f;
                if (h == 0 && mine) {
                    const size_t i = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + row;
                    const size_t plane = static_cast<size_t>(p.num_splits) * p.BH * p.Nq;
                    p.lse_part[i] = any ? m_ref * p.scale + logf(l_all) : -INFINITY;
                    p.lse_part[plane + i] = any ? m_ref * p.scale + logf(lhat_all) : -INFINITY;
                }
                const float inv = any ? 1.f / lhat_all : 0.f;
#pragma unroll 1
                for (int c = h * D / 64; c < (h + 1) * D / 64; ++c) {
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
                        ptx::tma_store_4d(&tm_o, stage, 32 * c, out_row, w.bh, w.split);
                        ptx::bulk_commit_group();
                    }
                }
            } else {
                // columns [64 h, 64 h + 64) of d = 128, all 64 of d = 64 from
                // the first warp; rows >= Nq and columns >= d are clipped
                const bool mine = row < p.Nq && !*abort;
                if (D == 128 || h == 0) {
                    const float inv = lhat_all > 0.f ? 1.f / lhat_all : 0.f;
                    const float2 iv = make_float2(inv, inv);
                    const int c0 = D == 128 ? 64 * h : 0;
                    if (lane == 0) ptx::bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        if (n > 0) {
                            ptx::tmem_ld_32x32b_x32(u_addr + c0 + cc * 32, ov);
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
                        ptx::tma_store_4d(&tm_o, stage, c0, out_row, h_idx, b_idx);
                        ptx::bulk_commit_group();
                    }
                }
                if (h == 0 && mine) {
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
    if (warp == kQtMmaWarp) ptx::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fa
