// fa_api.cu - host side of the C ABI declared in include/fa.h: argument
// checks, TMA tensor-map encoding, kernel selection and launch.
//
// The problem statement it validates is that of "CUDA 算子工程" ch. 14,
// section 14.5 (inputs Q, K, V [N, d]; outputs O [N, d] and LSE [N]), per
// (batch, head), with the explicit scale and causal flag of
// "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (sections
// "先固定一个例子" and "causal 模式在哪一步生效").
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/fa.h"
#include "../../include/fa_naive.h"
#include "fa_fwd_kernel.cuh"
#include "fa_fwd_qtile_kernel.cuh"
#include "fa_fwd_wide_kernel.cuh"
#include "naive_attention.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A 16-bit [B, H, rows, d] tensor with element strides (batch, head, row) and
// contiguous d, viewed by TMA in 4-D (d, rows, H, B) so that rows >= `rows`
// of one head are out of range (zero-filled on load, clipped on store)
// instead of belonging to the next head.  Columns >= d are out of range too:
// a kernel wider than d reads zeros there and never writes them.  Box: 64
// columns (128 bytes, one swizzle span) x box_rows rows (a query or key tile,
// one part of a V tile, or the 32 rows of O one softmax warp stores) x 1 x 1.
bool encode_4d(CUtensorMap* map, const void* ptr, int dtype, int64_t B, int64_t H, int64_t rows,
               int64_t d, const long long (&stride)[3], uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(stride[2]) * 2,
                                   static_cast<cuuint64_t>(stride[1]) * 2,
                                   static_cast<cuuint64_t>(stride[0]) * 2};
    const cuuint32_t box[4] = {64, box_rows, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == FA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return fn(map, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split-KV partials o_part [S][BH][Nq][kd] fp32 viewed by TMA in 4-D
// (kd, Nq, BH, S): rows >= Nq of a head are clipped on store.  Box: 32
// columns (128 bytes, one swizzle span) x 32 rows (one softmax warp's rows).
bool encode_partials(CUtensorMap* map, float* o_part, int64_t S, int64_t BH, int64_t Nq, int64_t kd) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kd), static_cast<cuuint64_t>(Nq),
                                static_cast<cuuint64_t>(BH), static_cast<cuuint64_t>(S)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kd) * 4,
                                   static_cast<cuuint64_t>(Nq * kd) * 4,
                                   static_cast<cuuint64_t>(BH * Nq * kd) * 4};
    const cuuint32_t box[4] = {32, 32, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, o_part, dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Width of the kernel that serves head dimension d: 64, 128, 192 or 256,
// the smallest that holds d (the columns beyond d are zeros: TMA fills them
// on load and clips them on store); 0 = unsupported (d must be a multiple of
// 8, a TMA stride rule, and at most 256).
int kernel_dim(int d) {
    if (d < 8 || d % 8 != 0 || d > 256) return 0;
    return d <= 64 ? 64 : d <= 128 ? 128 : d <= 192 ? 192 : 256;
}

struct KernelEntry {
    const void* fn;
    int smem;
    int threads;
    int block_m;  // query rows per unit of work
    int block_n;  // keys per K/V tile (rows of the K boxes)
    int v_rows;   // rows of the V boxes (a tile or a part of one)
};

// The kernel that serves a request.  Widths 192 and 256 have their own
// (one query tile per unit).  Widths 64 and 128 run units of two 128-row
// query tiles that share every K/V tile, except causal grids whose 256-row
// blocks fit in one wave: there units of one 128-row tile (twice as many,
// dealt longest first) share the SMs more evenly than two-tile units or key
// ranges do.
enum class Kind { kTwoTile, kOneTile, kWide };

int sm_count();

Kind kernel_kind(int kd, bool causal, int64_t BH, int64_t Nq) {
    if (kd > 128) return Kind::kWide;
    const int64_t blocks = BH * ((Nq + fa::kBlockM - 1) / fa::kBlockM);
    return (causal && blocks <= sm_count()) ? Kind::kOneTile : Kind::kTwoTile;
}

// Query rows per unit of work of a kernel kind.
int64_t unit_rows(Kind k) { return k == Kind::kTwoTile ? fa::kBlockM : fa::kTileM; }

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
KernelEntry entry(Kind k) {
    if constexpr (D <= 128) {
        if constexpr (CAUSAL)  // one-tile units serve causal grids only
            if (k == Kind::kOneTile)
                return KernelEntry{
                    reinterpret_cast<const void*>(&fa::fa_fwd_qtile_kernel<D, BF16, CAUSAL, SPLIT>),
                    fa::QtCfg<D>::kSmemBytes, fa::kQtThreads, fa::kTileM, fa::kQtBlockN, fa::kQtBlockN};
        return KernelEntry{
            reinterpret_cast<const void*>(&fa::fa_fwd_kernel<D, BF16, CAUSAL, SPLIT>),
            fa::Cfg<D>::kSmemBytes, fa::kThreads, fa::kBlockM, fa::kBlockN, fa::kBlockN};
    } else {
        return KernelEntry{
            reinterpret_cast<const void*>(&fa::fa_fwd_wide_kernel<D, BF16, CAUSAL, SPLIT>),
            fa::WideCfg<D>::kSmemBytes, fa::kWideThreads, fa::kTileM, fa::kWideBlockN,
            fa::WideCfg<D>::kVPartRows};
    }
}

template <int D, bool BF16>
KernelEntry select_d_dtype(Kind k, bool causal, bool split) {
    if (causal) return split ? entry<D, BF16, true, true>(k) : entry<D, BF16, true, false>(k);
    return split ? entry<D, BF16, false, true>(k) : entry<D, BF16, false, false>(k);
}

// kd: a kernel width from kernel_dim()
KernelEntry select_kernel(int kd, Kind k, int dtype, bool causal, bool split) {
    const bool bf = dtype == FA_BF16;
    switch (kd) {
        case 64: return bf ? select_d_dtype<64, true>(k, causal, split) : select_d_dtype<64, false>(k, causal, split);
        case 128: return bf ? select_d_dtype<128, true>(k, causal, split) : select_d_dtype<128, false>(k, causal, split);
        case 192: return bf ? select_d_dtype<192, true>(k, causal, split) : select_d_dtype<192, false>(k, causal, split);
        default: return bf ? select_d_dtype<256, true>(k, causal, split) : select_d_dtype<256, false>(k, causal, split);
    }
}

template <int D>
const void* merge_fn(bool bf, int num_splits) {
    if (num_splits <= 2)
        return bf ? reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, true, 2>)
                  : reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, false, 2>);
    if (num_splits <= 4)
        return bf ? reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, true, 4>)
                  : reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, false, 4>);
    return bf ? reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, true, 8>)
              : reinterpret_cast<const void*>(&fa::fa_split_merge_kernel<D, false, 8>);
}

const void* select_merge(int kd, int dtype, int num_splits) {
    const bool bf = dtype == FA_BF16;
    switch (kd) {
        case 64: return merge_fn<64>(bf, num_splits);
        case 128: return merge_fn<128>(bf, num_splits);
        case 192: return merge_fn<192>(bf, num_splits);
        default: return merge_fn<256>(bf, num_splits);
    }
}

// Opt each kernel into its dynamic shared memory once per device.
bool ensure_smem_attr(const void* fn, int smem, int device) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;  // (kernel, device) already set
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({fn, device})) return true;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return false;
    done.insert({fn, device});
    return true;
}

// Workspace layout of split-KV: o_part [S][BH][N][kd] fp32 (kd the kernel
// width), then (256-byte aligned) lse_part [2][S][BH][N] fp32.
size_t split_o_bytes(int64_t S, int64_t BH, int64_t N, int64_t d) {
    return (static_cast<size_t>(S * BH * N * d) * 4 + 255) & ~static_cast<size_t>(255);
}
size_t split_workspace_bytes(int64_t S, int64_t BH, int64_t N, int64_t d) {
    return split_o_bytes(S, BH, N, d) + static_cast<size_t>(2 * S * BH * N) * 4;
}

// SMs of the current device (GB300's 152 if it cannot be asked).
int sm_count() {
    int device = 0, sms = 152;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        sms = 152;
    return sms;
}

// Split count for num_splits = 0: BH heads of Nq query rows and Nk keys on
// a kernel of width kd.  Splitting costs fp32 partials and a merge.  Without
// the mask every query block takes as long as any other, so splitting pays
// only when the blocks leave more than half of the SMs idle: up to there one
// wave of whole blocks is as short as two waves of halves.  With the causal
// mask a wave lasts as long as its longest block (the one that sees every
// key), so a grid that fits in one wave is split as well: the halves of the
// long blocks then share CTAs with the short blocks in the persistent
// schedule.  The count aims at about one wave of CTAs, with at least 512 keys
// per range.
int choose_splits(int64_t BH, int Nq, int Nk, int kd, bool causal) {
    if (kd == 0) return 1;
    const int sms = sm_count();
    const int64_t block_m = unit_rows(kernel_kind(kd, causal, BH, Nq));
    const int64_t blocks = BH * ((Nq + block_m - 1) / block_m);
    if (blocks > sms || (!causal && 2 * blocks > sms)) return 1;
    int64_t s = (static_cast<int64_t>(sms) + blocks - 1) / blocks;
    s = std::min<int64_t>(s, std::max<int64_t>(1, static_cast<int64_t>(Nk) / 512));
    s = std::min<int64_t>(s, FA_MAX_SPLITS);
    return static_cast<int>(std::max<int64_t>(1, s));
}

// Contiguous [B, H, N, d] strides.
fa_fwd_args contiguous_args(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                            int H, int N, int d, float scale, int causal, int dtype, void* stream) {
    fa_fwd_args a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.B = B; a.H = H; a.Nq = N; a.Nk = N; a.d = d;
    const long long sn = d, sh = static_cast<long long>(N) * d, sb = sh * H;
    for (long long* st : {a.q_stride, a.k_stride, a.v_stride, a.o_stride}) {
        st[0] = sb; st[1] = sh; st[2] = sn;
    }
    a.lse_stride[0] = static_cast<long long>(H) * N;
    a.lse_stride[1] = N;
    a.scale = scale;
    a.mask = causal ? FA_MASK_CAUSAL_TOP_LEFT : FA_MASK_NONE;
    a.dtype = dtype;
    a.num_splits = 1;
    a.stream = stream;
    return a;
}

bool misaligned(const void* ptr, uintptr_t al) {
    return (reinterpret_cast<uintptr_t>(ptr) & (al - 1)) != 0;
}

// Testing controls of fa_fwd_debug (FA_OK in production calls).
enum FaultMode : int {
    kFaultNone = 0,
    kFaultSkipFirstKeyTile = 1,  // the loader never issues the first key tile: a wait times out
    kFaultLaunch = 2,            // the launch step reports failure instead of launching
};

// Every check that does not depend on the split count: pointers, sizes,
// dtype, scale, mask, strides and alignment.
int check_args(const fa_fwd_args& a, int fault_mode, double timeout_s) {
    if (!a.q || !a.k || !a.v || !a.o || !a.lse) return FA_ERR_INVALID_ARG;
    if (a.B < 1 || a.H < 1 || a.Nq < 1 || a.Nk < 1) return FA_ERR_INVALID_ARG;
    if (a.dtype != FA_FP16 && a.dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(a.scale) || !(a.scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (a.mask != FA_MASK_NONE && a.mask != FA_MASK_CAUSAL_TOP_LEFT &&
        a.mask != FA_MASK_CAUSAL_BOTTOM_RIGHT)
        return FA_ERR_INVALID_ARG;
    if (!(timeout_s > 0.0) || !std::isfinite(timeout_s)) return FA_ERR_INVALID_ARG;
    if (fault_mode < kFaultNone || fault_mode > kFaultLaunch) return FA_ERR_INVALID_ARG;
    const int kd = kernel_dim(a.d);
    if (kd == 0) return FA_ERR_UNSUPPORTED;
    const int64_t BH = static_cast<int64_t>(a.B) * a.H;
    const int64_t block_m = unit_rows(kernel_kind(kd, a.mask != FA_MASK_NONE, BH, a.Nq));
    const int64_t nq = (static_cast<int64_t>(a.Nq) + block_m - 1) / block_m;  // query blocks per head
    if (BH > INT32_MAX || BH * nq > INT32_MAX) return FA_ERR_INVALID_ARG;
    // TMA: every stride a positive multiple of 16 bytes (8 16-bit elements);
    // LSE rows contiguous, its strides positive
    for (const long long* st : {a.q_stride, a.k_stride, a.v_stride, a.o_stride})
        for (int i = 0; i < 3; ++i)
            if (st[i] <= 0 || st[i] % 8 != 0 || st[i] >= (1ll << 39)) return FA_ERR_MISALIGNED;
    if (a.lse_stride[0] <= 0 || a.lse_stride[1] <= 0) return FA_ERR_INVALID_ARG;
    if (misaligned(a.q, 16) || misaligned(a.k, 16) || misaligned(a.v, 16) || misaligned(a.o, 16) ||
        misaligned(a.lse, 4))
        return FA_ERR_MISALIGNED;
    return FA_OK;
}

int fwd_core(const fa_fwd_args& a, int fault_mode, double timeout_s) {
    const int st_args = check_args(a, fault_mode, timeout_s);
    if (st_args != FA_OK) return st_args;
    const int B = a.B, H = a.H, Nq = a.Nq, Nk = a.Nk, d = a.d, dtype = a.dtype;
    const int kd = kernel_dim(d);
    const bool causal = a.mask != FA_MASK_NONE;
    const int64_t BH = static_cast<int64_t>(B) * H;
    const Kind kind = kernel_kind(kd, causal, BH, Nq);
    const int64_t block_m = unit_rows(kind);
    const int64_t nq = (static_cast<int64_t>(Nq) + block_m - 1) / block_m;  // query blocks per head
    int num_splits = a.num_splits;
    if (num_splits == 0)
        num_splits = choose_splits(static_cast<int64_t>(B) * H, Nq, Nk, kernel_dim(d), causal);
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
    const bool split = num_splits > 1;
    if (split) {
        if (!a.workspace) return FA_ERR_INVALID_ARG;
        if (misaligned(a.workspace, 256)) return FA_ERR_MISALIGNED;
        if (a.workspace_bytes < split_workspace_bytes(num_splits, BH, Nq, kd)) return FA_ERR_INVALID_ARG;
        if (BH * nq * num_splits > INT32_MAX) return FA_ERR_INVALID_ARG;
    }

    const KernelEntry ke = select_kernel(kd, kind, dtype, causal, split);
    const uint32_t qrows = static_cast<uint32_t>(fa::kTileM);
    const uint32_t krows = static_cast<uint32_t>(ke.block_n);
    CUtensorMap tq, tk, tv, to;
    if (!encode_4d(&tq, a.q, dtype, B, H, Nq, d, a.q_stride, qrows) ||
        !encode_4d(&tk, a.k, dtype, B, H, Nk, d, a.k_stride, krows) ||
        !encode_4d(&tv, a.v, dtype, B, H, Nk, d, a.v_stride, static_cast<uint32_t>(ke.v_rows)) ||
        !encode_4d(&to, a.o, dtype, B, H, Nq, d, a.o_stride, 32u))  // one warp's rows per store
        return FA_ERR_CUDA;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
    if (!ensure_smem_attr(ke.fn, ke.smem, device)) return FA_ERR_CUDA;

    const int64_t units = BH * nq * num_splits;
    fa::FwdParams prm;
    prm.num_units = static_cast<int>(units);
    prm.lse = a.lse;
    prm.lse_sb = a.lse_stride[0];
    prm.lse_sh = a.lse_stride[1];
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.H = H;
    prm.mask_offset = a.mask == FA_MASK_CAUSAL_BOTTOM_RIGHT ? Nk - Nq : 0;
    prm.num_q_blocks = static_cast<int>(nq);
    prm.scale = a.scale;
    prm.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    prm.timeout_ns = static_cast<unsigned long long>(timeout_s * 1e9);
    prm.fault_mode = fault_mode;
    prm.num_splits = num_splits;
    prm.BH = static_cast<int>(BH);
    prm.o_part = split ? static_cast<float*>(a.workspace) : nullptr;
    prm.lse_part = split ? reinterpret_cast<float*>(static_cast<char*>(a.workspace) +
                                                    split_o_bytes(num_splits, BH, Nq, kd))
                         : nullptr;

    // split-KV kernels write no O: their last tensor map is that of the partials
    if (split && !encode_partials(&to, prm.o_part, num_splits, BH, Nq, kd)) return FA_ERR_CUDA;
    void* args[] = {&tq, &tk, &tv, &to, &prm};
    // the kernels are persistent: one CTA per SM walks the units
    const int64_t ctas = std::min<int64_t>(units, sm_count());
    const dim3 grid(static_cast<unsigned>(ctas));
    const dim3 block(static_cast<unsigned>(ke.threads));
    const cudaStream_t st = static_cast<cudaStream_t>(a.stream);
    if (fault_mode == kFaultLaunch) return FA_ERR_CUDA;  // as if cudaLaunchKernel had failed
    if (cudaLaunchKernel(ke.fn, grid, block, args, static_cast<size_t>(ke.smem), st) != cudaSuccess)
        return FA_ERR_CUDA;
    if (split) {
        fa::MergeParams mp;
        mp.o_part = prm.o_part;
        mp.lse_part = prm.lse_part;
        mp.o = a.o;
        mp.o_sb = a.o_stride[0];
        mp.o_sh = a.o_stride[1];
        mp.o_sn = a.o_stride[2];
        mp.lse = a.lse;
        mp.lse_sb = a.lse_stride[0];
        mp.lse_sh = a.lse_stride[1];
        mp.num_splits = num_splits;
        mp.H = H;
        mp.Nq = Nq;
        mp.d_out = d;
        mp.rows = BH * Nq;
        void* margs[] = {&mp};
        // a programmatic dependent launch: the merge grid is set up while the
        // attention kernel runs, and waits (griddepcontrol.wait) for its end
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t mcfg = {};
        mcfg.gridDim = dim3(static_cast<unsigned>((mp.rows + 7) / 8));
        mcfg.blockDim = dim3(256);
        mcfg.dynamicSmemBytes = 0;
        mcfg.stream = st;
        mcfg.attrs = attr;
        mcfg.numAttrs = 1;
        if (cudaLaunchKernelExC(&mcfg, select_merge(kd, dtype, num_splits), margs) != cudaSuccess) return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, int dtype, void* stream) {
    return fwd_core(contiguous_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream), 0,
                    2.0);
}

int fa_fwd_ex(const fa_fwd_args* args) {
    if (!args) return FA_ERR_INVALID_ARG;
    return fwd_core(*args, 0, 2.0);
}

int fa_fwd_debug(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, int dtype, void* stream, int fault_mode,
                 double timeout_s) {
    return fwd_core(contiguous_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream),
                    fault_mode, timeout_s);
}

int fa_splitkv_num_splits(int B, int H, int N, int d, int causal) {
    if (B < 1 || H < 1 || N < 1) return 1;
    return choose_splits(static_cast<int64_t>(B) * H, N, N, kernel_dim(d), causal != 0);
}

int fa_splitkv_num_splits_ex(const fa_fwd_args* a) {
    if (!a || a->B < 1 || a->H < 1 || a->Nq < 1 || a->Nk < 1) return 1;
    return choose_splits(static_cast<int64_t>(a->B) * a->H, a->Nq, a->Nk, kernel_dim(a->d),
                         a->mask != FA_MASK_NONE);
}

size_t fa_splitkv_workspace_size(int B, int H, int N, int d, int num_splits) {
    const int kd = kernel_dim(d);
    if (B < 1 || H < 1 || N < 1 || kd == 0 || num_splits < 2) return 0;
    return split_workspace_bytes(num_splits, static_cast<int64_t>(B) * H, N, kd);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int dtype, int num_splits,
                   void* workspace, size_t workspace_bytes, void* stream) {
    fa_fwd_args a = contiguous_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream);
    a.num_splits = num_splits;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return fwd_core(a, 0, 2.0);
}

// ---- split-KV without any allocation by the library or its caller --------
// Some callers cannot call cudaMalloc: a plugin whose host framework owns all
// device memory and forbids other allocations, or a latency-critical path that
// cannot take cudaMalloc's implicit device synchronisation.  For them the
// split-KV partials live in this fixed array, which every GPU that loads the
// library holds until the process exits.  In host code the name is only a
// host-side stand-in, so its device address is looked up per device.
static __device__ __align__(256) unsigned char g_fa_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {
// Device address of g_fa_noalloc_scratch on the current device, looked up by
// the first call made with that device current and kept for the process
// (nullptr if the lookup fails).  cudaDeviceReset unloads the module, after
// which the kept address is stale: the entry point is not for use after a
// reset of a device it has already run on.
void* noalloc_scratch() {
    static std::mutex mu;
    static void* addr[64] = {};
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[device] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_fa_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[device] = ptr;
    }
    return addr[device];
}
}  // namespace

int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal, int dtype,
                           int num_splits, void* stream) {
    fa_fwd_args a = contiguous_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream);
    // the same argument checks, in the same order, as every other entry point
    const int st_args = check_args(a, kFaultNone, 2.0);
    if (st_args != FA_OK) return st_args;
    if (num_splits < 0 || num_splits > FA_MAX_SPLITS) return FA_ERR_INVALID_ARG;
    if (num_splits == 0) {
        // the library's choice, lowered until its partials fit the array
        // (down to 1: plain fa_fwd, which needs no scratch at all)
        num_splits = fa_splitkv_num_splits(B, H, N, d, causal);
        while (num_splits > 1 &&
               fa_splitkv_workspace_size(B, H, N, d, num_splits) > FA_NOALLOC_SCRATCH_BYTES)
            --num_splits;
    }
    if (num_splits == 1) return fwd_core(a, kFaultNone, 2.0);
    // an explicit count whose partials do not fit is refused
    if (fa_splitkv_workspace_size(B, H, N, d, num_splits) > FA_NOALLOC_SCRATCH_BYTES)
        return FA_ERR_UNSUPPORTED;
    // Nothing in the partials needs to start at zero: every range writes both
    // of its log-sums for every row, and the merge reads O only where they
    // are finite.  Calls share the array, so calls that may overlap on the GPU
    // race; callers must order them (one stream, or events).
    void* scratch = noalloc_scratch();
    if (scratch == nullptr) return FA_ERR_CUDA;
    a.num_splits = num_splits;
    a.workspace = scratch;
    a.workspace_bytes = FA_NOALLOC_SCRATCH_BYTES;
    return fwd_core(a, kFaultNone, 2.0);
}

int fa_check_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
    unsigned int st = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&st, fa::g_fa_status, sizeof(st)) != cudaSuccess) return FA_ERR_CUDA;
    if (st != 0 && cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess)
        return FA_ERR_CUDA;
    return static_cast<int>(st);
}

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

int fa_version(void) { return 100; }

}  // extern "C"

// ---- the step-by-step baseline (S and P in HBM) ---------------------------
namespace {

size_t naive_matrix_bytes(int64_t BH, int64_t N) {
    return (static_cast<size_t>(BH * N * N) * 2 + 255) & ~static_cast<size_t>(255);
}

template <int D, bool BF16>
int naive_launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& to, const CUtensorMap& ts, const CUtensorMap& tp,
                 const uint16_t* S, uint16_t* P, float* lse, int H, int64_t BH, int N,
                 float scale, int causal, cudaStream_t st) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
    const unsigned long long tmo = 2000000000ull;
    const void* f1 = reinterpret_cast<const void*>(&fa::fa_naive_scores_kernel<D, BF16>);
    const void* f2 = reinterpret_cast<const void*>(&fa::fa_naive_softmax_kernel<BF16>);
    const void* f3 = reinterpret_cast<const void*>(&fa::fa_naive_pv_kernel<D, BF16>);
    const int sm1 = fa::NaiveScoresCfg<D>::kSmemBytes, sm3 = fa::NaivePvCfg<D>::kSmemBytes;
    if (!ensure_smem_attr(f1, sm1, device) || !ensure_smem_attr(f3, sm3, device)) return FA_ERR_CUDA;
    const unsigned nt = static_cast<unsigned>((N + 127) / 128);
    {
        int h = H;
        float sc = scale;
        unsigned long long t = tmo;
        void* args[] = {const_cast<CUtensorMap*>(&tq), const_cast<CUtensorMap*>(&tk),
                        const_cast<CUtensorMap*>(&ts), &h, &sc, &t};
        if (cudaLaunchKernel(f1, dim3(nt, nt, static_cast<unsigned>(BH)), dim3(fa::kNaiveThreads),
                             args, sm1, st) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    {
        const uint16_t* s_ = S;
        uint16_t* p_ = P;
        float* l_ = lse;
        int n = N, c = causal, off = 0;
        void* args[] = {&s_, &p_, &l_, &n, &c, &off};
        if (cudaLaunchKernel(f2, dim3(static_cast<unsigned>(BH * N)), dim3(fa::kNaiveSoftmaxThreads),
                             args, 0, st) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    {
        int h = H, n = N;
        unsigned long long t = tmo;
        void* args[] = {const_cast<CUtensorMap*>(&tp), const_cast<CUtensorMap*>(&tv),
                        const_cast<CUtensorMap*>(&to), &h, &n, &t};
        if (cudaLaunchKernel(f3, dim3(nt, static_cast<unsigned>(BH)), dim3(fa::kNaivePvThreads),
                             args, sm3, st) != cudaSuccess)
            return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace

extern "C" {

size_t fa_naive_workspace_size(int B, int H, int N) {
    if (B < 1 || H < 1 || N < 1) return 0;
    return 2 * naive_matrix_bytes(static_cast<int64_t>(B) * H, N);
}

int fa_naive_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, int dtype, void* workspace,
                 size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP16 && dtype != FA_BF16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (N % 8 != 0) return FA_ERR_UNSUPPORTED;
    const int64_t BH = static_cast<int64_t>(B) * H;
    if (BH > 65535 || (N + 127) / 128 > 65535 || BH * N > INT32_MAX) return FA_ERR_INVALID_ARG;
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
        misaligned(lse, 4) || misaligned(workspace, 256))
        return FA_ERR_MISALIGNED;
    if (workspace_bytes < fa_naive_workspace_size(B, H, N)) return FA_ERR_INVALID_ARG;
    uint16_t* S = static_cast<uint16_t*>(workspace);
    uint16_t* P = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + naive_matrix_bytes(BH, N));
    fa_fwd_args a = contiguous_args(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream);
    const long long mat[3] = {BH * N * N, static_cast<long long>(N) * N, N};
    CUtensorMap tq, tk, tv, to, ts, tp;
    if (!encode_4d(&tq, q, dtype, B, H, N, d, a.q_stride, 128) ||
        !encode_4d(&tk, k, dtype, B, H, N, d, a.k_stride, 128) ||
        !encode_4d(&tv, v, dtype, B, H, N, d, a.v_stride, 128) ||
        !encode_4d(&to, o, dtype, B, H, N, d, a.o_stride, 128) ||
        !encode_4d(&ts, S, dtype, 1, BH, N, N, mat, 128) ||
        !encode_4d(&tp, P, dtype, 1, BH, N, N, mat, 128))
        return FA_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = dtype == FA_BF16;
    if (d == 64)
        return bf ? naive_launch<64, true>(tq, tk, tv, to, ts, tp, S, P, lse, H, BH, N, scale, causal, st)
                  : naive_launch<64, false>(tq, tk, tv, to, ts, tp, S, P, lse, H, BH, N, scale, causal, st);
    return bf ? naive_launch<128, true>(tq, tk, tv, to, ts, tp, S, P, lse, H, BH, N, scale, causal, st)
              : naive_launch<128, false>(tq, tk, tv, to, ts, tp, S, P, lse, H, BH, N, scale, causal, st);
}

}  // extern "C"
