// ceilings.cu - microbenchmarks of the two secondary ceilings of the fused
// attention kernel besides the tensor core: the rate of the exponential unit
// (one 2^x per score) and the L2 -> SM read bandwidth (every CTA streams the
// K and V tiles of its head; after the first CTA of a head they come from L2).
// "CUDA 算子工程" ch. 14, section 14.2 counts the work of attention in FLOPs
// and bytes; these give the rates to divide those counts by.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa_ceilings.h"

namespace {

__device__ __forceinline__ float ex2_neg(float x) {
    float r;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(-x));
    return r;
}

// 8 independent chains per thread, x -> 2^-x (stays in [0.5, 1)).
constexpr int kChains = 8;

__global__ void __launch_bounds__(1024) ex2_rate_kernel(float* out, int iters) {
    float v[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) v[i] = 0.1f * (i + 1) + threadIdx.x * 1e-7f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) v[i] = ex2_neg(v[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += v[i];
    if (s == 1234.5f) out[blockIdx.x] = s;  // never true; keeps the chains live
}

// Grid-stride 16-byte loads cached in L2 only (ld.global.cg), `iters` passes.
__global__ void __launch_bounds__(512) l2_read_kernel(const uint4* buf, size_t n16, int iters,
                                                     uint32_t* out) {
    uint32_t acc = 0;
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    for (int it = 0; it < iters; ++it)
        for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
             i += stride) {
            const uint4 v = __ldcg(buf + i);
            acc ^= v.x ^ v.y ^ v.z ^ v.w;
        }
    if (acc == 0x9E3779B9u) out[0] = acc;  // never true in practice; keeps the loads
}

struct Events {
    cudaEvent_t a = nullptr, b = nullptr;
    bool ok = false;
    Events() { ok = cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess; }
    ~Events() {
        if (a) cudaEventDestroy(a);
        if (b) cudaEventDestroy(b);
    }
};

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

}  // namespace

extern "C" {

int fa_ceiling_ex2_rate(double* per_second, void* stream) {
    if (!per_second) return FA_CEIL_ERR_ARG;
    const int sms = sm_count();
    if (sms <= 0) return FA_CEIL_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int blocks = 2 * sms, threads = 1024, iters = 4096;
    Events ev;
    if (!ev.ok) return FA_CEIL_ERR_CUDA;
    ex2_rate_kernel<<<blocks, threads, 0, st>>>(nullptr, 256);  // warm-up (clocks, code)
    cudaEventRecord(ev.a, st);
    ex2_rate_kernel<<<blocks, threads, 0, st>>>(nullptr, iters);
    cudaEventRecord(ev.b, st);
    if (cudaEventSynchronize(ev.b) != cudaSuccess) return FA_CEIL_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev.a, ev.b) != cudaSuccess || ms <= 0.f) return FA_CEIL_ERR_CUDA;
    const double ops = static_cast<double>(blocks) * threads * kChains * iters;
    *per_second = ops / (ms * 1e-3);
    return FA_CEIL_OK;
}

int fa_ceiling_l2_read(const void* buf, size_t bytes, double* bytes_per_second, void* stream) {
    if (!buf || !bytes_per_second || bytes < 16 || bytes % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(buf) & 15u) != 0)
        return FA_CEIL_ERR_ARG;
    const int sms = sm_count();
    if (sms <= 0) return FA_CEIL_ERR_CUDA;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n16 = bytes / 16;
    const int blocks = 4 * sms, threads = 512, iters = 20;
    Events ev;
    if (!ev.ok) return FA_CEIL_ERR_CUDA;
    const uint4* p = static_cast<const uint4*>(buf);
    l2_read_kernel<<<blocks, threads, 0, st>>>(p, n16, 2, nullptr);  // bring the buffer into L2
    cudaEventRecord(ev.a, st);
    l2_read_kernel<<<blocks, threads, 0, st>>>(p, n16, iters, nullptr);
    cudaEventRecord(ev.b, st);
    if (cudaEventSynchronize(ev.b) != cudaSuccess) return FA_CEIL_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, ev.a, ev.b) != cudaSuccess || ms <= 0.f) return FA_CEIL_ERR_CUDA;
    *bytes_per_second = static_cast<double>(bytes) * iters / (ms * 1e-3);
    return FA_CEIL_OK;
}

}  // extern "C"
