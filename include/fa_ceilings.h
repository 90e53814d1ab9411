/*
 * fa_ceilings.h - microbenchmarks of the fused attention kernel's secondary
 * ceilings, exported by the same library as fa.h.
 *
 * Besides the tensor core (FLOPs, "CUDA 算子工程" ch. 14, section 14.2), the
 * kernel is bounded by the exponential unit (one 2^x per visible score, the
 * weights of "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程", section
 * "第四步") and by the L2 -> SM bandwidth (each CTA streams its head's K and V
 * tiles; all but the first read of a tile hit L2).  These two calls measure
 * those rates on the current device so that a benchmark can turn the
 * kernel's exp count and L2 bytes into time floors.
 *
 * Both synchronise `stream` (cudaStream_t as void*, NULL = legacy default)
 * and take a few milliseconds.  Not thread-safe with respect to other work on
 * the same device if the numbers are to mean anything.
 */
#ifndef FA_GB300_FA_CEILINGS_H
#define FA_GB300_FA_CEILINGS_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_CEIL_OK 0
#define FA_CEIL_ERR_ARG 1   /* null pointer, size not a positive multiple of 16, misaligned */
#define FA_CEIL_ERR_CUDA 4  /* a CUDA call failed */

/* 2^x evaluations per second (ex2.approx.ftz.f32, the instruction the kernel's
 * weights use) over the whole device: two CTAs of 1024 threads per SM, eight
 * independent chains per thread.  Result in *per_second. */
int fa_ceiling_ex2_rate(double* per_second, void* stream);

/* Read bandwidth from L2 into the SMs, bytes per second: 16-byte loads cached
 * in L2 only (ld.global.cg) over `bytes` of device memory at `buf` (16-byte
 * aligned; choose bytes well below the L2 size so that it stays resident),
 * read once to warm L2 and then 20 times timed.  `buf` is read, not written. */
int fa_ceiling_l2_read(const void* buf, size_t bytes, double* bytes_per_second, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_CEILINGS_H */
