/*
 * fa_naive.h - attention computed step by step with S and P in HBM: the
 * "standard attention" of "CUDA 算子工程" ch. 14, sections 14.1-14.2
 * (S = Q K^T, P = softmax(S), O = P V, each step a separate pass over HBM).
 * It exists to measure the HBM traffic and time of that baseline next to
 * the fused kernel of fa.h on the same inputs; it is not the fused path.
 *
 * fa_naive_fwd computes, for every (b, h) and row i < N:
 *   S[i, j] = scale * q_i . k_j, rounded to the 16-bit input type and stored;
 *   P[i, j] = exp(S[i, j] - m_i) / l_i over the visible keys (0 for the
 *             others), from three passes over the stored row of S (maximum
 *             m_i, sum l_i, then the weights), rounded to 16 bits and stored;
 *   O[i, :] = sum_j P[i, j] v_j (fp32 accumulation, rounded to 16 bits);
 *   LSE[i]  = m_i + ln l_i (fp32).
 * q, k, v, o, lse, B, H, d, scale, causal, dtype, stream: as fa_fwd in fa.h.
 * N       : a multiple of 8 (16-byte rows of S and P), else FA_ERR_UNSUPPORTED.
 * d       : 64 or 128, else FA_ERR_UNSUPPORTED.
 * workspace, workspace_bytes : caller-owned device memory, 256-byte aligned,
 *           at least fa_naive_workspace_size(B, H, N) bytes: S then P, each
 *           [B, H, N, N] 16-bit.  Overwritten.
 * Three kernels are enqueued on `stream`; status codes as fa.h.
 */
#ifndef FA_GB300_FA_NAIVE_H
#define FA_GB300_FA_NAIVE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

size_t fa_naive_workspace_size(int B, int H, int N);

int fa_naive_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, int dtype, void* workspace,
                 size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_NAIVE_H */
