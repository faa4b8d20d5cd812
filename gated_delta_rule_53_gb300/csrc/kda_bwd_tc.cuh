// Operand tiles of the tensor-core reverse pass of kda_chunk_bwd, per (chunk slot, head), written by
// bwd_prep_kernel and read by bwd_state_tc_kernel.  Each fp32 tile is stored as bf16 hi then bf16 lo
// (x = hi + lo), in the 128-byte-swizzled layouts of kda_tc.cuh:
//   Kr, scale Qg, Kg   [64 tokens][128 channels]: two regions of [64][64] (channels 0-63, 64-127)
//   scale A_qk, T      [64][64]: one region, row s, column t
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr uint32_t kBB_KR = 0;          // Kr = K e^{G_last - G}: hi 16 KB, lo 16 KB
constexpr uint32_t kBB_QG = 32768;      // scale Q e^G
constexpr uint32_t kBB_KG = 65536;      // K e^G
constexpr uint32_t kBB_AQ = 98304;      // scale A_qk: hi 8 KB, lo 8 KB
constexpr uint32_t kBB_TT = 114688;     // T = (I + A_kk)^-1
constexpr uint32_t kBB_GAM = 131072;    // gamma = e^{G_last}, fp32 [128]
constexpr uint32_t kBB_BETA = 131584;   // beta, fp32 [64] (0 past the chunk's end)
constexpr uint32_t kBwdBlobBytes = 131840;

// Per (chunk, head) the tiles above (Kr, scale Qg, Kg, scale A_qk, T, gamma, beta) for bf16 q, k, with the
// products A_qk and A_kk on the tensor cores; raises the gate and beta range bits of `err` as the forward does.
cudaError_t launch_bwd_prep_tc(const void* q, const void* k, const float* g, const float* beta, const int32_t* cu_seqlens,
                               int N, int64_t T_total, int H, float scale, void* blobs, unsigned int* err,
                               cudaStream_t stream);

// The forward pass along the chains on the tensor cores for bf16 v (v [T_total, H, 128]): the state entering
// every chunk, R and V'; outputs as the CUDA-core pass.
cudaError_t launch_bwd_fwd_state_tc(const void* v, const float* init_state, const int32_t* cu_seqlens, int N,
                                    int64_t T_total, int H, const void* blobs, float* S0s, float* R, float* Vp,
                                    unsigned int* err, cudaStream_t stream);

// The reverse pass on the tensor cores for bf16 dO (dO [T_total, H, 128]); outputs as the CUDA-core pass.
cudaError_t launch_bwd_state_tc(const void* d_o, const float* d_final, const int32_t* cu_seqlens, int N,
                                int64_t T_total, int H, const void* blobs, float* d_init, float* dS_next, float* dZ,
                                unsigned int* err, cudaStream_t stream);

// Per (chunk, head), on the tensor cores for bf16 q, k and dO: the products with S0 and dS_next, dA_qk, dA_kk,
// dv, dgamma and dbeta's first term (outputs as bwd_chunk_a_kernel), then the position-pair sums, dq, dk, dg and
// the two channel halves' parts of dbeta's second term (as bwd_chunk_b_kernel), one CTA per item: XQ, XK, XR
// and dA pass through the workspace but are read back by the CTA that wrote them.
cudaError_t launch_bwd_chunk_ab_tc(const void* q, const void* k, const float* g, const float* beta, const void* d_o,
                                   const int32_t* cu_seqlens, int N, int64_t T_total, int H, float scale,
                                   const float* S0s, const float* dS_next, const float* R, const float* Vp,
                                   const float* dZ, float* XQ, float* XK, float* XR, float* dgam, float* dAqk,
                                   float* dAkk, float* dv, float* dbeta, float* dq, float* dk, float* dg,
                                   float* dbeta_part, unsigned int* err, cudaStream_t stream);

}  // namespace kda
