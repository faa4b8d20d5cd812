// The intra-chunk blocks of the fp32 CUDA-core path, shared by its forward and backward kernels.
//
// For a chunk of kChunk tokens with G the running sum of g (per key channel), every position
// pair (i, j) of the chunk contributes with the decay e^{G_ic - G_jc} of that pair, never a
// positive exponent:
//   A_kk[i][j] = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}   (j < i)
//   A_qk[i][j] =        sum_c q_ic k_jc e^{G_ic - G_jc}   (j <= i)
// ("Kimi-K3 深度解析", section 三, "KDA 的关键改进", unrolled over a chunk.)
#pragma once

#include "kda_common.cuh"

namespace kda {

// sQ, sK, sG: [kChunk][kHeadDim] (q, k and the running sum G; rows past the chunk are zero);
// sB: beta [kChunk].  Writes sAk = A_kk and sAq = A_qk, [kChunk][kChunk], zero above their
// diagonals (either may be in global memory).  256 threads; the first 136 each take one 4 x 4 tile
// of the lower triangle.  kFastExp: the decays by the hardware exponential (__expf, relative error
// of order 1e-6 for these arguments) instead of expf.
template <bool kFastExp = false>
__device__ __forceinline__ void simt_pair_blocks(const float* sQ, const float* sK, const float* sG, const float* sB,
                                                 float* sAk, float* sAq, int tid) {
    constexpr int C = kChunk, D = kHeadDim;
    for (int idx = tid; idx < C * C; idx += 256) {  // zero the strict upper parts
        const int i = idx / C, j = idx % C;
        if ((j >> 2) > (i >> 2)) { sAk[idx] = 0.f; sAq[idx] = 0.f; }
    }
    if (tid < 136) {
        int bi = (int)((sqrtf(8.f * tid + 1.f) - 1.f) * 0.5f);
        while ((bi + 1) * (bi + 2) / 2 <= tid) ++bi;
        while (bi * (bi + 1) / 2 > tid) --bi;
        const int bj = tid - bi * (bi + 1) / 2;
        float akk[4][4] = {}, aqk[4][4] = {};
        for (int cc = 0; cc < D; ++cc) {
            const int c = (cc + tid) & (D - 1);  // rotate so that threads hit different banks
            float gi[4], ki[4], qi[4], gj[4], kj[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                gi[a] = sG[(4 * bi + a) * D + c];
                ki[a] = sK[(4 * bi + a) * D + c];
                qi[a] = sQ[(4 * bi + a) * D + c];
                gj[a] = sG[(4 * bj + a) * D + c];
                kj[a] = sK[(4 * bj + a) * D + c];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const float x = fminf(gi[a] - gj[b], 0.f);
                    const float e = kFastExp ? __expf(x) : expf(x);
                    akk[a][b] = fmaf(ki[a] * kj[b], e, akk[a][b]);
                    aqk[a][b] = fmaf(qi[a] * kj[b], e, aqk[a][b]);
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int i = 4 * bi + a, j = 4 * bj + b;
                sAk[i * C + j] = j < i ? sB[i] * akk[a][b] : 0.f;
                sAq[i * C + j] = j <= i ? aqk[a][b] : 0.f;
            }
    }
}

}  // namespace kda
