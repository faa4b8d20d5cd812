// The prefill front end of one warp run: ShortConv(kernel 4) + SiLU on one of q, k, v and, for q
// and k, the L2 norm over the head ("深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA; kernel
// size 4 from "Kimi K3 架构全景", section 02).  Shared by the stand-alone front end
// (kda_frontend.cu) and the fused prefill (kda_chunk_tc.cu), so both compute identical values.
//
// One warp owns one (part, head) and a run of RUN tokens; each lane owns 4 adjacent channels,
// so a token row of the head is one 256-byte coalesced load.  The warp loads its rows and their
// 3-token history up front, computes every token's convolution and SiLU, then reduces all the
// run's squared norms together (the shuffles of different tokens overlap).  A run that crosses a
// sequence start takes a general path that reads the carried state.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace fe {

constexpr int kFeRun = 8;  // tokens per warp run of the fused prefill (8 warps x 8 = one 64-token chunk)

__device__ __forceinline__ float4 bf16x4(uint2 u) {
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

// Largest n with cu[n] <= t < cu[n + 1] (skips empty sequences).
__device__ __forceinline__ int find_seq(const int32_t* cu, int N, int64_t t) {
    int lo = 0, hi = N;  // invariant: cu[lo] <= t, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// SiLU y / (1 + e^-y).  For bf16 outputs as 0.5 y (1 + tanh(y / 2)) with the hardware tanh
// approximation (relative error about 2^-11, under the 2^-9 of the bf16 rounding that follows);
// for fp32 outputs with exp and a divide.
template <typename OutT>
__device__ __forceinline__ float silu(float y) {
    return __fdividef(y, 1.0f + __expf(-y));
}
template <>
__device__ __forceinline__ float silu<__nv_bfloat16>(float y) {
    const float hy = 0.5f * y;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hy));
    return fmaf(hy, t, hy);
}

// y[i][e]: part p (0 q, 1 k, 2 v) of token t0 + i, channel 4 lane + e of head h, after the convolution
// and SiLU; for p < 2, ss[i] = the token's squared norm over the head (the caller scales by
// 1 / sqrt(ss + eps)).  Tokens at or past T_total give zeros.  x: raw rows of part p.
template <typename OutT, int RUN = kFeRun>
__device__ __forceinline__ void frontend_run(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                                             const __nv_bfloat16* __restrict__ conv_w,
                                             const int32_t* __restrict__ cu, int N, int64_t T_total, int H, int p,
                                             int h, int lane, int64_t t0, const __nv_bfloat16* __restrict__ cs_in,
                                             float (&y)[RUN][4], float (&ss)[RUN]) {
    const int64_t C = (int64_t)H * kHeadDim;
    const int64_t ch = (int64_t)h * kHeadDim + 4 * lane;
    const int64_t gc = p * C + ch;
    // raw rows t0 - 3 .. t0 + RUN - 1 (zero outside the tensor), loaded before any arithmetic
    uint2 xr[RUN + 3];
#pragma unroll
    for (int i = 0; i < RUN + 3; ++i) {
        const int64_t s = t0 - 3 + i;
        xr[i] = (s >= 0 && s < T_total) ? *reinterpret_cast<const uint2*>(x + s * x_stride + ch) : make_uint2(0, 0);
    }
    // taps of the lane's 4 channels: w[e][0..3], oldest .. current
    const uint4 w01 = *reinterpret_cast<const uint4*>(conv_w + gc * 4);
    const uint4 w23 = *reinterpret_cast<const uint4*>(conv_w + gc * 4 + 8);
    const uint32_t wr[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    float w[4][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        w[e][0] = bf16_lo(wr[2 * e]); w[e][1] = bf16_hi(wr[2 * e]);
        w[e][2] = bf16_lo(wr[2 * e + 1]); w[e][3] = bf16_hi(wr[2 * e + 1]);
    }

    // Sequence bounds.  Fast path: the run and its 3-token history lie inside one sequence.
    int n = cu ? find_seq(cu, N, t0) : 0;
    int64_t bos = cu ? cu[n] : 0, eos = cu ? cu[n + 1] : T_total;
    const int64_t t_last = (t0 + RUN < T_total ? t0 + RUN : T_total);  // one past the run's last real token
    const bool simple = (t0 - 3 >= bos) && (t_last <= eos);

    if (simple) {
#pragma unroll
        for (int i = 0; i < RUN; ++i) {
            const float4 a0 = bf16x4(xr[i]), a1 = bf16x4(xr[i + 1]), a2 = bf16x4(xr[i + 2]), a3 = bf16x4(xr[i + 3]);
            const float h0[4] = {a0.x, a0.y, a0.z, a0.w}, h1[4] = {a1.x, a1.y, a1.z, a1.w};
            const float h2[4] = {a2.x, a2.y, a2.z, a2.w}, h3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float acc = w[e][0] * h0[e];
                acc = fmaf(w[e][1], h1[e], acc);
                acc = fmaf(w[e][2], h2[e], acc);
                acc = fmaf(w[e][3], h3[e], acc);
                y[i][e] = silu<OutT>(acc);
            }
            ss[i] = y[i][0] * y[i][0] + y[i][1] * y[i][1] + y[i][2] * y[i][2] + y[i][3] * y[i][3];
        }
    } else {
        // general path: a sequence starts inside the window; earlier positions read the carried state (or zero)
#pragma unroll
        for (int i = 0; i < RUN; ++i) {
            const int64_t t = t0 + i;
            if (t < T_total && cu) {
                while ((int64_t)cu[n + 1] <= t) ++n;
                bos = cu[n];
            }
            float hist[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // position t - 3 + j
                const int64_t s2 = t - 3 + j;
                float4 a;
                if (s2 >= bos) {
                    a = bf16x4(xr[i + j]);
                } else {
                    const int64_t back = bos - s2;
                    a = (cs_in && back <= 3)
                            ? bf16x4(*reinterpret_cast<const uint2*>(cs_in + ((int64_t)n * 3 + (3 - back)) * 3 * C + gc))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                hist[j][0] = a.x; hist[j][1] = a.y; hist[j][2] = a.z; hist[j][3] = a.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float acc = w[e][0] * hist[0][e];
                acc = fmaf(w[e][1], hist[1][e], acc);
                acc = fmaf(w[e][2], hist[2][e], acc);
                acc = fmaf(w[e][3], hist[3][e], acc);
                y[i][e] = silu<OutT>(acc);
            }
            ss[i] = y[i][0] * y[i][0] + y[i][1] * y[i][1] + y[i][2] * y[i][2] + y[i][3] * y[i][3];
        }
    }
    // squared norms of q and k over the head: all the run's reductions interleaved
    if (p < 2) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < RUN; ++i) ss[i] += __shfl_xor_sync(0xFFFFFFFFu, ss[i], o);
    }
}

}  // namespace fe
}  // namespace kda
