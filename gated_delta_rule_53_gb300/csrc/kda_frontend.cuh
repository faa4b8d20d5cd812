// The prefill front end of one warp run: ShortConv(kernel 4) + SiLU on one of q, k, v and, for q
// and k, the L2 norm over the head ("深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA; kernel
// size 4 from "Kimi K3 架构全景", section 02).  Shared by the stand-alone front end
// (kda_frontend.cu) and the fused prefill (kda_chunk_tc.cu), so both compute identical values.
//
// One warp owns one (part, head) and a run of RUN tokens; each lane owns 4 adjacent channels,
// so a token row of the head is one 256-byte coalesced load.  The warp loads its rows and their
// 3-token history up front, computes every token's convolution and SiLU (two channels per packed
// fp32 instruction), then reduces all the run's squared norms together.  A run that crosses a
// sequence start takes a general path that reads the carried state.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace fe {

constexpr int kFeRun = 8;  // tokens per warp run of the fused prefill (8 warps x 8 = one 64-token chunk)

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

// Two adjacent channels as a float2, computed with the packed fp32 instructions of sm_100 and later: one
// instruction for both, each half rounded exactly as the scalar multiply or fma.
__device__ __forceinline__ float2 bf16x2f(uint32_t u) { return make_float2(bf16_lo(u), bf16_hi(u)); }

// ShortConv of a channel pair over the window h0 (oldest) .. h3 (current): w0 h0 + w1 h1 + w2 h2 + w3 h3,
// accumulated in that order.
__device__ __forceinline__ float2 conv4(const float2 (&w)[4], float2 h0, float2 h1, float2 h2, float2 h3) {
    float2 acc = __fmul2_rn(w[0], h0);
    acc = __ffma2_rn(w[1], h1, acc);
    acc = __ffma2_rn(w[2], h2, acc);
    return __ffma2_rn(w[3], h3, acc);
}

template <typename OutT>
__device__ __forceinline__ float2 silu2(float2 y) {
    return make_float2(silu<OutT>(y.x), silu<OutT>(y.y));
}
template <>
__device__ __forceinline__ float2 silu2<__nv_bfloat16>(float2 y) {
    const float2 hy = __fmul2_rn(y, make_float2(0.5f, 0.5f));
    float tx, ty;
    asm("tanh.approx.f32 %0, %1;" : "=f"(tx) : "f"(hy.x));
    asm("tanh.approx.f32 %0, %1;" : "=f"(ty) : "f"(hy.y));
    return __ffma2_rn(hy, make_float2(tx, ty), hy);
}

// Squared norm of a lane's four channels (y0, y1) and (y2, y3): (y0^2 + y2^2) + (y1^2 + y3^2).
__device__ __forceinline__ float sq4(float2 a, float2 b) {
    const float2 s = __ffma2_rn(b, b, __fmul2_rn(a, a));
    return s.x + s.y;
}

// y[i][e]: part p (0 q, 1 k, 2 v) of token t0 + i, channel 4 lane + e of head h, after the convolution
// and SiLU; inv[i]: for p < 2, 1 / sqrt(the token's squared norm over the head + eps), the factor the
// caller scales y by (1 for p = 2).  Tokens at or past T_total give zeros.  x: raw rows of part p.
template <typename OutT, int RUN = kFeRun>
__device__ __forceinline__ void frontend_run(const __nv_bfloat16* __restrict__ x, int64_t x_stride,
                                             const __nv_bfloat16* __restrict__ conv_w,
                                             const int32_t* __restrict__ cu, int N, int64_t T_total, int H, int p,
                                             int h, int lane, int64_t t0, const __nv_bfloat16* __restrict__ cs_in,
                                             float eps, float (&y)[RUN][4], float (&inv)[RUN]) {
    const int64_t C = (int64_t)H * kHeadDim;
    const int64_t ch = (int64_t)h * kHeadDim + 4 * lane;
    const int64_t gc = p * C + ch;
    // raw rows t0 - 3 .. t0 + RUN - 1 (zero outside the tensor), loaded before any arithmetic
    uint2 xr[RUN + 3];
    if (t0 >= 3 && t0 + RUN <= T_total) {  // the whole window inside the tensor (the warp agrees)
        const __nv_bfloat16* xp = x + (t0 - 3) * x_stride + ch;
#pragma unroll
        for (int i = 0; i < RUN + 3; ++i) xr[i] = *reinterpret_cast<const uint2*>(xp + i * x_stride);
    } else {
#pragma unroll
        for (int i = 0; i < RUN + 3; ++i) {
            const int64_t s = t0 - 3 + i;
            xr[i] = (s >= 0 && s < T_total) ? *reinterpret_cast<const uint2*>(x + s * x_stride + ch) : make_uint2(0, 0);
        }
    }
    // taps of the lane's 4 channels: w[e][0..3], oldest .. current
    const uint4 w01 = *reinterpret_cast<const uint4*>(conv_w + gc * 4);
    const uint4 w23 = *reinterpret_cast<const uint4*>(conv_w + gc * 4 + 8);
    const uint32_t wr[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
    // as channel pairs: wp[c][j] = tap j of channels 2c and 2c + 1
    float2 wp[2][4];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        wp[c][0] = make_float2(bf16_lo(wr[4 * c]), bf16_lo(wr[4 * c + 2]));
        wp[c][1] = make_float2(bf16_hi(wr[4 * c]), bf16_hi(wr[4 * c + 2]));
        wp[c][2] = make_float2(bf16_lo(wr[4 * c + 1]), bf16_lo(wr[4 * c + 3]));
        wp[c][3] = make_float2(bf16_hi(wr[4 * c + 1]), bf16_hi(wr[4 * c + 3]));
    }

    float ss[RUN];  // squared norms over the lane's channels, then over the head
    // Sequence bounds.  Fast path: the run and its 3-token history lie inside one sequence.
    int n = cu ? find_seq(cu, N, t0) : 0;
    int64_t bos = cu ? cu[n] : 0, eos = cu ? cu[n + 1] : T_total;
    const int64_t t_last = (t0 + RUN < T_total ? t0 + RUN : T_total);  // one past the run's last real token
    const bool simple = (t0 - 3 >= bos) && (t_last <= eos);

    if (simple) {
#pragma unroll
        for (int i = 0; i < RUN; ++i) {
            const float2 y01 = silu2<OutT>(conv4(wp[0], bf16x2f(xr[i].x), bf16x2f(xr[i + 1].x), bf16x2f(xr[i + 2].x),
                                                 bf16x2f(xr[i + 3].x)));
            const float2 y23 = silu2<OutT>(conv4(wp[1], bf16x2f(xr[i].y), bf16x2f(xr[i + 1].y), bf16x2f(xr[i + 2].y),
                                                 bf16x2f(xr[i + 3].y)));
            y[i][0] = y01.x; y[i][1] = y01.y; y[i][2] = y23.x; y[i][3] = y23.y;
            ss[i] = p < 2 ? sq4(y01, y23) : 0.f;
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
            uint2 hist[4];  // position t - 3 + j, raw bf16
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t s2 = t - 3 + j;
                if (s2 >= bos) {
                    hist[j] = xr[i + j];
                } else {
                    const int64_t back = bos - s2;
                    hist[j] = (cs_in && back <= 3)
                                  ? *reinterpret_cast<const uint2*>(cs_in + ((int64_t)n * 3 + (3 - back)) * 3 * C + gc)
                                  : make_uint2(0, 0);
                }
            }
            // the same arithmetic as the fast path
            const float2 y01 = silu2<OutT>(conv4(wp[0], bf16x2f(hist[0].x), bf16x2f(hist[1].x), bf16x2f(hist[2].x),
                                                 bf16x2f(hist[3].x)));
            const float2 y23 = silu2<OutT>(conv4(wp[1], bf16x2f(hist[0].y), bf16x2f(hist[1].y), bf16x2f(hist[2].y),
                                                 bf16x2f(hist[3].y)));
            y[i][0] = y01.x; y[i][1] = y01.y; y[i][2] = y23.x; y[i][3] = y23.y;
            ss[i] = p < 2 ? sq4(y01, y23) : 0.f;
        }
    }
    // squared norms of q and k over the head (the sum over the 32 lanes), and the scale factors
#pragma unroll
    for (int i = 0; i < RUN; ++i) inv[i] = 1.0f;
    if (p < 2) {
        if constexpr (RUN == 8) {
            // Reduce-scatter: in each of the first three steps a lane keeps half of its tokens and adds its
            // partner's partial sums of them, so that lane L ends with token 4 b4 + 2 b3 + b2 (bits of L); two
            // more steps finish that sum, then every lane reads each token's total from a lane holding it.  The
            // additions pair lanes in the order of a plain xor-shuffle reduction (16, 8, 4, 2, 1), with the
            // lane's own partial sum first, so every lane gets the bits that reduction would give; the lanes
            // holding a token's total take its reciprocal square root, which the others then read.
            constexpr unsigned kAll = 0xFFFFFFFFu;
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float r4[4], r2[2];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float keep = b4 ? ss[4 + j] : ss[j], send = b4 ? ss[j] : ss[4 + j];
                r4[j] = keep + __shfl_xor_sync(kAll, send, 16);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float keep = b3 ? r4[2 + j] : r4[j], send = b3 ? r4[j] : r4[2 + j];
                r2[j] = keep + __shfl_xor_sync(kAll, send, 8);
            }
            float r = (b2 ? r2[1] : r2[0]) + __shfl_xor_sync(kAll, b2 ? r2[0] : r2[1], 4);
            r += __shfl_xor_sync(kAll, r, 2);
            r += __shfl_xor_sync(kAll, r, 1);
            const float ri = rsqrtf(r + eps);
#pragma unroll
            for (int i = 0; i < 8; ++i) inv[i] = __shfl_sync(kAll, ri, ((i & 4) << 2) | ((i & 2) << 2) | ((i & 1) << 2));
        } else {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int i = 0; i < RUN; ++i) ss[i] += __shfl_xor_sync(0xFFFFFFFFu, ss[i], o);
#pragma unroll
            for (int i = 0; i < RUN; ++i) inv[i] = rsqrtf(ss[i] + eps);
        }
    }
}

}  // namespace fe
}  // namespace kda
