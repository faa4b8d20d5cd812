// kda_shortconv_l2norm: the prefill front end.  ShortConv(kernel 4) + SiLU on
// each of q, k, v and the L2 norm of q and k over each head ("深入 Kimi-K3:
// Hugging Face 仓库分析", paragraph on KDA; kernel size 4 from "Kimi K3 架构全景",
// section 02).
//
// Memory-bound elementwise work: every raw element is read once and every
// output written once.  One warp owns one (part, head) and a run of 8 tokens;
// each lane owns 4 adjacent channels, so a token row of the head is one 256-byte
// coalesced load.  The warp loads its 8 rows and their 3-token history up front,
// computes every token's convolution and SiLU, then reduces all the run's squared
// norms of q / k together (the shuffles of different tokens overlap).  A run that
// crosses a sequence start takes a general path that reads the carried state.  A second small kernel writes the carried
// convolution state (last three raw inputs per sequence) after the first has
// finished reading the incoming one, so the two buffers may alias.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kRun = 8;           // tokens per warp
constexpr int kWarps = 8;         // warps per CTA (64 tokens of one part and head); 4 CTAs per SM

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

template <typename OutT>
__device__ __forceinline__ void store4(OutT* p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float a, float b, float c, float d) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(a, b), pack_bf16x2(c, d));
}

template <typename OutT>
__global__ void __launch_bounds__(kWarps * 32, 4)
shortconv_kernel(const __nv_bfloat16* __restrict__ xq, const __nv_bfloat16* __restrict__ xk,
                 const __nv_bfloat16* __restrict__ xv, int64_t x_stride,
                 const __nv_bfloat16* __restrict__ conv_w, const int32_t* __restrict__ cu, int N,
                 int64_t T_total, int H, const __nv_bfloat16* __restrict__ cs_in, float eps,
                 OutT* __restrict__ q_out, OutT* __restrict__ k_out, OutT* __restrict__ v_out) {
    const int p = blockIdx.z, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * kRun;
    if (t0 >= T_total) return;
    const int64_t C = (int64_t)H * kHeadDim;
    const int64_t ch = (int64_t)h * kHeadDim + 4 * lane;
    const int64_t gc = p * C + ch;
    const __nv_bfloat16* x = p == 0 ? xq : (p == 1 ? xk : xv);
    OutT* out = p == 0 ? q_out : (p == 1 ? k_out : v_out);

    // raw rows t0 - 3 .. t0 + kRun - 1 (zero outside the tensor), loaded before any arithmetic
    uint2 xr[kRun + 3];
#pragma unroll
    for (int i = 0; i < kRun + 3; ++i) {
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
    const int64_t t_last = (t0 + kRun < T_total ? t0 + kRun : T_total);  // one past the run's last real token
    const bool simple = (t0 - 3 >= bos) && (t_last <= eos);

    float y[kRun][4];
    float ss[kRun];
    if (simple) {
#pragma unroll
        for (int i = 0; i < kRun; ++i) {
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
        for (int i = 0; i < kRun; ++i) {
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
    // L2 norms of q and k: all the run's reductions interleaved
    if (p < 2) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < kRun; ++i) ss[i] += __shfl_xor_sync(0xFFFFFFFFu, ss[i], o);
    }
#pragma unroll
    for (int i = 0; i < kRun; ++i) {
        const int64_t t = t0 + i;
        if (t < T_total) {
            const float inv = p < 2 ? rsqrtf(ss[i] + eps) : 1.0f;
            store4<OutT>(out + (t * H + h) * kHeadDim + 4 * lane, y[i][0] * inv, y[i][1] * inv, y[i][2] * inv,
                         y[i][3] * inv);
        }
    }
}

// conv_state_out[n][r][gc] = raw input at position eos - 3 + r of sequence n.
__global__ void conv_state_out_kernel(const __nv_bfloat16* __restrict__ xq, const __nv_bfloat16* __restrict__ xk,
                                      const __nv_bfloat16* __restrict__ xv, int64_t x_stride,
                                      const int32_t* __restrict__ cu, int64_t T_total, int H,
                                      const __nv_bfloat16* cs_in, __nv_bfloat16* cs_out) {
    const int n = blockIdx.y;
    const int64_t C = (int64_t)H * kHeadDim;
    const int64_t gc = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gc >= 3 * C) return;
    const int p = (int)(gc / C);
    const int64_t ch = gc - p * C;
    const __nv_bfloat16* x = p == 0 ? xq : (p == 1 ? xk : xv);
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    __nv_bfloat16 val[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const int64_t s = eos - 3 + r;
        if (s >= bos) {
            val[r] = x[s * x_stride + ch];
        } else {
            const int64_t back = bos - s;
            val[r] = (cs_in && back <= 3) ? cs_in[((int64_t)n * 3 + (3 - back)) * 3 * C + gc] : __float2bfloat16_rn(0.f);
        }
    }
#pragma unroll
    for (int r = 0; r < 3; ++r) cs_out[((int64_t)n * 3 + r) * 3 * C + gc] = val[r];
}

}  // namespace

cudaError_t launch_shortconv_l2norm(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                    const void* conv_w, const int32_t* cu_seqlens, int N, int64_t T_total,
                                    int H, const void* conv_state_in, void* conv_state_out, float eps,
                                    kda_dtype out_dtype, void* q, void* k, void* v, cudaStream_t stream) {
    const auto* bq = static_cast<const __nv_bfloat16*>(xq);
    const auto* bk = static_cast<const __nv_bfloat16*>(xk);
    const auto* bv = static_cast<const __nv_bfloat16*>(xv);
    const auto* w = static_cast<const __nv_bfloat16*>(conv_w);
    const auto* cs_in = static_cast<const __nv_bfloat16*>(conv_state_in);
    if (T_total > 0) {
        const int64_t per_cta = (int64_t)kWarps * kRun;
        dim3 grid((unsigned)((T_total + per_cta - 1) / per_cta), (unsigned)H, 3);
        if (out_dtype == KDA_DTYPE_BF16)
            shortconv_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
                bq, bk, bv, x_stride, w, cu_seqlens, N, T_total, H, cs_in, eps, static_cast<__nv_bfloat16*>(q),
                static_cast<__nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(v));
        else
            shortconv_kernel<float><<<grid, kWarps * 32, 0, stream>>>(
                bq, bk, bv, x_stride, w, cu_seqlens, N, T_total, H, cs_in, eps, static_cast<float*>(q),
                static_cast<float*>(k), static_cast<float*>(v));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (conv_state_out) {
        const int64_t C3 = 3 * (int64_t)H * kHeadDim;
        dim3 grid((unsigned)((C3 + 255) / 256), (unsigned)N);
        conv_state_out_kernel<<<grid, 256, 0, stream>>>(bq, bk, bv, x_stride, cu_seqlens, T_total, H, cs_in,
                                                        static_cast<__nv_bfloat16*>(conv_state_out));
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace kda
