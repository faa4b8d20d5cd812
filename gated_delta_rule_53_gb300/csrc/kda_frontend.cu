// kda_shortconv_l2norm: the prefill front end, as a pass of its own (the per-run arithmetic is in
// kda_frontend.cuh, shared with the fused prefill).  Memory-bound elementwise work: every raw
// element is read once and every output written once.  A second small kernel writes the carried
// convolution state (last three raw inputs per sequence) after the first has finished reading the
// incoming one, so the two buffers may alias.
#include "kda_frontend.cuh"

namespace kda {
namespace {

constexpr int kRun = 8;     // tokens per warp
constexpr int kWarps = 1;   // one warp per CTA: 32 CTAs per SM schedule independently

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
__global__ void __launch_bounds__(kWarps * 32, 32)
shortconv_kernel(const __nv_bfloat16* __restrict__ xq, const __nv_bfloat16* __restrict__ xk,
                 const __nv_bfloat16* __restrict__ xv, int64_t x_stride,
                 const __nv_bfloat16* __restrict__ conv_w, const int32_t* __restrict__ cu, int N,
                 int64_t T_total, int H, const __nv_bfloat16* __restrict__ cs_in, float eps,
                 OutT* __restrict__ q_out, OutT* __restrict__ k_out, OutT* __restrict__ v_out, int p0) {
    const int p = p0 + (int)blockIdx.z, h = blockIdx.y;  // parts p0 .. p0 + gridDim.z - 1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * kRun;
    if (t0 >= T_total) return;
    const __nv_bfloat16* x = p == 0 ? xq : (p == 1 ? xk : xv);
    OutT* out = p == 0 ? q_out : (p == 1 ? k_out : v_out);
    float y[kRun][4], inv[kRun];
    fe::frontend_run<OutT, kRun>(x, x_stride, conv_w, cu, N, T_total, H, p, h, lane, t0, cs_in, eps, y, inv);
#pragma unroll
    for (int i = 0; i < kRun; ++i) {
        const int64_t t = t0 + i;
        if (t < T_total) {
            store4<OutT>(out + (t * H + h) * kHeadDim + 4 * lane, y[i][0] * inv[i], y[i][1] * inv[i],
                         y[i][2] * inv[i], y[i][3] * inv[i]);
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
                static_cast<__nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(v), 0);
        else
            shortconv_kernel<float><<<grid, kWarps * 32, 0, stream>>>(
                bq, bk, bv, x_stride, w, cu_seqlens, N, T_total, H, cs_in, eps, static_cast<float*>(q),
                static_cast<float*>(k), static_cast<float*>(v), 0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (conv_state_out)
        return launch_conv_state_out(xq, xk, xv, x_stride, cu_seqlens, N, T_total, H, conv_state_in, conv_state_out,
                                     stream);
    return cudaSuccess;
}

// v alone (bf16), for the fused prefill, which computes q and k inside its chunk pass.
cudaError_t launch_frontend_v(const void* xv, int64_t x_stride, const void* conv_w, const int32_t* cu_seqlens, int N,
                              int64_t T_total, int H, const void* conv_state_in, void* v, cudaStream_t stream) {
    if (T_total <= 0) return cudaSuccess;
    const int64_t per_cta = (int64_t)kWarps * kRun;
    dim3 grid((unsigned)((T_total + per_cta - 1) / per_cta), (unsigned)H, 1);
    const auto* bv = static_cast<const __nv_bfloat16*>(xv);
    shortconv_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, stream>>>(
        bv, bv, bv, x_stride, static_cast<const __nv_bfloat16*>(conv_w), cu_seqlens, N, T_total, H,
        static_cast<const __nv_bfloat16*>(conv_state_in), 0.f, nullptr, nullptr, static_cast<__nv_bfloat16*>(v), 2);
    return cudaGetLastError();
}

cudaError_t launch_conv_state_out(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                  const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                                  const void* conv_state_in, void* conv_state_out, cudaStream_t stream) {
    const int64_t C3 = 3 * (int64_t)H * kHeadDim;
    dim3 grid((unsigned)((C3 + 255) / 256), (unsigned)N);
    conv_state_out_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(xq), static_cast<const __nv_bfloat16*>(xk),
        static_cast<const __nv_bfloat16*>(xv), x_stride, cu_seqlens, T_total, H,
        static_cast<const __nv_bfloat16*>(conv_state_in), static_cast<__nv_bfloat16*>(conv_state_out));
    return cudaGetLastError();
}

}  // namespace kda
