// kda_recurrent_step: one fused decode step (the fused_recurrent_kda operator of
// "Kimi K3 架构全景", section 02) for N sequences of one token each.
//
// Four CTAs of 4 warps per (sequence, head), 32 state rows each (eight such CTAs per SM).  Every CTA
// runs the front end of its head on the token (warps 0-2: ShortConv(4) + SiLU for q, k and v, L2 norm
// of q and k by warp shuffles, "深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA; warp 3:
// alpha = exp(g)) -- a few hundred values, recomputed rather than shared -- while the 128-bit loads
// of its 32 state rows are already in flight.  Then each row r of S (dv x dk) is updated on its own
// ("Kimi-K3 深度解析", section 三, "KDA 的关键改进"):
//     s~ = s * alpha;  p = s~ . k;  s = s~ + beta (v_r - p) k;  o_r = scale s . q
// with both dot products reduced by warp shuffles, and written back in place.  The convolution
// state is shifted by a second small kernel once every CTA has read it.  The step streams the state
// once in and once out: it is bound by HBM.  g outside [-5, 0] or beta outside [0, 1] sets a bit of
// the device error word (the update itself needs neither bound).
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kParts = 4;      // CTAs per (sequence, head)
constexpr int kRowsPerWarp = 8;

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 u) {
    return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}

__global__ void __launch_bounds__(kThreads, 8)
recurrent_step_kernel(const __nv_bfloat16* __restrict__ xq, const __nv_bfloat16* __restrict__ xk,
                      const __nv_bfloat16* __restrict__ xv, int64_t x_stride,
                      const __nv_bfloat16* __restrict__ conv_w, const float* __restrict__ g,
                      const float* __restrict__ beta, float* __restrict__ state,
                      __nv_bfloat16* __restrict__ conv_state, int H, float scale, float eps,
                      __nv_bfloat16* __restrict__ o, unsigned int* err) {
    __shared__ float4 s_q[32], s_k[32], s_v[32], s_alpha[32];
    __shared__ float s_beta;

    const int nh = blockIdx.x / kParts, pt = blockIdx.x % kParts;
    const int n = nh / H, h = nh % H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t C = (int64_t)H * kHeadDim;

    // 1. state rows of this warp: issue all loads first (streamed, read once).
    float* S = state + (int64_t)nh * kHeadDim * kHeadDim;
    float4 s[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = (pt * (kThreads / 32) + warp) * kRowsPerWarp + i;
        s[i] = __ldcs(reinterpret_cast<const float4*>(S + r * kHeadDim) + lane);
    }

    // 2. front end (warps 0..2) and decay (warp 3), for the whole head in every CTA.
    if (warp < 3) {
        const int p = warp;
        const __nv_bfloat16* x = p == 0 ? xq : (p == 1 ? xk : xv);
        const int64_t ch = (int64_t)h * kHeadDim + 4 * lane;  // channel within the part
        const int64_t gc = p * C + ch;                        // channel within q|k|v
        __nv_bfloat16* cs = conv_state + (int64_t)n * 3 * 3 * C;
        const uint2 old0 = *reinterpret_cast<const uint2*>(cs + gc);
        const uint2 old1 = *reinterpret_cast<const uint2*>(cs + 3 * C + gc);
        const uint2 old2 = *reinterpret_cast<const uint2*>(cs + 6 * C + gc);
        const uint2 xt = *reinterpret_cast<const uint2*>(x + (int64_t)n * x_stride + ch);
        const uint4 w01 = *reinterpret_cast<const uint4*>(conv_w + gc * 4);      // channels 0, 1
        const uint4 w23 = *reinterpret_cast<const uint4*>(conv_w + gc * 4 + 8);  // channels 2, 3
        const float4 a0 = bf16x4_to_f4(old0), a1 = bf16x4_to_f4(old1), a2 = bf16x4_to_f4(old2);
        const float4 a3 = bf16x4_to_f4(xt);
        // taps of channel e: w[e][0..3] (oldest .. current)
        const uint32_t wr[8] = {w01.x, w01.y, w01.z, w01.w, w23.x, w23.y, w23.z, w23.w};
        float y[4];
        const float h0[4] = {a0.x, a0.y, a0.z, a0.w}, h1[4] = {a1.x, a1.y, a1.z, a1.w};
        const float h2[4] = {a2.x, a2.y, a2.z, a2.w}, h3[4] = {a3.x, a3.y, a3.z, a3.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float w0 = bf16_lo(wr[2 * e]), w1 = bf16_hi(wr[2 * e]);
            const float w2 = bf16_lo(wr[2 * e + 1]), w3 = bf16_hi(wr[2 * e + 1]);
            float acc = w0 * h0[e];
            acc = fmaf(w1, h1[e], acc);
            acc = fmaf(w2, h2[e], acc);
            acc = fmaf(w3, h3[e], acc);
            y[e] = acc / (1.0f + expf(-acc));  // SiLU
        }
        float inv = 1.0f;
        if (p < 2) {
            const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
            inv = 1.0f / sqrtf(ss + eps);
        }
        float4* dst = p == 0 ? s_q : (p == 1 ? s_k : s_v);
        dst[lane] = make_float4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);

    } else if (warp == 3) {
        const float4 gv = *(reinterpret_cast<const float4*>(g + (int64_t)nh * kHeadDim) + lane);
        s_alpha[lane] = make_float4(expf(gv.x), expf(gv.y), expf(gv.z), expf(gv.w));
        const float bv = beta[nh];
        if (lane == 0) s_beta = bv;
        if (pt == 0) {  // inputs in the ranges of the pages (g in [-5, 0], beta in [0, 1]), once per head
            const float lo = fminf(fminf(gv.x, gv.y), fminf(gv.z, gv.w));
            const float hi = fmaxf(fmaxf(gv.x, gv.y), fmaxf(gv.z, gv.w));
            const float sum = gv.x + gv.y + gv.z + gv.w;  // NaN-propagating
            if (__any_sync(0xFFFFFFFFu, !(lo >= -5.f && hi <= 0.f && sum == sum)) && lane == 0)
                raise_device_error(err, kErrGateRange);
            if (lane == 0 && !(bv >= 0.f && bv <= 1.f)) raise_device_error(err, kErrBetaRange);
        }
    }
    __syncthreads();

    // 3. the recurrence, one state row per (warp, i).
    const float4 kv = s_k[lane], qv = s_q[lane], av = s_alpha[lane];
    const float b = s_beta;
    const float* vrow = reinterpret_cast<const float*>(s_v);
    float part[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        s[i].x *= av.x; s[i].y *= av.y; s[i].z *= av.z; s[i].w *= av.w;
        part[i] = s[i].x * kv.x + s[i].y * kv.y + s[i].z * kv.z + s[i].w * kv.w;
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) part[i] = warp_sum(part[i]);
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = (pt * (kThreads / 32) + warp) * kRowsPerWarp + i;
        const float e = b * (vrow[r] - part[i]);
        s[i].x = fmaf(e, kv.x, s[i].x); s[i].y = fmaf(e, kv.y, s[i].y);
        s[i].z = fmaf(e, kv.z, s[i].z); s[i].w = fmaf(e, kv.w, s[i].w);
        __stcs(reinterpret_cast<float4*>(S + r * kHeadDim) + lane, s[i]);
        part[i] = s[i].x * qv.x + s[i].y * qv.y + s[i].z * qv.z + s[i].w * qv.w;
    }
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) part[i] = warp_sum(part[i]);
    __nv_bfloat16* orow = o + (int64_t)nh * kHeadDim + (pt * (kThreads / 32) + warp) * kRowsPerWarp;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i)
        if (lane == i) orow[i] = __float2bfloat16_rn(scale * part[i]);
}

// conv_state[n]: rows 1, 2 move up, the raw token enters as row 2 (after recurrent_step_kernel has read it).
__global__ void conv_shift_kernel(const __nv_bfloat16* __restrict__ xq, const __nv_bfloat16* __restrict__ xk,
                                  const __nv_bfloat16* __restrict__ xv, int64_t x_stride,
                                  __nv_bfloat16* __restrict__ conv_state, int H) {
    const int n = blockIdx.y;
    const int64_t C = (int64_t)H * kHeadDim;
    const int64_t q4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // 4-channel group within q|k|v
    if (q4 * 4 >= 3 * C) return;
    const int64_t gc = q4 * 4;
    const int p = (int)(gc / C);
    const int64_t ch = gc - p * C;
    const __nv_bfloat16* x = p == 0 ? xq : (p == 1 ? xk : xv);
    __nv_bfloat16* cs = conv_state + (int64_t)n * 3 * 3 * C;
    const uint2 old1 = *reinterpret_cast<const uint2*>(cs + 3 * C + gc);
    const uint2 old2 = *reinterpret_cast<const uint2*>(cs + 6 * C + gc);
    const uint2 xt = *reinterpret_cast<const uint2*>(x + (int64_t)n * x_stride + ch);
    *reinterpret_cast<uint2*>(cs + gc) = old1;
    *reinterpret_cast<uint2*>(cs + 3 * C + gc) = old2;
    *reinterpret_cast<uint2*>(cs + 6 * C + gc) = xt;
}

}  // namespace

cudaError_t launch_recurrent_step(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                  const void* conv_w, const float* g, const float* beta, float* state,
                                  void* conv_state, int N, int H, float scale, float eps, void* o,
                                  unsigned int* err, cudaStream_t stream) {
    const int64_t blocks = (int64_t)N * H;
    if (blocks == 0) return cudaSuccess;
    if (blocks * kParts > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    recurrent_step_kernel<<<(unsigned)(blocks * kParts), kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(xq), static_cast<const __nv_bfloat16*>(xk),
        static_cast<const __nv_bfloat16*>(xv), x_stride, static_cast<const __nv_bfloat16*>(conv_w), g, beta, state,
        static_cast<__nv_bfloat16*>(conv_state), H, scale, eps, static_cast<__nv_bfloat16*>(o), err);
    const int64_t groups = 3 * (int64_t)H * kHeadDim / 4;
    conv_shift_kernel<<<dim3((unsigned)((groups + 255) / 256), (unsigned)N), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(xq), static_cast<const __nv_bfloat16*>(xk),
        static_cast<const __nv_bfloat16*>(xv), x_stride, static_cast<__nv_bfloat16*>(conv_state), H);
    return cudaGetLastError();
}

}  // namespace kda
