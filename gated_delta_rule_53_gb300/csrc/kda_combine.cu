// kda_state_combine: S_out = S_in M + E for a batch of 128 x 128 fp32 matrices.
//
// Carrying a state across segments of one sequence ("Kimi K3 架构全景", section 02: the
// chunk_kda operator over long contexts; the state update of "Kimi-K3 深度解析", section 三,
// "KDA 的关键改进"): the update S_t = S_{t-1} Diag(alpha_t)(I - beta_t k_t k_t^T) + beta_t v_t k_t^T
// is affine in S_{t-1}, so a segment maps its entering state S to S M + E, with M the product of
// its per-token operators and E its end state from zero.  This kernel applies that map.
//
// One CTA per matrix, 256 threads, each an 8 x 8 tile of the output; both operands are staged in
// shared memory (rows padded to 132 floats) before any output is written, so S_out may alias any
// input.  fp32 throughout, k summed in order.
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kCombThreads = 256;
constexpr int kCombLd = 132;  // padded row stride, in floats
constexpr size_t kCombSmem = (size_t)2 * 128 * kCombLd * sizeof(float);

__global__ void __launch_bounds__(kCombThreads) state_combine_kernel(const float* S_in, const float* M,
                                                                     const float* E, float* S_out) {
    extern __shared__ float sh[];
    const int64_t base = (int64_t)blockIdx.x * 128 * 128;
    const int tid = threadIdx.x;
    if (!S_in) {  // no entering state: the map gives E
        for (int idx = tid; idx < 128 * 32; idx += kCombThreads)
            reinterpret_cast<float4*>(S_out + base)[idx] = reinterpret_cast<const float4*>(E + base)[idx];
        return;
    }
    float* A = sh;
    float* B = sh + 128 * kCombLd;
    for (int idx = tid; idx < 128 * 32; idx += kCombThreads) {
        const int r = idx >> 5, c4 = idx & 31;
        *reinterpret_cast<float4*>(A + r * kCombLd + 4 * c4) =
            *reinterpret_cast<const float4*>(S_in + base + r * 128 + 4 * c4);
        *reinterpret_cast<float4*>(B + r * kCombLd + 4 * c4) =
            *reinterpret_cast<const float4*>(M + base + r * 128 + 4 * c4);
    }
    __syncthreads();
    const int ty = tid >> 4, tx = tid & 15;  // rows 8 ty .. +7, columns 8 tx .. +7
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;
#pragma unroll 1
    for (int k = 0; k < 128; k += 4) {
        float a[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r)
            *reinterpret_cast<float4*>(a[r]) = *reinterpret_cast<const float4*>(A + (8 * ty + r) * kCombLd + k);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float b[8];
            *reinterpret_cast<float4*>(b) = *reinterpret_cast<const float4*>(B + (k + kk) * kCombLd + 8 * tx);
            *reinterpret_cast<float4*>(b + 4) = *reinterpret_cast<const float4*>(B + (k + kk) * kCombLd + 8 * tx + 4);
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[r][c] = fmaf(a[r][kk], b[c], acc[r][c]);
        }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int64_t at = base + (int64_t)(8 * ty + r) * 128 + 8 * tx;
        const float4 e0 = *reinterpret_cast<const float4*>(E + at);
        const float4 e1 = *reinterpret_cast<const float4*>(E + at + 4);
        *reinterpret_cast<float4*>(S_out + at) =
            make_float4(acc[r][0] + e0.x, acc[r][1] + e0.y, acc[r][2] + e0.z, acc[r][3] + e0.w);
        *reinterpret_cast<float4*>(S_out + at + 4) =
            make_float4(acc[r][4] + e1.x, acc[r][5] + e1.y, acc[r][6] + e1.z, acc[r][7] + e1.w);
    }
}

}  // namespace

cudaError_t launch_state_combine(const float* S_in, const float* M, const float* E, float* S_out, int64_t count,
                                 cudaStream_t stream) {
    if (count <= 0) return cudaSuccess;
    if (count > 0x7FFFFFFF) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(state_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kCombSmem);
    if (e != cudaSuccess) return e;
    state_combine_kernel<<<(unsigned)count, kCombThreads, S_in ? kCombSmem : 0, stream>>>(S_in, M, E, S_out);
    return cudaGetLastError();
}

}  // namespace kda
