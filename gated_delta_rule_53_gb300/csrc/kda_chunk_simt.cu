// kda_chunk_fwd, fp32 path: chunkwise prefill in fp32 on the CUDA cores.
//
// The chunk form of the recurrence ("Kimi-K3 深度解析", section 三, subsection
// "KDA 的关键改进", unrolled over a chunk of C = 64 tokens; the chunk_kda operator
// of "Kimi K3 架构全景", section 02).  With G_t the running sum of g inside the
// chunk (per key channel), S0 the state entering the chunk and Gamma = e^G:
//   A_kk[i][j] = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}      (j < i)
//   A_qk[i][j] =        sum_c q_ic k_jc e^{G_ic - G_jc}      (j <= i)
//   Z  = diag(beta) (V - (K . Gamma) S0^T)
//   U  = (I + A_kk)^{-1} Z                                    (forward substitution)
//   O  = scale ((Q . Gamma) S0^T + A_qk U)
//   S  = S0 Diag(e^{G_C}) + U^T (K . e^{G_C - G})
// This path evaluates every decay factor e^{G_ic - G_jc} of a position pair
// directly (the exponent is never positive), so it is exact to fp32 rounding
// for any g <= 0 and does not rely on the -5 bound.  It is the path for fp32
// inputs and a second, independent GPU form for the bf16 tensor-core path.
//
// Grid: one CTA per (sequence, head, slice of 32 value rows); the CTA walks its
// sequence chunk by chunk with its state slice S[r0:r0+32, :] in shared memory
// (stored transposed so that a warp's lanes read consecutive words).  The key
// side (A_kk, A_qk) is recomputed by each of the 4 slices of a head.
#include "kda_common.cuh"
#include "kda_simt_blocks.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kSlice = 32;       // value rows per CTA
constexpr int kUStride = 36;     // row stride of U: 4*row + col hits distinct banks in the solve
constexpr int kC = kChunk;       // 64
constexpr int kD = kHeadDim;     // 128

constexpr size_t kSmemFloats = 3 * kC * kD + 2 * kC * kC + kC * kUStride + kD * kSlice + kC + kD;
constexpr size_t kSmemBytes = kSmemFloats * sizeof(float);

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1)
chunk_simt_kernel(const InT* __restrict__ q, const InT* __restrict__ k, const InT* __restrict__ v,
                  const float* __restrict__ g, const float* __restrict__ beta, const float* init_state,
                  const int32_t* __restrict__ cu, int64_t T_total, int H, float scale,
                  const __nv_bfloat16* __restrict__ gate, InT* __restrict__ o, float* final_state) {
    extern __shared__ float smem[];
    float* sQ = smem;                    // [C][D] q, then q * Gamma
    float* sK = sQ + kC * kD;            // [C][D] k, then k * Gamma
    float* sG = sK + kC * kD;            // [C][D] G, then k * e^{G_C - G}
    float* sAk = sG + kC * kD;           // [C][C] beta_i A_kk, strictly lower
    float* sAq = sAk + kC * kC;          // [C][C] A_qk, lower with diagonal
    float* sU = sAq + kC * kC;           // [C][kUStride] v -> Z -> U (slice columns)
    float* sSt = sU + kC * kUStride;     // [D][kSlice] sSt[c][r] = S[r0 + r][c]
    float* sB = sSt + kD * kSlice;       // [C] beta
    float* sGl = sB + kC;                // [D] G at the chunk's last row

    const int chain = blockIdx.x;
    const int n = chain / H, h = chain % H;
    const int r0 = blockIdx.y * kSlice;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t state_off = (int64_t)chain * kD * kD;

    for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
        const int r = idx / kD, c = idx % kD;
        sSt[c * kSlice + r] = init_state ? init_state[state_off + (int64_t)(r0 + r) * kD + c] : 0.0f;
    }

    for (int64_t c0 = bos; c0 < eos; c0 += kC) {
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        __syncthreads();  // previous chunk done with every buffer
        // ---- tiles of this chunk (rows past L are zero: they change nothing)
        for (int idx = tid; idx < kC * kD; idx += kThreads) {
            const int i = idx / kD, c = idx % kD;
            if (i < L) {
                const int64_t base = ((c0 + i) * H + h) * kD + c;
                sQ[idx] = load_as_float(q + base);
                sK[idx] = load_as_float(k + base);
                sG[idx] = g[base];
            } else {
                sQ[idx] = 0.f; sK[idx] = 0.f; sG[idx] = 0.f;
            }
        }
        for (int idx = tid; idx < kC * kSlice; idx += kThreads) {
            const int i = idx / kSlice, r = idx % kSlice;
            sU[i * kUStride + r] = i < L ? load_as_float(v + ((c0 + i) * H + h) * kD + r0 + r) : 0.f;
        }
        if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        __syncthreads();
        // ---- running sum of g per key channel
        if (tid < kD) {
            float acc = 0.f;
            for (int i = 0; i < kC; ++i) {
                acc += sG[i * kD + tid];
                sG[i * kD + tid] = acc;
            }
            sGl[tid] = acc;
        }
        __syncthreads();
        // ---- A_kk and A_qk: 4x4 tiles of the lower triangle, position-pair decays
        simt_pair_blocks(sQ, sK, sG, sB, sAk, sAq, tid);
        __syncthreads();
        // ---- decayed operands: q Gamma (sQ), k Gamma (sK), k e^{G_C - G} (sG)
        for (int idx = tid; idx < kC * kD; idx += kThreads) {
            const int c = idx % kD;
            const float G = sG[idx], kk = sK[idx];
            const float gam = expf(G);
            sQ[idx] *= gam;
            sK[idx] = kk * gam;
            sG[idx] = kk * expf(sGl[c] - G);
        }
        __syncthreads();
        // ---- Z = beta (V - (K Gamma) S0^T); lanes over value rows, warps over tokens
        {
            float acc[8] = {};
            for (int c = 0; c < kD; ++c) {
                const float s = sSt[c * kSlice + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaf(sK[(warp * 8 + a) * kD + c], s, acc[a]);
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const int i = warp * 8 + a;
                sU[i * kUStride + lane] = sB[i] * (sU[i * kUStride + lane] - acc[a]);
            }
        }
        __syncthreads();
        // ---- U = (I + A_kk)^{-1} Z by forward substitution; warp w owns columns 4w..4w+3
        {
            const int col = warp * 4 + (lane & 3), grp = lane >> 2;
            for (int i = 1; i < kC; ++i) {
                float part = 0.f;
                for (int j = grp; j < i; j += 8) part = fmaf(sAk[i * kC + j], sU[j * kUStride + col], part);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 4);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 8);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 16);
                if (grp == 0) sU[i * kUStride + col] -= part;
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- O = scale ((Q Gamma) S0^T + A_qk U), optional output gate
        {
            float acc[8] = {};
            for (int c = 0; c < kD; ++c) {
                const float s = sSt[c * kSlice + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaf(sQ[(warp * 8 + a) * kD + c], s, acc[a]);
            }
            for (int j = 0; j < kC; ++j) {
                const float u = sU[j * kUStride + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaf(sAq[(warp * 8 + a) * kC + j], u, acc[a]);
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const int i = warp * 8 + a;
                if (i < L) {
                    const int64_t at = ((c0 + i) * H + h) * kD + r0 + lane;
                    float val = scale * acc[a];
                    if (gate) val *= 1.0f / (1.0f + expf(-__bfloat162float(gate[at])));
                    store_from_float(o + at, val);
                }
            }
        }
        __syncthreads();
        // ---- S = S0 Diag(e^{G_C}) + U^T (K e^{G_C - G}); lanes over value rows, warps over key channels
        {
            float acc[16];
#pragma unroll
            for (int a = 0; a < 16; ++a) {
                const int c = warp * 16 + a;
                acc[a] = sSt[c * kSlice + lane] * expf(sGl[c]);
            }
            for (int j = 0; j < kC; ++j) {
                const float u = sU[j * kUStride + lane];
                const float4* kr = reinterpret_cast<const float4*>(sG + j * kD + warp * 16);
#pragma unroll
                for (int a4 = 0; a4 < 4; ++a4) {
                    const float4 kv = kr[a4];
                    acc[4 * a4 + 0] = fmaf(u, kv.x, acc[4 * a4 + 0]);
                    acc[4 * a4 + 1] = fmaf(u, kv.y, acc[4 * a4 + 1]);
                    acc[4 * a4 + 2] = fmaf(u, kv.z, acc[4 * a4 + 2]);
                    acc[4 * a4 + 3] = fmaf(u, kv.w, acc[4 * a4 + 3]);
                }
            }
#pragma unroll
            for (int a = 0; a < 16; ++a) sSt[(warp * 16 + a) * kSlice + lane] = acc[a];
        }
    }
    __syncthreads();
    if (final_state) {
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int r = idx / kD, c = idx % kD;
            final_state[state_off + (int64_t)(r0 + r) * kD + c] = sSt[c * kSlice + r];
        }
    }
}

template <typename InT>
cudaError_t launch_typed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* init_state, const int32_t* cu, int N, int64_t T_total, int H, float scale,
                         const void* gate, void* o, float* final_state, cudaStream_t stream) {
    auto kern = chunk_simt_kernel<InT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((int64_t)N * H), kD / kSlice);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(
        static_cast<const InT*>(q), static_cast<const InT*>(k), static_cast<const InT*>(v), g, beta, init_state, cu,
        T_total, H, scale, static_cast<const __nv_bfloat16*>(gate), static_cast<InT*>(o), final_state);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total,
                              int H, float scale, kda_dtype dtype, const void* out_gate, void* o,
                              float* final_state, cudaStream_t stream) {
    if (dtype == KDA_DTYPE_F32)
        return launch_typed<float>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, out_gate, o,
                                   final_state, stream);
    return launch_typed<__nv_bfloat16>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, out_gate,
                                       o, final_state, stream);
}

}  // namespace kda
