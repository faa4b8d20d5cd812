// kda_chunk_bwd: the backward of the chunk prefill, fp32 on the CUDA cores.
//
// The forward ("Kimi-K3 深度解析", section 三, "KDA 的关键改进", unrolled over chunks of
// C = 64 tokens: the chunk_kda operator of "Kimi K3 架构全景", section 02, which
// "月之暗面发布Kimi K3开源大模型技术报告", 架构, presents as a training-speed design) maps, per
// chunk with S0 entering it,
// G the running sum of g, Gamma = e^G, gamma = e^{G_last}, Kg = K Gamma, Qg = Q Gamma,
// Kr = K e^{G_last - G}:
//   R  = V - Kg S0^T,   V' = (I + A_kk)^-1 Diag(beta) R
//   O  = scale (Qg S0^T + A_qk V'),   S_next = S0 Diag(gamma) + V'^T Kr
// Given dO and dS_next, the chain rule through these lines gives
//   dV' = scale A_qk^T dO + Kr dS_next^T,      dZ = (I + A_kk)^-T dV'
//   dS0 = dS_next Diag(gamma) + scale dO^T Qg - (Diag(beta) dZ)^T Kg          (the reverse state pass)
// and, inside the chunk,
//   dQg = scale dO S0,  dKg = -Diag(beta) dZ S0,  dKr = V' dS_next,  dgamma = colsum(dS_next . S0)
//   dA_qk = scale dO V'^T (j <= i),  dA_kk = -dZ V'^T (j < i),  dv = Diag(beta) dZ
//   dbeta_i = sum_r dZ_ir R_ir + sum_j dA_kk[i][j] B[i][j]      (A_kk = Diag(beta) B)
// and the position-pair products of A_qk and A_kk taken back to q, k and G channel by channel; dg is
// the reverse running sum of dG inside the chunk.
//
// Six kernels (one stream, in order):
//   1. bwd_prep_kernel: per (chunk, head) at once, what does not depend on the state: G, A_qk,
//      T = (I + A_kk)^-1 (forward substitution, one column per thread), Qg, Kg, Kr, gamma;
//   2. bwd_fwd_state_kernel: per (sequence, head, 32 value rows) the chunks in order from S0, keeping
//      the state entering every chunk, R = V - Kg S0^T and V' = T Diag(beta) R;
//   3. bwd_state_kernel: per (sequence, head, 32 value rows) the chunks in reverse, dS in shared
//      memory (the state's rows are independent), keeping dS_next of every chunk and dZ = T^T dV';
//      with bf16 inputs bwd_fwd_state_tc_kernel and bwd_state_tc_kernel (kda_chunk_bwd_tc.cu) do passes 2
//      and 3 on the tensor cores instead, one CTA per chain, from bf16 hi/lo tiles that bwd_prep_tc_kernel
//      writes for them, and bwd_chunk_ab_tc_kernel does steps 4 and 5 on one CTA per (chunk, head);
//   4. bwd_chunk_a_kernel: per (chunk, head) the products with S0 and dS_next, dA_qk, dA_kk, dv and
//      the first term of dbeta;
//   5. bwd_chunk_b_kernel: per (chunk, head, half of the key channels) the position-pair products, dq,
//      dk, dg and the channel half's part of dbeta's second term; bwd_dbeta_kernel adds the parts.
// The two passes along the chains are plain products on shared-memory tiles (no exponentials, no
// triangular solve), small enough in shared memory for two or three CTAs per SM.
// Chunk slot of chunk j of sequence n: (bos_n + 64 j) / 64 + n, distinct for all chunks of a batch
// and below T_total / 64 + N + 1.
#include "kda_bwd_tc.cuh"
#include "kda_common.cuh"
#include "kda_simt_blocks.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr int kSlice = 32;
constexpr int kSS = kSlice + 1;  // row stride of the [D][kSlice] state tiles (consecutive channels on distinct banks)
constexpr int kUS = 36;       // row stride of [C][kSlice] tiles
constexpr int kHC = kD / 2;   // channels of a half-width [C][kHC] tile
constexpr int kPS = 132;      // row stride of [C][D] tiles read across rows (float4 rows on distinct banks)

int64_t n_slots(int N, int64_t T_total) { return T_total / kC + N + 1; }

// The chunk of a slot: sequence n with slot in [bos_n / C + n, bos_n / C + n + chunks_n); false if none.
__device__ bool slot_chunk(const int32_t* cu, int N, int64_t T_total, int64_t slot, int& n, int64_t& c0,
                           int64_t& eos) {
    int lo = 0, hi = N;  // f(n) = bos_n / C + n is increasing; the last n with f(n) <= slot
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        const int64_t b = cu ? (int64_t)cu[mid] : 0;
        if (b / kC + mid <= slot) lo = mid; else hi = mid;
    }
    int64_t bos;
    seq_bounds(cu, lo, T_total, bos, eos);
    n = lo;
    c0 = bos + (slot - (bos / kC + lo)) * kC;
    return slot >= bos / kC + lo && c0 < eos;
}

// ============================ per chunk: what does not depend on the state ============================
constexpr size_t kPrepFloats = 3 * kC * kD + kC * kC + kC + kD;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 2)
bwd_prep_kernel(const InT* __restrict__ q, const InT* __restrict__ k, const float* __restrict__ g,
                const float* __restrict__ beta, const int32_t* __restrict__ cu, int N, int64_t T_total, int H,
                float* __restrict__ gQg, float* __restrict__ gKg, float* __restrict__ gKr, float* __restrict__ gAqk,
                float* __restrict__ gT, float* __restrict__ gGam) {
    extern __shared__ float smem[];
    float* sQ = smem;             // [C][D] q
    float* sK = sQ + kC * kD;     // [C][D] k
    float* sG = sK + kC * kD;     // [C][D] g, then G
    float* sAk = sG + kC * kD;    // [C][C] A_kk (beta-scaled)
    float* sB = sAk + kC * kC;    // [C]
    float* sGl = sB + kC;         // [D]
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n;
    int64_t c0, eos;
    if (!slot_chunk(cu, N, T_total, slot, n, c0, eos)) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int tid = threadIdx.x;
    const int64_t base = slot * H + h;
    for (int idx = tid; idx < kC * kD; idx += kThreads) {
        const int i = idx / kD, c = idx % kD;
        if (i < L) {
            const int64_t at = ((c0 + i) * H + h) * kD + c;
            sQ[idx] = load_as_float(q + at);
            sK[idx] = load_as_float(k + at);
            sG[idx] = g[at];
        } else {
            sQ[idx] = 0.f; sK[idx] = 0.f; sG[idx] = 0.f;
        }
    }
    if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
    __syncthreads();
    if (tid < kD) {
        float acc = 0.f;
        for (int i = 0; i < kC; ++i) {
            acc += sG[i * kD + tid];
            sG[i * kD + tid] = acc;
        }
        sGl[tid] = acc;
        gGam[base * kD + tid] = expf(acc);
    }
    __syncthreads();
    simt_pair_blocks<true>(sQ, sK, sG, sB, sAk, gAqk + base * kC * kC, tid);  // A_qk straight to global memory
    __syncthreads();
    if (tid < kC) {  // column j = tid of T = (I + A_kk)^-1: x_i = [i == j] - sum_{m < i} A_kk[i][m] x_m
        const int j = tid;
        float x[kC];
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            float s = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m) s = fmaf(-sAk[i * kC + m], x[m], s);
            x[i] = s;
        }
#pragma unroll
        for (int i = 0; i < kC; ++i) gT[base * kC * kC + i * kC + j] = x[i];
    }
    // Qg, Kg, Kr in fp32 for the passes along the chains
    for (int idx = tid; idx < kC * kD; idx += kThreads) {
        const int c = idx % kD;
        const float G = sG[idx], kk = sK[idx];
        const float gam = expf(G);
        gQg[base * kC * kD + idx] = sQ[idx] * gam;
        gKg[base * kC * kD + idx] = kk * gam;
        gKr[base * kC * kD + idx] = kk * expf(sGl[c] - G);
    }
}

// [C][D] (or [C][C]) fp32 tile from global memory into shared memory, 16-byte pieces
__device__ __forceinline__ void tile_in(float* dst, const float* src, int floats, int tid) {
    for (int idx = tid; idx < floats / 4; idx += kThreads)
        reinterpret_cast<float4*>(dst)[idx] = reinterpret_cast<const float4*>(src)[idx];
}

// ============================ forward along the chains, keeping what the backward reads ============================
constexpr size_t kFwdFloats = kD * kSS + kC * kD + kC * kC + kC * kUS + kC + kD;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 3)
bwd_fwd_state_kernel(const InT* __restrict__ v, const float* __restrict__ beta, const float* __restrict__ init_state,
                     const int32_t* __restrict__ cu, int64_t T_total, int H, const float* __restrict__ gKg,
                     const float* __restrict__ gKr, const float* __restrict__ gT, const float* __restrict__ gGam,
                     float* __restrict__ S0s, float* __restrict__ Rb, float* __restrict__ Vp) {
    extern __shared__ float smem[];
    float* sSt = smem;                 // [D][kSS] sSt[c][r] = S[r0 + r][c]
    float* sX = sSt + kD * kSS;        // [C][D] Kg, then Kr
    float* sA = sX + kC * kD;          // [C][C] T
    float* sR = sA + kC * kC;          // [C][kUS] v, then beta R, then V'
    float* sB = sR + kC * kUS;         // [C]
    float* sGam = sB + kC;             // [D]
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int r0 = blockIdx.y * kSlice;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
        const int r = idx / kD, c = idx % kD;
        sSt[c * kSS + r] = init_state ? init_state[(int64_t)chain * kD * kD + (int64_t)(r0 + r) * kD + c] : 0.0f;
    }
    const int64_t nch = (eos - bos + kC - 1) / kC;
    for (int64_t ci = 0; ci < nch; ++ci) {
        const int64_t c0 = bos + ci * kC;
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        const int64_t base = (c0 / kC + n) * H + h;
        __syncthreads();  // the previous chunk is done with every buffer
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int r = idx / kD, c = idx % kD;
            S0s[(base * kD + r0 + r) * kD + c] = sSt[c * kSS + r];
        }
        tile_in(sX, gKg + base * kC * kD, kC * kD, tid);
        for (int idx = tid; idx < kC * kSlice; idx += kThreads) {
            const int i = idx / kSlice, r = idx % kSlice;
            sR[i * kUS + r] = i < L ? load_as_float(v + ((c0 + i) * H + h) * kD + r0 + r) : 0.f;
        }
        if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        if (tid < kD) sGam[tid] = gGam[base * kD + tid];
        __syncthreads();
        // ---- R = V - Kg S0^T: lanes over value rows, warps over tokens 8w .. 8w+7
        float br[8];
        {
            float acc[8] = {};
            for (int c = 0; c < kD; c += 4) {
                const float s0 = sSt[c * kSS + lane], s1 = sSt[(c + 1) * kSS + lane];
                const float s2 = sSt[(c + 2) * kSS + lane], s3 = sSt[(c + 3) * kSS + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const float4 x = *reinterpret_cast<const float4*>(sX + (warp * 8 + a) * kD + c);
                    acc[a] = fmaf(x.x, s0, fmaf(x.y, s1, fmaf(x.z, s2, fmaf(x.w, s3, acc[a]))));
                }
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const int t = warp * 8 + a;
                const float r = sR[t * kUS + lane] - acc[a];
                if (t < L) Rb[((c0 + t) * H + h) * kD + r0 + lane] = r;
                br[a] = sB[t] * r;
            }
        }
        __syncthreads();  // v and Kg consumed
#pragma unroll
        for (int a = 0; a < 8; ++a) sR[(warp * 8 + a) * kUS + lane] = br[a];
        tile_in(sA, gT + base * kC * kC, kC * kC, tid);
        tile_in(sX, gKr + base * kC * kD, kC * kD, tid);
        __syncthreads();
        // ---- V' = T (beta R)
        float vp[8];
        {
#pragma unroll
            for (int a = 0; a < 8; ++a) vp[a] = 0.f;
            for (int m = 0; m < kC; m += 4) {
                const float x0 = sR[m * kUS + lane], x1 = sR[(m + 1) * kUS + lane];
                const float x2 = sR[(m + 2) * kUS + lane], x3 = sR[(m + 3) * kUS + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const float4 t4 = *reinterpret_cast<const float4*>(sA + (warp * 8 + a) * kC + m);
                    vp[a] = fmaf(t4.x, x0, fmaf(t4.y, x1, fmaf(t4.z, x2, fmaf(t4.w, x3, vp[a]))));
                }
            }
        }
        __syncthreads();  // beta R consumed
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const int t = warp * 8 + a;
            sR[t * kUS + lane] = vp[a];
            if (t < L) Vp[((c0 + t) * H + h) * kD + r0 + lane] = vp[a];
        }
        __syncthreads();
        // ---- S = S0 Diag(gamma) + V'^T Kr: lanes over value rows, warps over key channels 16w .. 16w+15
        {
            float acc[16];
#pragma unroll
            for (int a = 0; a < 16; ++a) {
                const int c = warp * 16 + a;
                acc[a] = sSt[c * kSS + lane] * sGam[c];
            }
            for (int t = 0; t < kC; ++t) {
                const float u = sR[t * kUS + lane];
                const float4* kr = reinterpret_cast<const float4*>(sX + t * kD + warp * 16);
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
            for (int a = 0; a < 16; ++a) sSt[(warp * 16 + a) * kSS + lane] = acc[a];
        }
    }
}

// ============================ reverse state pass ============================
// Three CTAs per SM (384 CTAs for 96 chains fit one wave of 456): registers capped at 80 by the launch
// bounds, and the [C][D] tiles staged half a row (64 channels) at a time, 69 KB of shared memory.
constexpr size_t kStateFloats = kD * kSS + kC * kHC + kC * kC + 2 * kC * kUS + kC + kD;

// [C][kHC] half-width tile: channels hc * kHC .. + kHC - 1 of a [C][D] fp32 tile, 16-byte pieces
__device__ __forceinline__ void half_tile_in(float* dst, const float* src, int hc, int tid) {
    for (int idx = tid; idx < kC * kHC / 4; idx += kThreads) {
        const int i = idx / (kHC / 4), c4 = idx % (kHC / 4);
        reinterpret_cast<float4*>(dst)[idx] = reinterpret_cast<const float4*>(src + i * kD + hc * kHC)[c4];
    }
}

template <typename InT>
__global__ void __launch_bounds__(kThreads, 3)
bwd_state_kernel(const InT* __restrict__ d_o, const float* __restrict__ beta, const float* __restrict__ d_final,
                 const int32_t* __restrict__ cu, int64_t T_total, int H, float scale, const float* __restrict__ gQg,
                 const float* __restrict__ gKg, const float* __restrict__ gKr, const float* __restrict__ gAqk,
                 const float* __restrict__ gT, const float* __restrict__ gGam, float* __restrict__ d_init,
                 float* __restrict__ dS_next, float* __restrict__ dZ_out) {
    extern __shared__ float smem[];
    float* sDS = smem;                 // [D][kSS] sDS[c][r] = dS[r0 + r][c]
    float* sX = sDS + kD * kSS;        // [C][kHC] half of Kr, Qg or Kg
    float* sA = sX + kC * kHC;         // [C][C] A_qk, then T
    float* sDO = sA + kC * kC;         // [C][kUS] dO, slice columns
    float* sDV = sDO + kC * kUS;       // [C][kUS] dV', then beta dZ
    float* sB = sDV + kC * kUS;        // [C]
    float* sGam = sB + kC;             // [D]
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int r0 = blockIdx.y * kSlice;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t state_off = (int64_t)chain * kD * kD;
    for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
        const int r = idx / kD, c = idx % kD;
        sDS[c * kSS + r] = d_final ? d_final[state_off + (int64_t)(r0 + r) * kD + c] : 0.0f;
    }
    const int64_t nch = (eos - bos + kC - 1) / kC;
    for (int64_t ci = nch - 1; ci >= 0; --ci) {
        const int64_t c0 = bos + ci * kC;
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        const int64_t base = (c0 / kC + n) * H + h;
        const float* Kr = gKr + base * kC * kD;
        const float* Qg = gQg + base * kC * kD;
        const float* Kg = gKg + base * kC * kD;
        __syncthreads();  // the previous (later) chunk is done with every buffer
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int r = idx / kD, c = idx % kD;
            dS_next[(base * kD + r0 + r) * kD + c] = sDS[c * kSS + r];
        }
        half_tile_in(sX, Kr, 0, tid);
        tile_in(sA, gAqk + base * kC * kC, kC * kC, tid);
        for (int idx = tid; idx < kC * kSlice; idx += kThreads) {
            const int i = idx / kSlice, r = idx % kSlice;
            sDO[i * kUS + r] = i < L ? load_as_float(d_o + ((c0 + i) * H + h) * kD + r0 + r) : 0.f;
        }
        if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        if (tid < kD) sGam[tid] = gGam[base * kD + tid];
        __syncthreads();
        // ---- dV'[t][r] = sum_c Kr[t][c] dS[r][c] + scale sum_s A_qk[s][t] dO[s][r]; lanes over r, warps over t
        float dvp[8];
        {
            float acc[8] = {}, acc2[8] = {};
            for (int s = 0; s < kC; ++s) {
                const float x = sDO[s * kUS + lane];
                const float4 a0 = *reinterpret_cast<const float4*>(sA + s * kC + warp * 8);
                const float4 a1 = *reinterpret_cast<const float4*>(sA + s * kC + warp * 8 + 4);
                acc2[0] = fmaf(a0.x, x, acc2[0]); acc2[1] = fmaf(a0.y, x, acc2[1]);
                acc2[2] = fmaf(a0.z, x, acc2[2]); acc2[3] = fmaf(a0.w, x, acc2[3]);
                acc2[4] = fmaf(a1.x, x, acc2[4]); acc2[5] = fmaf(a1.y, x, acc2[5]);
                acc2[6] = fmaf(a1.z, x, acc2[6]); acc2[7] = fmaf(a1.w, x, acc2[7]);
            }
#pragma unroll 1
            for (int hc = 0; hc < 2; ++hc) {
                if (hc) {
                    __syncthreads();  // the first half of Kr consumed
                    half_tile_in(sX, Kr, 1, tid);
                    __syncthreads();
                }
                for (int c = 0; c < kHC; c += 4) {
                    const int cc = hc * kHC + c;
                    const float s0 = sDS[cc * kSS + lane], s1 = sDS[(cc + 1) * kSS + lane];
                    const float s2 = sDS[(cc + 2) * kSS + lane], s3 = sDS[(cc + 3) * kSS + lane];
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        const float4 x = *reinterpret_cast<const float4*>(sX + (warp * 8 + a) * kHC + c);
                        acc[a] = fmaf(x.x, s0, fmaf(x.y, s1, fmaf(x.z, s2, fmaf(x.w, s3, acc[a]))));
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) dvp[a] = fmaf(scale, acc2[a], acc[a]);
        }
        __syncthreads();  // Kr and A_qk consumed
#pragma unroll
        for (int a = 0; a < 8; ++a) sDV[(warp * 8 + a) * kUS + lane] = dvp[a];
        tile_in(sA, gT + base * kC * kC, kC * kC, tid);
        half_tile_in(sX, Qg, 0, tid);
        __syncthreads();
        // ---- dZ = T^T dV': dZ[t][r] = sum_s T[s][t] dV'[s][r]
        float bz[8];
        {
            float acc[8] = {};
            for (int s = 0; s < kC; ++s) {
                const float x = sDV[s * kUS + lane];
                const float4 a0 = *reinterpret_cast<const float4*>(sA + s * kC + warp * 8);
                const float4 a1 = *reinterpret_cast<const float4*>(sA + s * kC + warp * 8 + 4);
                acc[0] = fmaf(a0.x, x, acc[0]); acc[1] = fmaf(a0.y, x, acc[1]);
                acc[2] = fmaf(a0.z, x, acc[2]); acc[3] = fmaf(a0.w, x, acc[3]);
                acc[4] = fmaf(a1.x, x, acc[4]); acc[5] = fmaf(a1.y, x, acc[5]);
                acc[6] = fmaf(a1.z, x, acc[6]); acc[7] = fmaf(a1.w, x, acc[7]);
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const int t = warp * 8 + a;
                if (t < L) dZ_out[((c0 + t) * H + h) * kD + r0 + lane] = acc[a];
                bz[a] = sB[t] * acc[a];
            }
        }
        // ---- dS <- dS Diag(gamma) + scale dO^T Qg - (Diag(beta) dZ)^T Kg, one half of the channels at a time;
        //      lanes over r, warps over channels hc * 64 + 8w .. + 7
#pragma unroll 1
        for (int hc = 0; hc < 2; ++hc) {
            if (hc) {
                __syncthreads();  // Kg's first half consumed
                half_tile_in(sX, Qg, 1, tid);
                __syncthreads();
            }
            float ds[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const int c = hc * kHC + warp * 8 + a;
                ds[a] = sDS[c * kSS + lane] * sGam[c];
            }
            for (int t = 0; t < kC; ++t) {
                const float x = scale * sDO[t * kUS + lane];
                const float4 q0 = *reinterpret_cast<const float4*>(sX + t * kHC + warp * 8);
                const float4 q1 = *reinterpret_cast<const float4*>(sX + t * kHC + warp * 8 + 4);
                ds[0] = fmaf(x, q0.x, ds[0]); ds[1] = fmaf(x, q0.y, ds[1]);
                ds[2] = fmaf(x, q0.z, ds[2]); ds[3] = fmaf(x, q0.w, ds[3]);
                ds[4] = fmaf(x, q1.x, ds[4]); ds[5] = fmaf(x, q1.y, ds[5]);
                ds[6] = fmaf(x, q1.z, ds[6]); ds[7] = fmaf(x, q1.w, ds[7]);
            }
            __syncthreads();  // this half of Qg consumed (and, the first time, dV' and T)
            if (hc == 0) {
#pragma unroll
                for (int a = 0; a < 8; ++a) sDV[(warp * 8 + a) * kUS + lane] = bz[a];
            }
            half_tile_in(sX, Kg, hc, tid);
            __syncthreads();
            for (int t = 0; t < kC; ++t) {
                const float y = sDV[t * kUS + lane];
                const float4 k0 = *reinterpret_cast<const float4*>(sX + t * kHC + warp * 8);
                const float4 k1 = *reinterpret_cast<const float4*>(sX + t * kHC + warp * 8 + 4);
                ds[0] = fmaf(-y, k0.x, ds[0]); ds[1] = fmaf(-y, k0.y, ds[1]);
                ds[2] = fmaf(-y, k0.z, ds[2]); ds[3] = fmaf(-y, k0.w, ds[3]);
                ds[4] = fmaf(-y, k1.x, ds[4]); ds[5] = fmaf(-y, k1.y, ds[5]);
                ds[6] = fmaf(-y, k1.z, ds[6]); ds[7] = fmaf(-y, k1.w, ds[7]);
            }
            // only this thread reads these channels of its row again (the other half's terms read their own)
#pragma unroll
            for (int a = 0; a < 8; ++a) sDS[(hc * kHC + warp * 8 + a) * kSS + lane] = ds[a];
        }
    }
    __syncthreads();
    if (d_init) {
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int r = idx / kD, c = idx % kD;
            d_init[state_off + (int64_t)(r0 + r) * kD + c] = sDS[c * kSS + r];
        }
    }
}

// ============================ per chunk: products with S0 and dS_next ============================
constexpr int kSlab = 16;  // rows of S0 and dS_next in shared memory at a time
constexpr size_t kChunkAFloats = 3 * kC * kPS + 2 * kSlab * kD + kC;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_a_kernel(const float* __restrict__ beta, const InT* __restrict__ d_o, const int32_t* __restrict__ cu,
                   int N, int64_t T_total, int H, float scale, const float* __restrict__ S0s,
                   const float* __restrict__ dS_next, const float* __restrict__ Rb, const float* __restrict__ Vp,
                   const float* __restrict__ dZ, float* __restrict__ XQ, float* __restrict__ XK,
                   float* __restrict__ XR, float* __restrict__ dgam, float* __restrict__ dAqk,
                   float* __restrict__ dAkk, float* __restrict__ dv, float* __restrict__ dbeta) {
    extern __shared__ float smem[];
    float* sDO = smem;               // [C][kPS]
    float* sDZ = sDO + kC * kPS;     // [C][kPS]
    float* sVP = sDZ + kC * kPS;     // [C][kPS]
    float* sS = sVP + kC * kPS;      // [kSlab][D] rows of S0
    float* sD = sS + kSlab * kD;     // [kSlab][D] rows of dS_next
    float* sB = sD + kSlab * kD;     // [C]
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n;
    int64_t c0, eos;
    if (!slot_chunk(cu, N, T_total, slot, n, c0, eos)) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int idx = tid; idx < kC * kD; idx += kThreads) {
        const int i = idx / kD, c = idx % kD;
        float o = 0.f, z = 0.f, p = 0.f;
        if (i < L) {
            const int64_t at = ((c0 + i) * H + h) * kD + c;
            o = load_as_float(d_o + at);
            z = dZ[at];
            p = Vp[at];
            dv[at] = beta[(c0 + i) * H + h] * z;
        }
        sDO[i * kPS + c] = o;
        sDZ[i * kPS + c] = z;
        sVP[i * kPS + c] = p;
    }
    if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
    // dbeta, first term: sum_r dZ[t][r] R[t][r]; warp w takes rows 8w .. 8w+7
    for (int a = 0; a < 8; ++a) {
        const int i = warp * 8 + a;
        if (i < L) {
            const int64_t at = ((c0 + i) * H + h) * kD;
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) s = fmaf(dZ[at + lane + 32 * e], Rb[at + lane + 32 * e], s);
            s = warp_sum(s);
            if (lane == 0) dbeta[(c0 + i) * H + h] = s;
        }
    }
    // ---- dQg = scale dO S0, dKg = -Diag(beta) dZ S0, dKr = V' dS_next, dgamma: thread (channels 4 cq .. 4 cq + 3,
    //      tokens 8 tg .. 8 tg + 7); a warp shares its tokens, so their values are broadcast loads
    {
        const int cq = tid & 31, tg = tid >> 5;
        float aq[8][4], ak[8][4], ar[8][4];
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
            for (int e = 0; e < 4; ++e) { aq[a][e] = 0.f; ak[a][e] = 0.f; ar[a][e] = 0.f; }
        float4 dg4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const int64_t sbase = ((slot * H + h) * kD) * kD;
        for (int sb = 0; sb < kD / kSlab; ++sb) {
            __syncthreads();  // previous slab consumed (and, the first time, the tiles above stored)
            for (int idx = tid; idx < kSlab * kD / 4; idx += kThreads) {
                const int64_t at = sbase + (int64_t)(kSlab * sb) * kD;
                reinterpret_cast<float4*>(sS)[idx] = reinterpret_cast<const float4*>(S0s + at)[idx];
                reinterpret_cast<float4*>(sD)[idx] = reinterpret_cast<const float4*>(dS_next + at)[idx];
            }
            __syncthreads();
#pragma unroll 2
            for (int r = 0; r < kSlab; ++r) {
                const float4 s4 = *reinterpret_cast<const float4*>(sS + r * kD + 4 * cq);
                const float4 d4 = *reinterpret_cast<const float4*>(sD + r * kD + 4 * cq);
                if (tg == 0) {
                    dg4.x = fmaf(s4.x, d4.x, dg4.x); dg4.y = fmaf(s4.y, d4.y, dg4.y);
                    dg4.z = fmaf(s4.z, d4.z, dg4.z); dg4.w = fmaf(s4.w, d4.w, dg4.w);
                }
                const int rr = kSlab * sb + r;
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int t = 8 * tg + a;
                    const float o = sDO[t * kPS + rr], z = sDZ[t * kPS + rr], p = sVP[t * kPS + rr];
                    aq[a][0] = fmaf(o, s4.x, aq[a][0]); aq[a][1] = fmaf(o, s4.y, aq[a][1]);
                    aq[a][2] = fmaf(o, s4.z, aq[a][2]); aq[a][3] = fmaf(o, s4.w, aq[a][3]);
                    ak[a][0] = fmaf(z, s4.x, ak[a][0]); ak[a][1] = fmaf(z, s4.y, ak[a][1]);
                    ak[a][2] = fmaf(z, s4.z, ak[a][2]); ak[a][3] = fmaf(z, s4.w, ak[a][3]);
                    ar[a][0] = fmaf(p, d4.x, ar[a][0]); ar[a][1] = fmaf(p, d4.y, ar[a][1]);
                    ar[a][2] = fmaf(p, d4.z, ar[a][2]); ar[a][3] = fmaf(p, d4.w, ar[a][3]);
                }
            }
        }
        if (tg == 0) *reinterpret_cast<float4*>(dgam + (slot * H + h) * kD + 4 * cq) = dg4;
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const int t = 8 * tg + a;
            if (t < L) {
                const int64_t at = ((c0 + t) * H + h) * kD + 4 * cq;
                const float b = -sB[t];
                *reinterpret_cast<float4*>(XQ + at) =
                    make_float4(scale * aq[a][0], scale * aq[a][1], scale * aq[a][2], scale * aq[a][3]);
                *reinterpret_cast<float4*>(XK + at) = make_float4(b * ak[a][0], b * ak[a][1], b * ak[a][2], b * ak[a][3]);
                *reinterpret_cast<float4*>(XR + at) = make_float4(ar[a][0], ar[a][1], ar[a][2], ar[a][3]);
            }
        }
    }
    // ---- dA_qk = scale dO V'^T (j <= i), dA_kk = -dZ V'^T (j < i): thread (i, j = jq + 4 e)
    {
        const int i = tid >> 2, jq = tid & 3;
        float sq[16], sk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) { sq[e] = 0.f; sk[e] = 0.f; }
        for (int r = 0; r < kD; r += 4) {
            const float4 o4 = *reinterpret_cast<const float4*>(sDO + i * kPS + r);
            const float4 z4 = *reinterpret_cast<const float4*>(sDZ + i * kPS + r);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float4 p4 = *reinterpret_cast<const float4*>(sVP + (jq + 4 * e) * kPS + r);
                sq[e] = fmaf(o4.x, p4.x, fmaf(o4.y, p4.y, fmaf(o4.z, p4.z, fmaf(o4.w, p4.w, sq[e]))));
                sk[e] = fmaf(z4.x, p4.x, fmaf(z4.y, p4.y, fmaf(z4.z, p4.z, fmaf(z4.w, p4.w, sk[e]))));
            }
        }
        const int64_t at = ((slot * H + h) * kC + i) * kC;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int j = jq + 4 * e;
            dAqk[at + j] = j <= i ? scale * sq[e] : 0.f;
            dAkk[at + j] = j < i ? -sk[e] : 0.f;
        }
    }
}

// ============================ per chunk: position-pair products and the inputs' gradients ==========
// One CTA per (chunk, head, half of the key channels): the pair sums run channel by channel, so the two
// halves are independent except for dbeta's sum over channels, which each half leaves as a part.
constexpr int kHalf = kD / 2;
constexpr size_t kChunkBFloats = 4 * kC * kHalf + 2 * kC * kC + kC + kC * 2 + 4 * kHalf;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 2)
bwd_chunk_b_kernel(const InT* __restrict__ q, const InT* __restrict__ k, const float* __restrict__ g,
                   const float* __restrict__ beta, const int32_t* __restrict__ cu, int N, int64_t T_total, int H,
                   const float* __restrict__ XQ, const float* __restrict__ XK, const float* __restrict__ XR,
                   const float* __restrict__ dgam, const float* __restrict__ dAqk, const float* __restrict__ dAkk,
                   float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dg,
                   float* __restrict__ dbeta_part) {
    extern __shared__ float smem[];
    float* sQ = smem;                 // [C][kHalf] q (then dG, for the reverse running sum)
    float* sK = sQ + kC * kHalf;      // [C][kHalf] k
    float* sG = sK + kC * kHalf;      // [C][kHalf] G
    float* sAl = sG + kC * kHalf;     // [C][kHalf] alpha = e^g: the decay of a pair is a product of these
    float* sAq = sAl + kC * kHalf;    // [C][C] dA_qk
    float* sAk = sAq + kC * kC;       // [C][C] dA_kk
    float* sB = sAk + kC * kC;        // [C]
    float* sRed = sB + kC;            // [C][2] per-warp parts of sum_c k_ic rowK'_ic
    float* sLast = sRed + kC * 2;     // [4][kHalf] parts of sum_t dKr_t Kr_t
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y, half = blockIdx.z;
    int n;
    int64_t c0, eos;
    if (!slot_chunk(cu, N, T_total, slot, n, c0, eos)) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cb = kHalf * half;  // first channel of this half
    for (int idx = tid; idx < kC * kHalf; idx += kThreads) {
        const int i = idx / kHalf, cl = idx % kHalf;
        if (i < L) {
            const int64_t at = ((c0 + i) * H + h) * kD + cb + cl;
            sQ[idx] = load_as_float(q + at);
            sK[idx] = load_as_float(k + at);
            const float gv = g[at];
            sG[idx] = gv;
            sAl[idx] = expf(gv);
        } else {
            sQ[idx] = 0.f; sK[idx] = 0.f; sG[idx] = 0.f; sAl[idx] = 1.f;
        }
    }
    {
        const int64_t at = (slot * H + h) * kC * kC;
        for (int idx = tid; idx < kC * kC / 4; idx += kThreads) {
            reinterpret_cast<float4*>(sAq)[idx] = reinterpret_cast<const float4*>(dAqk + at)[idx];
            reinterpret_cast<float4*>(sAk)[idx] = reinterpret_cast<const float4*>(dAkk + at)[idx];
        }
    }
    if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
    __syncthreads();
    if (tid < kHalf) {
        float acc = 0.f;
        for (int i = 0; i < kC; ++i) {
            acc += sG[i * kHalf + tid];
            sG[i * kHalf + tid] = acc;
        }
    }
    __syncthreads();
    // thread (channel cl, group p): tokens i = p + 4 m of channel cl, as rows and then as columns of the pairs
    const int cl = tid & (kHalf - 1), p = tid >> 6;
    const float Gl = sG[(kC - 1) * kHalf + cl];
    float dka[16], dGa[16];
    float last = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = p + 4 * m;
        if (i >= L) {  // warp-uniform: i depends on the warp's group only
            dka[m] = 0.f;
            dGa[m] = 0.f;
            continue;
        }
        const float Gi = sG[i * kHalf + cl];
        // sum_j dA_qk[i][j] k_jc e_ij (j <= i) and sum_j dA_kk[i][j] k_jc e_ij (j < i), with
        // e_ij = e^{G_ic - G_jc} = alpha_{j+1} ... alpha_i taken as a running product from j = i down
        float rq = 0.f, rk = 0.f, e = 1.f;
        for (int j = i; j >= 0; --j) {
            const float kj = sK[j * kHalf + cl] * e;
            rq = fmaf(sAq[i * kC + j], kj, rq);
            rk = fmaf(sAk[i * kC + j], kj, rk);  // dA_kk is zero on the diagonal
            e *= sAl[j * kHalf + cl];
        }
        const float qi = sQ[i * kHalf + cl], ki = sK[i * kHalf + cl], bi = sB[i];
        const int64_t at = ((c0 + i) * H + h) * kD + cb + cl;
        const float xq = XQ[at], xk = XK[at], xr = XR[at];
        const float gam = expf(Gi), red = expf(fminf(Gl - Gi, 0.f));
        dq[at] = fmaf(xq, gam, rq);
        dka[m] = bi * rk + xk * gam + xr * red;
        dGa[m] = qi * rq + ki * bi * rk + (xq * qi + xk * ki) * gam - xr * ki * red;
        last = fmaf(xr * ki, red, last);
        const float part = warp_sum(ki * rk);
        if (lane == 0) sRed[i * 2 + (warp & 1)] = part;
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int j = p + 4 * m;
        if (j >= L) continue;
        // sum_i dA_qk[i][j] q_ic e_ij (i >= j) and sum_i dA_kk[i][j] beta_i k_ic e_ij (i > j), e_ij again
        // a running product, from i = j up
        float cq = 0.f, ck = 0.f, e = 1.f;
        for (int i = j; i < L; ++i) {
            cq = fmaf(sAq[i * kC + j], sQ[i * kHalf + cl] * e, cq);
            ck = fmaf(sAk[i * kC + j] * sB[i], sK[i * kHalf + cl] * e, ck);
            if (i + 1 < L) e *= sAl[(i + 1) * kHalf + cl];
        }
        dka[m] += cq + ck;
        dGa[m] -= sK[j * kHalf + cl] * (cq + ck);
    }
    sLast[p * kHalf + cl] = last;
    __syncthreads();  // every read of q, dA_qk and dA_kk done; sLast, sRed complete
    if (((L - 1) & 3) == p) {  // G_last = G at the chunk's last token: dKr and dgamma reach it
        const int m = (L - 1) >> 2;
        const float extra = sLast[cl] + sLast[kHalf + cl] + sLast[2 * kHalf + cl] + sLast[3 * kHalf + cl] +
                            dgam[(slot * H + h) * kD + cb + cl] * expf(Gl);
#pragma unroll
        for (int mm = 0; mm < 16; ++mm)
            if (mm == m) dGa[mm] += extra;
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = p + 4 * m;
        if (i < L) dk[((c0 + i) * H + h) * kD + cb + cl] = dka[m];
        sQ[i * kHalf + cl] = i < L ? dGa[m] : 0.f;
    }
    if (tid < L) dbeta_part[((int64_t)half * T_total + c0 + tid) * H + h] = sRed[tid * 2] + sRed[tid * 2 + 1];
    __syncthreads();
    if (tid < kHalf) {  // dg_t = sum_{s >= t} dG_s inside the chunk
        float acc = 0.f;
        for (int t = L - 1; t >= 0; --t) {
            acc += sQ[t * kHalf + tid];
            dg[((c0 + t) * H + h) * kD + cb + tid] = acc;
        }
    }
}

// dbeta = its first term (from bwd_chunk_a_kernel) + the two channel halves' parts, in that order
__global__ void bwd_dbeta_kernel(float* __restrict__ dbeta, const float* __restrict__ part, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dbeta[i] = (dbeta[i] + part[i]) + part[n + i];
}

struct BwdWorkspace {
    float *S0, *dSn, *R, *Vp, *dZ, *XQ, *XK, *XR, *dgam, *dAqk, *dAkk, *Qg, *Kg, *Kr, *Aqk, *T, *gam, *dbp;
    uint8_t* tc;  // the tensor-core reverse pass's tiles, kBwdBlobBytes per (chunk slot, head)
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t layout(int N, int64_t T_total, int H, uint8_t* base, BwdWorkspace* w) {
    const int64_t S = n_slots(N, T_total);
    const size_t state = align256((size_t)S * H * kD * kD * 4), tok = align256((size_t)T_total * H * kD * 4);
    const size_t gam = align256((size_t)S * H * kD * 4), amat = align256((size_t)S * H * kC * kC * 4);
    const size_t tile = align256((size_t)S * H * kC * kD * 4);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        float* p = base ? reinterpret_cast<float*>(base + off) : nullptr;
        off += bytes;
        return p;
    };
    BwdWorkspace x;
    x.S0 = take(state); x.dSn = take(state);
    x.R = take(tok); x.Vp = take(tok); x.dZ = take(tok); x.XQ = take(tok); x.XK = take(tok); x.XR = take(tok);
    x.dgam = take(gam); x.dAqk = take(amat); x.dAkk = take(amat);
    x.Qg = take(tile); x.Kg = take(tile); x.Kr = take(tile); x.Aqk = take(amat); x.T = take(amat); x.gam = take(gam);
    x.dbp = take(align256((size_t)2 * T_total * H * 4));
    x.tc = reinterpret_cast<uint8_t*>(take(align256((size_t)S * H * kBwdBlobBytes)));
    if (w) *w = x;
    return off;
}

template <typename InT>
cudaError_t launch_bwd_typed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu, int N, int64_t T_total, int H, float scale,
                             kda_dtype dtype, const void* d_o, const float* d_final, float* dq, float* dk,
                             float* dv, float* dg, float* dbeta, float* d_init, void* workspace, unsigned int* err,
                             cudaStream_t stream) {
    BwdWorkspace w;
    // bf16 inputs: the reverse pass on the tensor cores (dO reaches it by TMA: 32-bit token coordinates)
    const bool tc_state = sizeof(InT) == 2 && T_total > 0 && T_total < ((int64_t)1 << 31);
    layout(N, T_total, H, static_cast<uint8_t*>(workspace), &w);
    cudaError_t e;
    const size_t smP = kPrepFloats * 4, smF = kFwdFloats * 4, smS = kStateFloats * 4, smA = kChunkAFloats * 4,
                 smB = kChunkBFloats * 4;
    if ((e = cudaFuncSetAttribute(bwd_prep_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smP)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_fwd_state_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smF)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_state_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smS)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_chunk_a_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smA)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_chunk_b_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smB)) !=
            cudaSuccess)
        return e;
    const InT* qt = static_cast<const InT*>(q);
    const InT* kt = static_cast<const InT*>(k);
    const InT* vt = static_cast<const InT*>(v);
    const InT* ot = static_cast<const InT*>(d_o);
    const dim3 grid((unsigned)n_slots(N, T_total), (unsigned)H);
    const dim3 chains((unsigned)((int64_t)N * H), kD / kSlice);
    if (T_total > 0) {
        if (tc_state) {
            e = launch_bwd_prep_tc(q, k, g, beta, cu, N, T_total, H, scale, w.tc, err, stream);
        } else {
            bwd_prep_kernel<InT><<<grid, kThreads, smP, stream>>>(qt, kt, g, beta, cu, N, T_total, H, w.Qg, w.Kg,
                                                                  w.Kr, w.Aqk, w.T, w.gam);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
        if (tc_state) {
            e = launch_bwd_fwd_state_tc(v, init_state, cu, N, T_total, H, w.tc, w.S0, w.R, w.Vp, err, stream);
        } else {
            bwd_fwd_state_kernel<InT><<<chains, kThreads, smF, stream>>>(vt, beta, init_state, cu, T_total, H, w.Kg,
                                                                         w.Kr, w.T, w.gam, w.S0, w.R, w.Vp);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
    }
    if (tc_state) {
        e = launch_bwd_state_tc(d_o, d_final, cu, N, T_total, H, w.tc, d_init, w.dSn, w.dZ, err, stream);
    } else {
        bwd_state_kernel<InT><<<chains, kThreads, smS, stream>>>(ot, beta, d_final, cu, T_total, H, scale, w.Qg, w.Kg,
                                                                 w.Kr, w.Aqk, w.T, w.gam, d_init, w.dSn, w.dZ);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    if (T_total == 0) return cudaSuccess;
    if (tc_state) {  // both per-chunk steps in one kernel
        e = launch_bwd_chunk_ab_tc(q, k, g, beta, d_o, cu, N, T_total, H, scale, w.S0, w.dSn, w.R, w.Vp, w.dZ, w.XQ,
                                   w.XK, w.XR, w.dgam, w.dAqk, w.dAkk, dv, dbeta, dq, dk, dg, w.dbp, err, stream);
    } else {
        bwd_chunk_a_kernel<InT><<<grid, kThreads, smA, stream>>>(beta, ot, cu, N, T_total, H, scale, w.S0, w.dSn,
                                                                 w.R, w.Vp, w.dZ, w.XQ, w.XK, w.XR, w.dgam, w.dAqk,
                                                                 w.dAkk, dv, dbeta);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    if (!tc_state) {
        bwd_chunk_b_kernel<InT><<<dim3(grid.x, grid.y, 2), kThreads, smB, stream>>>(
            qt, kt, g, beta, cu, N, T_total, H, w.XQ, w.XK, w.XR, w.dgam, w.dAqk, w.dAkk, dq, dk, dg, w.dbp);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    const int64_t nb = T_total * H;
    bwd_dbeta_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, stream>>>(dbeta, w.dbp, nb);
    return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int N, int64_t T_total, int H) { return layout(N, T_total, H, nullptr, nullptr); }

cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                             float scale, kda_dtype dtype, const void* d_o, const float* d_final, float* dq,
                             float* dk, float* dv, float* dg, float* dbeta, float* d_init, void* workspace,
                             unsigned int* err, cudaStream_t stream) {
    if (dtype == KDA_DTYPE_F32)
        return launch_bwd_typed<float>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype, d_o,
                                       d_final, dq, dk, dv, dg, dbeta, d_init, workspace, err, stream);
    return launch_bwd_typed<__nv_bfloat16>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype, d_o,
                                           d_final, dq, dk, dv, dg, dbeta, d_init, workspace, err, stream);
}

}  // namespace kda
