// kda_chunk_bwd: the backward of the chunk prefill, fp32 on the CUDA cores.
//
// The forward ("Kimi-K3 深度解析", section 三, "KDA 的关键改进", unrolled over chunks of
// C = 64 tokens; the chunk_kda operator of "Kimi K3 架构全景", section 02, whose training speed
// "月之暗面发布Kimi K3开源大模型技术报告", 架构, is about) maps, per chunk with S0 entering it,
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
//   dbeta_i = sum_r dZ_ir R_ir + sum_j dA_kk[i][j] A_kk[i][j] / beta_i
// and the position-pair products of A_qk and A_kk taken back to q, k and G channel by channel; dg is
// the reverse running sum of dG inside the chunk.
//
// Four kernels (one stream, in order):
//   1. the fp32 forward (chunk_simt_kernel) keeping S0 of every chunk, R and V';
//   2. bwd_state_kernel: per (sequence, head, 32 value rows) the chunks in reverse, dS in shared
//      memory (the state's rows are independent, as in the forward), keeping dS_next of every chunk
//      and dZ;
//   3. bwd_chunk_a_kernel: per (chunk, head) the products with S0 and dS_next, dA_qk, dA_kk, dv and
//      the first term of dbeta;
//   4. bwd_chunk_b_kernel: per (chunk, head) the position-pair products, dq, dk, dg, the rest of dbeta.
// Chunk slot of chunk j of sequence n: (bos_n + 64 j) / 64 + n, distinct for all chunks of a batch
// and below T_total / 64 + N + 1.
#include "kda_common.cuh"
#include "kda_simt_blocks.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr int kSlice = 32;
constexpr int kUS = 36;       // row stride of [C][kSlice] tiles
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

// ============================ reverse state pass ============================
constexpr size_t kStateFloats = 3 * kC * kD + 2 * kC * kC + 2 * kC * kUS + kD * kSlice + kC + kD;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_state_kernel(const InT* __restrict__ q, const InT* __restrict__ k, const float* __restrict__ g,
                 const float* __restrict__ beta, const InT* __restrict__ d_o, const float* __restrict__ d_final,
                 const int32_t* __restrict__ cu, int64_t T_total, int H, float scale, float* __restrict__ d_init,
                 float* __restrict__ dS_next, float* __restrict__ dZ_out) {
    extern __shared__ float smem[];
    float* sQ = smem;                // [C][D] q, then Qg
    float* sK = sQ + kC * kD;        // [C][D] k, then Kg
    float* sG = sK + kC * kD;        // [C][D] G, then Kr
    float* sAk = sG + kC * kD;       // [C][C] A_kk (beta-scaled, strictly lower)
    float* sAq = sAk + kC * kC;      // [C][C] A_qk
    float* sDO = sAq + kC * kC;      // [C][kUS] dO, slice columns
    float* sDV = sDO + kC * kUS;     // [C][kUS] dV', then dZ
    float* sDS = sDV + kC * kUS;     // [D][kSlice] sDS[c][r] = dS[r0 + r][c]
    float* sB = sDS + kD * kSlice;   // [C]
    float* sGl = sB + kC;            // [D]

    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int r0 = blockIdx.y * kSlice;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t state_off = (int64_t)chain * kD * kD;
    for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
        const int r = idx / kD, c = idx % kD;
        sDS[c * kSlice + r] = d_final ? d_final[state_off + (int64_t)(r0 + r) * kD + c] : 0.0f;
    }
    const int64_t nch = (eos - bos + kC - 1) / kC;
    for (int64_t ci = nch - 1; ci >= 0; --ci) {
        const int64_t c0 = bos + ci * kC;
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        __syncthreads();  // the previous (later) chunk is done with every buffer
        {  // dS_next of this chunk
            const int64_t at = (((c0 / kC + n) * H + h) * kD + r0) * kD;
            for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
                const int r = idx / kD, c = idx % kD;
                dS_next[at + (int64_t)r * kD + c] = sDS[c * kSlice + r];
            }
        }
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
            sDO[i * kUS + r] = i < L ? load_as_float(d_o + ((c0 + i) * H + h) * kD + r0 + r) : 0.f;
        }
        if (tid < kC) sB[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        __syncthreads();
        if (tid < kD) {  // running sum of g per key channel
            float acc = 0.f;
            for (int i = 0; i < kC; ++i) {
                acc += sG[i * kD + tid];
                sG[i * kD + tid] = acc;
            }
            sGl[tid] = acc;
        }
        __syncthreads();
        simt_pair_blocks(sQ, sK, sG, sB, sAk, sAq, tid);
        __syncthreads();
        for (int idx = tid; idx < kC * kD; idx += kThreads) {  // Qg, Kg, Kr
            const int c = idx % kD;
            const float G = sG[idx], kk = sK[idx];
            const float gam = expf(G);
            sQ[idx] *= gam;
            sK[idx] = kk * gam;
            sG[idx] = kk * expf(sGl[c] - G);
        }
        __syncthreads();
        // ---- dV'[t][r] = sum_c Kr[t][c] dS[r][c] + scale sum_s A_qk[s][t] dO[s][r]; lanes over r, warps over t
        {
            float acc[8] = {};
            for (int c = 0; c < kD; ++c) {
                const float s = sDS[c * kSlice + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = fmaf(sG[(warp * 8 + a) * kD + c], s, acc[a]);
            }
            float acc2[8] = {};
            for (int s = 0; s < kC; ++s) {
                const float x = sDO[s * kUS + lane];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc2[a] = fmaf(sAq[s * kC + warp * 8 + a], x, acc2[a]);
            }
#pragma unroll
            for (int a = 0; a < 8; ++a) sDV[(warp * 8 + a) * kUS + lane] = fmaf(scale, acc2[a], acc[a]);
        }
        __syncthreads();
        // ---- dZ = (I + A_kk)^-T dV' by back substitution; warp w owns columns 4w .. 4w+3
        {
            const int col = warp * 4 + (lane & 3), grp = lane >> 2;
            for (int t = kC - 2; t >= 0; --t) {
                float part = 0.f;
                for (int s = t + 1 + grp; s < kC; s += 8) part = fmaf(sAk[s * kC + t], sDV[s * kUS + col], part);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 4);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 8);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 16);
                if (grp == 0) sDV[t * kUS + col] -= part;
                __syncwarp();
            }
        }
        __syncthreads();
        for (int idx = tid; idx < kC * kSlice; idx += kThreads) {
            const int i = idx / kSlice, r = idx % kSlice;
            if (i < L) dZ_out[((c0 + i) * H + h) * kD + r0 + r] = sDV[i * kUS + r];
        }
        // ---- dS <- dS Diag(gamma) + scale dO^T Qg - (Diag(beta) dZ)^T Kg; lanes over r, warps over c
        {
            float acc[16];
#pragma unroll
            for (int a = 0; a < 16; ++a) {
                const int c = warp * 16 + a;
                acc[a] = sDS[c * kSlice + lane] * expf(sGl[c]);
            }
            for (int t = 0; t < kC; ++t) {
                const float x = scale * sDO[t * kUS + lane];
                const float y = -sB[t] * sDV[t * kUS + lane];
                const float4* qg = reinterpret_cast<const float4*>(sQ + t * kD + warp * 16);
                const float4* kg = reinterpret_cast<const float4*>(sK + t * kD + warp * 16);
#pragma unroll
                for (int a4 = 0; a4 < 4; ++a4) {
                    const float4 qv = qg[a4], kv = kg[a4];
                    acc[4 * a4 + 0] = fmaf(y, kv.x, fmaf(x, qv.x, acc[4 * a4 + 0]));
                    acc[4 * a4 + 1] = fmaf(y, kv.y, fmaf(x, qv.y, acc[4 * a4 + 1]));
                    acc[4 * a4 + 2] = fmaf(y, kv.z, fmaf(x, qv.z, acc[4 * a4 + 2]));
                    acc[4 * a4 + 3] = fmaf(y, kv.w, fmaf(x, qv.w, acc[4 * a4 + 3]));
                }
            }
#pragma unroll
            for (int a = 0; a < 16; ++a) sDS[(warp * 16 + a) * kSlice + lane] = acc[a];
        }
    }
    __syncthreads();
    if (d_init) {
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int r = idx / kD, c = idx % kD;
            d_init[state_off + (int64_t)(r0 + r) * kD + c] = sDS[c * kSlice + r];
        }
    }
}

// ============================ per chunk: products with S0 and dS_next ============================
constexpr size_t kChunkAFloats = 3 * kC * kPS + 2 * kSlice * kD + kC;

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
    float* sS = sVP + kC * kPS;      // [kSlice][D] rows of S0
    float* sD = sS + kSlice * kD;    // [kSlice][D] rows of dS_next
    float* sB = sD + kSlice * kD;    // [C]
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
    // ---- dQg = scale dO S0, dKg = -Diag(beta) dZ S0, dKr = V' dS_next, dgamma; thread (c, half of the tokens)
    const int c = tid & (kD - 1), hf = tid >> 7;
    float aq[32], ak[32], ar[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) { aq[e] = 0.f; ak[e] = 0.f; ar[e] = 0.f; }
    float dgc = 0.f;
    const int64_t sbase = ((slot * H + h) * kD) * kD;
    for (int sb = 0; sb < kD / kSlice; ++sb) {
        __syncthreads();  // previous slab consumed (and, the first time, the tiles above stored)
        for (int idx = tid; idx < kSlice * kD; idx += kThreads) {
            const int64_t at = sbase + (int64_t)(kSlice * sb) * kD + idx;
            sS[idx] = S0s[at];
            sD[idx] = dS_next[at];
        }
        __syncthreads();
#pragma unroll 2
        for (int r = 0; r < kSlice; ++r) {
            const float s = sS[r * kD + c], d = sD[r * kD + c];
            dgc = fmaf(s, d, dgc);
            const int rr = kSlice * sb + r;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int t = 32 * hf + e;
                aq[e] = fmaf(sDO[t * kPS + rr], s, aq[e]);
                ak[e] = fmaf(sDZ[t * kPS + rr], s, ak[e]);
                ar[e] = fmaf(sVP[t * kPS + rr], d, ar[e]);
            }
        }
    }
    if (hf == 0) dgam[(slot * H + h) * kD + c] = dgc;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int t = 32 * hf + e;
        if (t < L) {
            const int64_t at = ((c0 + t) * H + h) * kD + c;
            XQ[at] = scale * aq[e];
            XK[at] = -sB[t] * ak[e];
            XR[at] = ar[e];
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
constexpr size_t kChunkBFloats = 3 * kC * kD + 2 * kC * kC + kC + kC * 4 + 2 * kD;

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_chunk_b_kernel(const InT* __restrict__ q, const InT* __restrict__ k, const float* __restrict__ g,
                   const float* __restrict__ beta, const int32_t* __restrict__ cu, int N, int64_t T_total, int H,
                   const float* __restrict__ XQ, const float* __restrict__ XK, const float* __restrict__ XR,
                   const float* __restrict__ dgam, const float* __restrict__ dAqk, const float* __restrict__ dAkk,
                   float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dg,
                   float* __restrict__ dbeta) {
    extern __shared__ float smem[];
    float* sQ = smem;                 // [C][D] q (then dG, for the reverse running sum)
    float* sK = sQ + kC * kD;         // [C][D] k
    float* sG = sK + kC * kD;         // [C][D] G
    float* sAq = sG + kC * kD;        // [C][C] dA_qk
    float* sAk = sAq + kC * kC;       // [C][C] dA_kk
    float* sB = sAk + kC * kC;        // [C]
    float* sRed = sB + kC;            // [C][4] per-warp parts of sum_c k_ic rowK'_ic
    float* sLast = sRed + kC * 4;     // [2][D] parts of sum_t dKr_t Kr_t
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n;
    int64_t c0, eos;
    if (!slot_chunk(cu, N, T_total, slot, n, c0, eos)) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    {
        const int64_t at = (slot * H + h) * kC * kC;
        for (int idx = tid; idx < kC * kC; idx += kThreads) {
            sAq[idx] = dAqk[at + idx];
            sAk[idx] = dAkk[at + idx];
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
    }
    __syncthreads();
    // thread (c, parity p): tokens i = p + 2 m of channel c, as rows and then as columns of the pairs
    const int c = tid & (kD - 1), p = tid >> 7;
    const float Gl = sG[(kC - 1) * kD + c];
    float dka[32], dGa[32];
    float last = 0.f;
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        const int i = p + 2 * m;
        if (i >= L) {  // warp-uniform: i depends on the warp's parity only
            dka[m] = 0.f;
            dGa[m] = 0.f;
            continue;
        }
        const float Gi = sG[i * kD + c];
        float rq = 0.f, rk = 0.f;  // sum_j dA_qk[i][j] k_jc e_ij (j <= i), sum_j dA_kk[i][j] k_jc e_ij (j < i)
        for (int j = 0; j <= i; ++j) {
            const float e = expf(fminf(Gi - sG[j * kD + c], 0.f));
            const float kj = sK[j * kD + c] * e;
            rq = fmaf(sAq[i * kC + j], kj, rq);
            rk = fmaf(sAk[i * kC + j], kj, rk);  // dA_kk is zero on the diagonal
        }
        const float qi = sQ[i * kD + c], ki = sK[i * kD + c], bi = sB[i];
        const int64_t at = ((c0 + i) * H + h) * kD + c;
        const float xq = XQ[at], xk = XK[at], xr = XR[at];
        const float gam = expf(Gi), red = expf(fminf(Gl - Gi, 0.f));
        dq[at] = fmaf(xq, gam, rq);
        dka[m] = bi * rk + xk * gam + xr * red;
        dGa[m] = qi * rq + ki * bi * rk + (xq * qi + xk * ki) * gam - xr * ki * red;
        last = fmaf(xr * ki, red, last);
        const float part = warp_sum(ki * rk);
        if (lane == 0) sRed[i * 4 + (warp & 3)] = part;
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        const int j = p + 2 * m;
        if (j >= L) continue;
        const float Gj = sG[j * kD + c];
        float cq = 0.f, ck = 0.f;  // sum_i dA_qk[i][j] q_ic e_ij (i >= j), sum_i dA_kk[i][j] beta_i k_ic e_ij (i > j)
        for (int i = j; i < L; ++i) {
            const float e = expf(fminf(sG[i * kD + c] - Gj, 0.f));
            cq = fmaf(sAq[i * kC + j], sQ[i * kD + c] * e, cq);
            ck = fmaf(sAk[i * kC + j] * sB[i], sK[i * kD + c] * e, ck);
        }
        dka[m] += cq + ck;
        dGa[m] -= sK[j * kD + c] * (cq + ck);
    }
    sLast[p * kD + c] = last;
    __syncthreads();  // every read of q, dA_qk and dA_kk done; sLast, sRed complete
    if (((L - 1) & 1) == p) {  // G_last = G at the chunk's last token: dKr and dgamma reach it
        const int m = (L - 1) >> 1;
        const float extra = sLast[c] + sLast[kD + c] + dgam[(slot * H + h) * kD + c] * expf(Gl);
#pragma unroll
        for (int mm = 0; mm < 32; ++mm)
            if (mm == m) dGa[mm] += extra;
    }
#pragma unroll
    for (int m = 0; m < 32; ++m) {
        const int i = p + 2 * m;
        if (i < L) dk[((c0 + i) * H + h) * kD + c] = dka[m];
        sQ[i * kD + c] = i < L ? dGa[m] : 0.f;
    }
    if (tid < L) {
        const float s = sRed[tid * 4] + sRed[tid * 4 + 1] + sRed[tid * 4 + 2] + sRed[tid * 4 + 3];
        dbeta[(c0 + tid) * H + h] += s;
    }
    __syncthreads();
    if (tid < kD) {  // dg_t = sum_{s >= t} dG_s inside the chunk
        float acc = 0.f;
        for (int t = L - 1; t >= 0; --t) {
            acc += sQ[t * kD + tid];
            dg[((c0 + t) * H + h) * kD + tid] = acc;
        }
    }
}

struct BwdWorkspace {
    float *S0, *dSn, *R, *Vp, *dZ, *XQ, *XK, *XR, *dgam, *dAqk, *dAkk;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t layout(int N, int64_t T_total, int H, uint8_t* base, BwdWorkspace* w) {
    const int64_t S = n_slots(N, T_total);
    const size_t state = align256((size_t)S * H * kD * kD * 4), tok = align256((size_t)T_total * H * kD * 4);
    const size_t gam = align256((size_t)S * H * kD * 4), amat = align256((size_t)S * H * kC * kC * 4);
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
    if (w) *w = x;
    return off;
}

template <typename InT>
cudaError_t launch_bwd_typed(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu, int N, int64_t T_total, int H, float scale,
                             kda_dtype dtype, const void* d_o, const float* d_final, float* dq, float* dk,
                             float* dv, float* dg, float* dbeta, float* d_init, void* workspace,
                             cudaStream_t stream) {
    BwdWorkspace w;
    layout(N, T_total, H, static_cast<uint8_t*>(workspace), &w);
    cudaError_t e = launch_chunk_simt(q, k, v, g, beta, init_state, cu, N, T_total, H, scale, dtype, nullptr,
                                      nullptr, nullptr, stream, w.S0, w.R, w.Vp);
    if (e != cudaSuccess) return e;
    const size_t smS = kStateFloats * 4, smA = kChunkAFloats * 4, smB = kChunkBFloats * 4;
    if ((e = cudaFuncSetAttribute(bwd_state_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smS)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_chunk_a_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smA)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_chunk_b_kernel<InT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smB)) !=
            cudaSuccess)
        return e;
    const InT* qt = static_cast<const InT*>(q);
    const InT* kt = static_cast<const InT*>(k);
    const InT* ot = static_cast<const InT*>(d_o);
    bwd_state_kernel<InT><<<dim3((unsigned)((int64_t)N * H), kD / kSlice), kThreads, smS, stream>>>(
        qt, kt, g, beta, ot, d_final, cu, T_total, H, scale, d_init, w.dSn, w.dZ);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (T_total == 0) return cudaSuccess;
    const dim3 grid((unsigned)n_slots(N, T_total), (unsigned)H);
    bwd_chunk_a_kernel<InT><<<grid, kThreads, smA, stream>>>(beta, ot, cu, N, T_total, H, scale, w.S0, w.dSn, w.R,
                                                             w.Vp, w.dZ, w.XQ, w.XK, w.XR, w.dgam, w.dAqk, w.dAkk, dv,
                                                             dbeta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_chunk_b_kernel<InT><<<grid, kThreads, smB, stream>>>(qt, kt, g, beta, cu, N, T_total, H, w.XQ, w.XK, w.XR,
                                                             w.dgam, w.dAqk, w.dAkk, dq, dk, dg, dbeta);
    return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int N, int64_t T_total, int H) { return layout(N, T_total, H, nullptr, nullptr); }

cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                             float scale, kda_dtype dtype, const void* d_o, const float* d_final, float* dq,
                             float* dk, float* dv, float* dg, float* dbeta, float* d_init, void* workspace,
                             cudaStream_t stream) {
    if (dtype == KDA_DTYPE_F32)
        return launch_bwd_typed<float>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype, d_o,
                                       d_final, dq, dk, dv, dg, dbeta, d_init, workspace, stream);
    return launch_bwd_typed<__nv_bfloat16>(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype, d_o,
                                           d_final, dq, dk, dv, dg, dbeta, d_init, workspace, stream);
}

}  // namespace kda
