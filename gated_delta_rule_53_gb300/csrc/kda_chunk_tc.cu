// kda_chunk_fwd, bf16 path: chunkwise prefill on the tcgen05 tensor cores.
//
// Math (chunk of C = 64 tokens, state S0 entering it; "Kimi-K3 深度解析",
// section 三, "KDA 的关键改进", unrolled over the chunk as in the chunk_kda
// operator of "Kimi K3 架构全景", section 02).  G_t is the running sum of g
// inside the chunk, per key channel:
//   A_kk[i][j] = beta_i sum_c k_ic k_jc e^{G_ic - G_jc}  (j < i),   T = (I + A_kk)^-1
//   A_qk[i][j] =        sum_c q_ic k_jc e^{G_ic - G_jc}  (j <= i)
//   Z^T  = (beta V)^T - S0 (beta K . e^G)^T              V'^T = Z^T T^T
//   O^T  = scale (S0 (Q . e^G)^T + V'^T A_qk^T)
//   S    = S0 Diag(e^{G_C}) + V'^T (K . e^{G_C - G})
//
// Dense intra-chunk blocks.  The position-pair factor e^{G_ic - G_jc} is split
// as e^{G_ic - R_c} e^{R_c - G_jc} around a reference R, which turns each block
// into a plain matrix product.  With the log-decay bounded below by -5 ("Kimi K3
// 架构全景", section 02: gate lower_bound -5.0; "月之暗面发布Kimi K3开源大模型技术
// 报告", 架构: the bound lets the diagonal blocks run as dense tensor-core
// products), 16 tokens span at most 5 * 15 = 75 in the exponent, and e^75 fits
// fp32 / bf16 (max ~ e^88.7).  Column block J (16 tokens) uses R = G at its last
// token: the column factor e^{R - G_j} is in [e^-75, 1], the row factor of a row
// in block J is in [1, e^75], and rows of later blocks get factors <= 1 whose
// underflow only drops terms that are below e^-87 in truth.  So A_kk and A_qk
// are four M=128 (64 k-rows + 64 q-rows) x N=16 x K=128 MMAs, one per column block.
//
// State path.  S0 (fp32) lives in registers: thread (r, half) of the 256 holds
// row r, key channels [64 half, 64 half + 64); a bf16 copy in shared memory is
// the A operand of the S0 products, so every product has M = 128 = dv and maps
// row r to TMEM lane r.  The UT solve (I + A_kk)^-1 runs in fp32 on the CUDA
// cores.  All tensor-core products take bf16 operands and accumulate in fp32.
//
// This first tensor-core version runs the phases of a chunk one after another
// in one CTA per (sequence, head); operands are written to shared memory by the
// threads (all of them are decay-scaled), so no operand comes raw from memory.
#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr int kAStride = 65;  // fp32 row stride of A_kk / T work arrays
constexpr uint32_t kWaitLimit = 1u << 22;

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_STK = 0;          // k staging bf16 [64][128]   | later Z^T / V'^T operand [128][64]
constexpr uint32_t OFF_STQ = 16384;      // q staging bf16 [64][128]   | later T operand [64][64] and A_qk [64][64]
constexpr uint32_t OFF_STV = 32768;      // v staging bf16 [64][128]
constexpr uint32_t OFF_STG = 49152;      // g -> G fp32 [64][128]      | later T fp32 work [64][65]
constexpr uint32_t OFF_KT = 81920;       // K~ operand [64][128]  (2 regions of 8 KB)
constexpr uint32_t OFF_B1 = 98304;       // [beta K e^G ; Q e^G] operand [128][128] (2 regions of 16 KB)
constexpr uint32_t OFF_KP = 131072;      // K e^{G_C - G} operand [64 tokens][128] (MN-major B)
constexpr uint32_t OFF_R = 147456;       // row operand of column block J [128][128] | later A_kk fp32 [64][65]
constexpr uint32_t OFF_S = 180224;       // bf16 S0 operand [128][128]
constexpr uint32_t OFF_BETA = 212992;    // fp32 [64]
constexpr uint32_t OFF_GEND = OFF_BETA + 256;     // fp32 [4][128] G at the end of each 16-token block
constexpr uint32_t OFF_EGL = OFF_GEND + 2048;     // fp32 [128] e^{G_C}
constexpr uint32_t OFF_BAR = OFF_EGL + 512;       // mbarrier
constexpr uint32_t OFF_MISC = OFF_BAR + 16;       // TMEM base, abort flag
constexpr uint32_t kSmemUsed = OFF_MISC + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base

// TMEM columns
constexpr uint32_t TM_A = 0;     // [A_kk raw ; A_qk raw] 64 columns
constexpr uint32_t TM_V = 64;    // V'^T 64 columns
constexpr uint32_t TM_Y = 128;   // Y^T = S0 (beta K e^G)^T 64 columns, then O^T 64 columns
constexpr uint32_t TM_O = 192;
constexpr uint32_t TM_DS = 256;  // delta S 128 columns
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// MMA with a K = 128 (two-region) A operand of 128 rows and a K-major B operand.
__device__ __forceinline__ void mma_k128(uint32_t d, uint32_t a_base, uint32_t a_region, uint32_t b_base,
                                         uint32_t b_region, uint32_t idesc, bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t reg = ks >> 2, off = (ks & 3) * 32;
        mma_bf16(d, sdesc_sw128(a_base + reg * a_region + off, 16, 1024), sdesc_sw128(b_base + reg * b_region + off, 16, 1024),
                 idesc, (ks > 0 || accumulate_first) ? 1u : 0u);
    }
}

// MMA with a K = 64 (one-region) A operand and a K-major one-region B operand.
__device__ __forceinline__ void mma_k64(uint32_t d, uint32_t a_base, uint32_t b_base, uint32_t idesc,
                                        bool accumulate_first) {
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
        mma_bf16(d, sdesc_sw128(a_base + ks * 32, 16, 1024), sdesc_sw128(b_base + ks * 32, 16, 1024), idesc,
                 (ks > 0 || accumulate_first) ? 1u : 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                const __nv_bfloat16* __restrict__ v, const float* __restrict__ g, const float* __restrict__ beta,
                const float* init_state, const int32_t* __restrict__ cu, int64_t T_total, int H, float scale,
                const __nv_bfloat16* __restrict__ gate, __nv_bfloat16* __restrict__ o, float* final_state,
                unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    float* sBeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* sGend = reinterpret_cast<float*>(sm + OFF_GEND);
    float* sEGl = reinterpret_cast<float*>(sm + OFF_EGL);
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);
    float* sG = reinterpret_cast<float*>(sm + OFF_STG);
    float* sAkk = reinterpret_cast<float*>(sm + OFF_R);
    float* sTf = reinterpret_cast<float*>(sm + OFF_STG);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int row = tid & 127, half = tid >> 7;  // state row / TMEM lane, key-channel half
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t state_off = (int64_t)chain * kD * kD + (int64_t)row * kD + 64 * half;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        *sAbort = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, kTmemCols);

    // state rows in registers, bf16 copy as the S0 operand
    float s[64];
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
        float4 x = init_state ? *reinterpret_cast<const float4*>(init_state + state_off + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        s[j] = x.x; s[j + 1] = x.y; s[j + 2] = x.z; s[j + 3] = x.w;
    }
    auto write_state_operand = [&]() {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = s[8 * ch + e];
            *reinterpret_cast<uint4*>(sm + OFF_S + half * 16384 + sw128(row, ch)) = pack8(f);
        }
    };
    write_state_operand();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    uint32_t phase = 0;

    auto wait_mma = [&]() {
        if (!mbar_wait(bar, phase, kWaitLimit)) {
            *sAbort = 1;
            raise_device_error(err, kErrMbarTimeout);
        }
        phase ^= 1u;
        tc_fence_after();
    };

    const uint32_t id_a = idesc_bf16_f32(128, 16, false, false);
    const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_64 = idesc_bf16_f32(128, 64, false, false);
    const uint32_t id_ds = idesc_bf16_f32(128, 128, false, true);

    for (int64_t c0 = bos; c0 < eos; c0 += kC) {
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        // ---- (1) staging loads (rows past L are zero)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int id = tid + kThreads * m, i = id >> 4, cc = id & 15;
            uint4 uk = make_uint4(0, 0, 0, 0), uq = uk, uv = uk;
            if (i < L) {
                const int64_t at = ((c0 + i) * H + h) * kD + cc * 8;
                uk = *reinterpret_cast<const uint4*>(k + at);
                uq = *reinterpret_cast<const uint4*>(q + at);
                uv = *reinterpret_cast<const uint4*>(v + at);
            }
            *reinterpret_cast<uint4*>(sm + OFF_STK + i * 256 + cc * 16) = uk;
            *reinterpret_cast<uint4*>(sm + OFF_STQ + i * 256 + cc * 16) = uq;
            *reinterpret_cast<uint4*>(sm + OFF_STV + i * 256 + cc * 16) = uv;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int id = tid + kThreads * m, i = id >> 5, cc = id & 31;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < L) x = *reinterpret_cast<const float4*>(g + ((c0 + i) * H + h) * kD + cc * 4);
            *reinterpret_cast<float4*>(sm + OFF_STG + i * 512 + cc * 16) = x;
        }
        if (tid < kC) sBeta[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        __syncthreads();
        // ---- (2) running sum of g per key channel; block-end references
        if (tid < kD) {
            float acc = 0.f;
#pragma unroll 16
            for (int i = 0; i < kC; ++i) {
                acc += sG[i * kD + tid];
                sG[i * kD + tid] = acc;
                if ((i & 15) == 15) sGend[(i >> 4) * kD + tid] = acc;
            }
            sEGl[tid] = expf(acc);
        }
        __syncthreads();
        // ---- (3) operands that do not depend on the column block, and the row operand of block 0
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
            const int id = tid + kThreads * m, i = id >> 4, cc = id & 15, c = cc * 8;
            const uint32_t reg = cc >> 3, ch = cc & 7;
            float kv[8], qv[8], Gv[8];
            unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STK + i * 256 + cc * 16), kv);
            unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STQ + i * 256 + cc * 16), qv);
#pragma unroll
            for (int e = 0; e < 8; ++e) Gv[e] = sG[i * kD + c + e];
            const float b = sBeta[i];
            const float* gb = sGend + (i >> 4) * kD + c;
            const float* gl = sGend + 3 * kD + c;
            const float* g0 = sGend + c;
            float f0[8], f1[8], f2[8], f3[8], f4[8], f5[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float eg = __expf(Gv[e]);
                f0[e] = kv[e] * __expf(gb[e] - Gv[e]);    // K~
                f1[e] = b * kv[e] * eg;                   // beta K e^G
                f2[e] = qv[e] * eg;                       // Q e^G
                f3[e] = kv[e] * __expf(gl[e] - Gv[e]);    // K e^{G_C - G}
                const float r0 = __expf(Gv[e] - g0[e]);   // row factor of column block 0
                f4[e] = kv[e] * r0;
                f5[e] = qv[e] * r0;
            }
            *reinterpret_cast<uint4*>(sm + OFF_KT + reg * 8192 + sw128(i, ch)) = pack8(f0);
            *reinterpret_cast<uint4*>(sm + OFF_B1 + reg * 16384 + sw128(i, ch)) = pack8(f1);
            *reinterpret_cast<uint4*>(sm + OFF_B1 + reg * 16384 + sw128(64 + i, ch)) = pack8(f2);
            *reinterpret_cast<uint4*>(sm + OFF_KP + reg * 8192 + sw128(i, ch)) = pack8(f3);
            *reinterpret_cast<uint4*>(sm + OFF_R + reg * 16384 + sw128(i, ch)) = pack8(f4);
            *reinterpret_cast<uint4*>(sm + OFF_R + reg * 16384 + sw128(64 + i, ch)) = pack8(f5);
        }
        fence_proxy_async();
        __syncthreads();
        // ---- (4) A block 0 and the S0 products
        if (tid == 0) {
            tc_fence_after();
            mma_k128(tbase + TM_A, sbase + OFF_R, 16384, sbase + OFF_KT, 8192, id_a, false);
            mma_k128(tbase + TM_Y, sbase + OFF_S, 16384, sbase + OFF_B1, 16384, id_s, false);
            mma_commit(bar);
        }
        wait_mma();
        for (int J = 1; J < 4; ++J) {
            const int rows = kC - 16 * J;  // rows of blocks >= J, for the k half and the q half
#pragma unroll 1
            for (int id = tid; id < rows * 16; id += kThreads) {
                const int i = 16 * J + (id >> 4), cc = id & 15, c = cc * 8;
                const uint32_t reg = cc >> 3, ch = cc & 7;
                float kv[8], qv[8], f4[8], f5[8];
                unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STK + i * 256 + cc * 16), kv);
                unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STQ + i * 256 + cc * 16), qv);
                const float* gj = sGend + J * kD + c;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float r = __expf(sG[i * kD + c + e] - gj[e]);
                    f4[e] = kv[e] * r;
                    f5[e] = qv[e] * r;
                }
                *reinterpret_cast<uint4*>(sm + OFF_R + reg * 16384 + sw128(i, ch)) = pack8(f4);
                *reinterpret_cast<uint4*>(sm + OFF_R + reg * 16384 + sw128(64 + i, ch)) = pack8(f5);
            }
            fence_proxy_async();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                // B = rows [16J, 16J + 16) of K~: 16 rows = two 8-row groups, so the sub-tile starts 2048 J bytes in
                mma_k128(tbase + TM_A + 16 * J, sbase + OFF_R, 16384, sbase + OFF_KT + 2048 * J, 8192, id_a, false);
                mma_commit(bar);
            }
            wait_mma();
        }
        // ---- (5) A_kk (fp32 work array), A_qk (bf16 operand) and Z^T (bf16 operand)
        {
            float a[32];
            tmem_ld32(tbase + lane_base + TM_A + 32 * half, a);
            if (row < kC) {
                const int i = row;
                const float b = sBeta[i];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 32 * half + e;
                    sAkk[i * kAStride + j] = j < i ? b * a[e] : 0.f;
                }
            } else {
                const int i = row - kC;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 32 * half + 8 * c4 + e;
                        f[e] = j <= i ? a[8 * c4 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4*>(sm + OFF_STQ + 8192 + sw128(i, 4 * half + c4)) = pack8(f);
                }
            }
            float y[32];
            tmem_ld32(tbase + lane_base + TM_Y + 32 * half, y);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 32 * half + 8 * c4 + e;
                    const float vj = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STV)[j * kD + row]);
                    f[e] = sBeta[j] * vj - y[8 * c4 + e];
                }
                *reinterpret_cast<uint4*>(sm + OFF_STK + sw128(row, 4 * half + c4)) = pack8(f);
            }
        }
        __syncthreads();
        // ---- (6) T = (I + A_kk)^-1 by forward substitution (fp32); warp w owns columns 8w .. 8w+7
        {
            const int col = 8 * warp + (lane & 7), grp = lane >> 3;
            for (int i = 0; i < kC; ++i) {
                float p0 = 0.f, p1 = 0.f;
                int j = grp;
                for (; j + 4 < i; j += 8) {
                    p0 = fmaf(sAkk[i * kAStride + j], sTf[j * kAStride + col], p0);
                    p1 = fmaf(sAkk[i * kAStride + j + 4], sTf[(j + 4) * kAStride + col], p1);
                }
                if (j < i) p0 = fmaf(sAkk[i * kAStride + j], sTf[j * kAStride + col], p0);
                float part = p0 + p1;
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 8);
                part += __shfl_xor_sync(0xFFFFFFFFu, part, 16);
                if (grp == 0) sTf[i * kAStride + col] = col < i ? -part : (col == i ? 1.f : 0.f);
                __syncwarp();
            }
        }
        __syncthreads();
        for (int id = tid; id < kC * 8; id += kThreads) {
            const int i = id >> 3, ch = id & 7;
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = sTf[i * kAStride + 8 * ch + e];
            *reinterpret_cast<uint4*>(sm + OFF_STQ + sw128(i, ch)) = pack8(f);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        if (*sAbort) break;
        // ---- (7) V'^T = Z^T T^T
        if (tid == 0) {
            tc_fence_after();
            mma_k64(tbase + TM_V, sbase + OFF_STK, sbase + OFF_STQ, id_64, false);
            mma_commit(bar);
        }
        wait_mma();
        {
            float x[32];
            tmem_ld32(tbase + lane_base + TM_V + 32 * half, x);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = x[8 * c4 + e];
                *reinterpret_cast<uint4*>(sm + OFF_STK + sw128(row, 4 * half + c4)) = pack8(f);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // ---- (8) O^T += V'^T A_qk^T;  dS = V'^T (K e^{G_C - G})
        if (tid == 0) {
            tc_fence_after();
            mma_k64(tbase + TM_O, sbase + OFF_STK, sbase + OFF_STQ + 8192, id_64, true);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tbase + TM_DS, sdesc_sw128(sbase + OFF_STK + ks * 32, 16, 1024),
                         sdesc_sw128(sbase + OFF_KP + ks * 2048, 8192, 1024), id_ds, ks > 0 ? 1u : 0u);
            mma_commit(bar);
        }
        wait_mma();
        // ---- (9) outputs and the state update
        {
            float x[32];
            tmem_ld32(tbase + lane_base + TM_O + 32 * half, x);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = 32 * half + e;
                if (j < L) {
                    const int64_t at = ((c0 + j) * H + h) * kD + row;
                    float val = scale * x[e];
                    if (gate) val *= 1.0f / (1.0f + __expf(-__bfloat162float(gate[at])));
                    o[at] = __float2bfloat16_rn(val);
                }
            }
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tmem_ld32(tbase + lane_base + TM_DS + 64 * half + 32 * part, x);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int jj = 32 * part + e;
                    s[jj] = fmaf(s[jj], sEGl[64 * half + jj], x[e]);
                }
            }
        }
        write_state_operand();
        tc_fence_before();
        __syncthreads();
        if (*sAbort) break;
    }

    if (final_state && !*sAbort) {
#pragma unroll
        for (int j = 0; j < 64; j += 4)
            *reinterpret_cast<float4*>(final_state + state_off + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                            float scale, const void* out_gate, void* o, float* final_state, unsigned int* err,
                            cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    chunk_tc_kernel<<<(unsigned)((int64_t)N * H), kThreads, kSmemBytes, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), g,
        beta, init_state, cu_seqlens, T_total, H, scale, static_cast<const __nv_bfloat16*>(out_gate),
        static_cast<__nv_bfloat16*>(o), final_state, err);
    return cudaGetLastError();
}

}  // namespace kda
