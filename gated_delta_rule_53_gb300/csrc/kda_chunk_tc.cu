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
// around a reference as e^{G_ic - R_c} e^{R_c - G_jc}, which turns each block of
// A into a plain matrix product.  With the log-decay bounded below by -5 ("Kimi K3
// 架构全景", section 02: gate lower_bound -5.0; "月之暗面发布Kimi K3开源大模型技术
// 报告", 架构: the bound lets the diagonal blocks run as dense tensor-core
// products), a 16-token block spans at most 5 * 15 = 75 in the exponent and e^75
// fits fp32 and bf16 (max ~ e^88.7).  Row block I (tokens 16I .. 16I+15) takes
// R = E_I, the value of G at its last token:
//   row operand     x_i e^{G_i - E_I(i)}     in [1, e^75] x |x|   (one operand for all I)
//   column operand  k_j e^{E_I - G_j}        <= |k|, for j <= 16I + 15
// so row block I of A_kk and A_qk is one MMA of M = 128 (64 k-rows on top of 64
// q-rows) x N = 16(I+1) x K = 128, and the four are issued together.  A column
// factor that underflows fp32 (below e^-87.3) drops a term smaller than e^-12.3
// |x k| against a row factor of at most e^75: at most 4.5e-6 per entry of A, far
// under the bf16 rounding of the operands.  The column operand of block 3 is
// K e^{G_C - G}, the same tile the state update uses.
//
// State path.  S0 (fp32) lives in registers: thread (r, half) of the 256 holds
// row r, key channels [64 half, 64 half + 64); a bf16 copy in shared memory is
// the A operand of the S0 products, so every product has M = 128 = dv and maps
// row r to TMEM lane r.  Products accumulate in fp32 in TMEM; their operands are
// bf16, except Z T^T and the output's A_qk V' term, which run on kind::tf32 (tf32
// operands): that halves the bf16 rounding in the output.  T = (I + A_kk)^-1 is computed in fp32 on the CUDA
// cores by 16 x 16 blocks: the four diagonal blocks D by forward substitution, then
// the blocks below them as (I - N + N^2 - N^3) D with N = D A_below (N^4 = 0).
//
// One CTA of 16 warps per (sequence, head) walks the chunks in order; thread
// (r, quarter) holds state row r, key channels [32 quarter, 32 quarter + 32).  The
// next chunk's inputs are copied into shared memory with cp.async while the
// current chunk computes (k, q, g once the operands are built, v once Z is built).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kThreads = 512;
constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr int kAS = 68;       // fp32 row stride of the A_kk / T work arrays (float4 rows on distinct banks)
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// shared-memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_STK = 0;        // k staging bf16 [64][128]
constexpr uint32_t OFF_STQ = 16384;    // q staging bf16 [64][128]
constexpr uint32_t OFF_STV = 32768;    // v staging bf16 [64][128]
constexpr uint32_t OFF_STG = 49152;    // g -> G fp32 [64][128]
constexpr uint32_t OFF_B1 = 81920;     // [beta K e^G ; Q e^G] [128][128] (B of the S0 products)
constexpr uint32_t OFF_KP = 114688;    // K e^{G_C - G} [64][128]: column operand of row block 3, B of dS
constexpr uint32_t OFF_RR = 131072;    // row operand [K e^{G-E} ; Q e^{G-E}] [128][128] | A_kk, A_qk, scratch | O fp32
constexpr uint32_t OFF_CC = 163840;    // column operands of row blocks 0..2 (16, 32, 48 rows) | T fp32, T bf16 | Z^T
constexpr uint32_t OFF_S = 188416;     // bf16 S0 [128][128]
constexpr uint32_t OFF_SMALL = 221184;
constexpr uint32_t OFF_BETA = OFF_SMALL;             // fp32 [2][64] (double-buffered)
constexpr uint32_t OFF_E = OFF_BETA + 512;           // fp32 [4][128] E_I = G at the last token of block I
constexpr uint32_t OFF_DT = OFF_E + 2048;            // fp32 [6][128] e^{E_J - E_I}, J > I
constexpr uint32_t OFF_EGL = OFF_DT + 3072;          // fp32 [128] e^{G_C}
constexpr uint32_t OFF_TOT = OFF_EGL + 512;          // fp32 [4][128] per-block sums of g
constexpr uint32_t OFF_BAR = OFF_TOT + 2048;         // mbarriers: A products, state products, k/q/g tiles, v tile
constexpr uint32_t OFF_MISC = OFF_BAR + 32;          // TMEM base, abort flag
constexpr uint32_t kSmemUsed = OFF_MISC + 64;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;    // slack for aligning the base

// After the A products complete (RR and CC are free; the S0 products may still read B1):
constexpr uint32_t OFF_AKK = OFF_CC;                 // A_kk fp32 [64][kAS] (17 KB)
constexpr uint32_t OFF_AQ = OFF_RR;                  // A_qk tf32 operand [64][64] (2 regions of 8 KB)
// After the S0 products complete (B1 is free):
constexpr uint32_t OFF_TF = OFF_B1;                  // T fp32 [64][kAS] (17 KB)
constexpr uint32_t OFF_NB = OFF_B1 + 64 * kAS * 4;   // N blocks of the solve, 9 x [16][20] fp32
// Once T is in registers:
constexpr uint32_t OFF_TT = OFF_CC;                  // T tf32 operand [64][64] (2 regions of 8 KB)
constexpr uint32_t OFF_ZT = OFF_B1;                  // Z^T, then V'^T, tf32 operand [128][64] (2 regions of 16 KB)
constexpr uint32_t OFF_VB = OFF_CC;                  // V'^T bf16 operand [128][64] (16 KB), once T is consumed
// column operand of row block I < 3: 16(I+1) rows, two regions of 16(I+1) * 128 bytes
__host__ __device__ constexpr uint32_t cc_off(int I) { return I == 0 ? 0u : (I == 1 ? 4096u : 12288u); }

// TMEM columns
constexpr uint32_t TM_A0 = 0, TM_A1 = 32, TM_A2 = 64, TM_A3 = 128;  // row blocks of A: 16, 32, 48, 64 columns
constexpr uint32_t TM_V = 192;    // V'^T
constexpr uint32_t TM_Y = 256;    // Y^T = S0 (beta K e^G)^T, then O^T at TM_O
constexpr uint32_t TM_O = 320;
constexpr uint32_t TM_DS = 384;   // delta S
constexpr uint32_t kTmemCols = 512;

static_assert(OFF_AKK + 64 * kAS * 4 <= OFF_S && OFF_AQ + 16384 <= OFF_CC, "A work overflows its region");
static_assert(OFF_NB + 9 * 16 * 20 * 4 <= OFF_KP, "T work overflows its region");
static_assert(kSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// D (+)= A B^T with a K = 128 (two-region) A of 128 rows and a K-major two-region B.  The
// descriptors of the operands' first bytes are passed in; moving the start address by `off`
// bytes adds off / 16 to the descriptor (shared addresses stay below 2^18, so no carry).
__device__ __forceinline__ void mma_k128(uint32_t d, uint64_t a_desc, uint32_t a_region, uint64_t b_desc,
                                         uint32_t b_region, uint32_t idesc) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const uint32_t reg = ks >> 2, off = (ks & 3) * 32;
        mma_bf16(d, a_desc + ((reg * a_region + off) >> 4), b_desc + ((reg * b_region + off) >> 4), idesc,
                 ks > 0 ? 1u : 0u);
    }
}

__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return sdesc_sw128(saddr, 16, 1024); }

// Loads of the chunk starting at token c0 of head h.  Thread 0 issues one TMA box per tensor
// ([64 tokens][1 head][128 channels]; rows past the end of the tensor read as zero) and arms the
// stage's mbarrier with the byte count; beta (64 strided words) comes by cp.async, zero past the
// chunk's L tokens.  Rows past L that belong to the next packed sequence are harmless in k, q
// and v (their beta is zero) and g is masked where it is summed.
constexpr uint32_t kKQGBytes = 2 * 16384 + 32768;
constexpr uint32_t kVBytes = 16384;

__device__ __forceinline__ void prefetch_kqg(uint8_t* sm, uint64_t* bar, float* beta_dst, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_q, const CUtensorMap* tm_g, const float* beta,
                                             int64_t c0, int L, int H, int h, int tid) {
    if (tid == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, kKQGBytes);
        tma_load_3d(sm + OFF_STK, tm_k, 0, h, (int)c0, bar);
        tma_load_3d(sm + OFF_STQ, tm_q, 0, h, (int)c0, bar);
        tma_load_3d(sm + OFF_STG, tm_g, 0, h, (int)c0, bar);
    }
    if (tid < kC) {
        const bool ok = tid < L;
        cp_async4(beta_dst + tid, beta + (ok ? (c0 + tid) * H + h : 0), ok ? 4u : 0u);
    }
}

__device__ __forceinline__ void prefetch_v(uint8_t* sm, uint64_t* bar, const CUtensorMap* tm_v, int64_t c0, int h,
                                           int tid) {
    if (tid == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar, kVBytes);
        tma_load_3d(sm + OFF_STV, tm_v, 0, h, (int)c0, bar);
    }
}

// One 16 x 16 fp32 block product for 64 threads (t = 0..63 owns row t / 4, columns 4 (t % 4) .. +3):
//   out = sign * (A0 + w1 A1 + w2 A2) B  [+ A3 B3]
// NA = number of A blocks combined on the fly (an entry of P = -N + N^2 - N^3); SECOND adds A3 B3.
struct Blk {
    const float* p;
    int ld;
};
template <int NA, bool SECOND>
__device__ __forceinline__ void blk_mma(float* out, int ldo, float sign, Blk a0, Blk a1, float w1, Blk a2, float w2,
                                        Blk b, Blk a3, Blk b3, int t) {
    const int r = t >> 2, c = 4 * (t & 3);
    float av[16];
#pragma unroll
    for (int m = 0; m < 16; m += 4) {
        float4 x = *reinterpret_cast<const float4*>(a0.p + r * a0.ld + m);
        if (NA > 1) {
            const float4 y = *reinterpret_cast<const float4*>(a1.p + r * a1.ld + m);
            x.x = fmaf(w1, y.x, x.x); x.y = fmaf(w1, y.y, x.y); x.z = fmaf(w1, y.z, x.z); x.w = fmaf(w1, y.w, x.w);
        }
        if (NA > 2) {
            const float4 y = *reinterpret_cast<const float4*>(a2.p + r * a2.ld + m);
            x.x = fmaf(w2, y.x, x.x); x.y = fmaf(w2, y.y, x.y); x.z = fmaf(w2, y.z, x.z); x.w = fmaf(w2, y.w, x.w);
        }
        av[m] = x.x; av[m + 1] = x.y; av[m + 2] = x.z; av[m + 3] = x.w;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), acc2 = acc;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float4 bv = *reinterpret_cast<const float4*>(b.p + m * b.ld + c);
        float4& ac = (m & 1) ? acc2 : acc;
        ac.x = fmaf(av[m], bv.x, ac.x); ac.y = fmaf(av[m], bv.y, ac.y);
        ac.z = fmaf(av[m], bv.z, ac.z); ac.w = fmaf(av[m], bv.w, ac.w);
    }
    if (SECOND) {
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 x = *reinterpret_cast<const float4*>(a3.p + r * a3.ld + m);
            av[m] = x.x; av[m + 1] = x.y; av[m + 2] = x.z; av[m + 3] = x.w;
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float4 bv = *reinterpret_cast<const float4*>(b3.p + m * b3.ld + c);
            float4& ac = (m & 1) ? acc2 : acc;
            ac.x = fmaf(av[m], bv.x, ac.x); ac.y = fmaf(av[m], bv.y, ac.y);
            ac.z = fmaf(av[m], bv.z, ac.z); ac.w = fmaf(av[m], bv.w, ac.w);
        }
    }
    *reinterpret_cast<float4*>(out + r * ldo + c) = make_float4(sign * (acc.x + acc2.x), sign * (acc.y + acc2.y),
                                                                  sign * (acc.z + acc2.z), sign * (acc.w + acc2.w));
}

// Blocks of T below the diagonal.  With D = diag(T_00 .. T_33) (inverses of the diagonal blocks of
// I + A_kk) and N = D A_off (A_off: the blocks of A_kk below the diagonal; N is strictly block-lower,
// so N^4 = 0):  (I + A_kk)^-1 = (I + N)^-1 D = (I - N + N^2 - N^3) D.
// Three levels, each a set of independent 16 x 16 products spread over the CTA's warps.
constexpr int kNB = 20;  // row stride of the N blocks (float4 rows, eight rows on distinct banks)
__device__ __forceinline__ void t_offdiag(const float* A, float* T, float* nb, int tid) {
    const int u = tid >> 6, t = tid & 63;
    auto Ablk = [&](int I, int J) { return Blk{A + 16 * I * kAS + 16 * J, kAS}; };
    auto Tblk = [&](int I, int J) { return Blk{T + 16 * I * kAS + 16 * J, kAS}; };
    // N_IJ at nb[slot]: (1,0) 0, (2,0) 1, (3,0) 2, (2,1) 3, (3,1) 4, (3,2) 5; N^2: (2,0) 6, (3,1) 7, (3,0) 8
    auto Nb = [&](int slot) { return Blk{nb + slot * 16 * kNB, kNB}; };
    const Blk none{nullptr, 0};
    if (u < 6) {  // slots 0..5: (1,0) (2,0) (3,0) (2,1) (3,1) (3,2)
        const int I = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3), J = u < 3 ? 0 : (u < 5 ? 1 : 2);
        blk_mma<1, false>(nb + u * 16 * kNB, kNB, 1.f, Tblk(I, I), none, 0.f, none, 0.f, Ablk(I, J), none, none, t);
    }
    __syncthreads();
    if (u == 0) blk_mma<1, false>(nb + 6 * 16 * kNB, kNB, 1.f, Nb(3), none, 0.f, none, 0.f, Nb(0), none, none, t);   // N21 N10
    if (u == 1) blk_mma<1, false>(nb + 7 * 16 * kNB, kNB, 1.f, Nb(5), none, 0.f, none, 0.f, Nb(3), none, none, t);   // N32 N21
    if (u == 2) blk_mma<1, true>(nb + 8 * 16 * kNB, kNB, 1.f, Nb(4), none, 0.f, none, 0.f, Nb(0), Nb(5), Nb(1), t);  // N31 N10 + N32 N20
    if (u == 3) blk_mma<1, false>(T + 16 * kAS * 1 + 0, kAS, -1.f, Nb(0), none, 0.f, none, 0.f, Tblk(0, 0), none, none, t);   // T10
    if (u == 4) blk_mma<1, false>(T + 16 * kAS * 2 + 16, kAS, -1.f, Nb(3), none, 0.f, none, 0.f, Tblk(1, 1), none, none, t);  // T21
    if (u == 5) blk_mma<1, false>(T + 16 * kAS * 3 + 32, kAS, -1.f, Nb(5), none, 0.f, none, 0.f, Tblk(2, 2), none, none, t);  // T32
    __syncthreads();
    // T_30 = (N^2_30 - N_30 - N^3_30) D_0 with N^3_30 D_0 = N^2_31 N_10 D_0 = -N^2_31 T_10
    if (u == 0) blk_mma<2, true>(T + 16 * kAS * 3 + 0, kAS, 1.f, Nb(8), Nb(2), -1.f, none, 0.f, Tblk(0, 0), Nb(7), Tblk(1, 0), t);
    if (u == 1) blk_mma<2, false>(T + 16 * kAS * 2 + 0, kAS, 1.f, Nb(6), Nb(1), -1.f, none, 0.f, Tblk(0, 0), none, none, t);  // T20
    if (u == 2) blk_mma<2, false>(T + 16 * kAS * 3 + 16, kAS, 1.f, Nb(7), Nb(4), -1.f, none, 0.f, Tblk(1, 1), none, none, t); // T31
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                const float* __restrict__ beta,
                const float* init_state, const int32_t* __restrict__ cu, int64_t T_total, int H, float scale,
                const __nv_bfloat16* __restrict__ gate, __nv_bfloat16* __restrict__ o, float* final_state,
                unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    float* sBetaBuf = reinterpret_cast<float*>(sm + OFF_BETA);
    float* sE = reinterpret_cast<float*>(sm + OFF_E);
    float* sDt = reinterpret_cast<float*>(sm + OFF_DT);
    float* sEGl = reinterpret_cast<float*>(sm + OFF_EGL);
    float* sTot = reinterpret_cast<float*>(sm + OFF_TOT);
    uint64_t* barA = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* barS = barA + 1;
    uint64_t* barL = barA + 2;  // k, q, g tiles
    uint64_t* barV = barA + 3;  // v tile
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + OFF_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + OFF_MISC + 4);
    float* sG = reinterpret_cast<float*>(sm + OFF_STG);
    float* sAkk = reinterpret_cast<float*>(sm + OFF_AKK);
    float* sTf = reinterpret_cast<float*>(sm + OFF_TF);
    float* sO = reinterpret_cast<float*>(sm + OFF_RR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int row = tid & 127, qq = tid >> 7;  // state row / TMEM lane; quarter of the key channels / tokens
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t state_off = (int64_t)chain * kD * kD + (int64_t)row * kD + 32 * qq;

    if (tid == 0) {
        mbar_init(barA, 1);
        mbar_init(barS, 1);
        mbar_init(barL, 1);
        mbar_init(barV, 1);
        fence_mbar_init();
        *sAbort = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, kTmemCols);
    __syncthreads();  // barriers initialised before the first copy lands on them
    if (bos < eos) {  // the first chunk's inputs
        const int L0 = (eos - bos) < kC ? (int)(eos - bos) : kC;
        prefetch_kqg(sm, barL, sBetaBuf, &tm_k, &tm_q, &tm_g, beta, bos, L0, H, h, tid);
        prefetch_v(sm, barV, &tm_v, bos, h, tid);
        cp_async_commit();
    }

    // state: row `row`, key channels [32 qq, 32 qq + 32) in registers; bf16 copy as the S0 operand
    float s[32];
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float4 x = init_state ? *reinterpret_cast<const float4*>(init_state + state_off + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        s[j] = x.x; s[j + 1] = x.y; s[j + 2] = x.z; s[j + 3] = x.w;
    }
    auto write_state_operand = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = s[8 * c + e];
            *reinterpret_cast<uint4*>(sm + OFF_S + (qq >> 1) * 16384 + sw128(row, 4 * (qq & 1) + c)) = pack8(f);
        }
    };
    write_state_operand();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    uint32_t phaseA = 0, phaseS = 0, phaseL = 0, phaseV = 0;

    auto wait_bar = [&](uint64_t* b, uint32_t& ph) {
        if (!mbar_wait(b, ph, kWaitLimit)) {
            *sAbort = 1;
            raise_device_error(err, kErrMbarTimeout);
        }
        ph ^= 1u;
        tc_fence_after();
    };
    auto wait_mma = [&]() { wait_bar(barS, phaseS); };

    const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_t64 = idesc_tf32_f32(128, 64);
    const uint32_t id_ds = idesc_bf16_f32(128, 128, false, true);

    int buf = 0;
    for (int64_t c0 = bos; c0 < eos; c0 += kC, buf ^= 1) {
        const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        const int64_t c1 = c0 + kC;
        const int L1 = c1 < eos ? ((eos - c1) < kC ? (int)(eos - c1) : kC) : 0;
        const float* sBeta = sBetaBuf + 64 * buf;
        cp_async_wait_all();
        wait_bar(barL, phaseL);
        wait_bar(barV, phaseV);
        __syncthreads();
        // ---- (1) running sum of g per key channel: thread (c, qq) sums the 16 tokens of block qq
        {
            const int c = row;
            float acc = 0.f;
#pragma unroll
            for (int i = 16 * qq; i < 16 * qq + 16; ++i) {  // in log2 units: every use is a power of e
                acc = fmaf(i < L ? sG[i * kD + c] : 0.f, kLog2e, acc);
                sG[i * kD + c] = acc;
            }
            sTot[qq * kD + c] = acc;
            __syncthreads();
            float base = 0.f;
#pragma unroll
            for (int p2 = 0; p2 < 3; ++p2)
                if (p2 < qq) base += sTot[p2 * kD + c];
            if (qq > 0) {
#pragma unroll
                for (int i = 16 * qq; i < 16 * qq + 16; ++i) sG[i * kD + c] += base;
            }
            sE[qq * kD + c] = base + acc;  // G at the last token of block qq
            __syncthreads();
            if (qq == 0) {
                float e[4];
#pragma unroll
                for (int I = 0; I < 4; ++I) e[I] = sE[I * kD + c];
                sEGl[c] = exp2f(e[3]);
                sDt[0 * kD + c] = ex2(e[1] - e[0]);
                sDt[1 * kD + c] = ex2(e[2] - e[0]);
                sDt[2 * kD + c] = ex2(e[3] - e[0]);
            } else if (qq == 1) {
                const float e1 = sE[1 * kD + c], e2 = sE[2 * kD + c], e3 = sE[3 * kD + c];
                sDt[3 * kD + c] = ex2(e2 - e1);
                sDt[4 * kD + c] = ex2(e3 - e1);
                sDt[5 * kD + c] = ex2(e3 - e2);
            }
            __syncthreads();
        }
        // ---- (2) operands: row operand RR, column operands CC / KP, B1 = [beta K e^G ; Q e^G]
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int id = tid + kThreads * m, i = id >> 4, cc = id & 15, c = cc * 8, I = i >> 4;
            const uint32_t reg = cc >> 3, ch = cc & 7;
            float kv[8], qv[8], Gv[8], Ev[8];
            unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STK + i * 256 + cc * 16), kv);
            unpack8(*reinterpret_cast<const uint4*>(sm + OFF_STQ + i * 256 + cc * 16), qv);
            *reinterpret_cast<float4*>(Gv) = *reinterpret_cast<const float4*>(sG + i * kD + c);
            *reinterpret_cast<float4*>(Gv + 4) = *reinterpret_cast<const float4*>(sG + i * kD + c + 4);
            *reinterpret_cast<float4*>(Ev) = *reinterpret_cast<const float4*>(sE + I * kD + c);
            *reinterpret_cast<float4*>(Ev + 4) = *reinterpret_cast<const float4*>(sE + I * kD + c + 4);
            const float b = sBeta[i];
            float rk[8], rq[8], bk[8], eq[8], kr[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float f = ex2(Gv[e] - Ev[e]);   // >= 1
                const float r = ex2(Ev[e] - Gv[e]);   // <= 1
                const float eg = ex2(Gv[e]);          // <= 1
                rk[e] = kv[e] * f;
                rq[e] = qv[e] * f;
                bk[e] = b * kv[e] * eg;
                eq[e] = qv[e] * eg;
                kr[e] = kv[e] * r;
            }
            *reinterpret_cast<uint4*>(sm + OFF_RR + reg * 16384 + sw128(i, ch)) = pack8(rk);
            *reinterpret_cast<uint4*>(sm + OFF_RR + reg * 16384 + sw128(64 + i, ch)) = pack8(rq);
            *reinterpret_cast<uint4*>(sm + OFF_B1 + reg * 16384 + sw128(i, ch)) = pack8(bk);
            *reinterpret_cast<uint4*>(sm + OFF_B1 + reg * 16384 + sw128(64 + i, ch)) = pack8(eq);
            // column operands of row blocks J >= I: k_j e^{E_J - G_j} = kr * e^{E_J - E_I}
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                if (J < I) continue;
                float cv[8];
                if (J == I) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) cv[e] = kr[e];
                } else {
                    const int pair = I == 0 ? J - 1 : (I == 1 ? J + 1 : 5);
                    const float* dt = sDt + pair * kD + c;
#pragma unroll
                    for (int e = 0; e < 8; ++e) cv[e] = kr[e] * dt[e];
                }
                if (J == 3)
                    *reinterpret_cast<uint4*>(sm + OFF_KP + reg * 8192 + sw128(i, ch)) = pack8(cv);
                else
                    *reinterpret_cast<uint4*>(sm + OFF_CC + cc_off(J) + reg * (16u * (J + 1) * 128u) + sw128(i, ch)) =
                        pack8(cv);
            }
        }
        fence_proxy_async();
        __syncthreads();
        // k, q, g of the next chunk may now land in the staging buffers
        if (L1 > 0) prefetch_kqg(sm, barL, sBetaBuf + 64 * (buf ^ 1), &tm_k, &tm_q, &tm_g, beta, c1, L1, H, h, tid);
        cp_async_commit();
        // ---- (3) the four row blocks of A (barrier A), then the S0 products (barrier S)
        if (tid == 0) {
            tc_fence_after();
            const uint64_t rr = kdesc(sbase + OFF_RR);
            mma_k128(tbase + TM_A0, rr, 16384, kdesc(sbase + OFF_CC + cc_off(0)), 2048, idesc_bf16_f32(128, 16, false, false));
            mma_k128(tbase + TM_A1, rr, 16384, kdesc(sbase + OFF_CC + cc_off(1)), 4096, idesc_bf16_f32(128, 32, false, false));
            mma_k128(tbase + TM_A2, rr, 16384, kdesc(sbase + OFF_CC + cc_off(2)), 6144, idesc_bf16_f32(128, 48, false, false));
            mma_k128(tbase + TM_A3, rr, 16384, kdesc(sbase + OFF_KP), 8192, idesc_bf16_f32(128, 64, false, false));
            mma_commit(barA);
            mma_k128(tbase + TM_Y, kdesc(sbase + OFF_S), 16384, kdesc(sbase + OFF_B1), 16384, id_s);
            mma_commit(barS);
        }
        wait_bar(barA, phaseA);
        // ---- (4) A_kk (fp32 work array) and A_qk (bf16 operand); warps of key quarters 0, 1
        if (qq < 2) {
            // lane quarter qt holds rows 32qt .. 32qt+31 of [k-rows ; q-rows]: lanes 0-15 belong to row block
            // 2(qt%2) and lanes 16-31 to 2(qt%2)+1; warps with qq = 0 read the first block's columns, qq = 1 the second's.
            const int qt = warp & 3, Ib = 2 * (qt & 1) + qq;
            const bool mine = ((lane >> 4) == qq);
            const int r = 32 * qt + lane;
            const int i = r & 63;
            const bool is_k = r < 64;
            // 64 columns from the block's first column; those past its 16(Ib+1) are masked below
            const uint32_t col0 = Ib == 0 ? TM_A0 : (Ib == 1 ? TM_A1 : (Ib == 2 ? TM_A2 : TM_A3));
            uint32_t a[64];
            {
                uint32_t t0[32], t1[32];
                tmem_ld32_async(tbase + lane_base + col0, t0);
                tmem_ld32_async(tbase + lane_base + col0 + 32, t1);
                tmem_wait_ld(); reg_fence(t0); reg_fence(t1);
#pragma unroll
                for (int e = 0; e < 32; ++e) { a[e] = t0[e]; a[32 + e] = t1[e]; }
            }
            const int ncols = 16 * (Ib + 1);
            if (mine) {
                if (is_k) {
                    const float b = sBeta[i];
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        float4 w;
                        float* wp = reinterpret_cast<float*>(&w);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * j4 + e;
                            wp[e] = (j < i && j < ncols) ? b * __uint_as_float(a[j]) : 0.f;
                        }
                        *reinterpret_cast<float4*>(sAkk + i * kAS + 4 * j4) = w;
                    }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {  // tf32: 32 columns per 128-byte region row
                        float f[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * c4 + e;
                            f[e] = (j <= i && j < ncols) ? to_tf32(__uint_as_float(a[j])) : 0.f;
                        }
                        *reinterpret_cast<float4*>(sm + OFF_AQ + (c4 >> 3) * 8192 + sw128(i, c4 & 7)) =
                            make_float4(f[0], f[1], f[2], f[3]);
                    }
                }
            }
        }
        wait_bar(barS, phaseS);  // the S0 products are done: B1 becomes the solve's work space
        __syncthreads();
        // ---- (5) T = (I + A_kk)^-1 by 16 x 16 blocks (fp32)
        if (lane < 16 && warp < 4) {  // diagonal block `warp`, column `lane`, right-looking (independent updates)
            const int I = warp, c = lane;
            const float* A = sAkk + 16 * I * kAS + 16 * I;
            float x[16];
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) x[r2] = (r2 == c) ? 1.f : 0.f;
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2)
#pragma unroll
                for (int r3 = r2 + 1; r3 < 16; ++r3) x[r3] = fmaf(-A[r3 * kAS + r2], x[r2], x[r3]);
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) sTf[(16 * I + r2) * kAS + 16 * I + c] = x[r2];
        }
        __syncthreads();
        t_offdiag(sAkk, sTf, reinterpret_cast<float*>(sm + OFF_NB), tid);
        {   // T as a tf32 operand (zero above the diagonal blocks); all of T is read before B1 / CC are reused
            float4 f[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int id = tid + kThreads * u, i = id >> 4, c4 = id & 15;
                if ((c4 >> 2) > (i >> 4)) {
                    f[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    const float4 x = *reinterpret_cast<const float4*>(sTf + i * kAS + 4 * c4);
                    f[u] = make_float4(to_tf32(x.x), to_tf32(x.y), to_tf32(x.z), to_tf32(x.w));
                }
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int id = tid + kThreads * u, i = id >> 4, c4 = id & 15;
                *reinterpret_cast<float4*>(sm + OFF_TT + (c4 >> 3) * 8192 + sw128(i, c4 & 7)) = f[u];
            }
        }
        // ---- Z^T = (beta V)^T - Y^T; thread (row, qq) owns tokens 16qq .. 16qq+15
        {
            uint32_t y[16];
            tmem_ld16_async(tbase + lane_base + TM_Y + 16 * qq, y);
            tmem_wait_ld(); reg_fence(y);
            const __nv_bfloat16* sv = reinterpret_cast<const __nv_bfloat16*>(sm + OFF_STV);
            // tf32 row `row` of Z^T: tokens 16qq .. 16qq+15 are 4 chunks of region qq >> 1
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float f[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 16 * qq + 4 * c4 + e;
                    f[e] = to_tf32(sBeta[j] * __bfloat162float(sv[j * kD + row]) - __uint_as_float(y[4 * c4 + e]));
                }
                *reinterpret_cast<float4*>(sm + OFF_ZT + (qq >> 1) * 16384 + sw128(row, 4 * (qq & 1) + c4)) =
                    make_float4(f[0], f[1], f[2], f[3]);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // v of the next chunk may now land
        if (L1 > 0) prefetch_v(sm, barV, &tm_v, c1, h, tid);
        cp_async_commit();
        if (*sAbort) break;
        // ---- (6) V'^T = Z^T T^T
        if (tid == 0) {
            tc_fence_after();
            const uint64_t za = kdesc(sbase + OFF_ZT), tb = kdesc(sbase + OFF_TT);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {  // K = 64 tokens, 8 per tf32 instruction
                const uint32_t reg = ks >> 2, off = (ks & 3) * 32;
                mma_tf32(tbase + TM_V, za + ((reg * 16384 + off) >> 4), tb + ((reg * 8192 + off) >> 4), id_t64,
                         ks > 0 ? 1u : 0u);
            }
            mma_commit(barS);
        }
        wait_mma();
        {
            uint32_t x[16];
            tmem_ld16_async(tbase + lane_base + TM_V + 16 * qq, x);
            tmem_wait_ld(); reg_fence(x);
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)  // tf32 copy for the output product
                *reinterpret_cast<float4*>(sm + OFF_ZT + (qq >> 1) * 16384 + sw128(row, 4 * (qq & 1) + c4)) =
                    make_float4(to_tf32(__uint_as_float(x[4 * c4])), to_tf32(__uint_as_float(x[4 * c4 + 1])),
                                to_tf32(__uint_as_float(x[4 * c4 + 2])), to_tf32(__uint_as_float(x[4 * c4 + 3])));
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {  // bf16 copy for the state update
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(x[8 * c2 + e]);
                *reinterpret_cast<uint4*>(sm + OFF_VB + sw128(row, 2 * qq + c2)) = pack8(f);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // ---- (7) O^T += V'^T A_qk^T;  dS = V'^T (K e^{G_C - G})
        if (tid == 0) {
            tc_fence_after();
            const uint64_t va = kdesc(sbase + OFF_ZT), aq = kdesc(sbase + OFF_AQ);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t reg = ks >> 2, off = (ks & 3) * 32;
                mma_tf32(tbase + TM_O, va + ((reg * 16384 + off) >> 4), aq + ((reg * 8192 + off) >> 4), id_t64, 1u);
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tbase + TM_DS, kdesc(sbase + OFF_VB) + ks * 2, sdesc_sw128(sbase + OFF_KP, 8192, 1024) + ks * 128,
                         id_ds, ks > 0 ? 1u : 0u);
            mma_commit(barS);
        }
        wait_mma();
        // ---- (8) outputs (fp32 staging, then coalesced) and the state update
        {
            uint32_t xo[16], d0[32];
            tmem_ld16_async(tbase + lane_base + TM_O + 16 * qq, xo);
            tmem_ld32_async(tbase + lane_base + TM_DS + 32 * qq, d0);
            tmem_wait_ld(); reg_fence(xo); reg_fence(d0);
#pragma unroll
            for (int e = 0; e < 16; ++e) sO[(16 * qq + e) * kD + row] = scale * __uint_as_float(xo[e]);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[e] = fmaf(s[e], sEGl[32 * qq + e], __uint_as_float(d0[e]));
        }
        write_state_operand();
        tc_fence_before();
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int id = tid + kThreads * m, j = id >> 4, c16 = id & 15;
            if (j < L) {
                float f[8];
                *reinterpret_cast<float4*>(f) = *reinterpret_cast<const float4*>(sO + j * kD + 8 * c16);
                *reinterpret_cast<float4*>(f + 4) = *reinterpret_cast<const float4*>(sO + j * kD + 8 * c16 + 4);
                const int64_t at = ((c0 + j) * H + h) * kD + 8 * c16;
                if (gate) {
                    float gv[8];
                    unpack8(*reinterpret_cast<const uint4*>(gate + at), gv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] *= 1.0f / (1.0f + __expf(-gv[e]));
                }
                *reinterpret_cast<uint4*>(o + at) = pack8(f);
            }
        }
        if (*sAbort) break;
    }

    cp_async_wait_all();
    if (*sAbort) {  // a chunk issued its successor's loads and then stopped: let them land (bounded)
        mbar_wait(barL, phaseL, kWaitLimit);
        mbar_wait(barV, phaseV, kWaitLimit);
    }
    if (final_state && !*sAbort) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(final_state + state_off + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [T, H, 128] tensor of `elem` bytes per value, boxes of [64 tokens][1 head][128 channels], no swizzle.
bool encode_chunk_map(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem, int64_t T, int H) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * elem, (cuuint64_t)H * 128 * elem};
    const cuuint32_t box[3] = {128, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                            float scale, const void* out_gate, void* o, float* final_state, unsigned int* err,
                            cudaStream_t stream) {
    CUtensorMap tq, tk, tv, tg;
    if (!encode_chunk_map(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T_total, H) ||
        !encode_chunk_map(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T_total, H) ||
        !encode_chunk_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, T_total, H) ||
        !encode_chunk_map(&tg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, T_total, H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    chunk_tc_kernel<<<(unsigned)((int64_t)N * H), kThreads, kSmemBytes, stream>>>(
        tq, tk, tv, tg, beta, init_state, cu_seqlens, T_total, H, scale, static_cast<const __nv_bfloat16*>(out_gate),
        static_cast<__nv_bfloat16*>(o), final_state, err);
    return cudaGetLastError();
}

}  // namespace kda
