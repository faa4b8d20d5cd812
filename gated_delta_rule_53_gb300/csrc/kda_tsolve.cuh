// T = (I + A)^-1 for a strictly lower-triangular 64 x 64 fp32 matrix A (the chunk's beta-scaled A_kk),
// by 16 x 16 blocks on the CUDA cores, shared by the forward and backward operand kernels.  The
// triangular solve of the chunk form ("Kimi-K3 深度解析", section 三, "KDA 的关键改进", unrolled over a
// chunk): the diagonal blocks by forward substitution, then the blocks below them from the block
// structure of the inverse.  A and T are [64][kAS] fp32 in shared memory; only the blocks on and below
// the diagonal are read and written.
#pragma once

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kAS = 68;  // fp32 row stride of the A / T work arrays (float4 rows on distinct banks)
constexpr int kNB = 20;  // row stride of the N blocks (float4 rows, eight rows on distinct banks)

// Diagonal block `warp` (warps 0-3), column `lane` (lanes 0-15) of T: right-looking substitution, whose
// updates of later rows are independent of one another.
__device__ __forceinline__ void t_diag_blocks(const float* A, float* T, int warp, int lane) {
    if (lane < 16 && warp < 4) {
        const int I = warp, cl = lane;
        const float* Ad = A + 16 * I * kAS + 16 * I;
        float x[16];
#pragma unroll
        for (int r2 = 0; r2 < 16; ++r2) x[r2] = (r2 == cl) ? 1.f : 0.f;
#pragma unroll
        for (int r2 = 0; r2 < 16; ++r2)
#pragma unroll
            for (int r3 = r2 + 1; r3 < 16; ++r3) x[r3] = fmaf(-Ad[r3 * kAS + r2], x[r2], x[r3]);
#pragma unroll
        for (int r2 = 0; r2 < 16; ++r2) T[(16 * I + r2) * kAS + 16 * I + cl] = x[r2];
    }
}

// One 16 x 16 fp32 block product for 32 threads; thread t owns rows 2 (t / 4) and 2 (t / 4) + 1, columns
// 4 (t % 4) .. +3:   out = sign * ((A0 + w1 A1) B + A3 B3), the A1 and A3 B3 terms optional.  Inlined into
// every call site, where its operands are known shared-memory addresses (shared loads, not generic ones)
// whenever the caller's pointers keep the shared address space.
struct BlkJob {
    const float* a0; const float* a1; const float* b; const float* a3; const float* b3;
    float* out;
    int lda0, lda1, ldb, lda3, ldb3, ldo;
    float w1, sign;
};
__device__ __forceinline__ void blk_job(BlkJob j, int t) {
    const int r0 = 2 * (t >> 2), c = 4 * (t & 3);
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const float* a = pass ? j.a3 : j.a0;
        if (!a) break;
        const int lda = pass ? j.lda3 : j.lda0;
        const float* bp = pass ? j.b3 : j.b;
        const int ldb = pass ? j.ldb3 : j.ldb;
        const float* a1 = pass ? nullptr : j.a1;
        float av[2][16];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int m = 0; m < 16; m += 4) {
                float4 x = *reinterpret_cast<const float4*>(a + (r0 + rr) * lda + m);
                if (a1) {
                    const float4 y = *reinterpret_cast<const float4*>(a1 + (r0 + rr) * j.lda1 + m);
                    x.x = fmaf(j.w1, y.x, x.x); x.y = fmaf(j.w1, y.y, x.y);
                    x.z = fmaf(j.w1, y.z, x.z); x.w = fmaf(j.w1, y.w, x.w);
                }
                av[rr][m] = x.x; av[rr][m + 1] = x.y; av[rr][m + 2] = x.z; av[rr][m + 3] = x.w;
            }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const float4 bv = *reinterpret_cast<const float4*>(bp + m * ldb + c);
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                acc[rr][0] = fmaf(av[rr][m], bv.x, acc[rr][0]); acc[rr][1] = fmaf(av[rr][m], bv.y, acc[rr][1]);
                acc[rr][2] = fmaf(av[rr][m], bv.z, acc[rr][2]); acc[rr][3] = fmaf(av[rr][m], bv.w, acc[rr][3]);
            }
        }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
        *reinterpret_cast<float4*>(j.out + (r0 + rr) * j.ldo + c) =
            make_float4(j.sign * acc[rr][0], j.sign * acc[rr][1], j.sign * acc[rr][2], j.sign * acc[rr][3]);
}

// Blocks of T below the diagonal.  With D = diag(T_00 .. T_33) (inverses of the diagonal blocks of
// I + A_kk) and N = D A_off (A_off: the blocks of A_kk below the diagonal; N is strictly block-lower,
// so N^4 = 0):  (I + A_kk)^-1 = (I + N)^-1 D = (I - N + N^2 - N^3) D.
// Three rounds of independent 16 x 16 products, one warp each: round 1 (the last reader of A) here,
// rounds 2 and 3 in t_offdiag_23.
// N_IJ at nb[slot]: (1,0) 0, (2,0) 1, (3,0) 2, (2,1) 3, (3,1) 4, (3,2) 5; N^2: (2,0) 6, (3,1) 7, (3,0) 8
__device__ __forceinline__ void t_offdiag_1(const float* A, const float* T, float* nb, int tid) {
    const int u = tid >> 5, t = tid & 31;
    BlkJob j{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, kAS, kNB, kAS, kNB, kAS, kAS, 0.f, 1.f};
    if (u < 6) {  // N blocks: (1,0) (2,0) (3,0) (2,1) (3,1) (3,2)
        const int I = u < 3 ? u + 1 : (u < 5 ? u - 1 : 3), J = u < 3 ? 0 : (u < 5 ? 1 : 2);
        j.a0 = T + 16 * I * kAS + 16 * I; j.b = A + 16 * I * kAS + 16 * J; j.out = nb + u * 16 * kNB; j.ldo = kNB;
        blk_job(j, t);
    }
    __syncthreads();
}
__device__ __forceinline__ void t_offdiag_23(float* T, float* nb, int tid) {
    auto Tb = [&](int I, int J) { return T + 16 * I * kAS + 16 * J; };
    auto Nb = [&](int slot) { return nb + slot * 16 * kNB; };
    const int u = tid >> 5, t = tid & 31;
    BlkJob j;
    if (u < 6) {
        j = BlkJob{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, kNB, kNB, kNB, kNB, kNB, kNB, 0.f, 1.f};
        switch (u) {
            case 0: j.a0 = Nb(3); j.b = Nb(0); j.out = Nb(6); break;                            // N21 N10
            case 1: j.a0 = Nb(5); j.b = Nb(3); j.out = Nb(7); break;                            // N32 N21
            case 2: j.a0 = Nb(4); j.b = Nb(0); j.a3 = Nb(5); j.b3 = Nb(1); j.out = Nb(8); break; // N31 N10 + N32 N20
            case 3: j.a0 = Nb(0); j.b = Tb(0, 0); j.ldb = kAS; j.out = Tb(1, 0); j.ldo = kAS; j.sign = -1.f; break;  // T10
            case 4: j.a0 = Nb(3); j.b = Tb(1, 1); j.ldb = kAS; j.out = Tb(2, 1); j.ldo = kAS; j.sign = -1.f; break;  // T21
            default: j.a0 = Nb(5); j.b = Tb(2, 2); j.ldb = kAS; j.out = Tb(3, 2); j.ldo = kAS; j.sign = -1.f; break; // T32
        }
        blk_job(j, t);
    }
    __syncthreads();
    // T_30 = (N^2_30 - N_30 - N^3_30) D_0 with N^3_30 D_0 = N^2_31 N_10 D_0 = -N^2_31 T_10
    if (u < 3) {
        j = BlkJob{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, kNB, kNB, kAS, kNB, kAS, kAS, -1.f, 1.f};
        switch (u) {
            case 0: j.a0 = Nb(8); j.a1 = Nb(2); j.b = Tb(0, 0); j.a3 = Nb(7); j.b3 = Tb(1, 0); j.out = Tb(3, 0); break;
            case 1: j.a0 = Nb(6); j.a1 = Nb(1); j.b = Tb(0, 0); j.out = Tb(2, 0); break;  // T20
            default: j.a0 = Nb(7); j.a1 = Nb(4); j.b = Tb(1, 1); j.out = Tb(3, 1); break; // T31
        }
        blk_job(j, t);
    }
    __syncthreads();
}

}  // namespace
}  // namespace kda
