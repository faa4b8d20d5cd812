// The two passes of kda_chunk_bwd along the chains on the tcgen05 tensor cores (bf16 inputs).
//
// Per chunk of a (sequence, head) chain, taken from the last chunk to the first, with dS the gradient of
// the state at the chunk's end ("Kimi-K3 深度解析", section 三, "KDA 的关键改进", unrolled over a chunk
// as in the chunk_kda operator of "Kimi K3 架构全景", section 02; the chain rule through the chunk form):
//   dV'^T = dS Kr^T + scale dO^T A_qk                      [dv x C]
//   dZ^T  = dV'^T T                                        [dv x C]   (T = (I + A_kk)^-1)
//   dS   <- dS Diag(gamma) + scale dO^T Qg - (Diag(beta) dZ)^T Kg      [dv x dk]
// One CTA per chain: 16 warps hold dS in fp32 registers (thread (r, quarter): row r, key channels
// 32 quarter .. +31) and do the element-wise work, one warp issues every product and copy.  Every
// product has M = dv = 128 (row r in TMEM lane r) and keeps fp32-level accuracy: each fp32 operand is
// split into bf16 hi + lo (x = hi + lo to about 16 bits) and the product taken as hi.hi + hi.lo + lo.hi
// (the bf16 dO is exact and enters once).  The state-side operands (dS, dV', -beta dZ) are written to
// TMEM by the state warps; the chunk's tiles (Kr, scale Qg, Kg, scale A_qk, T as bf16 hi/lo) come from
// bwd_prep_kernel in the layouts the products read, and dO by TMA from its tensor.
//
// Outputs as the CUDA-core reverse pass: dS_next of every chunk (the gradient at the chunk's end), dZ
// for every token, the gradient of the initial state.  The forward pass along the chains that the
// backward recomputes first (the state entering every chunk, R and V') runs the same way, below.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_bwd_tc.cuh"
#include "kda_common.cuh"
#include "kda_tc.cuh"
#include "kda_tsolve.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr int kSimt = 512;
constexpr int kThreads = kSimt + 32;
constexpr int kMmaWarp = kSimt / 32;
constexpr uint32_t kWaitLimit = 1u << 22;

// named barriers between the state warps and the product warp (id 0 is __syncthreads), all kThreads each
constexpr int NB_S = 1;  // state -> products: dS hi/lo in TMEM (and the previous chunk's gamma, beta read)
constexpr int NB_1 = 2;  // products -> state: dV'^T in TMEM
constexpr int NB_V = 3;  // state -> products: dV' hi/lo in TMEM
constexpr int NB_2 = 4;  // products -> state: dZ^T in TMEM
constexpr int NB_Z = 5;  // state -> products: -beta dZ hi/lo in TMEM (beta read)
constexpr int NB_3 = 6;  // products -> state: the dS increment in TMEM

// shared memory: one buffer per tile, two for scale A_qk + dO (the first product of a chunk is issued
// during the chunk after it)
constexpr uint32_t R_KR = 0;            // Kr hi, lo                     [64 t][128 c] x 2
constexpr uint32_t R_QG = 32768;        // scale Qg hi, lo               [64 t][128 c] x 2
constexpr uint32_t R_KG = 65536;        // Kg hi, lo                     [64 t][128 c] x 2
constexpr uint32_t R_TT = 98304;        // T hi, lo                      [64 s][64 t] x 2
constexpr uint32_t R_AQ = 114688;       // scale A_qk hi, lo, two chunks [64 s][64 t] x 2 x 2
constexpr uint32_t R_DO = 147456;       // dO, two chunks                [64 t][64 r] x 2 regions x 2
constexpr uint32_t R_GAM = 180224;      // gamma fp32 [128] (with Kg)
constexpr uint32_t R_BETA = 180736;     // beta fp32 [64] (with T)
constexpr uint32_t R_BAR = 181248;      // mbarriers: KR, QG, KG, TT, AQ/DO x2, D1, D2, D3
constexpr uint32_t R_MISC = R_BAR + 128;
constexpr uint32_t R_DSN = 182272;      // dS_next fp32 staged for its TMA store: two boxes of [128 rows][32 channels]
                                        // at a time (channels 0-63, then 64-127), 128-byte swizzle
constexpr uint32_t kSmem = R_DSN + 32768 + 1024;
static_assert(R_AQ % 1024 == 0 && R_DO % 1024 == 0 && R_TT % 1024 == 0 && R_BAR % 8 == 0 && R_DSN % 1024 == 0 &&
                  R_MISC + 16 <= R_DSN,
              "alignment");
static_assert(kSmem <= 232448, "shared memory");

// TMEM columns
constexpr uint32_t TM_D1 = 0, TM_D2 = 64, TM_D3 = 128, TM_SH = 256, TM_SL = 320, TM_VH = 384, TM_VL = 416,
                   TM_ZH = 448, TM_ZL = 480;

__device__ __forceinline__ void nb_sync(int id) { asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kThreads) : "memory"); }
// Element (token t, value row r) of a chunk's [64 t][128 r] fp32 tile staged as four boxes of [64 t][32 r]
// (boxes 8 KB apart, 128-byte swizzle): thread (r, quarter) writes its tokens 16 quarter .. +15.
__device__ __forceinline__ void stage_token_tile(uint8_t* tile, int r, int quarter, const float (&x)[16]) {
    uint8_t* box = tile + (r >> 5) * 8192;
    const int col = r & 31;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int t = 16 * quarter + e;
        *reinterpret_cast<float*>(box + t * 128 + ((((col >> 2) ^ (t & 7))) << 4) + (col & 3) * 4) = x[e];
    }
}

// The 16 state warps among themselves (named barrier 7; the product warp does not take part).
__device__ __forceinline__ void state_sync() { asm volatile("bar.sync 7, %0;" ::"n"(kSimt) : "memory"); }
__device__ __forceinline__ void nb_arrive(int id) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(kThreads) : "memory");
}
__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return sdesc_sw128(saddr, 16, 1024); }

// One chunk's tiles on their way to L2 ahead of the copies that read them: its blob (131,840 bytes) and its
// 64 rows of a bf16 [T, H, 128] tensor (rows past the sequence's end skipped); one 128-byte line per thread
// per round.
__device__ __forceinline__ void prefetch_chunk(const uint8_t* blob, const __nv_bfloat16* x, int64_t tok0, int L, int H,
                                               int h, int tid, int nthreads) {
    constexpr int kBlobLines = (int)(kBwdBlobBytes / 128);
    static_assert(kBwdBlobBytes % 128 == 0, "whole lines");
    for (int i = tid; i < kBlobLines + 2 * kC; i += nthreads) {
        if (i < kBlobLines) {
            prefetch_l2(blob + 128 * i);
        } else {
            const int r = (i - kBlobLines) >> 1;
            if (r < L) prefetch_l2(x + ((tok0 + r) * H + h) * kD + 64 * ((i - kBlobLines) & 1));
        }
    }
}

// x = hi + lo, both bf16 (round to nearest even), packed in pairs
__device__ __forceinline__ void split_pairs(const float* x, int n2, uint32_t* hi, uint32_t* lo) {
    for (int j = 0; j < n2; ++j) {
        const float a = x[2 * j], b = x[2 * j + 1];
        const uint32_t h = pack_bf16x2(a, b);
        hi[j] = h;
        lo[j] = pack_bf16x2(a - bf16_lo(h), b - bf16_hi(h));
    }
}

template <typename InT>
__global__ void __launch_bounds__(kThreads, 1)
bwd_state_tc_kernel(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dsn,
                    const __grid_constant__ CUtensorMap tm_dz,
                    const __nv_bfloat16* __restrict__ d_o,
                    const float* __restrict__ d_final, const int32_t* __restrict__ cu, int64_t T_total, int H,
                    const uint8_t* __restrict__ blobs, float* __restrict__ d_init, float* __restrict__ dS_next,
                    float* __restrict__ dZ_out, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array (accesses through `sm` stay shared ones)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int nch = (int)((eos - bos + kC - 1) / kC);
    const int row = tid & 127, qq = (tid >> 7) & 3;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int64_t state_off = (int64_t)chain * kD * kD;

    // copy barriers bKR + w: 0 Kr, 1 scale Qg, 2 Kg and gamma, 3 T and beta, 4 + j scale A_qk and dO (two)
    uint64_t* bKR = reinterpret_cast<uint64_t*>(sm + R_BAR);
    uint64_t* bAD = bKR + 4;
    uint64_t* bD1 = bKR + 6;
    uint64_t* bD2 = bKR + 7;
    uint64_t* bD3 = bKR + 8;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + R_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + R_MISC + 4);  // a wait ran out (product warp)
    volatile int* sStop = reinterpret_cast<volatile int*>(sm + R_MISC + 8);   // both sides stop after this chunk
    if (tid == 0) {
        for (int i = 0; i < 9; ++i) mbar_init(bKR + i, 1);
        fence_mbar_init();
        *sAbort = 0;
        *sStop = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    // chunk ci of the chain (0 = first): its slot's operands and its first token
    auto blob_of = [&](int ci) {
        const int64_t c0 = bos + (int64_t)kC * ci;
        return blobs + ((c0 / kC + n) * H + h) * (int64_t)kBwdBlobBytes;
    };

    if (warp == kMmaWarp) {
        // ======== products and copies (one warp; products from an elected lane, copies from lane 0) ========
        auto wait = [&](uint64_t* b, uint32_t ph) {
            if (!mbar_wait(b, ph, kWaitLimit)) {
                *sAbort = 1;
                raise_device_error(err, kErrMbarTimeout);
            }
        };
        // phase bit per barrier, flipped when the copy it counts is consumed; `iss` flips when one is issued
        uint32_t ph = 0, iss = 0;
        auto copy = [&](int which, uint32_t dst, const uint8_t* src, uint32_t bytes, uint32_t dst2, const uint8_t* src2,
                        uint32_t bytes2) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bKR + which, bytes + bytes2);
                bulk_load(sm + dst, src, bytes, bKR + which);
                if (bytes2) bulk_load(sm + dst2, src2, bytes2, bKR + which);
            }
            __syncwarp();
            iss ^= 1u << which;
        };
        auto load_kr = [&](int ci) { copy(0, R_KR, blob_of(ci) + kBB_KR, 32768, 0, nullptr, 0); };
        auto load_qg = [&](int ci) { copy(1, R_QG, blob_of(ci) + kBB_QG, 32768, 0, nullptr, 0); };
        auto load_kg = [&](int ci) { copy(2, R_KG, blob_of(ci) + kBB_KG, 32768, R_GAM, blob_of(ci) + kBB_GAM, 512); };
        auto load_tt = [&](int ci) { copy(3, R_TT, blob_of(ci) + kBB_TT, 16384, R_BETA, blob_of(ci) + kBB_BETA, 256); };
        auto load_ad = [&](int ci, int j) {  // scale A_qk from the workspace, dO by TMA from its tensor
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bAD + j, 16384 + 16384);
                bulk_load(sm + R_AQ + j * 16384, blob_of(ci) + kBB_AQ, 16384, bAD + j);
                const int tok = (int)(bos + (int64_t)kC * ci);
                tma_load_3d(sm + R_DO + j * 16384, &tm_do, 0, h, tok, bAD + j);
                tma_load_3d(sm + R_DO + j * 16384 + 8192, &tm_do, 64, h, tok, bAD + j);
            }
            __syncwarp();
            iss ^= 1u << (4 + j);
        };
        auto use = [&](int which) {
            wait(bKR + which, (ph >> which) & 1u);
            ph ^= 1u << which;
        };
        const uint32_t id_d1s = idesc_bf16_f32(128, 64, false, false);  // A = dS (TMEM), B = Kr (K-major)
        const uint32_t id_do64 = idesc_bf16_f32(128, 64, true, true);   // A = dO^T (MN-major), B = A_qk (MN-major)
        const uint32_t id_t = idesc_bf16_f32(128, 64, false, true);     // A = dV'^T (TMEM), B = T (MN-major)
        const uint32_t id_do128 = idesc_bf16_f32(128, 128, true, true); // A = dO^T, B = scale Qg (MN-major)
        const uint32_t id_z = idesc_bf16_f32(128, 128, false, true);    // A = -beta dZ^T (TMEM), B = Kg (MN-major)
        uint32_t p1 = 0, p2 = 0, p3 = 0;
        // D1 <- scale dO^T A_qk of chunk ci (buffer j): the part of dV' that does not depend on dS
        auto issue_1b = [&](int j) {
            use(4 + j);
            tc_fence_after();
            const uint64_t dd = sdesc_sw128(sbase + R_DO + j * 16384, 8192, 1024);
            const uint64_t ah = sdesc_sw128(sbase + R_AQ + j * 16384, 8192, 1024);
            const uint64_t al = sdesc_sw128(sbase + R_AQ + j * 16384 + 8192, 8192, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + TM_D1, dd + ks * 128, ah + ks * 128, id_do64, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + TM_D1, dd + ks * 128, al + ks * 128, id_do64, 1u);
        };
        const int last = nch - 1;
        if (nch > 0) {
            load_ad(last, last & 1);
            load_kr(last);
            load_qg(last);
            load_kg(last);
            load_tt(last);
            if (last >= 1) load_ad(last - 1, (last - 1) & 1);
            issue_1b(last & 1);
        }
        for (int ci = last; ci >= 0; --ci) {
            const int j = ci & 1;
            const bool more = ci >= 1;
            nb_sync(NB_S);  // dS hi/lo of this chunk in TMEM; gamma and beta of the chunk after it read
            if (ci < last) load_kg(ci);
            // ---- D1 += dS Kr^T (hi.hi + hi.lo + lo.hi): dV'^T
            use(0);
            tc_fence_after();
            {
                const uint32_t kh = sbase + R_KR, kl = sbase + R_KR + 16384;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + TM_D1, tbase + TM_SH + 8 * ks, kdesc(kh + (ks >> 2) * 8192) + (ks & 3) * 2, id_d1s, 1u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + TM_D1, tbase + TM_SH + 8 * ks, kdesc(kl + (ks >> 2) * 8192) + (ks & 3) * 2, id_d1s, 1u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + TM_D1, tbase + TM_SL + 8 * ks, kdesc(kh + (ks >> 2) * 8192) + (ks & 3) * 2, id_d1s, 1u);
            }
            mma_commit(bD1);
            // ---- D3 <- scale dO^T Qg (independent of the chain): issued behind D1, before it is read
            use(1);
            tc_fence_after();
            {
                const uint64_t dd = sdesc_sw128(sbase + R_DO + j * 16384, 8192, 1024);
                const uint64_t qh = sdesc_sw128(sbase + R_QG, 8192, 1024), ql = sdesc_sw128(sbase + R_QG + 16384, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + TM_D3, dd + ks * 128, qh + ks * 128, id_do128, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + TM_D3, dd + ks * 128, ql + ks * 128, id_do128, 1u);
            }
            wait(bD1, p1);
            p1 ^= 1u;
            tc_fence_before();
            nb_arrive(NB_1);
            if (more) load_kr(ci - 1);  // Kr consumed
            // ---- D2 = dV'^T T (hi.hi + hi.lo + lo.hi): dZ^T
            nb_sync(NB_V);
            use(3);
            tc_fence_after();
            {
                const uint64_t th = sdesc_sw128(sbase + R_TT, 8192, 1024), tl = sdesc_sw128(sbase + R_TT + 8192, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D2, tbase + TM_VH + 8 * ks, th + ks * 128, id_t, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D2, tbase + TM_VH + 8 * ks, tl + ks * 128, id_t, 1u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D2, tbase + TM_VL + 8 * ks, th + ks * 128, id_t, 1u);
            }
            mma_commit(bD2);
            wait(bD2, p2);
            p2 ^= 1u;
            tc_fence_before();
            nb_arrive(NB_2);
            if (more) load_qg(ci - 1);         // scale Qg consumed (the dO^T Qg product is complete)
            if (ci >= 2) load_ad(ci - 2, j);   // this chunk's A_qk and dO consumed
            // ---- D3 += (-beta dZ)^T Kg (hi.hi + hi.lo + lo.hi): the dS increment
            nb_sync(NB_Z);  // the state warps have read this chunk's beta
            if (more) load_tt(ci - 1);
            use(2);
            tc_fence_after();
            {
                const uint64_t gh = sdesc_sw128(sbase + R_KG, 8192, 1024), gl = sdesc_sw128(sbase + R_KG + 16384, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D3, tbase + TM_ZH + 8 * ks, gh + ks * 128, id_z, 1u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D3, tbase + TM_ZH + 8 * ks, gl + ks * 128, id_z, 1u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + TM_D3, tbase + TM_ZL + 8 * ks, gh + ks * 128, id_z, 1u);
            }
            mma_commit(bD3);
            wait(bD3, p3);
            p3 ^= 1u;
            const bool stop = *sAbort != 0;
            if (stop) *sStop = 1;  // written only here, read by the state warps after this hand-off
            tc_fence_before();
            nb_arrive(NB_3);
            if (stop) break;
            if (more) issue_1b(j ^ 1);  // D1 of the chunk before this one (D1 was read before NB_V)
        }
        if (*sAbort && lane == 0) {  // let copies still in flight land (bounded) before the CTA exits
            for (int w = 0; w < 6; ++w)
                if (((iss ^ ph) >> w) & 1u) mbar_wait(bKR + w, (ph >> w) & 1u, kWaitLimit);
        }
        __syncwarp();
    } else {
        // ======== the gradient of the state: thread (row, qq) holds row `row`, key channels 32 qq .. +31 ========
        float s[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 x = d_final ? *reinterpret_cast<const float4*>(d_final + state_off + (int64_t)row * kD + 32 * qq + e)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            s[e] = x.x; s[e + 1] = x.y; s[e + 2] = x.z; s[e + 3] = x.w;
        }
        const float* sGam = reinterpret_cast<const float*>(sm + R_GAM);
        const float* sBeta = reinterpret_cast<const float*>(sm + R_BETA);
        for (int ci = nch - 1; ci >= 0; --ci) {
            const int64_t c0 = bos + (int64_t)kC * ci;
            const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
            const int64_t base = (c0 / kC + n) * H + h;
            if (ci >= 2) {  // the tiles two chunks on (in this pass's order) on their way to L2
                const int64_t c2 = c0 - 2 * kC;
                prefetch_chunk(blob_of(ci - 2), d_o, c2, kC, H, h, tid, kSimt);
            }
            {  // dS as bf16 hi + lo, the A operand of dS Kr^T
                uint32_t hi[16], lo[16];
                split_pairs(s, 16, hi, lo);
                tmem_st16(tbase + lane_base + TM_SH + 16 * qq, hi);
                tmem_st16(tbase + lane_base + TM_SL + 16 * qq, lo);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_S);
            // dS at the chunk's end, for the per-chunk kernel, once the product warp has it: staged and stored by
            // TMA, channels 0-63 (quarters 0, 1) then 64-127 (the tile is free at the start: its previous copies
            // finished reading before NB_3)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                if (half) {
                    if (tid == 0) bulk_wait_read();
                    state_sync();
                }
                if ((qq >> 1) == half) {
                    uint8_t* box = sm + R_DSN + (qq & 1) * 16384 + row * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<float4*>(box + ((c ^ (row & 7)) << 4)) =
                            make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
                }
                fence_proxy_async();
                state_sync();
                if (tid == 0) {
                    tma_store_2d(&tm_dsn, sm + R_DSN, 64 * half, (int)(base * kD));
                    tma_store_2d(&tm_dsn, sm + R_DSN + 16384, 64 * half + 32, (int)(base * kD));
                    bulk_commit();
                }
            }
            // ---- dV'^T: tokens 16 qq .. +15 of row `row`, back to TMEM as hi + lo
            nb_sync(NB_1);
            tc_fence_after();
            {
                uint32_t y[16];
                tmem_ld16_async(tbase + lane_base + TM_D1 + 16 * qq, y);
                tmem_wait_ld(); reg_fence(y);
                float x[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(y[e]);
                uint32_t hi[8], lo[8];
                split_pairs(x, 8, hi, lo);
                tmem_st8(tbase + lane_base + TM_VH + 8 * qq, hi);
                tmem_st8(tbase + lane_base + TM_VL + 8 * qq, lo);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_V);
            // ---- dZ^T: out for every token of the chunk; -beta dZ back to TMEM as hi + lo
            nb_sync(NB_2);
            tc_fence_after();
            {
                uint32_t y[16];
                tmem_ld16_async(tbase + lane_base + TM_D2 + 16 * qq, y);
                tmem_wait_ld(); reg_fence(y);
                float z[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) z[e] = -sBeta[16 * qq + e] * __uint_as_float(y[e]);
                uint32_t hi[8], lo[8];
                split_pairs(z, 8, hi, lo);
                tmem_st8(tbase + lane_base + TM_ZH + 8 * qq, hi);
                tmem_st8(tbase + lane_base + TM_ZL + 8 * qq, lo);
                tmem_wait_st();
                tc_fence_before();
                nb_arrive(NB_Z);
                // dZ out, once the product warp has -beta dZ: a whole chunk through the dS_next tile by TMA (once
                // dS_next's copies have read it), the sequence's partial last chunk row by row
                float dzv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) dzv[e] = __uint_as_float(y[e]);
                if (L == kC) {
                    if (tid == 0) bulk_wait_read();
                    state_sync();
                    stage_token_tile(sm + R_DSN, row, qq, dzv);
                    fence_proxy_async();
                    state_sync();
                    if (tid == 0) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) tma_store_3d(&tm_dz, sm + R_DSN + b * 8192, 32 * b, h, (int)c0);
                        bulk_commit();
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int t = 16 * qq + e;
                        if (t < L) dZ_out[((c0 + t) * H + h) * kD + row] = dzv[e];
                    }
                }
            }
            // ---- dS <- dS Diag(gamma) + increment.  A stop is taken here only, where the product warp
            //      takes it (it reads the flag before this hand-off), so both sides leave at the same barrier.
            if (tid == 0) bulk_wait_read();  // the staging tile is free for the next chunk past NB_3
            nb_sync(NB_3);
            tc_fence_after();
            if (*sStop) break;
            {
                uint32_t d3[32];
                tmem_ld32_async(tbase + lane_base + TM_D3 + 32 * qq, d3);
                float gm[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(gm + e) = *reinterpret_cast<const float4*>(sGam + 32 * qq + e);
                tmem_wait_ld(); reg_fence(d3);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[e] = fmaf(s[e], gm[e], __uint_as_float(d3[e]));
            }
        }
        if (tid == 0) bulk_wait_all();  // the dS_next copies are complete before the CTA ends
        if (!*sStop && d_init) {
            float* dst = d_init + state_off + (int64_t)row * kD + 32 * qq;
#pragma unroll
            for (int e = 0; e < 32; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(s[e], s[e + 1], s[e + 2], s[e + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ============================ the forward pass along the chains ============================
// Per chunk, from the chain's initial state S0, the values the per-chunk gradient kernels read:
//   R^T  = V^T - S0 Kg^T            (kept, fp32)
//   V'^T = (Diag(beta) R)^T T^T     (kept, fp32; V' = T Diag(beta) R)
//   S   <- S0 Diag(gamma) + V'^T Kr  (S0 of every chunk kept, fp32)
// The same structure as the reverse pass: 16 state warps hold S in fp32 registers, one warp issues the
// products (bf16 hi.hi + hi.lo + lo.hi) and copies; v arrives by TMA from its tensor.
constexpr uint32_t F_KG = 0;          // Kg hi, lo      [64 t][128 c] x 2 (K-major B of S Kg^T)
constexpr uint32_t F_KR = 32768;      // Kr hi, lo      [64 t][128 c] x 2 (MN-major B of V'^T Kr)
constexpr uint32_t F_TT = 65536;      // T hi, lo       [64][64] x 2 (K-major B of (beta R)^T T^T)
constexpr uint32_t F_V = 81920;       // v              [64 t][64 r] x 2 regions
constexpr uint32_t F_GAM = 98304;     // gamma fp32 [128] (with Kr)
constexpr uint32_t F_BETA = 98816;    // beta fp32 [64] (with T)
constexpr uint32_t F_BAR = 99328;     // mbarriers: KG (even chunks), KR, TT, V, D1, D2, D3, KG (odd chunks)
constexpr uint32_t F_MISC = F_BAR + 64;
constexpr uint32_t F_KG1 = 100352;    // Kg hi, lo of odd chunks (even ones at F_KG): copied two chunks ahead
constexpr uint32_t F_S0 = 133120;     // S0 fp32 staged for its TMA store: four boxes of [128 rows][32 channels],
                                      // 128-byte swizzle
constexpr uint32_t F_RV = 198656;     // R, then V', of a whole chunk staged for their TMA stores: four boxes of
                                      // [64 tokens][32 rows], 128-byte swizzle
constexpr uint32_t kFwdSmem = F_RV + 32768 + 1024;
static_assert(F_V % 1024 == 0 && F_TT % 1024 == 0 && F_BAR % 8 == 0 && F_KG1 % 1024 == 0 && F_MISC + 16 <= F_KG1 &&
                  F_S0 % 1024 == 0 && F_S0 >= F_KG1 + 32768 && F_RV % 1024 == 0 && F_RV >= F_S0 + 65536 &&
                  kFwdSmem <= 232448,
              "alignment");

__global__ void __launch_bounds__(kThreads, 1)
bwd_fwd_state_tc_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_s0,
                        const __grid_constant__ CUtensorMap tm_r, const __grid_constant__ CUtensorMap tm_vp,
                        const __nv_bfloat16* __restrict__ v,
                        const float* __restrict__ init_state, const int32_t* __restrict__ cu, int64_t T_total, int H,
                        const uint8_t* __restrict__ blobs, float* __restrict__ S0s, float* __restrict__ Rb,
                        float* __restrict__ Vp, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array (accesses through `sm` stay shared ones)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int nch = (int)((eos - bos + kC - 1) / kC);
    const int row = tid & 127, qq = (tid >> 7) & 3;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // copy barriers bB + w: 0 Kg (even chunks), 1 Kr and gamma, 2 T and beta, 3 v; then the three product barriers;
    // bB + 7 Kg (odd chunks)
    uint64_t* bB = reinterpret_cast<uint64_t*>(sm + F_BAR);
    uint64_t* bD1 = bB + 4;
    uint64_t* bD2 = bB + 5;
    uint64_t* bD3 = bB + 6;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + F_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + F_MISC + 4);
    volatile int* sStop = reinterpret_cast<volatile int*>(sm + F_MISC + 8);
    if (tid == 0) {
        for (int i = 0; i < 8; ++i) mbar_init(bB + i, 1);
        fence_mbar_init();
        *sAbort = 0;
        *sStop = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    auto blob_of = [&](int ci) {
        const int64_t c0 = bos + (int64_t)kC * ci;
        return blobs + ((c0 / kC + n) * H + h) * (int64_t)kBwdBlobBytes;
    };
    // TMEM: D1 = S Kg^T, D2 = V'^T, D3 = the state increment; S, beta R and V' as bf16 hi/lo
    constexpr uint32_t F_D1 = 0, F_D2 = 64, F_D3 = 128, F_SH = 256, F_SL = 320, F_RH = 384, F_RL = 416,
                       F_VH = 448, F_VL = 480;

    if (warp == kMmaWarp) {
        auto wait = [&](uint64_t* b, uint32_t ph) {
            if (!mbar_wait(b, ph, kWaitLimit)) {
                *sAbort = 1;
                raise_device_error(err, kErrMbarTimeout);
            }
        };
        uint32_t ph = 0, iss = 0;
        auto copy = [&](int which, uint32_t dst, const uint8_t* src, uint32_t bytes, uint32_t dst2, const uint8_t* src2,
                        uint32_t bytes2) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bB + which, bytes + bytes2);
                bulk_load(sm + dst, src, bytes, bB + which);
                if (bytes2) bulk_load(sm + dst2, src2, bytes2, bB + which);
            }
            __syncwarp();
            iss ^= 1u << which;
        };
        auto load_kg = [&](int ci) {
            copy((ci & 1) ? 7 : 0, (ci & 1) ? F_KG1 : F_KG, blob_of(ci) + kBB_KG, 32768, 0, nullptr, 0);
        };
        auto load_kr = [&](int ci) { copy(1, F_KR, blob_of(ci) + kBB_KR, 32768, F_GAM, blob_of(ci) + kBB_GAM, 512); };
        auto load_tt = [&](int ci) { copy(2, F_TT, blob_of(ci) + kBB_TT, 16384, F_BETA, blob_of(ci) + kBB_BETA, 256); };
        auto load_v = [&](int ci) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(bB + 3, 16384);
                const int tok = (int)(bos + (int64_t)kC * ci);
                tma_load_3d(sm + F_V, &tm_v, 0, h, tok, bB + 3);
                tma_load_3d(sm + F_V + 8192, &tm_v, 64, h, tok, bB + 3);
            }
            __syncwarp();
            iss ^= 1u << 3;
        };
        auto use = [&](int which) {
            wait(bB + which, (ph >> which) & 1u);
            ph ^= 1u << which;
        };
        const uint32_t id_kg = idesc_bf16_f32(128, 64, false, false);   // A = S (TMEM), B = Kg (K-major)
        const uint32_t id_tt = idesc_bf16_f32(128, 64, false, false);   // A = (beta R)^T (TMEM), B = T (K-major)
        const uint32_t id_kr = idesc_bf16_f32(128, 128, false, true);   // A = V'^T (TMEM), B = Kr (MN-major)
        uint32_t p1 = 0, p2 = 0, p3 = 0;
        if (nch > 0) {
            load_kg(0);
            load_v(0);
            load_tt(0);
            load_kr(0);
            if (nch > 1) load_kg(1);
        }
        for (int ci = 0; ci < nch; ++ci) {
            const bool more = ci + 1 < nch;
            nb_sync(NB_S);  // S hi/lo in TMEM; gamma of the chunk before read
            if (ci > 0) load_kr(ci);
            // ---- D1 = S Kg^T (hi.hi + hi.lo + lo.hi)
            use((ci & 1) ? 7 : 0);
            tc_fence_after();
            {
                const uint32_t kh = sbase + ((ci & 1) ? F_KG1 : F_KG), kl = kh + 16384;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + F_D1, tbase + F_SH + 8 * ks, kdesc(kh + (ks >> 2) * 8192) + (ks & 3) * 2, id_kg, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + F_D1, tbase + F_SH + 8 * ks, kdesc(kl + (ks >> 2) * 8192) + (ks & 3) * 2, id_kg, 1u);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ta(tbase + F_D1, tbase + F_SL + 8 * ks, kdesc(kh + (ks >> 2) * 8192) + (ks & 3) * 2, id_kg, 1u);
            }
            mma_commit(bD1);
            use(3);  // v, read by the state warps after the next hand-off
            use(2);  // T and beta (beta read by the state warps)
            wait(bD1, p1);
            p1 ^= 1u;
            tc_fence_before();
            nb_arrive(NB_1);
            if (ci + 2 < nch) load_kg(ci + 2);  // this buffer's Kg consumed
            // ---- D2 = (beta R)^T T^T (hi.hi + hi.lo + lo.hi) = V'^T
            nb_sync(NB_V);  // beta R hi/lo in TMEM; v and beta read
            if (more) load_v(ci + 1);
            tc_fence_after();
            {
                const uint32_t th = sbase + F_TT, tl = sbase + F_TT + 8192;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D2, tbase + F_RH + 8 * ks, kdesc(th) + ks * 2, id_tt, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D2, tbase + F_RH + 8 * ks, kdesc(tl) + ks * 2, id_tt, 1u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D2, tbase + F_RL + 8 * ks, kdesc(th) + ks * 2, id_tt, 1u);
            }
            mma_commit(bD2);
            wait(bD2, p2);
            p2 ^= 1u;
            tc_fence_before();
            nb_arrive(NB_2);
            if (more) load_tt(ci + 1);  // T consumed, beta read before NB_V
            // ---- D3 = V'^T Kr (hi.hi + hi.lo + lo.hi)
            nb_sync(NB_Z);  // V' hi/lo in TMEM
            use(1);
            tc_fence_after();
            {
                const uint64_t rh = sdesc_sw128(sbase + F_KR, 8192, 1024), rl = sdesc_sw128(sbase + F_KR + 16384, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D3, tbase + F_VH + 8 * ks, rh + ks * 128, id_kr, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D3, tbase + F_VH + 8 * ks, rl + ks * 128, id_kr, 1u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(tbase + F_D3, tbase + F_VL + 8 * ks, rh + ks * 128, id_kr, 1u);
            }
            mma_commit(bD3);
            wait(bD3, p3);
            p3 ^= 1u;
            const bool stop = *sAbort != 0;
            if (stop) *sStop = 1;
            tc_fence_before();
            nb_arrive(NB_3);
            if (stop) break;
        }
        if (*sAbort && lane == 0) {
            for (int w = 0; w < 8; ++w)
                if (w < 4 || w == 7)
                    if (((iss ^ ph) >> w) & 1u) mbar_wait(bB + w, (ph >> w) & 1u, kWaitLimit);
        }
        __syncwarp();
    } else {
        float s[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 x = init_state ? *reinterpret_cast<const float4*>(init_state + (int64_t)chain * kD * kD +
                                                                            (int64_t)row * kD + 32 * qq + e)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
            s[e] = x.x; s[e + 1] = x.y; s[e + 2] = x.z; s[e + 3] = x.w;
        }
        const float* sGam = reinterpret_cast<const float*>(sm + F_GAM);
        const float* sBeta = reinterpret_cast<const float*>(sm + F_BETA);
        // Each operand goes to TMEM first and is handed to the product warp; its global copy (S0, R, V') is
        // stored after the hand-off, while the next product runs.
        for (int ci = 0; ci < nch; ++ci) {
            const int64_t c0 = bos + (int64_t)kC * ci;
            const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
            const int64_t base = (c0 / kC + n) * H + h;
            {  // the state entering the chunk, as hi + lo
                uint32_t hi[16], lo[16];
                split_pairs(s, 16, hi, lo);
                tmem_st16(tbase + lane_base + F_SH + 16 * qq, hi);
                tmem_st16(tbase + lane_base + F_SL + 16 * qq, lo);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_S);
            {  // ... and kept: staged (the tile is free: its previous copies finished reading before NB_3), then
               // stored by TMA as four boxes of channels 32 qq .. +31
                uint8_t* box = sm + F_S0 + qq * 16384 + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(box + ((c ^ (row & 7)) << 4)) =
                        make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]);
                fence_proxy_async();
                state_sync();
                if (tid == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) tma_store_2d(&tm_s0, sm + F_S0 + b * 16384, 32 * b, (int)(base * kD));
                    bulk_commit();
                }
            }
            // v[t][row] of the chunk's tokens 16 qq .. +15 (the TMA tile: [64 t][64 r] per half of the rows), read
            // as soon as its copy has landed (phase ci % 2 of its barrier), before the product S Kg^T is ready
            float x[16];
            {
                if (!mbar_wait(bB + 3, (uint32_t)(ci & 1), kWaitLimit)) raise_device_error(err, kErrMbarTimeout);
                const uint8_t* vt = sm + F_V + (row >> 6) * 8192;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qq + e;
                    const uint32_t at = sw128((uint32_t)t, (uint32_t)((row & 63) >> 3)) + (uint32_t)(row & 7) * 2u;
                    x[e] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(vt + at));
                }
            }
            // ---- R = V - Kg S^T (kept), beta R to TMEM as hi + lo
            nb_sync(NB_1);
            tc_fence_after();
            {
                uint32_t y[16];
                tmem_ld16_async(tbase + lane_base + F_D1 + 16 * qq, y);
                tmem_wait_ld(); reg_fence(y);
                float br[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    x[e] -= __uint_as_float(y[e]);
                    br[e] = sBeta[16 * qq + e] * x[e];
                }
                uint32_t hi[8], lo[8];
                split_pairs(br, 8, hi, lo);
                tmem_st8(tbase + lane_base + F_RH + 8 * qq, hi);
                tmem_st8(tbase + lane_base + F_RL + 8 * qq, lo);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_V);
            if (L == kC) {  // a whole chunk: staged and stored by TMA (the tile is free: see NB_3)
                stage_token_tile(sm + F_RV, row, qq, x);
                fence_proxy_async();
                state_sync();
                if (tid == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) tma_store_3d(&tm_r, sm + F_RV + b * 8192, 32 * b, h, (int)c0);
                    bulk_commit();
                }
            } else {  // the sequence's last, partial chunk: the rows past its end belong to the next sequence
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qq + e;
                    if (t < L) Rb[((c0 + t) * H + h) * kD + row] = x[e];
                }
            }
            // ---- V' (kept), to TMEM as hi + lo
            nb_sync(NB_2);
            tc_fence_after();
            {
                uint32_t y[16];
                tmem_ld16_async(tbase + lane_base + F_D2 + 16 * qq, y);
                tmem_wait_ld(); reg_fence(y);
#pragma unroll
                for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(y[e]);
                uint32_t hi[8], lo[8];
                split_pairs(x, 8, hi, lo);
                tmem_st8(tbase + lane_base + F_VH + 8 * qq, hi);
                tmem_st8(tbase + lane_base + F_VL + 8 * qq, lo);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_Z);
            if (L == kC) {  // as R, once R's copies have read the tile
                if (tid == 0) bulk_wait_read();
                state_sync();
                stage_token_tile(sm + F_RV, row, qq, x);
                fence_proxy_async();
                state_sync();
                if (tid == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) tma_store_3d(&tm_vp, sm + F_RV + b * 8192, 32 * b, h, (int)c0);
                    bulk_commit();
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * qq + e;
                    if (t < L) Vp[((c0 + t) * H + h) * kD + row] = x[e];
                }
            }
            // ---- S <- S Diag(gamma) + V'^T Kr
            if (tid == 0) bulk_wait_read();  // the S0 and R/V' tiles are free for the next chunk past NB_3
            nb_sync(NB_3);
            tc_fence_after();
            if (*sStop) break;
            {
                uint32_t d3[32];
                tmem_ld32_async(tbase + lane_base + F_D3 + 32 * qq, d3);
                float gm[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(gm + e) = *reinterpret_cast<const float4*>(sGam + 32 * qq + e);
                tmem_wait_ld(); reg_fence(d3);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[e] = fmaf(s[e], gm[e], __uint_as_float(d3[e]));
            }
        }
        if (tid == 0) bulk_wait_all();  // the S0 copies are complete before the CTA ends
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ============================ per chunk: the products with S0 and dS_next ============================
// Per (chunk, head), the products of bwd_chunk_a_kernel, with the channel (or token) dimension as M = 128:
//   [XQ / scale | -XK / beta]^T = S0^T [dO ; dZ]^T      (S0 as an MN-major A operand, [dO ; dZ] K-major)
//   XR^T                        = dS_next^T V'^T
//   [dA_qk / scale ; -dA_kk]    = [dO ; dZ] V'^T        (rows 0-63 dO, 64-127 dZ)
// every fp32 operand split as bf16 hi + lo (the bf16 dO is exact), products hi.hi + hi.lo + lo.hi.  S0 and
// dS_next take one shared-memory buffer in turn; dgamma = colsum(S0 . dS_next) and the first term of dbeta
// on the CUDA cores, in a fixed order.
constexpr int kAThreads = 512;
constexpr uint32_t A_BUF = 0;         // S0, then dS_next: hi, lo, each [128 r][128 c] (two regions of [128][64])
constexpr uint32_t A_QZH = 65536;     // [dO ; dZ_hi]  [128][128 r] K-major (two regions of [128][64])
constexpr uint32_t A_QZL = 98304;     // [0 ; dZ_lo]
constexpr uint32_t A_VH = 131072;     // V'_hi [64 s][128 r] (two regions of [64][64])
constexpr uint32_t A_VL = 147456;     // V'_lo
constexpr uint32_t A_RED = 163840;    // dgamma parts [32][128] fp32
constexpr uint32_t A_BETA = 180224;   // beta [64]
constexpr uint32_t A_BAR = 180480;    // mbarriers: X and dA products, XR product
constexpr uint32_t A_MISC = A_BAR + 16;
constexpr uint32_t kASmem = A_MISC + 16 + 1024;
// TMEM: X^T 128 columns, XR^T 64, dA 64
constexpr uint32_t A_TX = 0, A_TR = 128, A_TA = 192;

// 8 values as bf16 hi + lo, 16-byte chunks at `at` of two tiles `tile` bytes apart
__device__ __forceinline__ void put_hi_lo(uint8_t* base, uint32_t at, uint32_t tile, const float (&x)[8]) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        hi[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
        lo[j] = pack_bf16x2(x[2 * j] - bf16_lo(hi[j]), x[2 * j + 1] - bf16_hi(hi[j]));
    }
    *reinterpret_cast<uint4*>(base + at) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(base + at + tile) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Phase A of the per-chunk work (item (chunk at c0 with L tokens, head h; base = slot * H + h)): the products
// with S0 and dS_next, dA, dgamma, dv and dbeta's first term; XQ, XK, XR and dA go to global memory for phase B.
// TMEM columns 0-255 of the caller's allocation; ends with every thread past a barrier.
__device__ __forceinline__ void chunk_a_phase(const float* __restrict__ beta, const __nv_bfloat16* __restrict__ d_o,
                                              int64_t T_total, int H, float scale, const float* __restrict__ S0s,
                                              const float* __restrict__ dS_next, const float* __restrict__ Rb,
                                              const float* __restrict__ Vp, const float* __restrict__ dZ,
                                              float* __restrict__ XQ, float* __restrict__ XK, float* __restrict__ XR,
                                              float* __restrict__ dgam, float* __restrict__ dAqk,
                                              float* __restrict__ dAkk, float* __restrict__ dv,
                                              float* __restrict__ dbeta, unsigned int* err, uint8_t* sm, uint32_t tbase,
                                              int64_t c0, int L, int64_t base, int h) {
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* sRed = reinterpret_cast<float*>(sm + A_RED);
    float* sBeta = reinterpret_cast<float*>(sm + A_BETA);
    uint64_t* bX = reinterpret_cast<uint64_t*>(sm + A_BAR);
    uint64_t* bR = bX + 1;
    if (tid == 0) {
        mbar_init(bX, 1);
        mbar_init(bR, 1);
        fence_mbar_init();
    }
    if (tid < kC) sBeta[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
    const float* S0 = S0s + base * kD * kD;
    const float* dSn = dS_next + base * kD * kD;
    prefetch_l2(dSn + 32 * tid);  // dS_next (64 KB) on its way to L2: one 128-byte line per thread
    // ---- loads first (S0: thread (row r = tid / 16 + 32 it, channels 8 (tid % 16) ..); the chunk's tokens:
    //      (token t = tid / 16 + 32 it, value rows 8 (tid % 16) ..)), then the buffers
    float4 s0v[4][2];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kAThreads * it, r = idx >> 4, c8 = idx & 15;
        s0v[it][0] = *reinterpret_cast<const float4*>(S0 + r * kD + 8 * c8);
        s0v[it][1] = *reinterpret_cast<const float4*>(S0 + r * kD + 8 * c8 + 4);
    }
    uint4 ov[2];
    float4 zv[2][2], pv[2][2], rv[2][2];
    float btv[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kAThreads * it, t = idx >> 4, r8 = idx & 15;
        const int tc = t < L ? t : L - 1;  // rows past the end read the last row and are zeroed below
        const int64_t at = ((c0 + tc) * H + h) * kD + 8 * r8;
        ov[it] = *reinterpret_cast<const uint4*>(d_o + at);
        zv[it][0] = *reinterpret_cast<const float4*>(dZ + at);
        zv[it][1] = *reinterpret_cast<const float4*>(dZ + at + 4);
        pv[it][0] = *reinterpret_cast<const float4*>(Vp + at);
        pv[it][1] = *reinterpret_cast<const float4*>(Vp + at + 4);
        rv[it][0] = *reinterpret_cast<const float4*>(Rb + at);
        rv[it][1] = *reinterpret_cast<const float4*>(Rb + at + 4);
        btv[it] = beta[(c0 + tc) * H + h];
    }
    // ---- S0 -> the buffer (MN-major A: row r, channels c)
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kAThreads * it, r = idx >> 4, c8 = idx & 15;
        const float x[8] = {s0v[it][0].x, s0v[it][0].y, s0v[it][0].z, s0v[it][0].w,
                            s0v[it][1].x, s0v[it][1].y, s0v[it][1].z, s0v[it][1].w};
        put_hi_lo(sm + A_BUF, (uint32_t)(c8 >> 3) * 16384u + sw128((uint32_t)r, (uint32_t)(c8 & 7)), 32768, x);
    }
    // ---- [dO ; dZ] (rows past the chunk's end zero), V'; dv = beta dZ; dbeta's first term sum_r dZ R
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kAThreads * it, t = idx >> 4, r8 = idx & 15;
        const bool ok = t < L;
        const int64_t at = ((c0 + t) * H + h) * kD + 8 * r8;
        float z[8], vp[8];
        uint4 o = make_uint4(0, 0, 0, 0);
        float part = 0.f;
        if (ok) {
            o = ov[it];
            z[0] = zv[it][0].x; z[1] = zv[it][0].y; z[2] = zv[it][0].z; z[3] = zv[it][0].w;
            z[4] = zv[it][1].x; z[5] = zv[it][1].y; z[6] = zv[it][1].z; z[7] = zv[it][1].w;
            vp[0] = pv[it][0].x; vp[1] = pv[it][0].y; vp[2] = pv[it][0].z; vp[3] = pv[it][0].w;
            vp[4] = pv[it][1].x; vp[5] = pv[it][1].y; vp[6] = pv[it][1].z; vp[7] = pv[it][1].w;
            const float rr[8] = {rv[it][0].x, rv[it][0].y, rv[it][0].z, rv[it][0].w,
                                 rv[it][1].x, rv[it][1].y, rv[it][1].z, rv[it][1].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) part = fmaf(z[e], rr[e], part);
            const float bt = btv[it];
            *reinterpret_cast<float4*>(dv + at) = make_float4(bt * z[0], bt * z[1], bt * z[2], bt * z[3]);
            *reinterpret_cast<float4*>(dv + at + 4) = make_float4(bt * z[4], bt * z[5], bt * z[6], bt * z[7]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) { z[e] = 0.f; vp[e] = 0.f; }
        }
        const uint32_t c = (uint32_t)(r8 & 7), reg = (uint32_t)(r8 >> 3);
        *reinterpret_cast<uint4*>(sm + A_QZH + reg * 16384 + sw128((uint32_t)t, c)) = o;
        *reinterpret_cast<uint4*>(sm + A_QZL + reg * 16384 + sw128((uint32_t)t, c)) = make_uint4(0, 0, 0, 0);
        {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                hi[j] = pack_bf16x2(z[2 * j], z[2 * j + 1]);
                lo[j] = pack_bf16x2(z[2 * j] - bf16_lo(hi[j]), z[2 * j + 1] - bf16_hi(hi[j]));
            }
            *reinterpret_cast<uint4*>(sm + A_QZH + reg * 16384 + sw128((uint32_t)(64 + t), c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(sm + A_QZL + reg * 16384 + sw128((uint32_t)(64 + t), c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        put_hi_lo(sm + A_VH, reg * 8192 + sw128((uint32_t)t, c), 16384, vp);
        // a row's 16 parts are 16 consecutive lanes: reduce them in a fixed order
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o2);
        if (r8 == 0 && ok) dbeta[(c0 + t) * H + h] = part;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t id_x = idesc_bf16_f32(128, 128, true, false);   // A = S0^T (MN-major), B = [dO ; dZ] (K-major)
    const uint32_t id_r = idesc_bf16_f32(128, 64, true, false);    // A = dS_next^T (MN-major), B = V' (K-major)
    const uint32_t id_a = idesc_bf16_f32(128, 64, false, false);   // A = [dO ; dZ], B = V' (K-major)
    auto kd = [&](uint32_t tile, uint32_t region, int ks) { return sdesc_sw128(tile + (ks >> 2) * region, 16, 1024) + (ks & 3) * 2; };
    if (warp == 0) {
        const uint64_t sh = sdesc_sw128(sbase + A_BUF, 16384, 1024), sl = sdesc_sw128(sbase + A_BUF + 32768, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TX, sh + ks * 128, kd(sbase + A_QZH, 16384, ks), id_x, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TX, sl + ks * 128, kd(sbase + A_QZH, 16384, ks), id_x, 1u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TX, sh + ks * 128, kd(sbase + A_QZL, 16384, ks), id_x, 1u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tbase + A_TA, kd(sbase + A_QZH, 16384, ks), kd(sbase + A_VH, 8192, ks), id_a, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TA, kd(sbase + A_QZH, 16384, ks), kd(sbase + A_VL, 8192, ks), id_a, 1u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TA, kd(sbase + A_QZL, 16384, ks), kd(sbase + A_VH, 8192, ks), id_a, 1u);
        mma_commit(bX);
    }
    // ---- dS_next (and S0 again, from L2, for dgamma) in flight while the S0 products run; thread (row
    //      r = tid / 16 + 32 it, channels 8 (tid % 16) ..)
    float4 dv4[4][2];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kAThreads * it, r = idx >> 4, c8 = idx & 15;
        dv4[it][0] = *reinterpret_cast<const float4*>(dSn + r * kD + 8 * c8);
        dv4[it][1] = *reinterpret_cast<const float4*>(dSn + r * kD + 8 * c8 + 4);
    }
    {  // dgamma parts: sum over the thread's four rows of S0 . dS_next, per channel; 32 row groups x 128 channels
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int c8 = tid & 15;
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = (tid >> 4) + 32 * it;
            const float4 a0 = *reinterpret_cast<const float4*>(S0 + r * kD + 8 * c8);
            const float4 a1 = *reinterpret_cast<const float4*>(S0 + r * kD + 8 * c8 + 4);
            acc[0] = fmaf(a0.x, dv4[it][0].x, acc[0]); acc[1] = fmaf(a0.y, dv4[it][0].y, acc[1]);
            acc[2] = fmaf(a0.z, dv4[it][0].z, acc[2]); acc[3] = fmaf(a0.w, dv4[it][0].w, acc[3]);
            acc[4] = fmaf(a1.x, dv4[it][1].x, acc[4]); acc[5] = fmaf(a1.y, dv4[it][1].y, acc[5]);
            acc[6] = fmaf(a1.z, dv4[it][1].z, acc[6]); acc[7] = fmaf(a1.w, dv4[it][1].w, acc[7]);
        }
        float* dst = sRed + (tid >> 4) * kD + 8 * c8;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    // ---- the buffer takes dS_next once the S0 products are done
    if (tid == 0 && !mbar_wait(bX, 0, kWaitLimit)) raise_device_error(err, kErrMbarTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int idx = tid + kAThreads * it, r = idx >> 4, c8 = idx & 15;
        const float x[8] = {dv4[it][0].x, dv4[it][0].y, dv4[it][0].z, dv4[it][0].w,
                            dv4[it][1].x, dv4[it][1].y, dv4[it][1].z, dv4[it][1].w};
        put_hi_lo(sm + A_BUF, (uint32_t)(c8 >> 3) * 16384u + sw128((uint32_t)r, (uint32_t)(c8 & 7)), 32768, x);
    }
    if (tid < kD) {  // dgamma: the 32 row groups' parts in order
        float sum = 0.f;
        for (int g = 0; g < 32; ++g) sum += sRed[g * kD + tid];
        dgam[base * kD + tid] = sum;
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        const uint64_t dh = sdesc_sw128(sbase + A_BUF, 16384, 1024), dl = sdesc_sw128(sbase + A_BUF + 32768, 16384, 1024);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TR, dh + ks * 128, kd(sbase + A_VH, 8192, ks), id_r, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TR, dh + ks * 128, kd(sbase + A_VL, 8192, ks), id_r, 1u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tbase + A_TR, dl + ks * 128, kd(sbase + A_VH, 8192, ks), id_r, 1u);
        mma_commit(bR);
    }
    // ---- X^T out while XR^T is computed: warp w reads lanes 32 (w % 4) .. (channels c), columns 32 (w / 4) ..
    {
        const int q = warp & 3, cb = warp >> 2;  // column block: 0, 1 -> XQ tokens 0-31, 32-63; 2, 3 -> XK
        const int c = 32 * q + lane;
        uint32_t x[32];
        tmem_ld32_async(tbase + ((uint32_t)(32 * q) << 16) + A_TX + 32 * cb, x);
        tmem_wait_ld(); reg_fence(x);
        const bool is_q = cb < 2;
        const int t0 = 32 * (cb & 1);
        float* outp = is_q ? XQ : XK;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int t = t0 + e;
            if (t < L) outp[((c0 + t) * H + h) * kD + c] = (is_q ? scale : -sBeta[t]) * __uint_as_float(x[e]);
        }
    }
    // ---- dA: lanes 0-63 dO V'^T (dA_qk / scale, j <= i), lanes 64-127 dZ V'^T (-dA_kk, j < i)
    if (warp < 8) {
        const int q = warp & 3, hb = warp >> 2;  // columns 32 hb .. +31
        const int m = 32 * q + lane, i = m & 63;
        const bool is_q = m < 64;
        uint32_t x[32];
        tmem_ld32_async(tbase + ((uint32_t)(32 * q) << 16) + A_TA + 32 * hb, x);
        tmem_wait_ld(); reg_fence(x);
        float* row = (is_q ? dAqk : dAkk) + (base * kC + i) * kC + 32 * hb;
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
            float4 w;
            float* wp = reinterpret_cast<float*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 32 * hb + e4 + e;
                const float v = __uint_as_float(x[e4 + e]);
                wp[e] = is_q ? (j <= i ? scale * v : 0.f) : (j < i ? -v : 0.f);
            }
            *reinterpret_cast<float4*>(row + e4) = w;
        }
    }
    if (tid == 0 && !mbar_wait(bR, 0, kWaitLimit)) raise_device_error(err, kErrMbarTimeout);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- XR^T out: warp w reads lanes 32 (w % 4) .. (channels), tokens 16 (w / 4) .. +15
    {
        const int q = warp & 3, tb = warp >> 2;
        const int c = 32 * q + lane;
        uint32_t x[16];
        tmem_ld16_async(tbase + ((uint32_t)(32 * q) << 16) + A_TR + 16 * tb, x);
        tmem_wait_ld(); reg_fence(x);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int t = 16 * tb + e;
            if (t < L) XR[((c0 + t) * H + h) * kD + c] = __uint_as_float(x[e]);
        }
    }
    if (tid == 0) {  // phase B reuses this shared memory
        mbar_inval(bX);
        mbar_inval(bR);
    }
    tc_fence_before();
    __syncthreads();
}

// 2^x by the hardware approximation (results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ============================ per chunk: what does not depend on the state ============================
// bwd_prep_tc_kernel: per (chunk, head) the tiles the tensor-core passes read, as bf16 hi + lo in their
// layouts (kda_bwd_tc.cuh): Kr, scale Qg, Kg, gamma, beta, scale A_qk and T = (I + A_kk)^-1.  A_qk and A_kk
// are one tensor-core product with the block factorisation of the decay around E_I, G at the last token of
// 16-token block I ("月之暗面发布Kimi K3开源大模型技术报告", 架构: the -5 bound keeps the factors within fp32):
// for rows i of block I and columns j <= 16 I + 15,
//   e^{G_ic - G_jc} = e^{G_ic - E_Ic} e^{E_Ic - G_jc}     (the first factor >= 1, the second <= 1),
// so the row operand [k ; q] e^{G - E_I} (M = 128) meets, per row block, its own column operand
// k_j e^{E_I - G_j} (the four stacked, 16 + 32 + 48 + 64 = 160 rows, N = 160), K = 128 channels; each
// operand as bf16 hi + lo and the product hi.hi + hi.lo + lo.hi (fp32-level).  T by 16 x 16 blocks on the
// CUDA cores (kda_tsolve.cuh).
constexpr int kPThreads = 512;
constexpr uint32_t Q_ROW = 0;                 // [k ; q] e^{G - E_I}: hi, lo, each two regions of [128][64]
constexpr uint32_t Q_COL = 65536;             // stacked k e^{E_I - G}: hi, lo, each two regions of [160][64]
constexpr uint32_t kColRegion = 160 * 128;
constexpr uint32_t Q_G = Q_COL + 4 * kColRegion;  // G (log2 units) fp32 [64][128]
constexpr uint32_t Q_BETA = Q_G + 32768;      // beta [64]
constexpr uint32_t Q_BAR = Q_BETA + 256;
constexpr uint32_t Q_MISC = Q_BAR + 16;
constexpr uint32_t kQSmem = Q_MISC + 16 + 1024;
// once the product is complete (its operands are free)
constexpr uint32_t Q_AKK = 0;                 // beta-scaled A_kk fp32 [64][kAS] (blocks on and below the diagonal)
constexpr uint32_t Q_TF = 64 * kAS * 4;       // T fp32 [64][kAS]
constexpr uint32_t Q_NB = 2 * 64 * kAS * 4;   // N blocks of the solve, 9 x [16][kNB] fp32
constexpr uint32_t Q_AQS = Q_COL;             // scale A_qk hi, lo staged in the blob's layout (16 KB)
static_assert(Q_NB + 9 * 16 * kNB * 4 <= Q_COL && Q_G % 1024 == 0 && kQSmem <= 232448, "prep layout");

// 8 values as bf16 hi + lo (x = hi + lo), 16-byte chunks at `at` of two tiles `tile` bytes apart
__device__ __forceinline__ void put_2(uint8_t* base, uint32_t at, uint32_t tile, const float (&x)[8]) {
    uint32_t p1[4], p2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        p1[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
        p2[j] = pack_bf16x2(x[2 * j] - bf16_lo(p1[j]), x[2 * j + 1] - bf16_hi(p1[j]));
    }
    *reinterpret_cast<uint4*>(base + at) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
    *reinterpret_cast<uint4*>(base + at + tile) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
}

__device__ __forceinline__ void load8f(const float* p, float (&f)[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__global__ void __launch_bounds__(kPThreads, 1)
bwd_prep_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                   const float* __restrict__ g, const float* __restrict__ beta, const int32_t* __restrict__ cu, int N,
                   int64_t T_total, int H, float scale, uint8_t* __restrict__ blobs, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array (accesses through `sm` stay shared ones)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n = 0;
    {
        int lo = 0, hi = N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            const int64_t b = cu ? (int64_t)cu[mid] : 0;
            if (b / kC + mid <= slot) lo = mid; else hi = mid;
        }
        n = lo;
    }
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t c0 = bos + (slot - (bos / kC + n)) * kC;
    if (slot < bos / kC + n || c0 >= eos) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int64_t base = slot * H + h;
    const int64_t rs = (int64_t)H * kD, hoff = (int64_t)h * kD;
    constexpr float kLog2e = 1.4426950408889634f;
    uint8_t* blob = blobs + base * (int64_t)kBwdBlobBytes;
    float* sG = reinterpret_cast<float*>(sm + Q_G);
    float* sBeta = reinterpret_cast<float*>(sm + Q_BETA);
    uint64_t* bM = reinterpret_cast<uint64_t*>(sm + Q_BAR);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + Q_MISC);
    if (tid == 0) {
        mbar_init(bM, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sTmem, 256);
    // k and q of the thread's two (row, 8 channels) items, in flight while G is formed
    uint4 kx[2], qx[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kPThreads * it, i = idx >> 4, c8 = idx & 15;
        kx[it] = make_uint4(0, 0, 0, 0);
        qx[it] = make_uint4(0, 0, 0, 0);
        if (i < L) {
            const int64_t at = (c0 + i) * rs + hoff + 8 * c8;
            kx[it] = *reinterpret_cast<const uint4*>(k + at);
            qx[it] = *reinterpret_cast<const uint4*>(q + at);
        }
    }
    if (tid < kC) {
        const float b = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
        sBeta[tid] = b;
        if (__any_sync(0xFFFFFFFFu, !(b >= 0.f && b <= 1.f)) && lane == 0) raise_device_error(err, kErrBetaRange);
    }
    // ---- G: running sum of g per channel (log2 units), thread (c, half): tokens 32 half .. +31
    if (tid < 256) {
        const int c = tid & 127, hh = tid >> 7;
        float gv[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int t = 32 * hh + r;
            gv[r] = t < L ? g[(c0 + t) * rs + hoff + c] : 0.f;
        }
        float acc = 0.f, gmin = 0.f, gmax = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            gmin = fminf(gmin, gv[r]);
            gmax = fmaxf(gmax, gv[r]);
            acc = fmaf(gv[r], kLog2e, acc);
            gv[r] = acc;
        }
        // g in [-5, 0]: min and max skip a NaN, the running sum does not
        if (__any_sync(0xFFFFFFFFu, !(gmin >= -5.f && gmax <= 0.f && acc == acc)) && lane == 0)
            raise_device_error(err, kErrGateRange);
#pragma unroll
        for (int r = 0; r < 32; ++r) sG[(32 * hh + r) * kD + c] = gv[r];
    }
    __syncthreads();
    if (tid >= 128 && tid < 256) {  // the second half's running sum continues from the first's total
        const int c = tid & 127;
        const float t0 = sG[31 * kD + c];
#pragma unroll 4
        for (int r = 32; r < 64; ++r) sG[r * kD + c] += t0;
    }
    __syncthreads();
    if (tid < kD) reinterpret_cast<float*>(blob + kBB_GAM)[tid] = ex2f(sG[(kC - 1) * kD + tid]);
    if (tid < kC) reinterpret_cast<float*>(blob + kBB_BETA)[tid] = sBeta[tid];
    // ---- operands, and Kr, scale Qg, Kg to the blob
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kPThreads * it, i = idx >> 4, c8 = idx & 15, I = i >> 4;
        const uint32_t reg = (uint32_t)(c8 >> 3), ch = (uint32_t)(c8 & 7);
        float G[8], EI[8], kv[8], qv[8];
        load8f(sG + i * kD + 8 * c8, G);
        load8f(sG + (16 * I + 15) * kD + 8 * c8, EI);
        const uint32_t kw[4] = {kx[it].x, kx[it].y, kx[it].z, kx[it].w};
        const uint32_t qw[4] = {qx[it].x, qx[it].y, qx[it].z, qx[it].w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kv[e] = (e & 1) ? bf16_hi(kw[e >> 1]) : bf16_lo(kw[e >> 1]);
            qv[e] = (e & 1) ? bf16_hi(qw[e >> 1]) : bf16_lo(qw[e >> 1]);
        }
        float rk[8], rq[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float f = ex2f(G[e] - EI[e]);
            rk[e] = kv[e] * f;
            rq[e] = qv[e] * f;
        }
        put_2(sm + Q_ROW, reg * 16384u + sw128((uint32_t)i, ch), 32768, rk);
        put_2(sm + Q_ROW, reg * 16384u + sw128((uint32_t)(kC + i), ch), 32768, rq);
        for (int J = I; J < 4; ++J) {  // column operand of row block J >= I
            float EJ[8], cv[8];
            load8f(sG + (16 * J + 15) * kD + 8 * c8, EJ);
#pragma unroll
            for (int e = 0; e < 8; ++e) cv[e] = kv[e] * ex2f(EJ[e] - G[e]);
            put_2(sm + Q_COL, reg * kColRegion + sw128((uint32_t)(8 * J * (J + 1) + i), ch), 2 * kColRegion, cv);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    if (warp == 0) {  // D = [k ; q] rows x stacked columns: hi.hi + hi.lo + lo.hi, K = 128 in 8 steps
        const uint32_t id = idesc_bf16_f32(128, 160, false, false);
#pragma unroll
        for (int pr = 0; pr < 3; ++pr) {
            const uint32_t pa = pr == 2 ? 1u : 0u, pb = pr == 1 ? 1u : 0u;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t rg2 = (uint32_t)(ks >> 2), off = (uint32_t)(ks & 3) * 32u;
                mma_bf16(tbase, kdesc(sbase + Q_ROW + pa * 32768u + rg2 * 16384u + off),
                         kdesc(sbase + Q_COL + pb * 2u * kColRegion + rg2 * kColRegion + off), id,
                         (pr | ks) ? 1u : 0u);
            }
        }
        mma_commit(bM);
    }
    // ---- Kr, scale Qg, Kg to the blob while the product runs
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kPThreads * it, i = idx >> 4, c8 = idx & 15;
        float G[8], Gl[8], kv[8], qv[8];
        load8f(sG + i * kD + 8 * c8, G);
        load8f(sG + (kC - 1) * kD + 8 * c8, Gl);
        const uint32_t kw[4] = {kx[it].x, kx[it].y, kx[it].z, kx[it].w};
        const uint32_t qw[4] = {qx[it].x, qx[it].y, qx[it].z, qx[it].w};
        float kr[8], qg[8], kg[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kv[e] = (e & 1) ? bf16_hi(kw[e >> 1]) : bf16_lo(kw[e >> 1]);
            qv[e] = (e & 1) ? bf16_hi(qw[e >> 1]) : bf16_lo(qw[e >> 1]);
            const float eg = ex2f(G[e]);
            kr[e] = kv[e] * ex2f(Gl[e] - G[e]);
            qg[e] = scale * (qv[e] * eg);
            kg[e] = kv[e] * eg;
        }
        const uint32_t at = (uint32_t)(c8 >> 3) * 8192u + sw128((uint32_t)i, (uint32_t)(c8 & 7));
        put_2(blob + kBB_KR, at, 16384, kr);
        put_2(blob + kBB_QG, at, 16384, qg);
        put_2(blob + kBB_KG, at, 16384, kg);
    }
    if (!mbar_wait(bM, 0, kWaitLimit)) raise_device_error(err, kErrMbarTimeout);
    tc_fence_after();
    float* sAkk = reinterpret_cast<float*>(sm + Q_AKK);
    float* sTf = reinterpret_cast<float*>(sm + Q_TF);
    // ---- A_kk (fp32 work array) and scale A_qk (bf16 hi, lo staged): lane quarter qt holds rows 32 qt .. +31
    //      of [k-rows ; q-rows], lanes 0-15 of row block IbA = 2 (qt % 2), lanes 16-31 of IbA + 1; warp
    //      slice sl takes columns 16 sl .. +15 of each lane's own block (both blocks' columns are loaded)
    {
        const int qt = warp & 3, sl = warp >> 2, IbA = 2 * (qt & 1);
        const int r = 32 * qt + lane, i = r & 63, Ib = IbA + (lane >> 4);
        const bool is_k = r < kC;
        const uint32_t lane_base = (uint32_t)(32 * qt) << 16;
        uint32_t t0[16], t1[16];
        tmem_ld16_async(tbase + lane_base + 8 * IbA * (IbA + 1) + 16 * sl, t0);
        tmem_ld16_async(tbase + lane_base + 8 * (IbA + 1) * (IbA + 2) + 16 * sl, t1);
        tmem_wait_ld(); reg_fence(t0); reg_fence(t1);
        const bool second = lane >= 16, inb = sl <= Ib;  // this column block is one of the row block's
        float a[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) a[e] = __uint_as_float(second ? t1[e] : t0[e]);
        if (is_k) {
            if (inb) {
                const float b = sBeta[i];
#pragma unroll
                for (int j4 = 0; j4 < 16; j4 += 4) {
                    float4 w;
                    float* wp = reinterpret_cast<float*>(&w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) wp[e] = (16 * sl + j4 + e < i) ? b * a[j4 + e] : 0.f;
                    *reinterpret_cast<float4*>(sAkk + i * kAS + 16 * sl + j4) = w;
                }
            }
        } else {
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (inb && 16 * sl + 8 * h8 + e <= i) ? scale * a[8 * h8 + e] : 0.f;
                put_2(sm + Q_AQS, sw128((uint32_t)i, (uint32_t)(2 * sl + h8)), 8192, x);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    // ---- T = (I + A_kk)^-1 (warps 0-5); warps 8-15 copy scale A_qk out as whole rows meanwhile
    if (warp >= 8) {
        const int t = tid - 256;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            *reinterpret_cast<uint4*>(blob + kBB_AQ + 4096 * kk + 16 * t) =
                *reinterpret_cast<const uint4*>(sm + Q_AQS + 4096 * kk + 16 * t);
    }
    t_diag_blocks(sAkk, sTf, warp, lane);
    __syncthreads();
    t_offdiag_1(sAkk, sTf, reinterpret_cast<float*>(sm + Q_NB), tid);
    t_offdiag_23(sTf, reinterpret_cast<float*>(sm + Q_NB), tid);
    // ---- T as bf16 hi + lo: thread (row tid / 8, columns 8 (tid % 8) ..), zero above the diagonal blocks
    {
        const int i = tid >> 3, t8 = tid & 7;
        float x[8];
        const bool zero = (t8 >> 1) > (i >> 4);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = zero ? 0.f : sTf[i * kAS + 8 * t8 + e];
        put_2(blob + kBB_TT, sw128((uint32_t)i, (uint32_t)t8), 8192, x);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// ============================ per chunk: the position-pair sums ============================
// Per (chunk, head), the sums of bwd_chunk_b_kernel over position pairs with the decay e^{G_ic - G_jc}:
//   rq_ic = sum_{j<=i} dA_qk[i][j] k_jc e^{G_ic-G_jc},   rk_ic = sum_{j<i} dA_kk[i][j] k_jc e^{G_ic-G_jc}
//   cq_jc = sum_{i>=j} dA_qk[i][j] q_ic e^{G_ic-G_jc},   ck_jc = sum_{i>j} dA_kk[i][j] beta_i k_ic e^{G_ic-G_jc}
// as tensor-core products over blocks of 16 tokens.  E_b is G at block b's last token; the -5 bound on g keeps
// e^{+-(G_t - E_b)} for t in block b within fp32 ("月之暗面发布Kimi K3开源大模型技术报告", 架构).  With the
// block operands
//   K_b[j] = k_j e^{E_b - G_j},  Q_b[i] = q_i e^{G_i - E_b},  B_b[i] = beta_i k_i e^{G_i - E_b}  (t in block b)
// and, for blocks x >= y, the per-channel factor s_xy = e^{E_x - E_y} <= 1:
//   rq_i = e^{G_i - E_b} sum_{y <= b} s_by (K_y^T dA_qk[block b rows][block y cols])_i      (i in block b)
//   cq_j = e^{E_b - G_j} sum_{x >= b} s_xb (Q_x^T dA_qk[block x rows][block b cols])_j      (j in block b)
// and rk, ck alike with dA_kk and B_x.  Each operand is therefore built once, and every block pair is one
// 128 x 16 x 16 product (channels as M = 128), taken from three-piece bf16 splits (x = p1 + p2 + p3 to about
// 2^-27; p1p1 + p1p2 + p2p1 + p1p3 + p3p1 + p2p2): the gradient of G is a difference of these sums, where a
// two-piece split (2^-17) leaves too little.  The pairs land in their own TMEM columns and the epilogue weighs
// them in fp32.  Then, per (i, c), the element-wise part of bwd_chunk_b_kernel: dq, dk, the gradient of G,
// dbeta's second term (a part per channel half) and dg as the reverse running sum of the G gradient.
constexpr int kBThreads = 512;
constexpr uint32_t B_AR = 0;          // [dA_qk ; dA_kk]: [128 rows i][64 j], three pieces of 16 KB
constexpr uint32_t B_OPA = 49152;     // K then B operands: [64 rows][128 c] (two regions of [64][64]), three
constexpr uint32_t B_OPB = 98304;     // pieces of 16 KB; Q operand
constexpr uint32_t B_G = 147456;      // G (log2 units) fp32 [64][128]
constexpr uint32_t B_TOT = 180224;    // dG totals of the 16 four-row groups, fp32 [16][128]
constexpr uint32_t B_BETA = 188416;   // beta [64]
constexpr uint32_t B_LAST = 188672;   // per (row group, channel): sum over its rows of xr k e^{G_last - G}, fp32 [4][128]
constexpr uint32_t B_DBP = 190720;    // dbeta parts per (row, lane quarter): fp32 [64][4]
constexpr uint32_t B_BAR = 191744;    // two mbarriers
constexpr uint32_t B_MISC = B_BAR + 32;
constexpr uint32_t kBSmem = B_MISC + 16 + 1024;
// TMEM columns, 16 per block pair, laid out so that one product per operand block covers all of its pairs:
// RQ (b, y <= b) at 16 pair_hi(y, b) (block y's pairs: rows 16 y .. 63 from column 16 pair_hi(y, y)), RK at
// 160 + the same; CQ + CK (b, x >= b) at 320 + 16 pair_lo(x, b) (block x's pairs: columns 0 .. 16 x + 15 from
// 320 + 16 pair_lo(x, 0)); cq and ck carry the same weights, so their products share columns
constexpr uint32_t B_RK = 160, B_CS = 320;
__host__ __device__ constexpr int pair_lo(int b, int y) { return b * (b + 1) / 2 + y; }
__host__ __device__ constexpr int pair_hi(int b, int x) { return 4 * b - b * (b - 1) / 2 + x - b; }

// 8 values as three bf16 pieces (x = p1 + p2 + p3), 16-byte chunks at `at` of three tiles `tile` bytes apart
__device__ __forceinline__ void put_3(uint8_t* base, uint32_t at, uint32_t tile, const float (&x)[8]) {
    uint32_t p1[4], p2[4], p3[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float a = x[2 * j], b = x[2 * j + 1];
        p1[j] = pack_bf16x2(a, b);
        const float ra = a - bf16_lo(p1[j]), rb = b - bf16_hi(p1[j]);
        p2[j] = pack_bf16x2(ra, rb);
        p3[j] = pack_bf16x2(ra - bf16_lo(p2[j]), rb - bf16_hi(p2[j]));
    }
    *reinterpret_cast<uint4*>(base + at) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
    *reinterpret_cast<uint4*>(base + at + tile) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
    *reinterpret_cast<uint4*>(base + at + 2 * tile) = make_uint4(p3[0], p3[1], p3[2], p3[3]);
}

// One block operand (kOp 0: K_b, 1: Q_b, 2: B_b) of the chunk's 64 rows into `dst`; thread (row, 8 channels),
// two per thread, from the rows xv (k or q; zero past the sequence's end).
template <int kOp>
__device__ __forceinline__ void build_operand(uint8_t* sm, uint32_t dst, const uint4 (&xv)[2], int tid) {
    const float* sG = reinterpret_cast<const float*>(sm + B_G);
    const float* sBeta = reinterpret_cast<const float*>(sm + B_BETA);
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kBThreads * it, r = idx >> 4, c8 = idx & 15;
        const uint32_t xw[4] = {xv[it].x, xv[it].y, xv[it].z, xv[it].w};
        const float* gr = sG + r * kD + 8 * c8;
        const float* er = sG + (16 * (r >> 4) + 15) * kD + 8 * c8;
        const float4 g0 = *reinterpret_cast<const float4*>(gr), g1 = *reinterpret_cast<const float4*>(gr + 4);
        const float4 e0 = *reinterpret_cast<const float4*>(er), e1 = *reinterpret_cast<const float4*>(er + 4);
        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
        const float br = kOp == 2 ? sBeta[r] : 1.f;
        float val[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float xe = (e & 1) ? bf16_hi(xw[e >> 1]) : bf16_lo(xw[e >> 1]);
            const float f = kOp == 0 ? ex2f(ev[e] - gv[e]) : ex2f(gv[e] - ev[e]);
            val[e] = kOp == 2 ? (br * xe) * f : xe * f;
        }
        put_3(sm + dst, (uint32_t)(c8 >> 3) * 8192u + sw128((uint32_t)r, (uint32_t)(c8 & 7)), 16384, val);
    }
}

// Sum over the warp's 32 lanes of four values v[0..3]; lane l returns the total of v[(l >> 3) & 3].
__device__ __forceinline__ float warp_sum4(const float (&v)[4], int lane) {
    const bool u16 = lane & 16, u8 = lane & 8;
    float w0 = (u16 ? v[2] : v[0]) + __shfl_xor_sync(0xFFFFFFFFu, u16 ? v[0] : v[2], 16);
    float w1 = (u16 ? v[3] : v[1]) + __shfl_xor_sync(0xFFFFFFFFu, u16 ? v[1] : v[3], 16);
    float w = (u8 ? w1 : w0) + __shfl_xor_sync(0xFFFFFFFFu, u8 ? w0 : w1, 8);
    w += __shfl_xor_sync(0xFFFFFFFFu, w, 4);
    w += __shfl_xor_sync(0xFFFFFFFFu, w, 2);
    w += __shfl_xor_sync(0xFFFFFFFFu, w, 1);
    return w;
}

// Phase B of the per-chunk work: the position-pair sums, dq, dk, dg and dbeta's second term, reading phase A's
// XQ, XK, XR and dA back (from L2: this CTA has just written them) and then dropping their L2 lines, which
// nothing reads again, instead of writing them back.  TMEM columns 0-479 of the caller's allocation.
__device__ __forceinline__ void chunk_b_phase(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                                              const float* __restrict__ g, const float* __restrict__ beta,
                                              int64_t T_total, int H, const float* __restrict__ XQ,
                                              const float* __restrict__ XK, const float* __restrict__ XR,
                                              const float* __restrict__ dgam, const float* __restrict__ dAqk,
                                              const float* __restrict__ dAkk, float* __restrict__ dq,
                                              float* __restrict__ dk, float* __restrict__ dg,
                                              float* __restrict__ dbeta_part, unsigned int* err, uint8_t* sm,
                                              uint32_t tbase, int64_t c0, int L, int64_t base, int h) {
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t rs = (int64_t)H * kD;  // row stride of q, k, g and the per-channel tensors
    const int64_t hoff = (int64_t)h * kD;
    constexpr float kLog2e = 1.4426950408889634f;
    float* sG = reinterpret_cast<float*>(sm + B_G);
    float* sTot = reinterpret_cast<float*>(sm + B_TOT);
    float* sBeta = reinterpret_cast<float*>(sm + B_BETA);
    float* sLast = reinterpret_cast<float*>(sm + B_LAST);
    float* sDBP = reinterpret_cast<float*>(sm + B_DBP);
    uint64_t* bM = reinterpret_cast<uint64_t*>(sm + B_BAR);  // [0] the K operand's products, [1] every product
    if (tid == 0) {
        mbar_init(bM, 1);
        mbar_init(bM + 1, 1);
        fence_mbar_init();
    }
    if (tid < kC) sBeta[tid] = tid < L ? beta[(c0 + tid) * H + h] : 0.f;
    // k and q of the operand builder's two (row, 8 channels) items, held for the three builds
    uint4 kx[2], qx[2];
#pragma unroll
    for (int it = 0; it < 2; ++it) {
        const int idx = tid + kBThreads * it, r = idx >> 4, c8 = idx & 15;
        kx[it] = make_uint4(0, 0, 0, 0);
        qx[it] = make_uint4(0, 0, 0, 0);
        if (r < L) {
            kx[it] = *reinterpret_cast<const uint4*>(k + (c0 + r) * rs + hoff + 8 * c8);
            qx[it] = *reinterpret_cast<const uint4*>(q + (c0 + r) * rs + hoff + 8 * c8);
        }
    }
    // ---- G: running sum of g per channel (log2 units), thread (c, half): tokens 32 half .. +31
    if (tid < 256) {
        const int c = tid & 127, hh = tid >> 7;
        float gv[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int t = 32 * hh + r;
            gv[r] = t < L ? g[(c0 + t) * rs + hoff + c] * kLog2e : 0.f;
        }
#pragma unroll
        for (int r = 1; r < 32; ++r) gv[r] += gv[r - 1];
#pragma unroll
        for (int r = 0; r < 32; ++r) sG[(32 * hh + r) * kD + c] = gv[r];
    }
    // ---- dA_qk (rows 0-63), dA_kk (rows 64-127) as three bf16 pieces
    {
        float4 av[2][2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int idx = tid + kBThreads * it, m = idx >> 3, j8 = idx & 7;
            const float* src = (m < kC ? dAqk + (base * kC + m) * kC : dAkk + (base * kC + m - kC) * kC) + 8 * j8;
            av[it][0] = *reinterpret_cast<const float4*>(src);
            av[it][1] = *reinterpret_cast<const float4*>(src + 4);
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int idx = tid + kBThreads * it, m = idx >> 3, j8 = idx & 7;
            const float x[8] = {av[it][0].x, av[it][0].y, av[it][0].z, av[it][0].w,
                                av[it][1].x, av[it][1].y, av[it][1].z, av[it][1].w};
            put_3(sm + B_AR, sw128((uint32_t)m, (uint32_t)j8), 16384, x);
        }
    }
    __syncthreads();
    if (tid >= 128 && tid < 256) {  // the second half's running sum continues from the first's total
        const int c = tid & 127;
        const float t0 = sG[31 * kD + c];
#pragma unroll 4
        for (int r = 32; r < 64; ++r) sG[r * kD + c] += t0;
    }
    __syncthreads();
    // pieces (of the operand, of dA) of the six products p: nibble p of kPa, kPb
    // (11, 12, 21, 13, 31, 22 in one-based pieces)
    constexpr uint32_t kPa = 0x120100u, kPb = 0x102010u;
    // ---- K operand, then its products: RQ and RK of every pair (b, y <= b)
    build_operand<0>(sm, B_OPA, kx, tid);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
#pragma unroll 1
        for (int p = 0; p < 6; ++p) {
            const uint64_t ad = sdesc_sw128(sbase + B_OPA + 16384 * ((kPa >> (4 * p)) & 15u), 8192, 1024);
            const uint32_t bt = sbase + B_AR + 16384 * ((kPb >> (4 * p)) & 15u);
#pragma unroll
            for (int y = 0; y < 4; ++y) {  // block y's columns j against every row i >= 16 y: N = 64 - 16 y
                const uint32_t id = idesc_bf16_f32(128, 64 - 16 * y, true, false);
                mma_bf16(tbase + 16 * pair_hi(y, y), ad + y * 128, kdesc(bt + 2048 * y) + y * 2, id, p ? 1u : 0u);
                mma_bf16(tbase + B_RK + 16 * pair_hi(y, y), ad + y * 128, kdesc(bt + 8192 + 2048 * y) + y * 2, id,
                         p ? 1u : 0u);
            }
        }
        mma_commit(bM);
    }
    // ---- Q operand, then CQ of every pair (b, x >= b)
    build_operand<1>(sm, B_OPB, qx, tid);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
#pragma unroll 1
        for (int p = 0; p < 6; ++p) {
            const uint64_t ad = sdesc_sw128(sbase + B_OPB + 16384 * ((kPa >> (4 * p)) & 15u), 8192, 1024);
            const uint32_t bt = sbase + B_AR + 16384 * ((kPb >> (4 * p)) & 15u);
#pragma unroll
            for (int x = 0; x < 4; ++x)  // block x's rows i against every column j < 16 (x + 1): N = 16 (x + 1)
                mma_bf16(tbase + B_CS + 16 * pair_lo(x, 0), ad + x * 128, sdesc_sw128(bt + 2048 * x, 8192, 1024),
                         idesc_bf16_f32(128, 16 * (x + 1), true, true), p ? 1u : 0u);
        }
    }
    // ---- B operand once the K operand's products are complete, then CK of every pair onto CQ's columns
    if (!mbar_wait(bM, 0, kWaitLimit)) raise_device_error(err, kErrMbarTimeout);
    build_operand<2>(sm, B_OPA, kx, tid);
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
#pragma unroll 1
        for (int p = 0; p < 6; ++p) {
            const uint64_t ad = sdesc_sw128(sbase + B_OPA + 16384 * ((kPa >> (4 * p)) & 15u), 8192, 1024);
            const uint32_t bt = sbase + B_AR + 8192 + 16384 * ((kPb >> (4 * p)) & 15u);
#pragma unroll
            for (int x = 0; x < 4; ++x)
                mma_bf16(tbase + B_CS + 16 * pair_lo(x, 0), ad + x * 128, sdesc_sw128(bt + 2048 * x, 8192, 1024),
                         idesc_bf16_f32(128, 16 * (x + 1), true, true), 1u);
        }
        mma_commit(bM + 1);
    }
    // ---- epilogue: thread (channel c, row group rg), rows 16 b + 4 rg + a
    const int qr = warp & 3, rg = warp >> 2;
    const int c = 32 * qr + lane;
    const uint32_t lb = (uint32_t)(32 * qr) << 16;
    float E[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) E[b] = sG[(16 * b + 15) * kD + c];
    float sf[4][4];  // s_xy = e^{E_x - E_y}, x >= y
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y <= x; ++y) sf[x][y] = ex2f(E[x] - E[y]);
    const float Gl = sG[(kC - 1) * kD + c];
    const uint16_t* k16 = reinterpret_cast<const uint16_t*>(k);
    float dGs[16], last_acc = 0.f;  // the G gradient's running sums inside each four-row group
    // a block's per-token inputs, all loads issued together (rows past the end read the last row); the next
    // block's are in flight while one block is worked on
    float nxq[4], nxk[4], nxr[4], nq[4], nk[4];
    auto load_block = [&](int b) {
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = min(16 * b + 4 * rg + a, L - 1);
            const int64_t at = (c0 + i) * rs + hoff + c;
            nxq[a] = XQ[at];
            nxk[a] = XK[at];
            nxr[a] = XR[at];
            nq[a] = __bfloat162float(q[at]);
            nk[a] = __uint_as_float((uint32_t)k16[at] << 16);
        }
    };
    load_block(0);
    if (!mbar_wait(bM + 1, 0, kWaitLimit)) raise_device_error(err, kErrMbarTimeout);  // every product complete
    tc_fence_after();
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        float xqv[4], xkv[4], xrv[4], qv[4], kv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            xqv[a] = nxq[a]; xkv[a] = nxk[a]; xrv[a] = nxr[a]; qv[a] = nq[a]; kv[a] = nk[a];
        }
        if (b < 3) load_block(b + 1);
        uint32_t tq[4][4], tk[4][4], ts[4][4];
#pragma unroll
        for (int y = 0; y <= b; ++y) {
            tmem_ld4_async(tbase + lb + 16 * pair_hi(y, b) + 4 * rg, tq[y]);
            tmem_ld4_async(tbase + lb + B_RK + 16 * pair_hi(y, b) + 4 * rg, tk[y]);
        }
#pragma unroll
        for (int x = b; x < 4; ++x) tmem_ld4_async(tbase + lb + B_CS + 16 * pair_lo(x, b) + 4 * rg, ts[x - b]);
        tmem_wait_ld();
#pragma unroll
        for (int y = 0; y <= b; ++y) { reg_fence(tq[y]); reg_fence(tk[y]); }
#pragma unroll
        for (int x = b; x < 4; ++x) reg_fence(ts[x - b]);
        float dbv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = 16 * b + 4 * rg + a, m = 4 * b + a;
            float sq = 0.f, sk = 0.f, sc = 0.f;
#pragma unroll
            for (int y = 0; y <= b; ++y) {
                sq = fmaf(sf[b][y], __uint_as_float(tq[y][a]), sq);
                sk = fmaf(sf[b][y], __uint_as_float(tk[y][a]), sk);
            }
#pragma unroll
            for (int x = b; x < 4; ++x) sc = fmaf(sf[x][b], __uint_as_float(ts[x - b][a]), sc);
            const bool in = i < L;
            const float qi = qv[a], ki = kv[a], xq = xqv[a], xk = xkv[a], xr = xrv[a], bi = sBeta[i];
            const float Gi = sG[i * kD + c];
            const float rq = ex2f(Gi - E[b]) * sq, rk = ex2f(Gi - E[b]) * sk;
            const float cs = ex2f(E[b] - Gi) * sc;  // cq + ck
            const float gam = ex2f(Gi), red = ex2f(fminf(Gl - Gi, 0.f));
            const int64_t at = (c0 + i) * rs + hoff + c;
            if (in) {
                dq[at] = fmaf(xq, gam, rq);
                dk[at] = bi * rk + xk * gam + xr * red + cs;
                last_acc = fmaf(xr * ki, red, last_acc);
            }
            dGs[m] = in ? qi * rq + ki * bi * rk + (xq * qi + xk * ki) * gam - xr * ki * red - ki * cs : 0.f;
            dbv[a] = in ? ki * rk : 0.f;
        }
        // dbeta's second term of rows 16 b + 4 rg + a: this warp's 32 channels, in a fixed order
        const float tot = warp_sum4(dbv, lane);
        if ((lane & 7) == 0) sDBP[(16 * b + 4 * rg + ((lane >> 3) & 3)) * 4 + qr] = tot;
        // running sum from the group's last row; the group total goes to shared memory
        dGs[4 * b + 2] += dGs[4 * b + 3];
        dGs[4 * b + 1] += dGs[4 * b + 2];
        dGs[4 * b] += dGs[4 * b + 1];
        sTot[(4 * b + rg) * kD + c] = dGs[4 * b];
    }
    sLast[rg * kD + c] = last_acc;
    tc_fence_before();
    __syncthreads();
    // ---- dg_t = sum_{s >= t} dG_s inside the chunk, with the last token's extra (every row's
    //      xr k e^{G_last - G}, and dgamma e^{G_last}) in every dg_t.  G_t is the sum of g_s for s <= t and the
    //      factors above are natural exponentials, so dG is the gradient with respect to G in natural units.
    {
        const float extra = ((sLast[c] + sLast[kD + c]) + (sLast[2 * kD + c] + sLast[3 * kD + c])) +
                            dgam[base * kD + c] * ex2f(Gl);
        // totals of groups 4 b + rg + 1 .. 15, for each b, in a fixed order (from the chunk's end)
        float suff[4] = {0.f, 0.f, 0.f, 0.f};
        float acc = 0.f;
#pragma unroll
        for (int gi = 15; gi >= 0; --gi) {
            if ((gi & 3) == rg) suff[gi >> 2] = acc;
            acc += sTot[gi * kD + c];
        }
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                const int t = 16 * b + 4 * rg + a;
                if (t < L) dg[(c0 + t) * rs + hoff + c] = dGs[4 * b + a] + (suff[b] + extra);
            }
    }
    if (tid < L) {  // channel half 0 = lane quarters 0, 1; half 1 = 2, 3
        dbeta_part[(c0 + tid) * H + h] = sDBP[tid * 4] + sDBP[tid * 4 + 1];
        dbeta_part[(T_total + c0 + tid) * H + h] = sDBP[tid * 4 + 2] + sDBP[tid * 4 + 3];
    }
    tc_fence_before();
    __syncthreads();
    // XQ, XK, XR (the item's rows of its head) and dA: every read is done
    for (int idx = tid; idx < 3 * kC * 4 + 256; idx += kBThreads) {
        if (idx < 3 * kC * 4) {
            const int which = idx >> 8, r = (idx >> 2) & 63, part = idx & 3;
            if (r < L) discard_l2((which == 0 ? XQ : which == 1 ? XK : XR) + (c0 + r) * rs + hoff + 32 * part);
        } else {
            const int l = idx - 3 * kC * 4;
            discard_l2((l < 128 ? dAqk : dAkk) + base * kC * kC + 32 * (l & 127));
        }
    }
}

// The per-chunk work of one item, phase A then phase B on one CTA (512 threads; shared memory and TMEM
// reused from one phase to the next).
__global__ void __launch_bounds__(kBThreads, 1)
bwd_chunk_ab_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                       const float* __restrict__ g, const float* __restrict__ beta,
                       const __nv_bfloat16* __restrict__ d_o, const int32_t* __restrict__ cu, int N, int64_t T_total,
                       int H, float scale, const float* __restrict__ S0s, const float* __restrict__ dS_next,
                       const float* __restrict__ Rb, const float* __restrict__ Vp, const float* __restrict__ dZ,
                       float* __restrict__ XQ, float* __restrict__ XK, float* __restrict__ XR, float* __restrict__ dgam,
                       float* __restrict__ dAqk, float* __restrict__ dAkk, float* __restrict__ dv,
                       float* __restrict__ dbeta, float* __restrict__ dq, float* __restrict__ dk,
                       float* __restrict__ dg, float* __restrict__ dbeta_part, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n = 0;
    {
        int lo = 0, hi = N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            const int64_t b = cu ? (int64_t)cu[mid] : 0;
            if (b / kC + mid <= slot) lo = mid; else hi = mid;
        }
        n = lo;
    }
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);
    const int64_t c0 = bos + (slot - (bos / kC + n)) * kC;
    if (slot < bos / kC + n || c0 >= eos) return;
    const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
    const int64_t base = slot * H + h;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + B_MISC);  // outside phase A's shared memory
    if (warp == 0) tmem_alloc(sTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    chunk_a_phase(beta, d_o, T_total, H, scale, S0s, dS_next, Rb, Vp, dZ, XQ, XK, XR, dgam, dAqk, dAkk, dv, dbeta, err,
                  sm, tbase, c0, L, base, h);
    tc_fence_after();
    chunk_b_phase(q, k, g, beta, T_total, H, XQ, XK, XR, dgam, dAqk, dAkk, dq, dk, dg, dbeta_part, err, sm, tbase, c0,
                  L, base, h);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

}  // namespace

// [T, H, 128] bf16 tensor: boxes of [64 tokens][1 head][64 channels] with the 128-byte swizzle
static bool encode_token_map(CUtensorMap* tm, const void* base, int64_t T_total, int H) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * 2, (cuuint64_t)H * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A fp32 [T_total, H, 128] tensor stored in boxes of [64 tokens][1 head][32 channels] with the 128-byte swizzle.
static bool encode_token_rows_f32(CUtensorMap* tm, void* base, int64_t T_total, int H) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * 4, (cuuint64_t)H * 128 * 4};
    const cuuint32_t box[3] = {32, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Per-chunk states ([slot][head] of 128 x 128 fp32, slots below T_total / 64 + N + 1) as rows of 128 fp32, stored
// in boxes of [128 rows][32 channels] with the 128-byte swizzle.
static bool encode_state_rows_map(CUtensorMap* tm, void* base, int N, int64_t T_total, int H) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t rows = (cuuint64_t)(T_total / kC + N + 1) * (cuuint64_t)H * kD;
    if (rows >= ((cuuint64_t)1 << 31)) return false;  // 32-bit box coordinates
    const cuuint64_t dims[2] = {128, rows};
    const cuuint64_t strides[1] = {128 * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

cudaError_t launch_bwd_fwd_state_tc(const void* v, const float* init_state, const int32_t* cu_seqlens, int N,
                                    int64_t T_total, int H, const void* blobs, float* S0s, float* R, float* Vp,
                                    unsigned int* err, cudaStream_t stream) {
    CUtensorMap tm, tm_s0, tm_r, tm_vp;
    if (!encode_token_map(&tm, v, T_total, H)) return cudaErrorInvalidValue;
    if (!encode_state_rows_map(&tm_s0, S0s, N, T_total, H)) return cudaErrorInvalidValue;
    if (!encode_token_rows_f32(&tm_r, R, T_total, H) || !encode_token_rows_f32(&tm_vp, Vp, T_total, H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_fwd_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFwdSmem);
    if (e != cudaSuccess) return e;
    const int64_t chains = (int64_t)N * H;
    if (chains == 0) return cudaSuccess;
    bwd_fwd_state_tc_kernel<<<(unsigned)chains, kThreads, kFwdSmem, stream>>>(
        tm, tm_s0, tm_r, tm_vp, static_cast<const __nv_bfloat16*>(v), init_state, cu_seqlens, T_total, H, static_cast<const uint8_t*>(blobs),
        S0s, R, Vp, err);
    return cudaGetLastError();
}

cudaError_t launch_bwd_state_tc(const void* d_o, const float* d_final, const int32_t* cu_seqlens, int N,
                                int64_t T_total, int H, const void* blobs, float* d_init, float* dS_next, float* dZ,
                                unsigned int* err, cudaStream_t stream) {
    CUtensorMap tm, tm_dsn;
    if (!encode_token_map(&tm, d_o, T_total, H)) return cudaErrorInvalidValue;
    if (!encode_state_rows_map(&tm_dsn, dS_next, N, T_total, H)) return cudaErrorInvalidValue;
    CUtensorMap tm_dz;
    if (!encode_token_rows_f32(&tm_dz, dZ, T_total, H)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(bwd_state_tc_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmem);
    if (e != cudaSuccess) return e;
    const int64_t chains = (int64_t)N * H;
    if (chains == 0) return cudaSuccess;
    bwd_state_tc_kernel<__nv_bfloat16><<<(unsigned)chains, kThreads, kSmem, stream>>>(
        tm, tm_dsn, tm_dz, static_cast<const __nv_bfloat16*>(d_o), d_final, cu_seqlens, T_total, H, static_cast<const uint8_t*>(blobs),
        d_init, dS_next, dZ, err);
    return cudaGetLastError();
}

}  // namespace kda

namespace kda {

cudaError_t launch_bwd_chunk_ab_tc(const void* q, const void* k, const float* g, const float* beta, const void* d_o,
                                   const int32_t* cu_seqlens, int N, int64_t T_total, int H, float scale,
                                   const float* S0s, const float* dS_next, const float* R, const float* Vp,
                                   const float* dZ, float* XQ, float* XK, float* XR, float* dgam, float* dAqk,
                                   float* dAkk, float* dv, float* dbeta, float* dq, float* dk, float* dg,
                                   float* dbeta_part, unsigned int* err, cudaStream_t stream) {
    static_assert(kAThreads == kBThreads && kASmem <= kBSmem && A_MISC + 16 <= B_MISC,
                  "phase A fits the fused kernel's block and shared memory below its TMEM address slot");
    cudaError_t e =
        cudaFuncSetAttribute(bwd_chunk_ab_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBSmem);
    if (e != cudaSuccess) return e;
    const int64_t slots = T_total / kC + N + 1;
    bwd_chunk_ab_tc_kernel<<<dim3((unsigned)slots, (unsigned)H), kBThreads, kBSmem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g, beta,
        static_cast<const __nv_bfloat16*>(d_o), cu_seqlens, N, T_total, H, scale, S0s, dS_next, R, Vp, dZ, XQ, XK, XR,
        dgam, dAqk, dAkk, dv, dbeta, dq, dk, dg, dbeta_part, err);
    return cudaGetLastError();
}

cudaError_t launch_bwd_prep_tc(const void* q, const void* k, const float* g, const float* beta, const int32_t* cu_seqlens,
                               int N, int64_t T_total, int H, float scale, void* blobs, unsigned int* err,
                               cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(bwd_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmem);
    if (e != cudaSuccess) return e;
    const int64_t slots = T_total / kC + N + 1;
    bwd_prep_tc_kernel<<<dim3((unsigned)slots, (unsigned)H), kPThreads, kQSmem, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), g, beta, cu_seqlens, N, T_total, H,
        scale, static_cast<uint8_t*>(blobs), err);
    return cudaGetLastError();
}

}  // namespace kda
