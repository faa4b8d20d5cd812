// kda_chunk_fwd, bf16 path: chunkwise prefill on the tcgen05 tensor cores, as two kernels.
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
// Two kernels.  Everything except the state path is independent of S0: the running sum,
// the operand tiles, A_kk, A_qk, T, and with them
//   T_b = T Diag(beta)     W = T_b (K . e^G)     U = T_b V     (so that V'^T = U^T - S0 W^T).
// chunk_prep_kernel computes them for every (chunk, head) at once (256-thread CTAs, two per
// SM) and stores each chunk's state-path operands in the workspace, laid out exactly as the
// state path reads them (128-byte-swizzled tiles), so that one bulk copy brings each in:
//   B1    [-W ; Q e^G]      bf16 [128][128]   B of the S0 products
//   T_b   hi, lo            bf16 [64][64] x2  B of U^T = V^T T_b^T
//   A_qk  hi, lo            bf16 [64][64] x2  B of O^T += V'^T A_qk^T
//   KP    K e^{G_C - G}     bf16 [64][128]    B (MN-major) of dS = V'^T KP
//   e^{G_C}                 fp32 [128]
//   (v    bf16 [64][128], only when the front end runs inside the prep kernel)
// chunk_state_kernel then walks each (sequence, head) chain in order, one CTA of 16 warps
// per chain, with S0 (fp32) in registers: thread (r, quarter) holds row r, key channels
// [32 quarter, 32 quarter + 32); a bf16 copy in TMEM is the A operand of the S0 products, so
// every product has M = 128 = dv and maps row r to TMEM lane r.  Per chunk, U^T = V^T T_b^T is
// formed in TMEM ahead of time (v read straight from its tensor) and S0 (-W)^T is accumulated
// onto it, which leaves V'^T in TMEM; the serial path is that one product, the hi/lo split of
// V', one product (dS) and the state update; the output product and its store overlap the next
// chunk's first product.
//
// Precision.  Products accumulate in fp32 in TMEM.  W and U come from T Diag(beta) split as
// hi + lo in bf16 (two bf16 products each, T kept to about 16 bits; U - S0 W^T is summed in one
// fp32 accumulator); V'^T A_qk^T runs as
// three bf16 products of the hi/lo splits of both (hi hi + hi lo + lo hi); the state update
// V'^T KP takes V' as hi + lo (two bf16 products), so the rounding of V' does not build up in
// the state over a long chain; the other operands are bf16.  T = (I + A_kk)^-1 is computed in fp32 on the CUDA
// cores by 16 x 16 blocks: the four diagonal blocks D by forward substitution, then the blocks
// below them as (I - N + N^2 - N^3) D with N = D A_below (N^4 = 0).
//
// Packed sequences are numbered chunk by chunk (sequence-major); the workspace holds the
// operands of a range of chunk rows (all heads) at a time, and a chain that crosses the end
// of a range hands its fp32 state to the next range through the workspace.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_frontend.cuh"
#include "kda_tc.cuh"
#include "kda_tsolve.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int kC = kChunk;    // 64
constexpr int kD = kHeadDim;  // 128
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware approximation (relative error about 2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Operands of one (chunk, head) in the workspace, byte offsets (each tile in the layout its
// reader uses; A_qk and KP are contiguous so that one copy brings them in).
constexpr uint32_t BLOB_B1 = 0;        // [-W ; Q e^G] bf16, two regions of [128][64] (128-byte swizzle)
constexpr uint32_t BLOB_TB = 32768;    // T Diag(beta) as bf16 hi then lo, each [64][64] (one swizzled region)
constexpr uint32_t BLOB_AQ = 49152;    // A_qk as bf16 hi then lo, each [64][64]
constexpr uint32_t BLOB_KP = 65536;    // K e^{G_C - G} bf16, two regions of [64][64]
constexpr uint32_t BLOB_EGL = 81920;   // e^{G_C} fp32 [128]
constexpr uint32_t kBlobBytes = 82432;     // stride of the operands of one (chunk, head)
constexpr uint32_t kStateBytes = kD * kD * 4;


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

// One thread waits (bounded) for phase `ph` of an mbarrier; a wait that runs out marks the CTA aborted
// and reports.  The other warps meet that thread at a CTA barrier afterwards, blocked in bar.sync
// rather than polling the mbarrier (polling by every warp takes issue slots from the ones working).
__device__ __forceinline__ void solo_wait(uint64_t* b, uint32_t ph, volatile int* abort_flag, unsigned int* err) {
    if (!mbar_wait(b, ph, kWaitLimit)) {
        *abort_flag = 1;
        raise_device_error(err, kErrMbarTimeout);
    }
}

// All threads meet; TMEM accesses after it are ordered after the tcgen05 operations before it.
__device__ __forceinline__ void cta_sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Chunk offsets of the packed sequences: off[n] = sum over n' < n of ceil(L_n' / 64), off[N] = all.
// Without cu_seqlens (one sequence) the kernels take off = NULL as {0, ceil(T_total / 64)} instead.
__global__ void __launch_bounds__(1024) chunk_offsets_kernel(const int32_t* __restrict__ cu, int N, int64_t T_total,
                                                             int32_t* __restrict__ off) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < N; base += 1024) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            int64_t bos, eos;
            seq_bounds(cu, n, T_total, bos, eos);
            cnt = eos > bos ? (int)((eos - bos + kC - 1) / kC) : 0;
        }
        int incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, w, d);
                if (lane >= d) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - cnt;
        if (n < N) off[n] = before;
        __syncthreads();
        if (tid == 0) carry += warp_tot[31];
        __syncthreads();
    }
    if (tid == 0) off[N] = carry;
}

// =============================================================================================
// chunk_prep_kernel: the S0-independent part of every (chunk, head); persistent, two CTAs per SM,
// each taking items blockIdx.x, blockIdx.x + gridDim.x, ...; the next item's inputs are loaded while
// the current one's W and U are stored.
// =============================================================================================
constexpr int kPrepThreads = 256;
// Two 32 KB regions trade roles from one item to the next (offsets rr and gb, 0 and 32768 in turn):
//   rr: k (rows 0-63) and q (rows 64-127) land here by TMA in the layout of the row operand, two
//       regions of 16 KB, and are scaled in place; after the A products, A_kk fp32 [64][kAS]
//   gb: g fp32, four TMA boxes of [64][32]; the running sum G in place; then K e^G (two regions of
//       [64][64]): the MN-major B operand (N = 128) of W
// The next item's g lands in this item's rr once the solve has consumed A_kk, its k and q in gb once the
// W product is done.
constexpr uint32_t P_CT = 65536;      // column operands of the four row blocks stacked: 160 rows (block J from
                                      // row 16 J (J+1) / 2), two regions of 160 x 128 bytes; block 3 is K e^{G_C - G}
constexpr uint32_t kCTRegion = 160 * 128;
constexpr uint32_t P_BETA = P_CT + 2 * kCTRegion;  // fp32 [64]
constexpr uint32_t P_E = P_BETA + 256;     // fp32 [4][128]: G at the last token of each 16-token block
constexpr uint32_t P_TOT = P_E + 2048;     // fp32 [128]: sum of the first 32 tokens
constexpr uint32_t P_BAR = P_TOT + 512;    // mbarriers: k/q, (unused), A products, W product, g
constexpr uint32_t P_MISC = P_BAR + 40;    // TMEM base, abort flag
constexpr uint32_t kPrepSmem = P_MISC + 16 + 1024;
// After the A products complete (column operands free):
constexpr uint32_t P_TF = P_CT;                  // T fp32 [64][kAS]
constexpr uint32_t P_NB = P_CT + 64 * kAS * 4;   // N blocks of the solve, 9 x [16][20] fp32
constexpr uint32_t P_AQS = P_NB;                 // before them: A_qk hi, lo staged in the workspace layout (16 KB)
// Once T is in registers: T Diag(beta) as bf16 hi and lo, A operands of 128 rows (T twice: the product
// is M = 128, W lands in TMEM lanes 0-63 and again in 64-127)
constexpr uint32_t P_TH = P_CT, P_TL = P_CT + 16384;
constexpr uint32_t kPrepTmemCols = 256;
// row block I of A: 16 (I + 1) columns from 16 I (I + 1) / 2 (one product of N = 160)
// then [T ; T] K e^G: W = lanes 0-63 of columns 0-127
constexpr uint32_t kKQBytes = 4 * 8192;
constexpr uint32_t kGBytes = 4 * 8192;

static_assert(64 * kAS * 4 <= 32768 && P_NB + 9 * 16 * kNB * 4 <= P_BETA && P_TL + 16384 <= P_BETA &&
                  P_AQS + 16384 <= P_BETA && P_AQS % 128 == 0,
              "solve work overflows its region");
static_assert(2 * (kPrepSmem + 1024) <= 233472, "two prep CTAs per SM");

// Raw front-end inputs of the fused prefill (unused otherwise).
struct FrontendArgs {
    const __nv_bfloat16* xq;
    const __nv_bfloat16* xk;
    const __nv_bfloat16* xv;
    int64_t x_stride;
    const __nv_bfloat16* conv_w;
    const __nv_bfloat16* cs_in;
    float eps;
};

// Byte offset of g / G element (token i, channel c) in the four 128-byte-swizzled boxes of 32 channels.
__device__ __forceinline__ uint32_t g_off(int i, int c) {
    return (uint32_t)(c >> 5) * 8192u + sw128((uint32_t)i, (uint32_t)((c & 31) >> 2)) + (uint32_t)(c & 3) * 4u;
}

// FE: q and k are computed here from the raw front-end rows (ShortConv4 + SiLU + L2 norm, the same
// arithmetic as kda_shortconv_l2norm) instead of being read (v comes from the stand-alone front end).
template <bool FE>
__global__ void __launch_bounds__(kPrepThreads, 2)
chunk_prep_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_g,
                  const float* __restrict__ beta, const int32_t* __restrict__ cu, const int32_t* __restrict__ off,
                  int N, int64_t T_total, int H, int m0, int n_items, uint8_t* __restrict__ blobs,
                  FrontendArgs fe, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array, so that accesses through `sm` stay shared
    // ones (an integer round trip of the address would leave them generic)
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int offN = off ? off[N] : (int)((T_total + kC - 1) / kC);
    constexpr uint32_t kStride = kBlobBytes;

    float* sBeta = reinterpret_cast<float*>(sm + P_BETA);
    float* sE = reinterpret_cast<float*>(sm + P_E);
    float* sTot = reinterpret_cast<float*>(sm + P_TOT);
    uint64_t* barL = reinterpret_cast<uint64_t*>(sm + P_BAR);
    uint64_t* barA = barL + 2;
    uint64_t* barW = barL + 3;
    uint64_t* barG = barL + 4;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + P_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + P_MISC + 4);

    // item -> (head, chunk start, chunk length); false past the last chunk
    auto locate = [&](int item, int& h, int64_t& c0, int& L) {
        if (item >= n_items) return false;
        h = item % H;
        const int m = m0 + item / H;
        if (m >= offN) return false;
        int lo = 0, hi = N;  // off[lo] <= m < off[hi]
        while (off && hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (off[mid] <= m) lo = mid; else hi = mid;
        }
        int64_t bos, eos;
        seq_bounds(cu, lo, T_total, bos, eos);
        c0 = bos + (int64_t)kC * (m - (off ? off[lo] : 0));
        L = (eos - c0) < kC ? (int)(eos - c0) : kC;
        return true;
    };
    // Copies: issuing one takes its thread a few hundred cycles, so lane 0 of warps 0-3 issue one box each
    // (a box that lands before thread 0's expect_tx only makes the transaction count negative for a while).
    // g of an item (into region gb), and its beta (tokens past the chunk's end read as 0)
    auto load_g_tma = [&](int h, int64_t c0, uint32_t gb) {
        if (tid == 0) mbar_arrive_expect_tx(barG, kGBytes);
        if (lane == 0 && warp < 4) {
            fence_proxy_async();
            tma_load_3d(sm + gb + warp * 8192, &tm_g, 32 * warp, h, (int)c0, barG);
        }
    };
    auto load_beta = [&](int h, int64_t c0, int L) {
        if (tid < kC) {
            const bool ok = tid < L;
            cp_async4(sBeta + tid, beta + (ok ? (c0 + tid) * H + h : 0), ok ? 4u : 0u);
        }
        cp_async_commit();
    };
    // k, q into region rr in the row-operand layout (FE computes them instead)
    // box w: k (w even) or q (w odd), channels 64 (w / 2) ..; region w / 2, rows 0-63 (k) or 64-127 (q)
    auto load_kq = [&](int h, int64_t c0, uint32_t rr) {
        if (FE) return;
        if (tid == 0) mbar_arrive_expect_tx(barL, kKQBytes);
        if (lane == 0 && warp < 4) {
            fence_proxy_async();
            tma_load_3d(sm + rr + warp * 8192, (warp & 1) ? &tm_q : &tm_k, 64 * (warp >> 1), h, (int)c0, barL);
        }
    };
    // FE: an item's raw q and k rows (3 of history + 64; the head's 256 bytes each) into L2
    auto prefetch_rows = [&](int h, int64_t c0) {
        for (int i = tid; i < 2 * 67 * 2; i += kPrepThreads) {
            const int p = i / 134, r = (i % 134) >> 1, half = i & 1;
            const int64_t t = c0 - 3 + r;
            if (t >= 0 && t < T_total) {
                const __nv_bfloat16* x = p == 0 ? fe.xq : fe.xk;
                prefetch_l2(x + t * fe.x_stride + (int64_t)h * kD + 64 * half);
            }
        }
    };
    // FE: part p (q or k) of the chunk's 64 tokens, through the front end, as bf16 into a 128-byte-swizzled
    // operand tile in shared memory at `dst` (two regions of `region` bytes; token i at row row0 + i).  Warp w
    // takes tokens 8w .. 8w+7, lane the 4 channels from 4 lane.
    auto frontend_tile = [&](int p, int h, int64_t c0, uint8_t* dst, uint32_t region, int row0) {
        const __nv_bfloat16* x = p == 0 ? fe.xq : fe.xk;
        float y[fe::kFeRun][4], inv[fe::kFeRun];
        fe::frontend_run<__nv_bfloat16>(x, fe.x_stride, fe.conv_w, cu, N, T_total, H, p, h, lane,
                                        c0 + fe::kFeRun * warp, fe.cs_in, fe.eps, y, inv);
#pragma unroll
        for (int i = 0; i < fe::kFeRun; ++i) {
            float2 a = make_float2(y[i][0], y[i][1]), b = make_float2(y[i][2], y[i][3]);
            if (p < 2) {
                a = __fmul2_rn(a, make_float2(inv[i], inv[i]));
                b = __fmul2_rn(b, make_float2(inv[i], inv[i]));
            }
            const uint32_t at = (lane >> 4) * region + sw128(row0 + fe::kFeRun * warp + i, (lane & 15) >> 1) +
                                (lane & 1) * 8;
            *reinterpret_cast<uint2*>(dst + at) = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(b.x, b.y));
        }
    };

    if (tid == 0) {
        mbar_init(barL, 1);
        mbar_init(barA, 1);
        mbar_init(barW, 1);
        mbar_init(barG, 1);
        fence_mbar_init();
        *sAbort = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, kPrepTmemCols);
    cta_sync_tc();
    const uint32_t tbase = *sTmem;
    // thread 0: 1 = k/q loads in flight, 4 = A products, 8 = W product, 16 = g
    uint32_t pend = 0;

    int item = blockIdx.x, h = 0, L = 0;
    int64_t c0 = 0;
    bool have = locate(item, h, c0, L);
    if (have) {
        load_g_tma(h, c0, 32768);
        load_beta(h, c0, L);
        load_kq(h, c0, 0);
        if (FE) prefetch_rows(h, c0);  // the first item's rows: its q part then reads L2, not DRAM
        if (tid == 0) pend |= FE ? 16u : 17u;
    }
    for (uint32_t ph = 0; have; ph ^= 1u) {
        const uint32_t P_RR = ph ? 32768u : 0u, P_G = 32768u - P_RR;  // this item's two regions
        const uint32_t P_KG = P_G, P_AKK = P_RR;
        uint8_t* blob = blobs + (int64_t)item * kStride;
        // the next item's place, early: its global reads (and with FE its raw rows) complete while this item
        // is worked on
        const int next_item = item + gridDim.x;
        int h1 = 0, L1 = 0;
        int64_t c01 = 0;
        const bool have_next = locate(next_item, h1, c01, L1);
        if (FE && have_next) prefetch_rows(h1, c01);
        if (tid == 0) {
            solo_wait(barG, ph, sAbort, err);
            pend &= ~16u;
        }
        if (FE) {  // k and q into the row operand's space (free: the previous item's W/U products are done)
            frontend_tile(1, h, c0, sm + P_RR, 16384, 0);
            frontend_tile(0, h, c0, sm + P_RR, 16384, 64);
        }
        cp_async_wait_all();
        __syncthreads();
        if (*sAbort) break;
        // beta in [0, 1] (tokens past the chunk's end read as 0)
        if (warp < 2 && __any_sync(0xFFFFFFFFu, !(sBeta[tid] >= 0.f && sBeta[tid] <= 1.f)) && lane == 0)
            raise_device_error(err, kErrBetaRange);
        // ---- running sum of g per key channel (log2 units): thread (c, half) sums tokens 32 half .. +31
        {
            const int c = tid & 127, hh = tid >> 7;
            float gv[32];
#pragma unroll
            for (int r = 0; r < 32; ++r)
                gv[r] = (32 * hh + r) < L ? *reinterpret_cast<const float*>(sm + P_G + g_off(32 * hh + r, c)) : 0.f;
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
            if (hh == 0) sTot[c] = acc;
            __syncthreads();
            const float base = hh ? sTot[c] : 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) *reinterpret_cast<float*>(sm + P_G + g_off(32 * hh + r, c)) = gv[r] + base;
            sE[(2 * hh) * kD + c] = gv[15] + base;
            sE[(2 * hh + 1) * kD + c] = gv[31] + base;
            if (hh == 1) reinterpret_cast<float*>(blob + BLOB_EGL)[c] = exp2f(gv[31] + base);
            if (!FE && tid == 0) {  // k and q before the operands are built
                solo_wait(barL, ph, sAbort, err);
                pend &= ~1u;
            }
            __syncthreads();
        }
        // ---- operands.  Thread (cc, r4): channels 8cc .. 8cc+7 of rows i = r4 + 16 I (I = 0..3): the row
        // operand in place; Q e^G (workspace); column operands of blocks J >= I (KP also to the workspace);
        // K e^G, held until the running sum is no longer read.
        const int cc = lane & 15, r4 = 2 * warp + (lane >> 4), c8 = 8 * cc;  // a warp: rows r4 + 16 I, r4 + 1 + 16 I
        const uint32_t reg = cc >> 3, ch = cc & 7;
        uint4 kg_hold[4];
        {
            float E[4][8], dn[3][8];  // E_I, and e^{E_{J+1} - E_J}
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                *reinterpret_cast<float4*>(&E[I][0]) = *reinterpret_cast<const float4*>(sE + I * kD + c8);
                *reinterpret_cast<float4*>(&E[I][4]) = *reinterpret_cast<const float4*>(sE + I * kD + c8 + 4);
            }
#pragma unroll
            for (int J = 0; J < 3; ++J)
#pragma unroll
                for (int e = 0; e < 8; ++e) dn[J][e] = ex2(E[J + 1][e] - E[J][e]);
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                const int i = r4 + 16 * I;
                uint4* kp = reinterpret_cast<uint4*>(sm + P_RR + reg * 16384 + sw128(i, ch));
                uint4* qp = reinterpret_cast<uint4*>(sm + P_RR + reg * 16384 + sw128(64 + i, ch));
                float kv[8], qv[8], G[8];
                unpack8(*kp, kv);
                unpack8(*qp, qv);
                const uint8_t* gp = sm + P_G + (cc >> 2) * 8192;
                *reinterpret_cast<float4*>(&G[0]) = *reinterpret_cast<const float4*>(gp + sw128(i, 2 * (cc & 3)));
                *reinterpret_cast<float4*>(&G[4]) = *reinterpret_cast<const float4*>(gp + sw128(i, 2 * (cc & 3) + 1));
                float rk[8], rq[8], kg[8], qg[8], kr[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float f = ex2(G[e] - E[I][e]);   // >= 1
                    const float r = ex2(E[I][e] - G[e]);   // <= 1
                    const float eg = ex2(G[e]);            // <= 1
                    rk[e] = kv[e] * f;
                    rq[e] = qv[e] * f;
                    kg[e] = kv[e] * eg;
                    qg[e] = qv[e] * eg;
                    kr[e] = kv[e] * r;
                }
                *kp = pack8(rk);
                *qp = pack8(rq);
                kg_hold[I] = pack8(kg);
                *reinterpret_cast<uint4*>(blob + BLOB_B1 + reg * 16384 + sw128(64 + i, ch)) = pack8(qg);
                // column operands of row blocks J >= I: k_j e^{E_J - G_j} = kr * e^{E_J - E_I}
#pragma unroll
                for (int J = 0; J < 4; ++J) {
                    if (J < I) continue;
                    if (J > I) {
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 x = __fmul2_rn(make_float2(kr[e], kr[e + 1]),
                                                        make_float2(dn[J - 1][e], dn[J - 1][e + 1]));
                            kr[e] = x.x;
                            kr[e + 1] = x.y;
                        }
                    }
                    const uint4 u = pack8(kr);
                    *reinterpret_cast<uint4*>(sm + P_CT + reg * kCTRegion + sw128(8 * J * (J + 1) + i, ch)) = u;
                    if (J == 3) *reinterpret_cast<uint4*>(blob + BLOB_KP + reg * 8192 + sw128(i, ch)) = u;
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // ---- the four row blocks of A; then K e^G takes the place of the running sum
        if (warp == 0) {  // the products are issued by warp 0 (one elected lane)
            tc_fence_after();
            mma_k128(tbase, kdesc(sbase + P_RR), 16384, kdesc(sbase + P_CT), kCTRegion,
                     idesc_bf16_f32(128, 160, false, false));
            mma_commit(barA);
            if (tid == 0) pend |= 4u;
        }
#pragma unroll
        for (int I = 0; I < 4; ++I)
            *reinterpret_cast<uint4*>(sm + P_KG + reg * 8192 + sw128(r4 + 16 * I, ch)) = kg_hold[I];
        fence_proxy_async();
        if (tid == 0) {
            solo_wait(barA, ph, sAbort, err);
            pend &= ~4u;
        }
        cta_sync_tc();
        if (*sAbort) break;
        float* sAkk = reinterpret_cast<float*>(sm + P_AKK);
        float* sTf = reinterpret_cast<float*>(sm + P_TF);
        // ---- A_kk (fp32 work array) and A_qk (bf16 hi and lo operands, to the workspace)
        {
            // lane quarter qt holds rows 32qt .. 32qt+31 of [k-rows ; q-rows]: lanes 0-15 belong to row block
            // IbA = 2(qt%2), lanes 16-31 to IbA + 1; warp half hq takes columns 32hq .. 32hq+31 of each lane's own
            // block (both blocks' columns are loaded, each lane keeps its block's), so every lane works.
            const int qt = warp & 3, hq = warp >> 2, IbA = 2 * (qt & 1);
            const int r = 32 * qt + lane;
            const int i = r & 63;
            const bool is_k = r < 64;
            const int Ib = IbA + (lane >> 4);
            const uint32_t lane_base = (uint32_t)(32 * qt) << 16;
            uint32_t a[32];
            {
                uint32_t t0[32], t1[32];
                tmem_ld32_async(tbase + lane_base + 8 * IbA * (IbA + 1) + 32 * hq, t0);
                tmem_ld32_async(tbase + lane_base + 8 * (IbA + 1) * (IbA + 2) + 32 * hq, t1);
                tmem_wait_ld(); reg_fence(t0); reg_fence(t1);
                const bool second = lane >= 16;
#pragma unroll
                for (int e = 0; e < 32; ++e) a[e] = second ? t1[e] : t0[e];
            }
            const int ncols = 16 * (Ib + 1), j0 = 32 * hq;
            if (is_k) {  // columns past the block's are never read by the solve
                const float b = sBeta[i];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    float4 w;
                    float* wp = reinterpret_cast<float*>(&w);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = j0 + 4 * j4 + e;
                        wp[e] = (j < i && j < ncols) ? b * __uint_as_float(a[4 * j4 + e]) : 0.f;
                    }
                    *reinterpret_cast<float4*>(sAkk + i * kAS + j0 + 4 * j4) = w;
                }
            } else {
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {  // hi and lo bf16 tiles, 8 columns per 16-byte chunk
                    float fh[8], fl[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = j0 + 8 * c8 + e;
                        const float x = (j <= i && j < ncols) ? __uint_as_float(a[8 * c8 + e]) : 0.f;
                        fh[e] = __bfloat162float(__float2bfloat16_rn(x));
                        fl[e] = x - fh[e];
                    }
                    *reinterpret_cast<uint4*>(sm + P_AQS + sw128(i, 4 * hq + c8)) = pack8(fh);
                    *reinterpret_cast<uint4*>(sm + P_AQS + 8192 + sw128(i, 4 * hq + c8)) = pack8(fl);
                }
            }
        }
        __syncthreads();
        // ---- T = (I + A_kk)^-1 by 16 x 16 blocks (fp32); meanwhile warps 4-7 copy A_qk out as whole rows
        if (warp >= 4) {
            const int t = tid - 128;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                *reinterpret_cast<uint4*>(blob + BLOB_AQ + 2048 * k + 16 * t) =
                    *reinterpret_cast<const uint4*>(sm + P_AQS + 2048 * k + 16 * t);
        }
        t_diag_blocks(sAkk, sTf, warp, lane);
        __syncthreads();
        t_offdiag_1(sAkk, sTf, reinterpret_cast<float*>(sm + P_NB), tid);
        // A_kk (this item's rr) is consumed: the next item's g lands there while the solve goes on
        if (have_next) {
            load_g_tma(h1, c01, P_RR);
            if (tid == 0) pend |= 16u;
        }
        t_offdiag_23(sTf, reinterpret_cast<float*>(sm + P_NB), tid);
        // ---- T Diag(beta) = hi + lo (bf16 each): thread owns row tid / 4, columns 16 (tid % 4) ..
        {
            const int i = tid >> 2, j0 = 16 * (tid & 3);
            float tv[16];
#pragma unroll
            for (int j4 = 0; j4 < 16; j4 += 4) {
                const float4 x = *reinterpret_cast<const float4*>(sTf + i * kAS + j0 + j4);
                const float4 bb = *reinterpret_cast<const float4*>(sBeta + j0 + j4);
                const bool zero = (j0 >> 4) > (i >> 4);   // above the diagonal blocks
                tv[j4] = zero ? 0.f : x.x * bb.x; tv[j4 + 1] = zero ? 0.f : x.y * bb.y;
                tv[j4 + 2] = zero ? 0.f : x.z * bb.z; tv[j4 + 3] = zero ? 0.f : x.w * bb.w;
            }
            float hiv[16], lov[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                hiv[e] = __bfloat162float(__float2bfloat16_rn(tv[e]));
                lov[e] = tv[e] - hiv[e];
            }
            __syncthreads();  // every read of T is done: its space takes the two operands
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
                float a8[8], b8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) { a8[e] = hiv[8 * h8 + e]; b8[e] = lov[8 * h8 + e]; }
                const uint32_t at = sw128(i, (j0 >> 3) + h8), at2 = sw128(64 + i, (j0 >> 3) + h8);
                const uint4 hv = pack8(a8), lv = pack8(b8);
                *reinterpret_cast<uint4*>(sm + P_TH + at) = hv;
                *reinterpret_cast<uint4*>(sm + P_TH + at2) = hv;
                *reinterpret_cast<uint4*>(sm + P_TL + at) = lv;
                *reinterpret_cast<uint4*>(sm + P_TL + at2) = lv;
                *reinterpret_cast<uint4*>(blob + BLOB_TB + at) = hv;         // the state pass's U^T = V^T T_b^T
                *reinterpret_cast<uint4*>(blob + BLOB_TB + 8192 + at) = lv;
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // ---- the next item's beta (this item's is consumed); its g is on the way since the solve
        const int this_item = item;
        item = next_item;
        have = have_next;
        if (have) load_beta(h1, c01, L1);
        // ---- W = T Diag(beta) K e^G: [T ; T] K e^G (hi, then lo)
        if (warp == 0) {
            tc_fence_after();
            const uint32_t id_w = idesc_bf16_f32(128, 128, false, true);
            const uint64_t th = kdesc(sbase + P_TH), tl = kdesc(sbase + P_TL);
            const uint64_t kvd = sdesc_sw128(sbase + P_KG, 8192, 1024);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase, th + ks * 2, kvd + ks * 128, id_w, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase, tl + ks * 2, kvd + ks * 128, id_w, 1u);
            mma_commit(barW);
            pend |= 8u;
            solo_wait(barW, ph, sAbort, err);
            pend &= ~8u;
        }
        cta_sync_tc();
        if (*sAbort) break;
        // ---- the next item's k and q land in this item's gb while W goes out
        if (have) {
            load_kq(h1, c01, P_G);
            if (tid == 0 && !FE) pend |= 1u;
        }
        // -W (bf16, rows 0-63 of B1): warp w reads TMEM lanes 32 (w % 4) .. +31, i.e. rows 32 (w % 2) + lane
        // (lanes 64-127 hold rows 0-63 again), and columns 32 (w / 2) .. +31, stages them in 2 KB of the
        // column-operand region (free: T hi/lo are consumed; 16-byte chunks rotated by lane pair against
        // bank conflicts) and stores them as half rows of 64 bytes.
        {
            uint8_t* bl = blobs + (int64_t)this_item * kStride;
            const int q = warp & 3, cq = warp >> 1;  // lane quarter; column quarter
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            uint8_t* stg = sm + P_CT + warp * 2048;
            uint32_t x[32];
            tmem_ld32_async(tbase + lane_base + 32 * cq, x);
            tmem_wait_ld(); reg_fence(x);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = -__uint_as_float(x[8 * c + e]);
                *reinterpret_cast<uint4*>(stg + 64 * lane + 16 * (c ^ ((lane >> 1) & 3))) = pack8(f);
            }
            __syncwarp();
            // row 32 (q % 2) + r of region cq / 2, 16-byte chunks 4 (cq % 2) .. +3 of it (in the row's swizzle)
            uint8_t* dst = bl + BLOB_B1 + (cq >> 1) * 16384;
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // rows 8k .. 8k+7 of the warp's 32, four lanes per row
                const int r = 8 * k + (lane >> 2), c = lane & 3;
                const int row = 32 * (q & 1) + r;
                *reinterpret_cast<uint4*>(dst + sw128(row, 4 * (cq & 1) + c)) =
                    *reinterpret_cast<const uint4*>(stg + 64 * r + 16 * (c ^ ((r >> 1) & 3)));
            }
        }
        h = h1;
        c0 = c01;
        L = L1;
        tc_fence_before();
    }
    cp_async_wait_all();
    if (*sAbort && tid == 0) {  // copies or products still in flight end before the CTA does (bounded)
        if (pend & 1u) mbar_wait(barL, 0, kWaitLimit), mbar_wait(barL, 1, kWaitLimit);
        if (pend & 4u) mbar_wait(barA, 0, kWaitLimit), mbar_wait(barA, 1, kWaitLimit);
        if (pend & 8u) mbar_wait(barW, 0, kWaitLimit), mbar_wait(barW, 1, kWaitLimit);
        if (pend & 16u) mbar_wait(barG, 0, kWaitLimit), mbar_wait(barG, 1, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kPrepTmemCols);
}

// =============================================================================================
// chunk_state_kernel: one (sequence, head) chain through a range of its chunks
// =============================================================================================
constexpr int kSimt = 512;               // 16 warps hold the state and do the element-wise work
constexpr int kThreads = kSimt + 32;     // + one warp that issues the products and copies
constexpr int kMmaWarp = kSimt / 32;
// Named barriers between the two roles (id 0 is __syncthreads), each completed by all kThreads:
constexpr int NB_S = 1;  // SIMT -> MMA warp: bf16 state operand stored (e^{G_C} and the old B1 buffer free)
constexpr int NB_Y = 2;  // MMA warp -> SIMT: V'^T of the chunk in TMEM
constexpr int NB_V = 3;  // SIMT -> MMA warp: V' hi and lo stored
constexpr int NB_D = 4;  // MMA warp -> SIMT: dS in TMEM
constexpr int NB_O = 5;  // MMA warp -> SIMT: the chunk's output product complete
// Copies run ahead of their use: three B1 buffers, two of T_b/v and two of A_qk/KP, each chunk's data
// issued two chunks before it is needed.
constexpr uint32_t S_B1 = 0;            // [-W ; Q e^G] of three chunks, 32 KB each
constexpr uint32_t S_TB = 98304;        // T Diag(beta) bf16 hi, lo ([64][64] each) of two chunks
constexpr uint32_t S_V = 131072;        // v bf16, two regions of [64 tokens][64], of two chunks
constexpr uint32_t S_AQ = 163840;       // A_qk bf16 hi, lo (16 KB) then KP = K e^{G_C - G} bf16 (16 KB), two chunks
constexpr uint32_t S_EGL = 229376;      // e^{G_C} fp32 [128] of three chunks (copied with that chunk's B1)
constexpr uint32_t S_BAR = 230912;      // mbarriers: B1 x3, T_b/v x2, A_qk/KP x2, S0 products, dS, output product
constexpr uint32_t S_MISC = S_BAR + 128; // TMEM base, abort flag
constexpr uint32_t kStateSmem = S_MISC + 16 + 1008;
constexpr uint32_t kAQKBytes = BLOB_EGL - BLOB_AQ;
constexpr uint32_t kKPOff = BLOB_KP - BLOB_AQ;
// TMEM columns: products of chunk parity p at 128 p (V'^T = U^T - S0 W^T in 64 columns, then O^T in 64); dS at 256;
// the A operands of the products, bf16 packed two per column: S0 at 384 (64 columns), V'^T hi at 448
// and V'^T lo at 480 (32 columns each)
constexpr uint32_t TM_DS = 256, TM_SA = 384, TM_VH = 448, TM_VL = 480;
constexpr uint32_t kTmemCols = 512;

static_assert(kKPOff % 1024 == 0 && S_AQ % 1024 == 0 && S_TB % 1024 == 0 && S_V % 1024 == 0 &&
                  S_V + 2 * 16384 <= S_AQ && S_EGL + 1536 <= S_BAR, "alignment");
static_assert(kStateSmem <= 232448, "shared memory");

__device__ __forceinline__ void nb_sync(int id) { asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kThreads) : "memory"); }
__device__ __forceinline__ void nb_arrive(int id) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "n"(kThreads) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
chunk_state_kernel(const __grid_constant__ CUtensorMap tm_v, const float* init_state, const int32_t* __restrict__ cu,
                   const int32_t* __restrict__ off, int64_t T_total, int H, float scale,
                   const __nv_bfloat16* __restrict__ gate, __nv_bfloat16* __restrict__ o, float* final_state,
                   const float* carry_in, float* carry_out, int first_range, int m0, int m1,
                   const uint8_t* __restrict__ blobs, uint32_t blob_bytes, int mode, unsigned int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool zero_u = (mode & kStateZeroU) != 0;  // U taken as zero (v = 0): the transition operator
    const int chain = blockIdx.x, n = chain / H, h = chain % H;
    const int on = off ? off[n] : 0, on1 = off ? off[n + 1] : (int)((T_total + kC - 1) / kC);
    int lo = on > m0 ? on : m0, hi = on1 < m1 ? on1 : m1;
    const bool empty_seq = on == on1;
    if (empty_seq) {
        if (!first_range) return;  // an empty sequence passes its initial state through once
        lo = hi = 0;
    } else if (lo >= hi) {
        return;                    // no chunk of this chain in the range
    }
    const bool starts = empty_seq || lo == on;   // the chain begins here: initial state
    const bool ends = empty_seq || hi == on1;    // the chain ends here: final state
    const int row = tid & 127, qq = (tid >> 7) & 3;  // state row / TMEM lane; quarter of the key channels / tokens
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int64_t in_off = (starts ? (int64_t)chain : (int64_t)h) * kD * kD + (int64_t)row * kD + 32 * qq;
    const int64_t out_off = (ends ? (int64_t)chain : (int64_t)h) * kD * kD + (int64_t)row * kD + 32 * qq;
    const float* s_in = starts ? init_state : carry_in;
    float* s_out = ends ? final_state : carry_out;
    int64_t bos, eos;
    seq_bounds(cu, n, T_total, bos, eos);

    uint64_t* barB = reinterpret_cast<uint64_t*>(sm + S_BAR);  // [3] B1 and e^{G_C}
    uint64_t* barV = barB + 3;                                 // [2] T_b and v
    uint64_t* barK = barB + 5;                                 // [2] A_qk and KP
    uint64_t* barM = barB + 7;
    uint64_t* barD = barB + 8;
    uint64_t* barO = barB + 9;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + S_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + S_MISC + 4);

    if (tid == 0) {
        for (int i = 0; i < 10; ++i) mbar_init(barB + i, 1);
        fence_mbar_init();
        *sAbort = 0;
    }
    if (warp == 0) tmem_alloc(sTmem, kTmemCols);
    tc_fence_before();
    __syncthreads();  // barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tbase = *sTmem;

    float s[32];  // SIMT threads: the state, row `row`, key channels [32 qq, 32 qq + 32)
    if (warp == kMmaWarp) {
        // ======== products and copies: one warp, MMAs from an elected lane, copies from lane 0 ========
        auto blob_of = [&](int mm) { return blobs + ((int64_t)(mm - m0) * H + h) * blob_bytes; };
        // a bit flips per copy issued, as the phase bits flip per copy consumed: B1 buffers bits 0-2,
        // T_b/v buffers bits 3-4, A_qk/KP buffers bits 5-6
        uint32_t iss = 0;
        auto load_b1 = [&](int mm, int j) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(barB + j, 32768 + 512);
                bulk_load(sm + S_B1 + j * 32768, blob_of(mm) + BLOB_B1, 32768, barB + j);
                bulk_load(sm + S_EGL + j * 512, blob_of(mm) + BLOB_EGL, 512, barB + j);
            }
            __syncwarp();
            iss ^= 1u << j;
        };
        // T_b from the workspace; v straight from its tensor (token rows of the chunk; rows past the end of the
        // sequence meet zero columns of T_b)
        auto load_v = [&](int mm, int j) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(barV + j, 32768);
                bulk_load(sm + S_TB + j * 16384, blob_of(mm) + BLOB_TB, 16384, barV + j);
                const int tok = (int)(bos + (int64_t)kC * (mm - on));
                tma_load_3d(sm + S_V + j * 16384, &tm_v, 0, h, tok, barV + j);
                tma_load_3d(sm + S_V + j * 16384 + 8192, &tm_v, 64, h, tok, barV + j);
            }
            __syncwarp();
            iss ^= 8u << j;
        };
        auto load_aq = [&](int mm, int j) {
            if (lane == 0) {
                fence_proxy_async();
                mbar_arrive_expect_tx(barK + j, kAQKBytes);
                bulk_load(sm + S_AQ + j * 32768, blob_of(mm) + BLOB_AQ, kAQKBytes, barK + j);
            }
            __syncwarp();
            iss ^= 32u << j;
        };
        auto wait = [&](uint64_t* bar, uint32_t ph) { solo_wait(bar, ph, sAbort, err); };
        const uint32_t id_64 = idesc_bf16_f32(128, 64, false, false);
        const uint32_t id_u = idesc_bf16_f32(128, 64, true, false);   // A = V^T (MN-major), B = T_b (K-major)
        const uint32_t id_ds = idesc_bf16_f32(128, 128, false, true);
        uint32_t ph = 0;              // bit per buffer barrier, as iss
        uint32_t phM = 0, phD = 0, phO = 0;
        for (int i = 0; i < 2 && lo + i < hi; ++i) {
            load_b1(lo + i, i);
            if (!zero_u) load_v(lo + i, i);
            load_aq(lo + i, i);
        }
        int b = 0, b3 = 0;  // TMEM [V' | O] buffer and B1 buffer of this chunk; T_b/v and A_qk/KP buffers follow b
        for (int mm = lo; mm < hi; ++mm, b ^= 1, b3 = b3 == 2 ? 0 : b3 + 1) {
            const bool ahead = mm + 2 < hi;
            // ---- U^T = V^T T_b^T (hi, then lo) into the V' columns, while the state warps finish the previous
            //      chunk (those columns were last read two chunks ago)
            if (!zero_u) {
                wait(barV + b, (ph >> (3 + b)) & 1u);
                ph ^= 8u << b;
                tc_fence_after();
                const uint64_t vd = sdesc_sw128(sbase + S_V + b * 16384, 8192, 1024);
                const uint64_t th = kdesc(sbase + S_TB + b * 16384), tl = kdesc(sbase + S_TB + b * 16384 + 8192);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + 128 * b, vd + ks * 128, th + ks * 2, id_u, ks > 0 ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16(tbase + 128 * b, vd + ks * 128, tl + ks * 2, id_u, 1u);
            }
            // ---- V'^T = U^T + S0 (-W)^T (the V' pass waits for it), then O^T = S0 (Q e^G)^T; A = S0 from TMEM
            nb_sync(NB_S);
            wait(barB + b3, (ph >> b3) & 1u);
            ph ^= 1u << b3;
            tc_fence_after();
            const uint32_t b1 = sbase + S_B1 + b3 * 32768;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ta(tbase + 128 * b, tbase + TM_SA + 8 * ks,
                            kdesc(b1 + (ks >> 2) * 16384) + (ks & 3) * 2, id_64, (ks > 0 || !zero_u) ? 1u : 0u);
            mma_commit(barM);
            wait(barM, phM);
            phM ^= 1u;
            const bool stop = *sAbort != 0;
            tc_fence_before();
            nb_arrive(NB_Y);
            if (stop) break;
            if (ahead && !zero_u) load_v(mm + 2, b);  // T_b and v of this chunk are consumed (U^T is complete)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16_ta(tbase + 128 * b + 64, tbase + TM_SA + 8 * ks,
                            kdesc(b1 + (ks >> 2) * 16384 + 8192) + (ks & 3) * 2, id_64, ks > 0 ? 1u : 0u);
            if (ahead) load_b1(mm + 2, b3 == 0 ? 2 : b3 - 1);  // the previous chunk's B1 and e^{G_C} are consumed
            // ---- dS = (V'_hi + V'_lo)^T (K e^{G_C - G}) (the state waits for it), then O^T += V'^T A_qk^T
            //      as hi.hi + hi.lo + lo.hi; A = V'^T from TMEM
            nb_sync(NB_V);
            wait(barK + b, (ph >> (5 + b)) & 1u);
            ph ^= 32u << b;
            tc_fence_after();
            const uint32_t aq = sbase + S_AQ + b * 32768;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(tbase + TM_DS, tbase + TM_VH + 8 * ks, sdesc_sw128(aq + kKPOff, 8192, 1024) + ks * 128,
                            id_ds, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(tbase + TM_DS, tbase + TM_VL + 8 * ks, sdesc_sw128(aq + kKPOff, 8192, 1024) + ks * 128,
                            id_ds, 1u);
            mma_commit(barD);
            wait(barD, phD);
            phD ^= 1u;
            tc_fence_before();
            nb_arrive(NB_D);
            const uint32_t od = tbase + 128 * b + 64;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(od, tbase + TM_VH + 8 * ks, kdesc(aq) + ks * 2, id_64, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ta(od, tbase + TM_VH + 8 * ks, kdesc(aq + 8192) + ks * 2, id_64, 1u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_bf16_ta(od, tbase + TM_VL + 8 * ks, kdesc(aq) + ks * 2, id_64, 1u);
            mma_commit(barO);
            wait(barO, phO);
            phO ^= 1u;
            if (ahead) load_aq(mm + 2, b);  // A_qk and KP of this chunk are consumed
            tc_fence_before();
            nb_arrive(NB_O);
        }
        if (*sAbort && lane == 0) {  // let copies still in flight land (bounded) before the CTA exits
            for (int j = 0; j < 3; ++j)
                if (((iss ^ ph) >> j) & 1u) mbar_wait(barB + j, (ph >> j) & 1u, kWaitLimit);
            for (int j = 0; j < 2; ++j) {
                if (((iss ^ ph) >> (3 + j)) & 1u) mbar_wait(barV + j, (ph >> (3 + j)) & 1u, kWaitLimit);
                if (((iss ^ ph) >> (5 + j)) & 1u) mbar_wait(barK + j, (ph >> (5 + j)) & 1u, kWaitLimit);
            }
        }
        __syncwarp();
    } else {
        // ======== the state: thread (row, qq) holds row `row`, key channels [32 qq, 32 qq + 32) ========
        const bool ident = !s_in && (mode & kStateIdentity);  // a chain that starts from I (dv = dk)
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 x = s_in ? *reinterpret_cast<const float4*>(s_in + in_off + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            s[j] = x.x; s[j + 1] = x.y; s[j + 2] = x.z; s[j + 3] = x.w;
        }
        if (ident) {
#pragma unroll
            for (int j = 0; j < 32; ++j) s[j] = (row == 32 * qq + j) ? 1.f : 0.f;
        }
        auto write_state_operand = [&]() {  // bf16 copy in TMEM, the A operand of the S0 products
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(s[2 * j], s[2 * j + 1]);
            tmem_st16(tbase + lane_base + TM_SA + 16 * qq, w);
            tmem_wait_st();
        };
        // outputs of chunk mm (its product complete, in TMEM columns 128 p + 64): thread (row, qq) stores
        // tokens 16qq + 8 half .. + 7 of value row `row`; a warp writes 64 contiguous bytes per token.  The
        // two halves go out while the products of the next chunk run.
        // The output gate of chunk mm (when given), loaded right after the previous chunk's outputs are stored
        // and used when this chunk's are, an iteration later (the loads complete meanwhile, off the state
        // warps' path): thread (row, qq) holds tokens 16qq .. 16qq + 15 of value row `row` as bf16 pairs
        // (zero past the end of the sequence).  One buffer: the state warps' 96 registers hold no more.
        uint32_t g_cur[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) g_cur[j] = 0u;
        auto load_gate = [&](int mm) {
            const int64_t c0 = bos + (int64_t)kC * (mm - on);
            const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
            const int64_t stride = (int64_t)H * kD;
            const unsigned short* gp = reinterpret_cast<const unsigned short*>(gate) + ((c0 + 16 * qq) * H + h) * kD + row;
            if (16 * qq + 16 <= L) {  // all 16 tokens inside the sequence
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t a = __ldcs(gp), c = __ldcs(gp + stride);
                    g_cur[j] = a | (c << 16);
                    gp += 2 * stride;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t a = (16 * qq + 2 * j < L) ? (uint32_t)__ldcs(gp + (2 * j) * stride) : 0u;
                    const uint32_t c = (16 * qq + 2 * j + 1 < L) ? (uint32_t)__ldcs(gp + (2 * j + 1) * stride) : 0u;
                    g_cur[j] = a | (c << 16);
                }
            }
        };
        auto emit_o = [&](int mm, int p, int half) {
            const int64_t c0 = bos + (int64_t)kC * (mm - on);
            const int L = (eos - c0) < kC ? (int)(eos - c0) : kC;
            const int t0 = 16 * qq + 8 * half;
            uint32_t xo[8];
            tmem_ld8_async(tbase + lane_base + 128 * p + 64 + t0, xo);
            tmem_wait_ld(); reg_fence(xo);
            const int64_t stride = (int64_t)H * kD;
            const int64_t at0 = ((c0 + t0) * H + h) * kD + row;
            __nv_bfloat16* op = o + at0;
            if (gate) {
                // o sigma(gate) = o / (1 + e^-gate): the fast divide (2 ulp for a divisor in [1, 2^126); beyond,
                // where sigma < 1e-38, it gives 0) keeps this epilogue inside the dS product's wait
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (t0 + e < L) {
                        const uint32_t pr = half ? g_cur[4 + (e >> 1)] : g_cur[e >> 1];  // static indices
                        const float gv = (e & 1) ? bf16_hi(pr) : bf16_lo(pr);
                        op[e * stride] =
                            __float2bfloat16_rn(__fdividef(scale * __uint_as_float(xo[e]), 1.0f + __expf(-gv)));
                    }
            } else if (L == kC) {
#pragma unroll
                for (int e = 0; e < 8; ++e) op[e * stride] = __float2bfloat16_rn(scale * __uint_as_float(xo[e]));
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (t0 + e < L) op[e * stride] = __float2bfloat16_rn(scale * __uint_as_float(xo[e]));
            }
        };
        if (lo < hi) write_state_operand();
        int b = 0, b3 = 0;
        bool stopped = false;
        for (int mm = lo; mm < hi; ++mm, b ^= 1, b3 = b3 == 2 ? 0 : b3 + 1) {
            tc_fence_before();
            nb_arrive(NB_S);
            if (mm > lo) {
                nb_sync(NB_O);
                tc_fence_after();
            }
            nb_sync(NB_Y);
            tc_fence_after();
            if (*sAbort) {
                stopped = true;
                break;
            }
            // ---- V'^T (from TMEM); thread (row, qq) owns tokens 16qq .. 16qq+15, stored back to TMEM as bf16
            //      hi and lo (x = hi + lo to about 16 bits)
            {
                uint32_t y[16];
                tmem_ld16_async(tbase + lane_base + 128 * b + 16 * qq, y);
                tmem_wait_ld(); reg_fence(y);
                float hv[16], lv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float x = __uint_as_float(y[e]);
                    hv[e] = __bfloat162float(__float2bfloat16_rn(x));
                    lv[e] = x - hv[e];
                }
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    wh[j] = pack_bf16x2(hv[2 * j], hv[2 * j + 1]);
                    wl[j] = pack_bf16x2(lv[2 * j], lv[2 * j + 1]);
                }
                tmem_st8(tbase + lane_base + TM_VH + 8 * qq, wh);
                tmem_st8(tbase + lane_base + TM_VL + 8 * qq, wl);
                tmem_wait_st();
            }
            tc_fence_before();
            nb_arrive(NB_V);
            if (mm > lo && o) {
                emit_o(mm - 1, b ^ 1, 0);
                emit_o(mm - 1, b ^ 1, 1);
            }
            if (gate && o) load_gate(mm);
            // ---- the state update
            nb_sync(NB_D);
            tc_fence_after();
            {
                const float* sEGl = reinterpret_cast<const float*>(sm + S_EGL + b3 * 512);
                uint32_t d0[32];
                tmem_ld32_async(tbase + lane_base + TM_DS + 32 * qq, d0);
                float eg[32];
#pragma unroll
                for (int e4 = 0; e4 < 32; e4 += 4)
                    *reinterpret_cast<float4*>(eg + e4) = *reinterpret_cast<const float4*>(sEGl + 32 * qq + e4);
                tmem_wait_ld(); reg_fence(d0);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[e] = fmaf(s[e], eg[e], __uint_as_float(d0[e]));
            }
            if (mm + 1 < hi) write_state_operand();
        }
        if (lo < hi && !stopped) {
            nb_sync(NB_O);
            tc_fence_after();
            if (o) {
                emit_o(hi - 1, (hi - 1 - lo) & 1, 0);
                emit_o(hi - 1, (hi - 1 - lo) & 1, 1);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp != kMmaWarp && s_out && !*sAbort) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(s_out + out_off + j) = make_float4(s[j], s[j + 1], s[j + 2], s[j + 3]);
    }
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

// [T, H, 128] tensor of `elem` bytes per value, boxes of [64 tokens][1 head][inner channels], with the
// 128-byte swizzle (inner * elem = 128 bytes, the operand-tile layout).
bool encode_chunk_map(CUtensorMap* m, const void* base, CUtensorMapDataType type, int elem, int inner, int64_t T,
                      int H) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)128 * elem, (cuuint64_t)H * 128 * elem};
    const cuuint32_t box[3] = {(cuuint32_t)inner, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, type, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Overlapped ranges: about this many ranges of at least this many chunk rows, and (chunk, head) items per
// operand-kernel CTA there.  Measured on one GB300 (96 heads): 8K tokens (128 rows) run fastest as one
// range (0.842 ms against 0.863 for two overlapped ranges of 64 rows); 32K tokens (512 rows) in four
// ranges of 128 rows with four items per CTA (3.11 ms against 3.25 for eight ranges of 64 rows and one
// item per CTA, 3.30 for one range); 256K tokens (4,096 rows) in eight ranges of 512 rows (33.47 ms
// with the output gate, against 34.12 for four ranges of 1,024 rows and 33.43 for sixteen of 256).
constexpr int64_t kPipeRanges = 8, kPipeMinRows = 128, kPipeItemsPerCta = 4;

// Two streams per device (created once): a low-priority one for the operand kernel and a
// high-priority one for the state pass.
static cudaError_t side_streams(int dev, cudaStream_t* s_low, cudaStream_t* s_high) {
    static std::mutex mu;
    static cudaStream_t streams[64][2] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!streams[dev][0]) {
        int least = 0, greatest = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&streams[dev][0], cudaStreamNonBlocking, least);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&streams[dev][1], cudaStreamNonBlocking, greatest);
        if (e != cudaSuccess) {
            streams[dev][0] = streams[dev][1] = nullptr;
            return e;
        }
    }
    *s_low = streams[dev][0];
    *s_high = streams[dev][1];
    return cudaSuccess;
}

// Events of one call (released when the set goes out of scope; the driver keeps an event alive
// until the work it records has completed).
struct EventSet {
    explicit EventSet(int n) : n_(n), ev_(new cudaEvent_t[n]()) {
        for (int i = 0; i < n; ++i)
            if (cudaEventCreateWithFlags(&ev_[i], cudaEventDisableTiming) != cudaSuccess) ev_[i] = nullptr;
    }
    ~EventSet() {
        for (int i = 0; i < n_; ++i)
            if (ev_[i]) cudaEventDestroy(ev_[i]);
        delete[] ev_;
    }
    bool ok() const {
        for (int i = 0; i < n_; ++i)
            if (!ev_[i]) return false;
        return true;
    }
    cudaEvent_t operator[](int i) const { return ev_[i]; }
    EventSet(const EventSet&) = delete;
    EventSet& operator=(const EventSet&) = delete;

  private:
    int n_;
    cudaEvent_t* ev_;
};

// Workspace: [carried states, 2 x H x 128 x 128 fp32][chunk offsets, int32 N + 1][operands of
// `rows` chunk rows x H heads, kBlobBytes each] (the same with the fused front end).
static size_t ws_header_bytes(int N, int H) {
    return (size_t)2 * H * kStateBytes + (((size_t)(N + 1) * 4 + 1023) / 1024) * 1024;
}

// Upper bound of the number of chunks over all sequences (exact for one sequence without offsets).
static int64_t max_chunk_rows(int N, int64_t T_total, bool have_cu) {
    return have_cu ? T_total / kC + N : (T_total + kC - 1) / kC;
}

void chunk_tc_workspace(int N, int64_t T_total, int H, bool have_cu, size_t* full_bytes, size_t* min_bytes) {
    const size_t row = (size_t)H * kBlobBytes, hdr = ws_header_bytes(N, H);
    const int64_t rows = max_chunk_rows(N, T_total, have_cu);
    if (full_bytes) *full_bytes = hdr + row * (size_t)(rows > 0 ? rows : 1);
    if (min_bytes) *min_bytes = hdr + row;
}

cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                            float scale, const void* out_gate, void* o, float* final_state, void* workspace,
                            size_t workspace_bytes, const ChunkFrontend* front, unsigned int* err,
                            cudaStream_t stream, int state_mode, float* final_state2, int state_mode2,
                            bool overlap) {
    CUtensorMap tq = {}, tk = {}, tv = {}, tg;
    const uint32_t blob_bytes = kBlobBytes;
    // With the fused front end, v is computed by the stand-alone front end into `o` (the same shape) and read
    // back from there: each chunk's v tile is loaded before that chunk's outputs are written over it.
    if (front && !encode_chunk_map(&tv, o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, T_total, H)) return cudaErrorInvalidValue;
    if (!front && (!encode_chunk_map(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, T_total, H) ||
                   !encode_chunk_map(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, T_total, H) ||
                   !encode_chunk_map(&tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, T_total, H)))
        return cudaErrorInvalidValue;
    if (!encode_chunk_map(&tg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 32, T_total, H)) return cudaErrorInvalidValue;
    FrontendArgs fa = {};
    if (front)
        fa = FrontendArgs{static_cast<const __nv_bfloat16*>(front->xq), static_cast<const __nv_bfloat16*>(front->xk),
                          static_cast<const __nv_bfloat16*>(front->xv), front->x_stride,
                          static_cast<const __nv_bfloat16*>(front->conv_w),
                          static_cast<const __nv_bfloat16*>(front->conv_state_in), front->eps};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* carry = reinterpret_cast<float*>(ws);
    int32_t* off = reinterpret_cast<int32_t*>(ws + (size_t)2 * H * kStateBytes);
    uint8_t* blobs = ws + ws_header_bytes(N, H);
    const int64_t rows_max = max_chunk_rows(N, T_total, cu_seqlens != nullptr);
    int64_t rows = (int64_t)((workspace_bytes - ws_header_bytes(N, H)) / ((size_t)H * blob_bytes));
    if (rows < 1) return cudaErrorInvalidValue;
    if (rows > rows_max) rows = rows_max > 0 ? rows_max : 1;
    if (rows * H > 0x7FFFFFFF) rows = 0x7FFFFFFF / H;  // grid size of the prep kernel

    auto prep = front ? chunk_prep_kernel<true> : chunk_prep_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (cu_seqlens) chunk_offsets_kernel<<<1, 1024, 0, stream>>>(cu_seqlens, N, T_total, off);
    else off = nullptr;  // one sequence: the kernels use {0, ceil(T_total / 64)}
    // A second state pass on the same operands (final_state2, state_mode2) needs them all at once.
    if (final_state2 && rows < rows_max) return cudaErrorInvalidValue;
    if (overlap && !final_state2 && rows >= 2 * kPipeMinRows && rows_max >= 2 * kPipeMinRows) {
        // Overlapped ranges (when the call has, and the workspace holds, at least two ranges of
        // kPipeMinRows chunk rows): the chunk rows in about kPipeRanges ranges (of at least kPipeMinRows
        // rows: each extra range costs about 35 us of wave tails and state-pass start-up), their operands
        // in two alternating halves of the workspace; range r's state pass (high-priority stream, 96 of
        // the 152 SMs for 96 chains) runs while range r+1's operands are computed on the other SMs
        // (low-priority stream, short-lived CTAs of a few items each, so that the state pass's CTAs take SMs
        // first as they free up, while each item still loads the next one's inputs early).  Ordered by
        // events only.
        int64_t rr = (rows_max + kPipeRanges - 1) / kPipeRanges;
        if (rr < kPipeMinRows) rr = kPipeMinRows;
        if (rr > rows / 2) rr = rows / 2;
        cudaStream_t s_prep, s_state;
        e = side_streams(dev, &s_prep, &s_state);
        if (e != cudaSuccess) return e;
        const int nr = (int)((rows_max + rr - 1) / rr);
        EventSet ev(2 * nr + 1);
        if (!ev.ok()) return cudaErrorMemoryAllocation;
        cudaEvent_t ev_start = ev[2 * nr];
        e = cudaEventRecord(ev_start, stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_prep, ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_state, ev_start, 0);
        // v of the whole call ahead of the first state pass, beside the first range's operands (a pass bound by
        // memory beside one bound by its instruction stream)
        if (e == cudaSuccess && front)
            e = launch_frontend_v(front->xv, front->x_stride, front->conv_w, cu_seqlens, N, T_total, H,
                                  front->conv_state_in, o, s_state);
        for (int r = 0; r < nr && e == cudaSuccess; ++r) {
            const int64_t r0 = (int64_t)r * rr, r1 = r0 + rr < rows_max ? r0 + rr : rows_max;
            uint8_t* buf = blobs + (size_t)(r & 1) * (size_t)rr * H * blob_bytes;
            if (r >= 2) e = cudaStreamWaitEvent(s_prep, ev[nr + r - 2], 0);  // that half's state pass is done
            if (e != cudaSuccess) break;
            const int64_t items = (r1 - r0) * H;
            const int64_t grid = (items + kPipeItemsPerCta - 1) / kPipeItemsPerCta;
            prep<<<(unsigned)grid, kPrepThreads, kPrepSmem, s_prep>>>(tq, tk, tg, beta, cu_seqlens, off, N, T_total,
                                                                      H, (int)r0, (int)items, buf, fa, err);
            e = cudaGetLastError();
            if (e == cudaSuccess) e = cudaEventRecord(ev[r], s_prep);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s_state, ev[r], 0);
            if (e != cudaSuccess) break;
            float* c_out = carry + (size_t)(r & 1) * H * kD * kD;
            const float* c_in = carry + (size_t)((r + 1) & 1) * H * kD * kD;
            chunk_state_kernel<<<(unsigned)((int64_t)N * H), kThreads, kStateSmem, s_state>>>(
                tv, init_state, cu_seqlens, off, T_total, H, scale, static_cast<const __nv_bfloat16*>(out_gate),
                static_cast<__nv_bfloat16*>(o), final_state, c_in, c_out, r == 0 ? 1 : 0, (int)r0, (int)r1, buf,
                blob_bytes, state_mode, err);
            e = cudaGetLastError();
            if (e == cudaSuccess) e = cudaEventRecord(ev[nr + r], s_state);
        }
        // join: the caller's stream waits for both side streams' last work
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[nr - 1], 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[2 * nr - 1], 0);
        return e;
    }
    if (front) {
        e = launch_frontend_v(front->xv, front->x_stride, front->conv_w, cu_seqlens, N, T_total, H,
                              front->conv_state_in, o, stream);
        if (e != cudaSuccess) return e;
    }
    int range = 0;
    for (int64_t r0 = 0; range == 0 || r0 < rows_max; r0 += rows, ++range) {
        const int64_t r1 = r0 + rows < rows_max ? r0 + rows : rows_max;
        if (r1 > r0) {
            const int64_t items = (r1 - r0) * H;
            const int64_t grid = items < 2 * sms ? items : 2 * sms;
            prep<<<(unsigned)grid, kPrepThreads, kPrepSmem, stream>>>(
                tq, tk, tg, beta, cu_seqlens, off, N, T_total, H, (int)r0, (int)items, blobs, fa, err);
        }
        float* c_out = carry + (size_t)(range & 1) * H * kD * kD;
        const float* c_in = carry + (size_t)((range + 1) & 1) * H * kD * kD;
        chunk_state_kernel<<<(unsigned)((int64_t)N * H), kThreads, kStateSmem, stream>>>(
            tv, init_state, cu_seqlens, off, T_total, H, scale, static_cast<const __nv_bfloat16*>(out_gate),
            static_cast<__nv_bfloat16*>(o), final_state, c_in, c_out, range == 0 ? 1 : 0, (int)r0, (int)r1, blobs,
            blob_bytes, state_mode, err);
        if (final_state2)
            chunk_state_kernel<<<(unsigned)((int64_t)N * H), kThreads, kStateSmem, stream>>>(
                tv, nullptr, cu_seqlens, off, T_total, H, scale, nullptr, nullptr, final_state2, nullptr, nullptr, 1,
                (int)r0, (int)r1, blobs, blob_bytes, state_mode2, err);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace kda
