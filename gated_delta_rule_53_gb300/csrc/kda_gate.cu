// kda_gate_generator: the decay gate g and the full-rank output gate from the layer input x.
//
// "深入 Kimi-K3: Hugging Face 仓库分析", paragraph on KDA: the decay is per channel, driven by a
// low-rank projection plus a per-head parameter, with a lower bound of -5 (also "Kimi K3 架构
// 全景", section 02: gate lower_bound -5.0); the output gate is full rank.  Read here as
//   gate = x W_gate^T                              bf16 [T, H*d]
//   z    = x W_a^T                                 bf16 [T, r]     (rank r)
//   g    = max(-5, -softplus(z W_b^T + a_h))       fp32 [T, H, d]  (a_h: one parameter per head)
// The first two products share x, so they are one GEMM over the stacked weights [W_gate ; W_a];
// the second GEMM applies W_b with the bound in its epilogue.
//
// GEMM: C = A B^T, A [M, K] and B [N, K] bf16 with K innermost, fp32 accumulation in TMEM.
// Persistent CTAs (one per SM), tiles of 128 x 256 over (M, N) in groups of 16 row tiles (the CTAs
// running at one time share A and B bands in L2), K in blocks of 64 through a 4-stage TMA pipeline (128-byte
// swizzle, the tcgen05 K-major operand layout).  Warp 0 loads, warp 1 issues the products from
// one elected lane into one of two TMEM accumulators, warps 2-9 read the other accumulator out
// (lane quarter = warp % 4, half the columns each) and store it through shared memory as whole
// row segments, so a tile's epilogue overlaps the next tile's products.
// Every mbarrier wait is bounded; a wait that runs out stops the CTA and reports in the device
// error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr uint32_t kStageA = BM * BK * 2, kStageB = BN * BK * 2, kStageBytes = kStageA + kStageB;
// Two configurations: the x-side product (K = hidden, long main loop) keeps four stages of operands
// and eight epilogue warps; the rank product (K = rank, a short main loop and a transcendental epilogue)
// two stages and sixteen epilogue warps.  Shared memory: stages, 4 KB of staging per epilogue warp
// (32 rows x 128 bytes), then full[S], empty[S], acc_full[2], acc_empty[2], done, TMEM base, abort flag.
template <int S, int EW>
struct GemmCfg {
    static constexpr int kStages = S, kEpiWarps = EW, kThreads = 64 + 32 * EW;
    static constexpr uint32_t kStg = S * kStageBytes, kBar = kStg + EW * 4096, kMisc = kBar + 16 * 8;
    static constexpr uint32_t kSmem = kMisc + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(2 * S + 5 <= 16, "barrier space");
};
using CfgX = GemmCfg<4, 8>;
using CfgR = GemmCfg<2, 16>;
constexpr uint32_t kGemmWait = 1u << 24;

struct GemmEpi {
    int mode;                  // 0: gate (columns < n_split) and rank-r activations; 1: decay gate
    int n_split;               // mode 0
    __nv_bfloat16* c0;         // mode 0: [M, n_split]
    __nv_bfloat16* c1;         // mode 0: [M, N - n_split]
    float* g;                  // mode 1: [M, N]
    const float* a_head;       // mode 1: [N / d]
    int d;
};

// log(1 + e^x) by the hardware exponential and logarithm; above 15 it is x to fp32 precision
__device__ __forceinline__ float softplus(float x) { return x > 15.f ? x : __logf(1.f + __expf(x)); }

// Tile t of the persistent loop: groups of kGroupM m-tiles, n-tiles in turn inside a group, m fastest;
// the CTAs running at one time share a few A row bands and B column bands, which stay in L2.
constexpr int kGroupM = 16;
__device__ __forceinline__ void tile_coords(int t, int mt, int nt, int& m0, int& n0) {
    const int per_group = kGroupM * nt, gi = t / per_group, r = t - gi * per_group;
    const int gm = mt - gi * kGroupM < kGroupM ? mt - gi * kGroupM : kGroupM;
    m0 = (gi * kGroupM + r % gm) * BM;
    n0 = (r / gm) * BN;
}

// shared-memory descriptor of a K-major 128-byte-swizzled operand tile (8-row groups 1024 bytes apart)
__device__ __forceinline__ uint64_t kdesc_g(uint32_t saddr) { return sdesc_sw128(saddr, 16, 1024); }

// Columns [col, col + 32) of rows row0 .. row0 + 31 (this lane: row0 + lane) through the warp's
// staging rows (128 bytes each, 16-byte chunks swizzled by row), written back as whole row segments.
__device__ __forceinline__ void store_chunk(const GemmEpi& e, int64_t row0, int M, int col, int N,
                                            const uint32_t (&v)[32], uint8_t* stg, int lane) {
    __syncwarp();  // the previous chunk has been read back
    if (e.mode == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                w[i] = pack_bf16x2(__uint_as_float(v[8 * j + 2 * i]), __uint_as_float(v[8 * j + 2 * i + 1]));
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncwarp();
        const bool lo = col < e.n_split;
        __nv_bfloat16* base = lo ? e.c0 + col : e.c1 + (col - e.n_split);
        const int64_t ld = lo ? e.n_split : N - e.n_split;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // 8 rows of 64 bytes per instruction
            const int r = 8 * k + (lane >> 2), c = lane & 3;
            if (row0 + r < M)
                *reinterpret_cast<uint4*>(base + (row0 + r) * ld + 8 * c) =
                    *reinterpret_cast<const uint4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
        }
    } else {
        const float a = e.a_head[col / e.d];  // a chunk of 32 lies inside one head (d a multiple of 32)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = fmaxf(-5.f, -softplus(__uint_as_float(v[4 * j + i]) + a));
            *reinterpret_cast<float4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = make_float4(o[0], o[1], o[2], o[3]);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {  // 4 rows of 128 bytes per instruction
            const int r = 4 * k + (lane >> 3), c = lane & 7;
            if (row0 + r < M)
                *reinterpret_cast<float4*>(e.g + (row0 + r) * N + col + 4 * c) =
                    *reinterpret_cast<const float4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
gemm_gate_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                 GemmEpi epi, unsigned int* err) {
    constexpr int kStages = Cfg::kStages, kEpiWarps = Cfg::kEpiWarps;
    constexpr uint32_t G_STG = Cfg::kStg, G_BAR = Cfg::kBar, G_MISC = Cfg::kMisc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + G_BAR);
    uint64_t* empty = full + kStages;
    uint64_t* accf = empty + kStages;
    uint64_t* acce = accf + 2;
    uint64_t* done = acce + 2;
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + G_MISC);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + G_MISC + 4);
    const int mt = (M + BM - 1) / BM, nt = (N + BN - 1) / BN, kbn = (K + BK - 1) / BK;
    const int tiles = mt * nt;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accf + i, 1);
            mbar_init(acce + i, kEpiWarps);  // one arrival per epilogue warp
        }
        mbar_init(done, 1);
        fence_mbar_init();
        *sAbort = 0;
    }
    if (warp == 1) tmem_alloc(sTmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *sTmem;
    // bounded wait; false once this CTA has stopped
    auto wait = [&](uint64_t* b, uint32_t ph) -> bool {
        if (*sAbort) return false;
        if (mbar_wait(b, ph, kGemmWait)) return true;
        *sAbort = 1;
        raise_device_error(err, kErrMbarTimeout);
        return false;
    };

    if (warp == 0) {
        // ---- loads: stage s of round ph; a stage is refilled once the products that read it are done
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_ph = 0;  // bit s: stage s has a load in flight / its round
            bool ok = true;
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
                int m0, n0;
                tile_coords(t, mt, nt, m0, n0);
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!(ok = wait(empty + s, ph ^ 1u))) break;
                    fence_proxy_async();
                    mbar_arrive_expect_tx(full + s, kStageBytes);
                    tma_load_2d(sm + s * kStageBytes, &tmA, kb * BK, m0, full + s);
                    tma_load_2d(sm + s * kStageBytes + kStageA, &tmB, kb * BK, n0, full + s);
                    issued |= 1u << s;
                    issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
                    if (++s == kStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (*sAbort)  // let the copies in flight land (bounded) before the CTA exits
                for (int i = 0; i < kStages; ++i)
                    if ((issued >> i) & 1u) mbar_wait(full + i, (issued_ph >> i) & 1u, kGemmWait);
        }
    } else if (warp == 1) {
        // ---- products: accumulator a of tile `it` (two alternate), stage by stage
        const uint32_t id = idesc_bf16_f32(BM, BN, false, false);
        int s = 0, it = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++it) {
            const int a = it & 1;
            if (!(ok = wait(acce + a, ((aph >> a) & 1u) ^ 1u))) break;  // its previous tile has been read out
            aph ^= 1u << a;
            tc_fence_after();
            const uint32_t d = tbase + (uint32_t)(a * BN);
            for (int kb = 0; kb < kbn; ++kb) {
                if (!(ok = wait(full + s, ph))) break;
                tc_fence_after();
                const uint32_t sa = sbase + (uint32_t)(s * kStageBytes), sb = sa + kStageA;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(d, kdesc_g(sa) + ks * 2, kdesc_g(sb) + ks * 2, id, (kb | ks) ? 1u : 0u);
                mma_commit(empty + s);
                if (++s == kStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) mma_commit(accf + a);
        }
        mma_commit(done);  // every product issued has completed before the TMEM is released
        mbar_wait(done, 0, kGemmWait);
    } else {
        // ---- epilogue: warps 2 .. 2 + kEpiWarps - 1; lane quarter q = warp % 4 holds rows 32 q .. 32 q + 31
        //      of the tile, and part hf = (warp - 2) / 4 of the kEpiWarps / 4 parts takes BN / parts columns
        constexpr int kCols = BN / (kEpiWarps / 4);
        const int q = warp & 3, hf = (warp - 2) >> 2;
        uint8_t* stg = sm + G_STG + (warp - 2) * 4096;
        int it = 0;
        uint32_t fph = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int a = it & 1;
            if (!wait(accf + a, (fph >> a) & 1u)) break;
            fph ^= 1u << a;
            tc_fence_after();
            int m0, n0;
            tile_coords(t, mt, nt, m0, n0);
            const int64_t row0 = (int64_t)m0 + 32 * q;
#pragma unroll 1
            for (int c = kCols * hf; c < kCols * hf + kCols; c += 32) {
                uint32_t v[32];
                tmem_ld32_async(tbase + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * BN + c), v);
                tmem_wait_ld();
                reg_fence(v);
                if (row0 < M && n0 + c < N) store_chunk(epi, row0, M, n0 + c, N, v, stg, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce + a);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tbase, 512);
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

// bf16 [rows, K] with K innermost; boxes of [box_rows][64] with the 128-byte swizzle
bool encode_operand(CUtensorMap* m, const void* base, int64_t rows, int64_t K, int box_rows) {
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)(rows > 0 ? rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Cfg>
cudaError_t gemm(const void* A, const void* B, int M, int N, int K, const GemmEpi& epi, unsigned int* err,
                 cudaStream_t stream) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    CUtensorMap ta, tb;
    if (!encode_operand(&ta, A, M, K, BM) || !encode_operand(&tb, B, N, K, BN)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(gemm_gate_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    int dev = 0, sms = 0;
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int grid = (int)(tiles < sms ? tiles : sms);
    gemm_gate_kernel<Cfg><<<grid, Cfg::kThreads, Cfg::kSmem, stream>>>(ta, tb, M, N, K, epi, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_generator(const void* x, int64_t T, int hidden, const void* w_gate_a, const void* w_b,
                                  const float* a_head, int H, int d, int rank, void* gate, float* g, void* z,
                                  unsigned int* err, cudaStream_t stream) {
    const int hd = H * d;
    GemmEpi e1{0, hd, static_cast<__nv_bfloat16*>(gate), static_cast<__nv_bfloat16*>(z), nullptr, nullptr, d};
    cudaError_t e = gemm<CfgX>(x, w_gate_a, (int)T, hd + rank, hidden, e1, err, stream);
    if (e != cudaSuccess) return e;
    GemmEpi e2{1, hd, nullptr, nullptr, g, a_head, d};
    return gemm<CfgR>(z, w_b, (int)T, hd, rank, e2, err, stream);
}

}  // namespace kda
