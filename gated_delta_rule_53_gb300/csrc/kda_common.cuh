// Shared device helpers of libkda.so (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kHeadDim = 128;  // d = dk = dv supported by every kernel
constexpr int kChunk = 64;     // chunk length of the prefill

// Kernels get a pointer to the library's device error word (kda_api.cu) and OR a
// bit into it: a wait that runs out (instead of spinning forever), an input outside
// the range the arithmetic relies on.  The host reads and clears it through
// kda_device_error().  The bits are the KDA_DEVICE_ERR_* values of kda.h.
enum DeviceError : unsigned int {
    kErrNone = 0,
    kErrMbarTimeout = KDA_DEVICE_ERR_WAIT_TIMEOUT,
    kErrGateRange = KDA_DEVICE_ERR_GATE_RANGE,
    kErrBetaRange = KDA_DEVICE_ERR_BETA_RANGE,
};

__device__ __forceinline__ void raise_device_error(unsigned int* err, unsigned int code) {
    if (err) atomicOr(err, code);
}

__device__ __forceinline__ float bf16_lo(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t packed) { return __uint_as_float(packed & 0xFFFF0000u); }

// Round-to-nearest-even fp32 -> bf16 of two values, packed low | high << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void store_from_float(T* p, float x);
template <>
__device__ __forceinline__ void store_from_float<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void store_from_float<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }

// Sequence bounds of chain n (cu_seqlens may be null: one sequence).
__device__ __forceinline__ void seq_bounds(const int32_t* cu, int n, int64_t T_total, int64_t& bos, int64_t& eos) {
    if (cu) {
        bos = cu[n];
        eos = cu[n + 1];
    } else {
        bos = 0;
        eos = T_total;
    }
}

}  // namespace kda

// Kernel launchers (one per kernel file), called by the entry points in kda_api.cu
// after the arguments have been checked.  They return the launch's error.
namespace kda {

cudaError_t launch_recurrent_step(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                  const void* conv_w, const float* g, const float* beta, float* state,
                                  void* conv_state, int N, int H, float scale, float eps, void* o,
                                  unsigned int* err, cudaStream_t stream);

cudaError_t launch_shortconv_l2norm(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                    const void* conv_w, const int32_t* cu_seqlens, int N, int64_t T_total,
                                    int H, const void* conv_state_in, void* conv_state_out, float eps,
                                    kda_dtype out_dtype, void* q, void* k, void* v, cudaStream_t stream);
cudaError_t launch_frontend_v(const void* xv, int64_t x_stride, const void* conv_w, const int32_t* cu_seqlens, int N,
                              int64_t T_total, int H, const void* conv_state_in, void* v, cudaStream_t stream);

cudaError_t launch_chunk_simt(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total,
                              int H, float scale, kda_dtype dtype, const void* out_gate, void* o,
                              float* final_state, cudaStream_t stream);

// Backward of the chunk prefill (fp32 on the CUDA cores): gradients of q, k, v, g, beta and the initial
// state from those of o and of the final state.  Workspace: chunk_bwd_workspace_bytes().
size_t chunk_bwd_workspace_bytes(int N, int64_t T_total, int H);
cudaError_t launch_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                             float scale, kda_dtype dtype, const void* d_o, const float* d_final, float* dq,
                             float* dk, float* dv, float* dg, float* dbeta, float* d_init, void* workspace,
                             unsigned int* err, cudaStream_t stream);

// Raw inputs of the fused prefill: q and k are computed from them by the front end of
// kda_shortconv_l2norm (bf16) inside the chunk pass instead of being read, v by that front end
// into the output buffer, from which the state pass reads it.
struct ChunkFrontend {
    const void* xq;
    const void* xk;
    const void* xv;
    int64_t x_stride;
    const void* conv_w;
    const void* conv_state_in;
    float eps;
};

// Modes of a state pass: U taken as zero (the effect of v = 0), and chains that start without an
// initial state start from the identity (dv = dk).  Both together give a segment's transition
// operator  prod_t Diag(alpha_t) (I - beta_t k_t k_t^T)  as the final state.
constexpr int kStateZeroU = 1, kStateIdentity = 2;

// o may be null (no outputs).  final_state2 (with state_mode2): a second state pass over the same
// operands, from a zero / identity start, without outputs; it needs every chunk in one range of the
// workspace (cudaErrorInvalidValue otherwise).  overlap = false keeps every range on `stream`, one
// after the other (no internal streams or events).
cudaError_t launch_chunk_tc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                            const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                            float scale, const void* out_gate, void* o, float* final_state, void* workspace,
                            size_t workspace_bytes, const ChunkFrontend* front, unsigned int* err,
                            cudaStream_t stream, int state_mode = 0, float* final_state2 = nullptr,
                            int state_mode2 = 0, bool overlap = true);

// gate = x W_gate^T (bf16), z = x W_a^T (bf16 scratch [T, rank]), g = max(-5, -softplus(z W_b^T + a_h))
// (fp32); w_gate_a = [W_gate ; W_a] stacked, [H*d + rank, hidden].
cudaError_t launch_gate_generator(const void* x, int64_t T, int hidden, const void* w_gate_a, const void* w_b,
                                  const float* a_head, int H, int d, int rank, void* gate, float* g, void* z,
                                  unsigned int* err, cudaStream_t stream);

// S_out[i] = S_in[i] M[i] + E[i] for `count` 128 x 128 fp32 matrices (S_in null: S_out = E).
cudaError_t launch_state_combine(const float* S_in, const float* M, const float* E, float* S_out, int64_t count,
                                 cudaStream_t stream);

// conv_state_out of the front end (the last three raw inputs of each sequence), as a pass of its own.
cudaError_t launch_conv_state_out(const void* xq, const void* xk, const void* xv, int64_t x_stride,
                                  const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                                  const void* conv_state_in, void* conv_state_out, cudaStream_t stream);

// Workspace of launch_chunk_tc: all chunks in one range / the least accepted.
void chunk_tc_workspace(int N, int64_t T_total, int H, bool have_cu, size_t* full_bytes, size_t* min_bytes);

// Device address of the library's error word on the current device (nullptr if unavailable).
unsigned int* device_error_word();

}  // namespace kda
