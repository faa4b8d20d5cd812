// The C ABI of libkda.so (declared in include/kda.h): argument checks, error
// reporting and dispatch to the kernel launchers.  Nothing here allocates.
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

thread_local char t_last_error[512] = "";

}  // namespace

kda_status set_error(kda_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return s;
}

}  // namespace kda

__device__ unsigned int g_kda_device_error = 0;

namespace kda {

unsigned int* device_error_word() {
    static std::mutex mu;
    static unsigned int* cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int*>(p);
    }
    return cache[dev];
}

}  // namespace kda

using kda::set_error;

namespace {

// Scratch of kda_chunk_fwd_noalloc: part of the library's device image, so that entry point needs
// no allocation by anyone.  Calls that use it must not overlap (one stream, or ordered streams).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_chunk_scratch[kStaticScratchBytes];

// Device address of g_chunk_scratch on the current device.  In host code the array's name stands for a
// host-side shadow, not device memory, so the address is looked up once per device (the first call
// on that device, with it current) and kept.
cudaError_t static_scratch(void** out) {
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_chunk_scratch);
        if (e != cudaSuccess) return e;
        cache[dev] = p;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace

namespace {

// One thread waits on a barrier no one arrives at; the bounded wait gives up and reports.
__global__ void selftest_wait_kernel(unsigned int limit, unsigned int* err) {
    __shared__ uint64_t bar;
    kda::tc::mbar_init(&bar, 1);
    kda::tc::fence_mbar_init();
    if (!kda::tc::mbar_wait(&bar, 0, limit)) kda::raise_device_error(err, kda::kErrMbarTimeout);
}

}  // namespace

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte ranges [a, a + na) and [b, b + nb) share an address (NULL never does).
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

kda_status ok() {
    kda::t_last_error[0] = '\0';
    return KDA_OK;
}

kda_status from_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return set_error(KDA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define REQUIRE(cond, ...)                                        \
    do {                                                          \
        if (!(cond)) return set_error(KDA_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

#define REQUIRE_PTR(p)                                                          \
    do {                                                                        \
        REQUIRE((p) != nullptr, "%s must not be NULL", #p);                     \
        REQUIRE(aligned16(p), "%s must be 16-byte aligned", #p);                \
    } while (0)

#define OPTIONAL_PTR(p)                                                         \
    do {                                                                        \
        REQUIRE((p) == nullptr || aligned16(p), "%s must be 16-byte aligned", #p); \
    } while (0)

kda_status check_batch(const int32_t* cu, int N, int64_t T_total, int H) {
    REQUIRE(N >= 1, "N must be >= 1 (got %d)", N);
    REQUIRE(H >= 1 && H <= 65535, "H must be in [1, 65535] (got %d)", H);
    REQUIRE(T_total >= 0, "T_total must be >= 0");
    REQUIRE(cu != nullptr || N == 1, "cu_seqlens may be NULL only for N == 1 (got N = %d)", N);
    REQUIRE((int64_t)N * H <= 0x7FFFFFFF, "N * H too large");
    REQUIRE(T_total <= ((int64_t)1 << 40), "T_total too large");
    return KDA_OK;
}

}  // namespace

namespace {

// kda_chunk_fwd after its pointer checks; `overlap` as launch_chunk_tc.
kda_status chunk_fwd_checked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                             int dk, int dv, float scale, int chunk_size, kda_dtype dtype, const void* out_gate,
                             void* o, float* final_state, void* workspace, size_t workspace_bytes, void* stream,
                             bool overlap) {
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(dtype == KDA_DTYPE_F32 || dtype == KDA_DTYPE_BF16, "bad dtype");
    REQUIRE(std::isfinite(scale), "scale must be finite");
    if (dtype == KDA_DTYPE_F32)
        return from_cuda(kda::launch_chunk_simt(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype,
                                                out_gate, o, final_state, static_cast<cudaStream_t>(stream)),
                         "kda_chunk_fwd launch");
    REQUIRE(T_total < ((int64_t)1 << 31), "T_total must be below 2^31 for the bf16 path (tensor-map coordinates)");
    REQUIRE(T_total / 64 + N <= 0x7FFFFFFF, "too many chunks");
    size_t need = 0;
    kda::chunk_tc_workspace(N, T_total, H, cu_seqlens != nullptr, nullptr, &need);
    REQUIRE(workspace != nullptr && workspace_bytes >= need,
            "workspace must hold at least %zu bytes for these sizes (got %zu)", need, workspace_bytes);
    OPTIONAL_PTR(workspace);
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    return from_cuda(kda::launch_chunk_tc(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, out_gate, o,
                                          final_state, workspace, workspace_bytes, nullptr, err,
                                          static_cast<cudaStream_t>(stream), 0, nullptr, 0, overlap),
                     "kda_chunk_fwd launch");
}

}  // namespace

extern "C" {

const char* kda_status_string(kda_status s) {
    switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape or option";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
    case KDA_ERR_DEVICE: return "KDA_ERR_DEVICE: a kernel reported a fault";
    }
    return "unknown kda_status";
}

const char* kda_last_error(void) { return kda::t_last_error; }

const char* kda_version(void) { return "0.1.0"; }

kda_status kda_device_error(unsigned int* code) {
    REQUIRE(code != nullptr, "code must not be NULL");
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_kda_device_error, sizeof(v));
    if (e != cudaSuccess) return from_cuda(e, "reading the device error word");
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return from_cuda(e, "clearing the device error word");
    *code = v;
    return ok();
}

kda_status kda_selftest_bounded_wait(unsigned int poll_limit, void* stream) {
    REQUIRE(poll_limit >= 1 && poll_limit <= (1u << 24), "poll_limit must be in [1, 2^24]");
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(poll_limit, err);
    return from_cuda(cudaGetLastError(), "kda_selftest_bounded_wait launch");
}

kda_status kda_shortconv_l2norm(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                                const void* conv_w, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                                int d, const void* conv_state_in, void* conv_state_out, float eps,
                                kda_dtype out_dtype, void* q_out, void* k_out, void* v_out, void* stream) {
    REQUIRE_PTR(xq); REQUIRE_PTR(xk); REQUIRE_PTR(xv); REQUIRE_PTR(conv_w);
    REQUIRE_PTR(q_out); REQUIRE_PTR(k_out); REQUIRE_PTR(v_out);
    OPTIONAL_PTR(conv_state_in); OPTIONAL_PTR(conv_state_out);
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    if (d != kda::kHeadDim) return set_error(KDA_ERR_UNSUPPORTED, "only d = 128 is supported (got %d)", d);
    REQUIRE(x_row_stride >= (int64_t)H * d && x_row_stride % 8 == 0,
            "x_row_stride must be >= H*d and a multiple of 8 (got %lld)", (long long)x_row_stride);
    REQUIRE(out_dtype == KDA_DTYPE_F32 || out_dtype == KDA_DTYPE_BF16, "bad out_dtype");
    REQUIRE(std::isfinite(eps) && eps >= 0.f, "eps must be finite and >= 0");
    REQUIRE((T_total + 63) / 64 <= 0x7FFFFFFF, "T_total too large");
    return from_cuda(kda::launch_shortconv_l2norm(xq, xk, xv, x_row_stride, conv_w, cu_seqlens, N, T_total, H,
                                                  conv_state_in, conv_state_out, eps, out_dtype, q_out, k_out,
                                                  v_out, static_cast<cudaStream_t>(stream)),
                     "kda_shortconv_l2norm launch");
}

kda_status kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                         int dk, int dv, float scale, int chunk_size, kda_dtype dtype, const void* out_gate,
                         void* o, float* final_state, void* workspace, size_t workspace_bytes, void* stream) {
    REQUIRE_PTR(q); REQUIRE_PTR(k); REQUIRE_PTR(v); REQUIRE_PTR(g); REQUIRE_PTR(beta); REQUIRE_PTR(o);
    OPTIONAL_PTR(init_state); OPTIONAL_PTR(final_state); OPTIONAL_PTR(out_gate);
    return chunk_fwd_checked(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, chunk_size,
                             dtype, out_gate, o, final_state, workspace, workspace_bytes, stream, true);
}

kda_status kda_chunk_bwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv, int chunk_size,
                                        size_t* bytes) {
    REQUIRE_PTR(bytes);
    REQUIRE(N >= 1 && H >= 1 && T_total >= 0 && (int64_t)N * H <= 0x7FFFFFFF, "bad N, H or T_total");
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(T_total / 64 + N < 0x7FFFFFFF, "T_total too large");
    *bytes = kda::chunk_bwd_workspace_bytes(N, T_total, H);
    return ok();
}

kda_status kda_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H, int dk,
                         int dv, float scale, int chunk_size, kda_dtype dtype, const void* d_o,
                         const float* d_final_state, float* dq, float* dk_out, float* dv_out, float* dg, float* dbeta,
                         float* d_init_state, void* workspace, size_t workspace_bytes, void* stream) {
    REQUIRE_PTR(q); REQUIRE_PTR(k); REQUIRE_PTR(v); REQUIRE_PTR(g); REQUIRE_PTR(beta); REQUIRE_PTR(d_o);
    REQUIRE_PTR(dq); REQUIRE_PTR(dk_out); REQUIRE_PTR(dv_out); REQUIRE_PTR(dg); REQUIRE_PTR(dbeta);
    OPTIONAL_PTR(init_state); OPTIONAL_PTR(d_final_state); OPTIONAL_PTR(d_init_state);
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(dtype == KDA_DTYPE_F32 || dtype == KDA_DTYPE_BF16, "bad dtype");
    REQUIRE(std::isfinite(scale), "scale must be finite");
    REQUIRE(T_total / 64 + N < 0x7FFFFFFF, "T_total too large");
    const size_t need = kda::chunk_bwd_workspace_bytes(N, T_total, H);
    REQUIRE(workspace != nullptr && workspace_bytes >= need,
            "workspace must hold at least %zu bytes for these sizes (got %zu)", need, workspace_bytes);
    OPTIONAL_PTR(workspace);
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    return from_cuda(kda::launch_chunk_bwd(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, scale, dtype,
                                           d_o, d_final_state, dq, dk_out, dv_out, dg, dbeta, d_init_state,
                                           workspace, err, static_cast<cudaStream_t>(stream)),
                     "kda_chunk_bwd launch");
}

kda_status kda_chunk_segment_summary(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                     const int32_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv,
                                     int chunk_size, float* end_state, float* transition, void* workspace,
                                     size_t workspace_bytes, void* stream) {
    REQUIRE_PTR(k); REQUIRE_PTR(g); REQUIRE_PTR(beta);
    OPTIONAL_PTR(q); OPTIONAL_PTR(v); OPTIONAL_PTR(end_state); OPTIONAL_PTR(transition);
    REQUIRE(end_state != nullptr || transition != nullptr, "end_state and transition must not both be NULL");
    if (end_state) REQUIRE_PTR(v);
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(T_total < ((int64_t)1 << 31), "T_total must be below 2^31 (tensor-map coordinates)");
    REQUIRE(T_total / 64 + N <= 0x7FFFFFFF, "too many chunks");
    size_t full = 0, need = 0;
    kda::chunk_tc_workspace(N, T_total, H, cu_seqlens != nullptr, &full, &need);
    REQUIRE(workspace != nullptr && workspace_bytes >= need,
            "workspace must hold at least %zu bytes for these sizes (got %zu)", need, workspace_bytes);
    OPTIONAL_PTR(workspace);
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void* qq = q ? q : k;   // the outputs asked for do not depend on q
    const void* vv = v ? v : k;   // nor, for the transition alone, on v
    const int tr_mode = kda::kStateZeroU | kda::kStateIdentity;
    cudaError_t e;
    if (end_state && transition && workspace_bytes >= full) {  // one pass of chunk operands, two state passes
        e = kda::launch_chunk_tc(qq, k, vv, g, beta, nullptr, cu_seqlens, N, T_total, H, 1.0f, nullptr, nullptr,
                                 end_state, workspace, workspace_bytes, nullptr, err, st, 0, transition, tr_mode);
    } else {
        e = cudaSuccess;
        if (end_state)
            e = kda::launch_chunk_tc(qq, k, vv, g, beta, nullptr, cu_seqlens, N, T_total, H, 1.0f, nullptr, nullptr,
                                     end_state, workspace, workspace_bytes, nullptr, err, st, 0);
        if (e == cudaSuccess && transition)
            e = kda::launch_chunk_tc(qq, k, vv, g, beta, nullptr, cu_seqlens, N, T_total, H, 1.0f, nullptr, nullptr,
                                     transition, workspace, workspace_bytes, nullptr, err, st, tr_mode);
    }
    return from_cuda(e, "kda_chunk_segment_summary launch");
}

kda_status kda_gate_generator(const void* x, int64_t T, int hidden, const void* w_gate_a, const void* w_b,
                              const float* a_head, int H, int d, int rank, void* gate, float* g, void* z_workspace,
                              void* stream) {
    REQUIRE(T >= 0 && T < ((int64_t)1 << 31), "T must be in [0, 2^31) (got %lld)", (long long)T);
    REQUIRE(hidden >= 8 && hidden % 8 == 0, "hidden must be a positive multiple of 8 (got %d)", hidden);
    if (d != kda::kHeadDim) return set_error(KDA_ERR_UNSUPPORTED, "only d = 128 is supported (got %d)", d);
    REQUIRE(H >= 1 && H <= 65535, "H must be in [1, 65535] (got %d)", H);
    REQUIRE(rank >= 32 && rank <= 4096 && rank % 32 == 0, "rank must be a multiple of 32 in [32, 4096] (got %d)",
            rank);
    REQUIRE_PTR(w_gate_a); REQUIRE_PTR(w_b); REQUIRE_PTR(a_head);
    if (T == 0) return ok();  // nothing to compute; the per-token buffers may be empty
    REQUIRE_PTR(x); REQUIRE_PTR(gate); REQUIRE_PTR(g); REQUIRE_PTR(z_workspace);
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    return from_cuda(kda::launch_gate_generator(x, T, hidden, w_gate_a, w_b, a_head, H, d, rank, gate, g, z_workspace,
                                                err, static_cast<cudaStream_t>(stream)),
                     "kda_gate_generator launch");
}

kda_status kda_state_combine(const float* S_in, const float* M, const float* E, float* S_out, int64_t count,
                             void* stream) {
    OPTIONAL_PTR(S_in);
    REQUIRE_PTR(M); REQUIRE_PTR(E); REQUIRE_PTR(S_out);
    REQUIRE(count >= 0 && count <= 0x7FFFFFFF, "count must be in [0, 2^31) (got %lld)", (long long)count);
    return from_cuda(kda::launch_state_combine(S_in, M, E, S_out, count, static_cast<cudaStream_t>(stream)),
                     "kda_state_combine launch");
}

kda_status kda_chunk_fwd_frontend(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                                  const void* conv_w, const void* conv_state_in, void* conv_state_out, float eps,
                                  const float* g, const float* beta, const float* init_state,
                                  const int32_t* cu_seqlens, int N, int64_t T_total, int H, int d, float scale,
                                  int chunk_size, const void* out_gate, void* o, float* final_state,
                                  void* workspace, size_t workspace_bytes, void* stream) {
    REQUIRE_PTR(xq); REQUIRE_PTR(xk); REQUIRE_PTR(xv); REQUIRE_PTR(conv_w); REQUIRE_PTR(g); REQUIRE_PTR(beta);
    REQUIRE_PTR(o);
    OPTIONAL_PTR(conv_state_in); OPTIONAL_PTR(conv_state_out); OPTIONAL_PTR(init_state); OPTIONAL_PTR(final_state);
    OPTIONAL_PTR(out_gate);
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    if (d != kda::kHeadDim) return set_error(KDA_ERR_UNSUPPORTED, "only d = 128 is supported (got %d)", d);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(x_row_stride >= (int64_t)H * d && x_row_stride % 8 == 0,
            "x_row_stride must be >= H*d and a multiple of 8 (got %lld)", (long long)x_row_stride);
    REQUIRE(std::isfinite(eps) && eps >= 0.f, "eps must be finite and >= 0");
    REQUIRE(std::isfinite(scale), "scale must be finite");
    REQUIRE(T_total < ((int64_t)1 << 31), "T_total must be below 2^31 (tensor-map coordinates)");
    REQUIRE(T_total / 64 + N <= 0x7FFFFFFF, "too many chunks");
    {  // o holds v during the call: it must not share memory with an input
        const size_t ob = (size_t)T_total * H * d * 2, tb = (size_t)T_total * H;
        const size_t xb = T_total > 0 ? ((size_t)(T_total - 1) * x_row_stride + (size_t)H * d) * 2 : 0;
        REQUIRE(!overlaps(o, ob, xq, xb) && !overlaps(o, ob, xk, xb) && !overlaps(o, ob, xv, xb) &&
                    !overlaps(o, ob, out_gate, ob) && !overlaps(o, ob, g, tb * d * 4) &&
                    !overlaps(o, ob, beta, tb * 4),
                "o must not overlap an input (it holds v during the call)");
    }
    size_t need = 0;
    kda::chunk_tc_workspace(N, T_total, H, cu_seqlens != nullptr, nullptr, &need);
    REQUIRE(workspace != nullptr && workspace_bytes >= need,
            "workspace must hold at least %zu bytes for these sizes (got %zu)", need, workspace_bytes);
    OPTIONAL_PTR(workspace);
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    const kda::ChunkFrontend front{xq, xk, xv, x_row_stride, conv_w, conv_state_in, eps};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = kda::launch_chunk_tc(nullptr, nullptr, nullptr, g, beta, init_state, cu_seqlens, N, T_total, H,
                                         scale, out_gate, o, final_state, workspace, workspace_bytes, &front, err, st);
    if (e == cudaSuccess && conv_state_out)  // after the chunk pass has read conv_state_in: the two may alias
        e = kda::launch_conv_state_out(xq, xk, xv, x_row_stride, cu_seqlens, N, T_total, H, conv_state_in,
                                       conv_state_out, st);
    return from_cuda(e, "kda_chunk_fwd_frontend launch");
}

kda_status kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                 const float* init_state, const int32_t* cu_seqlens, int N, int64_t T_total, int H,
                                 int dk, int dv, float scale, int chunk_size, kda_dtype dtype, const void* out_gate,
                                 void* o, float* final_state, void* stream) {
    REQUIRE_PTR(q); REQUIRE_PTR(k); REQUIRE_PTR(v); REQUIRE_PTR(g); REQUIRE_PTR(beta); REQUIRE_PTR(o);
    OPTIONAL_PTR(init_state); OPTIONAL_PTR(final_state); OPTIONAL_PTR(out_gate);
    if (dtype == KDA_DTYPE_F32)  // the fp32 path needs no workspace
        return chunk_fwd_checked(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, chunk_size,
                                 dtype, out_gate, o, final_state, nullptr, 0, stream, false);
    kda_status s = check_batch(cu_seqlens, N, T_total, H);
    if (s != KDA_OK) return s;
    REQUIRE(dtype == KDA_DTYPE_BF16, "bad dtype");
    REQUIRE(T_total / 64 + N <= 0x7FFFFFFF, "too many chunks");
    size_t need = 0;
    kda::chunk_tc_workspace(N, T_total, H, cu_seqlens != nullptr, nullptr, &need);
    if (need > kStaticScratchBytes)
        return set_error(KDA_ERR_UNSUPPORTED, "the static scratch holds %zu bytes; these sizes need at least %zu",
                         kStaticScratchBytes, need);
    void* scratch = nullptr;
    cudaError_t e = static_scratch(&scratch);
    if (e != cudaSuccess) return from_cuda(e, "kda_chunk_fwd_noalloc: device address of the static scratch");
    // every range one after the other on `stream`: no internal streams or events
    return chunk_fwd_checked(q, k, v, g, beta, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, chunk_size,
                             dtype, out_gate, o, final_state, scratch, kStaticScratchBytes, stream, false);
}

kda_status kda_chunk_fwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv, int chunk_size,
                                        kda_dtype dtype, int have_cu_seqlens, size_t* full_bytes,
                                        size_t* min_bytes) {
    REQUIRE(N >= 1 && H >= 1 && T_total >= 0 && (int64_t)N * H <= 0x7FFFFFFF, "bad N, H or T_total");
    REQUIRE(have_cu_seqlens || N == 1, "several sequences need cu_seqlens");
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    if (chunk_size != kda::kChunk)
        return set_error(KDA_ERR_UNSUPPORTED, "only chunk_size = 64 is supported (got %d)", chunk_size);
    REQUIRE(dtype == KDA_DTYPE_F32 || dtype == KDA_DTYPE_BF16, "bad dtype");
    REQUIRE(T_total / 64 + N <= 0x7FFFFFFF, "T_total too large");
    size_t full = 0, least = 0;
    if (dtype == KDA_DTYPE_BF16) kda::chunk_tc_workspace(N, T_total, H, have_cu_seqlens != 0, &full, &least);
    if (full_bytes) *full_bytes = full;
    if (min_bytes) *min_bytes = least;
    return ok();
}

kda_status kda_recurrent_step(const void* xq, const void* xk, const void* xv, int64_t x_row_stride,
                              const void* conv_w, const float* g, const float* beta, float* state,
                              void* conv_state, int N, int H, int dk, int dv, float scale, float eps, void* o,
                              void* stream) {
    REQUIRE_PTR(xq); REQUIRE_PTR(xk); REQUIRE_PTR(xv); REQUIRE_PTR(conv_w); REQUIRE_PTR(g);
    REQUIRE_PTR(beta); REQUIRE_PTR(state); REQUIRE_PTR(conv_state); REQUIRE_PTR(o);
    REQUIRE(N >= 1, "N must be >= 1 (got %d)", N);
    REQUIRE(H >= 1 && (int64_t)N * H <= 0x7FFFFFFF, "bad H");
    if (dk != kda::kHeadDim || dv != kda::kHeadDim)
        return set_error(KDA_ERR_UNSUPPORTED, "only dk = dv = 128 is supported (got %d, %d)", dk, dv);
    REQUIRE(x_row_stride >= (int64_t)H * dk && x_row_stride % 8 == 0,
            "x_row_stride must be >= H*d and a multiple of 8 (got %lld)", (long long)x_row_stride);
    REQUIRE(std::isfinite(scale) && std::isfinite(eps) && eps >= 0.f, "scale and eps must be finite, eps >= 0");
    unsigned int* err = kda::device_error_word();
    if (!err) return set_error(KDA_ERR_CUDA, "device error word unavailable");
    return from_cuda(kda::launch_recurrent_step(xq, xk, xv, x_row_stride, conv_w, g, beta, state, conv_state, N,
                                                H, scale, eps, o, err, static_cast<cudaStream_t>(stream)),
                     "kda_recurrent_step launch");
}

}  // extern "C"
