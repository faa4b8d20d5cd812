/*
 * Counter-based synthetic input generator for the KDA hot path.
 *
 * Test and benchmark infrastructure.  Both the fp64 oracle and the CUDA
 * library are fed from the arrays this file fills; it holds none of the
 * attention arithmetic (no decay, no delta rule, no convolution): it draws
 * numbers, applies the input distribution of a workload, and rounds them to a
 * storage type.
 *
 * Every element is a pure function of (seed, tensor_id, flat element index),
 * so any slice of a tensor can be regenerated on its own (the oracle uses this
 * to rebuild one head of a 40 GB workload without holding the rest).
 *
 * Definition (stated here so that any other implementation can be checked):
 *   mix(z)        SplitMix64 finaliser:
 *                   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                   z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                   z =  z ^ (z >> 31)
 *   key(s, id)    mix(s * G ^ mix(id + G)),  G = 0x9E3779B97F4A7C15
 *   bits(s,id,i)  mix(key(s,id) + (i + 1) * G)                 (mod 2^64)
 *   unif(s,id,i)  ((bits(s,id,i) >> 11) + 0.5) * 2^-53           in (0, 1)
 *   z(s,id,i)     sqrt(-2 ln unif(s,id,2i)) * cos(2 pi unif(s,id,2i+1))
 *                 (Box-Muller, cosine branch; fp64)
 *
 * Portable C99: no intrinsics, no assumption on the signedness of char.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_G 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
    return mix64(seed * SYNTH_G ^ mix64(tid + SYNTH_G));
}

static inline uint64_t stream_bits(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1ULL) * SYNTH_G);
}

static inline double to_unif(uint64_t b) {
    return ((double)(b >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static inline double std_normal(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = to_unif(stream_bits(key, 2ULL * i));
    double u2 = to_unif(stream_bits(key, 2ULL * i + 1ULL));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* Distribution of one element, applied to a standard normal z. */
enum {
    SYNTH_NORMAL = 0,        /* p0 + p1 * z                                   */
    SYNTH_NEG5_SIGMOID = 1,  /* -5 / (1 + e^-z)             (log-decay g)      */
    SYNTH_SIGMOID = 2,       /* 1 / (1 + e^-z)              (beta)             */
    SYNTH_NEG_SOFTPLUS5 = 3, /* max(-5, -ln(1 + e^z))       (log-decay g)      */
    SYNTH_UNIT_GROUPS = 4    /* z / ||z|| over aligned groups of p1 elements   */
};

/* Storage type of the output array. */
enum { SYNTH_F64 = 0, SYNTH_F32 = 1, SYNTH_BF16 = 2 };

static inline double apply_kind(int kind, double z, double p0, double p1) {
    switch (kind) {
    case SYNTH_NORMAL: return p0 + p1 * z;
    case SYNTH_NEG5_SIGMOID: return -5.0 / (1.0 + exp(-z));
    case SYNTH_SIGMOID: return 1.0 / (1.0 + exp(-z));
    case SYNTH_NEG_SOFTPLUS5: {
        double sp = z > 0.0 ? z + log1p(exp(-z)) : log1p(exp(z));
        double gv = -sp;
        return gv < -5.0 ? -5.0 : gv;
    }
    default: return z;
    }
}

/* fp64 -> fp32 (round to nearest even by the C conversion) -> bf16 bits
 * (round to nearest even on the dropped 16 bits). */
static inline uint16_t f64_to_bf16_bits(double x) {
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline void store(void* out, int dtype, int64_t at, double x) {
    if (dtype == SYNTH_F64) ((double*)out)[at] = x;
    else if (dtype == SYNTH_F32) ((float*)out)[at] = (float)x;
    else ((uint16_t*)out)[at] = f64_to_bf16_bits(x);
}

typedef struct {
    uint64_t key;
    int kind;
    double p0, p1;
    int64_t row0, nrows, ld, col0, ncols;
    void* out;
    int dtype;
} fill_job;

static void fill_rows(const fill_job* j, int64_t r_begin, int64_t r_end) {
    for (int64_t r = r_begin; r < r_end; ++r) {
        uint64_t base = (uint64_t)((j->row0 + r) * j->ld + j->col0);
        int64_t at = r * j->ncols;
        if (j->kind == SYNTH_UNIT_GROUPS) {
            int64_t gsz = (int64_t)j->p1;
            double buf[1024];
            for (int64_t c0 = 0; c0 < j->ncols; c0 += gsz) {
                double ss = 0.0;
                for (int64_t c = 0; c < gsz; ++c) {
                    buf[c] = std_normal(j->key, base + (uint64_t)(c0 + c));
                    ss += buf[c] * buf[c];
                }
                double inv = 1.0 / sqrt(ss);
                for (int64_t c = 0; c < gsz; ++c) store(j->out, j->dtype, at + c0 + c, buf[c] * inv);
            }
        } else {
            for (int64_t c = 0; c < j->ncols; ++c) {
                double z = std_normal(j->key, base + (uint64_t)c);
                store(j->out, j->dtype, at + c, apply_kind(j->kind, z, j->p0, j->p1));
            }
        }
    }
}

typedef struct {
    const fill_job* job;
    int64_t r_begin, r_end;
} fill_slice;

static void* fill_thread(void* arg) {
    fill_slice* s = (fill_slice*)arg;
    fill_rows(s->job, s->r_begin, s->r_end);
    return NULL;
}

/*
 * Fill out[r, c] (row-major, nrows x ncols) with element
 *   flat index (row0 + r) * ld + col0 + c
 * of tensor (seed, tid) under distribution `kind`.  For SYNTH_UNIT_GROUPS,
 * p1 is the group length (<= 1024) and col0, ncols, ld must be multiples of it.
 * Returns 0 on success, -1 on a bad argument.
 */
int synth_fill(uint64_t seed, uint64_t tid, int kind, double p0, double p1,
               int64_t row0, int64_t nrows, int64_t ld, int64_t col0, int64_t ncols,
               void* out, int dtype, int nthreads) {
    if (!out || nrows < 0 || ncols < 0 || ld < ncols || row0 < 0 || col0 < 0 || col0 + ncols > ld) return -1;
    if (dtype < SYNTH_F64 || dtype > SYNTH_BF16 || kind < SYNTH_NORMAL || kind > SYNTH_UNIT_GROUPS) return -1;
    if (kind == SYNTH_UNIT_GROUPS) {
        int64_t gsz = (int64_t)p1;
        if (gsz < 1 || gsz > 1024 || (double)gsz != p1 || col0 % gsz || ncols % gsz || ld % gsz) return -1;
    }
    fill_job job = {stream_key(seed, tid), kind, p0, p1, row0, nrows, ld, col0, ncols, out, dtype};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
    if (nthreads == 1 || nrows * ncols < (1 << 16)) {
        fill_rows(&job, 0, nrows);
        return 0;
    }
    pthread_t th[256];
    fill_slice sl[256];
    int ok[256];
    for (int t = 0; t < nthreads; ++t) {
        sl[t].job = &job;
        sl[t].r_begin = nrows * t / nthreads;
        sl[t].r_end = nrows * (t + 1) / nthreads;
        ok[t] = pthread_create(&th[t], NULL, fill_thread, &sl[t]) == 0;
        if (!ok[t]) fill_rows(&job, sl[t].r_begin, sl[t].r_end);
    }
    for (int t = 0; t < nthreads; ++t)
        if (ok[t]) pthread_join(th[t], NULL);
    return 0;
}

/* Raw 64-bit draws bits(seed, tid, start + i), i < count (used for lengths). */
int synth_u64(uint64_t seed, uint64_t tid, int64_t start, int64_t count, uint64_t* out) {
    if (!out || start < 0 || count < 0) return -1;
    uint64_t key = stream_key(seed, tid);
    for (int64_t i = 0; i < count; ++i) out[i] = stream_bits(key, (uint64_t)(start + i));
    return 0;
}
