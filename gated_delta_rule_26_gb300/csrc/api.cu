// api.cu -- the extern "C" entry points of libkda: argument validation on the
// host, path selection, launch.  No exception crosses this boundary and
// nothing is launched when an argument is rejected.
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace kda {
cudaError_t launch_chunk_tc(const ChunkArgs& a, cudaStream_t s, int mode, bool* taken);
cudaError_t read_and_clear_carry_timeout(int* timed_out);
cudaError_t read_and_clear_decode_timeout(int* timed_out);
cudaError_t read_and_clear_bwd_timeout(int* timed_out);
cudaError_t launch_chunk_split_noalloc(const ChunkArgs& a, cudaStream_t s, bool* fits);
cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, cudaStream_t s);
cudaError_t read_and_clear_timeout(cudaStream_t s, int* timed_out);
}

namespace kda {
static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace kda

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int x) { return x >= 8 && x <= 128 && (x % 8) == 0; }

int check_dims(const kda_dims* d, bool need_v) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->B < 1 || d->H < 1 || d->T < 0 || d->K < 1 || (need_v && d->V < 1))
        return KDA_ERR_INVALID_ARG;
    if (!dim_ok(d->K) || (need_v && !dim_ok(d->V))) return KDA_ERR_UNSUPPORTED;
    if ((long long)d->B * d->H > 0x7fffffffLL) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

bool dtype_ok(int dt) { return dt == KDA_F32 || dt == KDA_BF16; }

bool aligned_to(const void* p, unsigned bytes) {
    return (reinterpret_cast<uintptr_t>(p) & (uintptr_t)(bytes - 1)) == 0;
}

// `required` must be non-null and 16-byte aligned; `optional` may be null, else 16-byte
// aligned; `elementwise` must be non-null and aligned to `elem_bytes` (read per element).
int check_ptrs(std::initializer_list<const void*> required,
               std::initializer_list<const void*> optional,
               std::initializer_list<const void*> elementwise = {}, unsigned elem_bytes = 4) {
    for (const void* p : required)
        if (!p) return KDA_ERR_INVALID_ARG;
    for (const void* p : elementwise)
        if (!p) return KDA_ERR_INVALID_ARG;
    for (const void* p : required)
        if (!aligned16(p)) return KDA_ERR_MISALIGNED;
    for (const void* p : optional)
        if (p && !aligned16(p)) return KDA_ERR_MISALIGNED;
    for (const void* p : elementwise)
        if (!aligned_to(p, elem_bytes)) return KDA_ERR_MISALIGNED;
    return KDA_OK;
}

unsigned io_bytes(kda_dtype dt) { return dt == KDA_BF16 ? 2u : 4u; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // namespace

extern "C" {

unsigned long long kda_launch_count(void) { return kda::g_launches.load(std::memory_order_relaxed); }

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported size or chunk";
        case KDA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_NO_MEMORY: return "out of device memory";
        case KDA_ERR_TIMEOUT: return "a kernel gave up on a bounded wait";
        default: return "unknown status";
    }
}

int kda_gate(const kda_dims* dims, kda_dtype z_dtype, const void* z, const float* A_log,
             const float* dt_bias, int chunk, float* g_out, kda_stream_t stream) {
    int st = check_dims(dims, false);
    if (st) return st;
    if (!dtype_ok(z_dtype)) return KDA_ERR_INVALID_ARG;
    if (chunk != 0 && chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    const int span = chunk > 0 ? chunk : 64;
    if ((dims->T + span - 1) / span > 65535) return KDA_ERR_UNSUPPORTED;
    if (dims->T == 0) return KDA_OK;
    st = check_ptrs({g_out}, {}, {z}, io_bytes(z_dtype));
    if (!st) st = check_ptrs({}, {}, {A_log, dt_bias}, 4);
    if (st) return st;
    return from_cuda(kda::launch_gate(dims->B, dims->H, dims->T, dims->K, z_dtype, z, A_log,
                                      dt_bias, chunk, g_out, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// mode 0: the faster tensor-core form (or the fp32 path where it does not apply);
// 1 / 2 / 3: only the fused / split / split-with-scan tensor-core form, KDA_ERR_UNSUPPORTED
// elsewhere.
int chunk_forward(int mode, const kda_dims* dims, kda_dtype io_dtype, const void* q,
                  const void* k, const void* v, const void* z, const void* beta,
                  const float* A_log, const float* dt_bias, float scale, const float* h0,
                  int chunk, void* out, float* hT, kda_stream_t stream) {
    int st = check_dims(dims, true);
    if (st) return st;
    if (!dtype_ok(io_dtype)) return KDA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (dims->T > 0) {
        st = check_ptrs({q, k, v, z, out}, {h0, hT}, {beta}, io_bytes(io_dtype));
        if (!st) st = check_ptrs({}, {}, {A_log, dt_bias}, 4);
    } else {
        st = check_ptrs({}, {h0, hT});
    }
    if (st) return st;
    if (mode != 0 && dims->T == 0) return KDA_ERR_UNSUPPORTED;
    if (dims->T == 0 && !hT) return KDA_OK;
    kda::ChunkArgs a{dims->B, dims->H, dims->T, dims->K, dims->V, chunk, io_dtype, q, k, v, z,
                     beta, A_log, dt_bias, h0, scale, out, hT};
    bool taken = false;
    cudaError_t e = kda::launch_chunk_tc(a, (cudaStream_t)stream, mode, &taken);
    if (taken) return e == cudaErrorMemoryAllocation ? KDA_ERR_NO_MEMORY : from_cuda(e);
    if (mode != 0) return KDA_ERR_UNSUPPORTED;
    return from_cuda(kda::launch_chunk_simt(a, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

int kda_chunk_forward(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                      const void* v, const void* z, const void* beta, const float* A_log,
                      const float* dt_bias, float scale, const float* h0, int chunk, void* out,
                      float* hT, kda_stream_t stream) {
    return chunk_forward(0, dims, io_dtype, q, k, v, z, beta, A_log, dt_bias, scale, h0, chunk,
                         out, hT, stream);
}

int kda_chunk_forward_split(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                            const void* k, const void* v, const void* z, const void* beta,
                            const float* A_log, const float* dt_bias, float scale,
                            const float* h0, int chunk, void* out, float* hT,
                            kda_stream_t stream) {
    return chunk_forward(2, dims, io_dtype, q, k, v, z, beta, A_log, dt_bias, scale, h0, chunk,
                         out, hT, stream);
}

int kda_chunk_forward_fused(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                            const void* k, const void* v, const void* z, const void* beta,
                            const float* A_log, const float* dt_bias, float scale,
                            const float* h0, int chunk, void* out, float* hT,
                            kda_stream_t stream) {
    return chunk_forward(1, dims, io_dtype, q, k, v, z, beta, A_log, dt_bias, scale, h0, chunk,
                         out, hT, stream);
}

int kda_chunk_forward_scan(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                           const void* k, const void* v, const void* z, const void* beta,
                           const float* A_log, const float* dt_bias, float scale,
                           const float* h0, int chunk, void* out, float* hT,
                           kda_stream_t stream) {
    return chunk_forward(3, dims, io_dtype, q, k, v, z, beta, A_log, dt_bias, scale, h0, chunk,
                         out, hT, stream);
}

int kda_chunk_forward_split_noalloc(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                                    const void* k, const void* v, const void* z,
                                    const void* beta, const float* A_log, const float* dt_bias,
                                    float scale, const float* h0, int chunk, void* out,
                                    float* hT, kda_stream_t stream) {
    int st = check_dims(dims, true);
    if (st) return st;
    if (!dtype_ok(io_dtype)) return KDA_ERR_INVALID_ARG;
    if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (dims->T == 0) return KDA_ERR_UNSUPPORTED;
    st = check_ptrs({q, k, v, z, out}, {h0, hT}, {beta}, io_bytes(io_dtype));
    if (!st) st = check_ptrs({}, {}, {A_log, dt_bias}, 4);
    if (st) return st;
    kda::ChunkArgs a{dims->B, dims->H, dims->T, dims->K, dims->V, chunk, io_dtype, q, k, v, z,
                     beta, A_log, dt_bias, h0, scale, out, hT};
    bool fits = false;
    const cudaError_t e = kda::launch_chunk_split_noalloc(a, (cudaStream_t)stream, &fits);
    if (!fits) return KDA_ERR_UNSUPPORTED;
    return from_cuda(e);
}

int kda_fused_recurrent(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                        const void* v, const void* z, const void* beta, const float* A_log,
                        const float* dt_bias, float scale, float* state, void* out,
                        kda_stream_t stream) {
    int st = check_dims(dims, true);
    if (st) return st;
    if (!dtype_ok(io_dtype)) return KDA_ERR_INVALID_ARG;
    if ((long long)dims->B * dims->H > 0x3fffffffLL) return KDA_ERR_UNSUPPORTED;
    if (dims->T == 0) return check_ptrs({state}, {});
    st = check_ptrs({state}, {}, {q, k, v, z, beta, out}, io_bytes(io_dtype));
    if (!st) st = check_ptrs({}, {}, {A_log, dt_bias}, 4);
    if (st) return st;
    kda::StepArgs a{dims->B, dims->H, dims->K, dims->V, io_dtype, q, k, v, z, beta,
                    A_log, dt_bias, scale, state, out};
    if (dims->T == 1) return from_cuda(kda::launch_decode(a, (cudaStream_t)stream));
    return from_cuda(kda::launch_recurrent(a, dims->T, (cudaStream_t)stream));
}

int kda_chunk_backward(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                       const void* v, const void* z, const void* beta, const float* A_log,
                       const float* dt_bias, float scale, const float* h0, const void* d_o,
                       const float* dhT, float* dq, float* dk, float* dv, float* dz,
                       float* dbeta, float* dA_log, float* ddt_bias, float* dh0,
                       kda_stream_t stream) {
    int st = check_dims(dims, true);
    if (st) return st;
    if (!dtype_ok(io_dtype)) return KDA_ERR_INVALID_ARG;
    if (dims->T > 0) {
        st = check_ptrs({q, k, v, z, d_o, dq, dk, dv, dz}, {h0, dhT, dh0}, {beta}, io_bytes(io_dtype));
        if (!st) st = check_ptrs({}, {}, {A_log, dt_bias, dbeta, dA_log, ddt_bias}, 4);
    } else {
        st = check_ptrs({}, {h0, dhT, dh0}, {A_log, dt_bias, dA_log, ddt_bias}, 4);
    }
    if (st) return st;
    kda::BwdLaunch L{dims->B, dims->H, dims->T, dims->K, dims->V, io_dtype, q, k, v, z, beta, d_o,
                     A_log, dt_bias, h0, dhT, scale, dq, dk, dv, dz, dbeta, dA_log, ddt_bias, dh0};
    const cudaError_t e = kda::launch_chunk_backward(L, (cudaStream_t)stream);
    if (e == cudaErrorMemoryAllocation) {
        (void)cudaGetLastError();
        return KDA_ERR_NO_MEMORY;
    }
    return from_cuda(e);
}

int kda_device_status(kda_stream_t stream) {
    int timed_out = 0;
    int carry_timed_out = 0, decode_timed_out = 0, bwd_timed_out = 0;
    if (kda::read_and_clear_timeout((cudaStream_t)stream, &timed_out) != cudaSuccess ||
        kda::read_and_clear_carry_timeout(&carry_timed_out) != cudaSuccess ||
        kda::read_and_clear_decode_timeout(&decode_timed_out) != cudaSuccess ||
        kda::read_and_clear_bwd_timeout(&bwd_timed_out) != cudaSuccess)
        return KDA_ERR_CUDA;
    timed_out |= carry_timed_out | decode_timed_out | bwd_timed_out;
    return timed_out ? KDA_ERR_TIMEOUT : KDA_OK;
}

int kda_release_scratch(void) { return from_cuda(kda::scratch_release()); }

int kda_selftest_bounded_wait(unsigned long long limit_ns, kda_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 10000000000ull) return KDA_ERR_INVALID_ARG;
    return from_cuda(kda::launch_bounded_wait_selftest(limit_ns, (cudaStream_t)stream));
}

int kda_recurrent_step(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                       const void* v, const void* z, const void* beta, const float* A_log,
                       const float* dt_bias, float scale, float* state, void* out,
                       kda_stream_t stream) {
    int st = check_dims(dims, true);
    if (st) return st;
    if (!dtype_ok(io_dtype)) return KDA_ERR_INVALID_ARG;
    if (dims->T != 1) return KDA_ERR_INVALID_ARG;
    st = check_ptrs({state}, {}, {q, k, v, z, beta, out}, io_bytes(io_dtype));
    if (!st) st = check_ptrs({}, {}, {A_log, dt_bias}, 4);
    if (st) return st;
    kda::StepArgs a{dims->B, dims->H, dims->K, dims->V, io_dtype, q, k, v, z, beta,
                    A_log, dt_bias, scale, state, out};
    return from_cuda(kda::launch_decode(a, (cudaStream_t)stream));
}

}  // extern "C"
