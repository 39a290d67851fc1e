/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) Kimi Delta Attention forward.
 *
 * The method (kdafix-2026-10-02, "Fix 1 -- decay form" and "Fix 2 -- read
 * scale"): per (batch b, head h) a state S of shape K x V; per token t and key
 * channel c the log decay
 *
 *     g[t,c] = -exp(A_log[h]) * softplus(z[t,c] + dt_bias[h,c]),   alpha = exp(g),
 *
 * and the step
 *
 *     S <- diag(alpha_t) S;   u = v_t - S^T k_t;   S <- S + beta_t k_t u^T;
 *     o_t = S^T (scale * q_t).
 *
 * The scale (default K**-0.5) is folded into q: it enters the read only and
 * never the state.  kda_chunk_forward computes the same function chunk-parallel
 * in WY form; its inter-chunk carry uses exp(G_last - G) with G the in-chunk
 * cumulative log decay (kda-adjoint-2026-10-01, section 2).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers to contiguous, head-major arrays:
 *       q, k, z   : (B, H, T, K)        v, out : (B, H, T, V)
 *       beta      : (B, H, T)           A_log  : (H)          dt_bias : (H, K)
 *       h0, hT, state : (B, H, K, V)    float32 always
 *   q, k, v, z, beta and out have the I/O dtype (KDA_F32 or KDA_BF16);
 *   A_log, dt_bias and the state are float32.
 * - Alignment (else KDA_ERR_MISALIGNED): q, k, v, z, out, h0, hT and state
 *   must be 16-byte aligned for kda_chunk_forward (tiles are moved in 16-byte
 *   units); kda_recurrent_step needs 16 bytes only for `state`; beta, A_log,
 *   dt_bias (and, for kda_recurrent_step and kda_gate, the per-token vectors)
 *   need only their element alignment.
 * - The caller owns every buffer.  The library keeps no state between calls
 *   except the CUDA resources the runtime itself caches, the split form's second
 *   stream, the no-alloc form's fixed array (both below) and its scratch pool; it
 *   is re-entrant.  Scratch memory, where a path needs it, is taken stream-ordered
 *   on the caller's stream from a memory pool of the library's own on the current
 *   device (cudaMallocFromPoolAsync) and returned to it on the same stream before
 *   the call returns.  The pool keeps the blocks returned to it for later calls
 *   (the device's default pool hands them back to the system at every
 *   synchronisation, and mapping them again cost as much as a backward kernel):
 *   it holds up to the largest scratch in use at once until kda_release_scratch()
 *   or the end of the process.
 * - Work is enqueued on `stream` (NULL = the legacy default stream); calls
 *   return as soon as it is enqueued.  Argument errors are detected on the host
 *   before anything is launched; a launch error is reported as KDA_ERR_CUDA;
 *   errors during execution surface at the caller's next synchronisation.
 *   No C++ exception crosses this boundary.
 * - Supported sizes: B, H >= 1; T >= 0 (T = 0 is a no-op apart from hT = h0);
 *   K and V multiples of 8 in [8, 128]; chunk in {16, 32, 64}.  Anything else
 *   returns KDA_ERR_UNSUPPORTED.  T need not be a multiple of chunk.
 */
#ifndef KDA_H_
#define KDA_H_

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* kda_stream_t; /* the same type as cudaStream_t */

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef struct {
    int B, H, T, K, V;
} kda_dims;

enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad enum */
    KDA_ERR_UNSUPPORTED = -2, /* size or chunk outside the supported set */
    KDA_ERR_MISALIGNED = -3,  /* a pointer not 16-byte aligned */
    KDA_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    KDA_ERR_NO_MEMORY = -5,   /* scratch allocation failed */
    KDA_ERR_TIMEOUT = -6      /* a kernel gave up on a bounded wait (see kda_device_status) */
};

/*
 * kda_gate -- the decay gate alone (kdafix-2026-10-02, "Fix 1").
 *   g_out[b,h,t,c] = -exp(A_log[h]) * softplus(z[b,h,t,c] + dt_bias[h,c])   (chunk == 0)
 *   or its inclusive cumulative sum over the tokens of each chunk of `chunk`
 *   tokens (chunk in {16, 32, 64}): G[t] = sum of g over the chunk's tokens up to t.
 * z has dtype z_dtype, shape (B, H, T, K); g_out is float32 (B, H, T, K).
 * dims->V is ignored.
 */
int kda_gate(const kda_dims* dims, kda_dtype z_dtype, const void* z, const float* A_log,
             const float* dt_bias, int chunk, float* g_out, kda_stream_t stream);

/*
 * kda_chunk_forward -- the KDA forward over T tokens, chunk-parallel WY form.
 *   scale : the read scale folded into q (pass K**-0.5 for the default).
 *   h0    : initial state (B,H,K,V) float32, or NULL for zero.
 *   out   : (B,H,T,V) in io_dtype.
 *   hT    : final state (B,H,K,V) float32, or NULL if not wanted.
 * h0 and hT may be the same buffer (the state is then advanced in place).
 */
int kda_chunk_forward(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                      const void* v, const void* z, const void* beta, const float* A_log,
                      const float* dt_bias, float scale, const float* h0, int chunk, void* out,
                      float* hT, kda_stream_t stream);

/*
 * kda_chunk_forward_split / kda_chunk_forward_fused -- kda_chunk_forward restricted to one of
 * its tensor-core forms (bf16 I/O, K = V = 128, chunk 64, T >= 1; anything else returns
 * KDA_ERR_UNSUPPORTED).  kda_chunk_forward picks among them (and kda_chunk_forward_scan below)
 * by the shape; these exist to run and compare each form on any shape.
 *   fused : the whole forward in one kernel that reads each input once, the state on chip.
 *           With at most one sequence per SM, one CTA per (b, h) walks its chunks.  With more
 *           sequences than SMs, one CTA per SM takes (segment, sequence) work items of a few
 *           chunks in order and the fp32 state passes between a sequence's segments through
 *           hT (or, when hT is NULL, a B*H*K*V*4-byte scratch buffer); a counter and one flag
 *           per sequence (4*(B*H + 1) bytes) are taken from the scratch pool, cleared and
 *           returned on `stream` by the call (KDA_ERR_NO_MEMORY if the allocation fails).
 *   split : the chunk-parallel WY form of kda-adjoint-2026-10-01 section 2 as two kernels.  A
 *           prep kernel spreads every chunk of every sequence over the GPU and writes, per
 *           chunk, the state-independent operands ([W^T | (Q Gamma)^T], U^T, K~ =
 *           K e^{G_last - G} and the masked score matrix M in bf16, Gamma_last in fp32:
 *           74,240 bytes); a carry kernel then walks the chunks of each sequence with the
 *           fp32 state on chip (Delta = U - W S, S <- Gamma_last S + K~^T Delta,
 *           o = scale (Q Gamma S + M Delta)).  Suited to few, long sequences, where
 *           the fused form leaves most of the GPU idle.  The operands live in scratch that
 *           the call takes from the scratch pool and returns on `stream` (at most 1 GiB:
 *           longer inputs run as consecutive segments of chunks); KDA_ERR_NO_MEMORY if that
 *           allocation fails.  With B*H at most half the SMs and four or more chunks,
 *           the call runs each segment's carry on a second stream, beside the next segment's
 *           prep, with two operand buffers, and joins it back into `stream` (events) before
 *           it returns.  That stream and its five events are created on the first such call
 *           on a device (and again after the device's context was reset) and kept until the
 *           process exits; calls on one device enqueue this part one at a time (a lock), and
 *           their carries share that stream.
 */
int kda_chunk_forward_split(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                            const void* k, const void* v, const void* z, const void* beta,
                            const float* A_log, const float* dt_bias, float scale,
                            const float* h0, int chunk, void* out, float* hT,
                            kda_stream_t stream);
int kda_chunk_forward_fused(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                            const void* k, const void* v, const void* z, const void* beta,
                            const float* A_log, const float* dt_bias, float scale,
                            const float* h0, int chunk, void* out, float* hT,
                            kda_stream_t stream);

/*
 * kda_chunk_forward_scan -- kda_chunk_forward_split with the chunk-parallel state scan: for few
 * sequences over many chunks, where the split form's one-CTA-per-sequence carry would walk
 * every chunk of a sequence in order.  Per chunk n the carry is affine in the state,
 *     S_{n+1} = P_n S_n + Z_n,   P_n = diag(Gamma_last) - K~^T W,   Z_n = K~^T U
 * (the chunk carry of kda-adjoint-2026-10-01 section 2), so the chunks of a sequence are cut
 * into sub-segments whose maps (P, the product of their P_n, and Z, the state they reach from
 * S = 0) are computed in parallel by the carry kernel, combined in order in fp32 into every
 * sub-segment's entering state, and then every sub-segment runs its plain carry (writing o)
 * in parallel.  About three times the carry work of the split form, but the sequential part
 * is one K x K by K x V product per sub-segment instead of one chunk step per chunk.
 * kda_chunk_forward takes this form by itself where it is the faster one.
 * Shapes, arguments and errors as kda_chunk_forward_split.  Scratch (from the scratch pool on
 * `stream`, at most 1 GiB, longer inputs in segments of chunks): the
 * per-chunk operands, 3 x B*H*K*V*4 bytes per sub-segment for the maps and the entering
 * states, and B*H*K*V*4 for the carried state when hT is NULL; KDA_ERR_NO_MEMORY if that
 * allocation fails.  The result equals the split form's to rounding (the state reaches each
 * sub-segment along another order of products), not bit for bit.
 */
int kda_chunk_forward_scan(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                           const void* k, const void* v, const void* z, const void* beta,
                           const float* A_log, const float* dt_bias, float scale,
                           const float* h0, int chunk, void* out, float* hT,
                           kda_stream_t stream);

/*
 * kda_chunk_forward_split_noalloc -- kda_chunk_forward_split for callers that cannot allocate
 * device memory during the call (memory budgeted up front by a serving runtime, code where an
 * allocation may stall or fail at the wrong moment).  The pages this library follows have no
 * counterpart: it is the same computation, with the per-chunk operands kept in one fixed
 * array of 64 MiB, reserved on each GPU where this entry point is called (the library loads
 * its module lazily), until the process exits.  The call makes no cudaMalloc /
 * cudaMallocAsync / cudaFree call of its own.
 *   Limit: one chunk of every sequence must fit, i.e. B*H*74,240 bytes, plus B*H*65,536 when
 *   hT is NULL (the carried state then lives in the array too), at most 64 MiB: B*H <= 903
 *   with hT, B*H <= 480 without.  Larger B*H returns KDA_ERR_UNSUPPORTED and launches
 *   nothing.  Any T: longer inputs run as consecutive segments of chunks.
 *   Shapes as kda_chunk_forward_split (bf16, K = V = 128, chunk 64, T >= 1).
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress
 *   with that device current); make that first call before any stream capture.  After a
 *   cudaDeviceReset the next call looks it up again (the array may have moved), so that
 *   call too belongs outside a capture.
 *   All calls share the array and it keeps the last call's contents; nothing needs clearing
 *   (every byte a call reads, the same call wrote first).  Calls that overlap on the GPU
 *   (other streams, other host threads) race on it: serialise them.
 */
int kda_chunk_forward_split_noalloc(const kda_dims* dims, kda_dtype io_dtype, const void* q,
                                    const void* k, const void* v, const void* z,
                                    const void* beta, const float* A_log, const float* dt_bias,
                                    float scale, const float* h0, int chunk, void* out,
                                    float* hT, kda_stream_t stream);

/*
 * kda_recurrent_step -- one decode token per (b, h): the step above applied
 * once, in place on `state` (B,H,K,V) float32.  dims->T must be 1; q, k, z are
 * (B,H,1,K), v and out (B,H,1,V), beta (B,H,1), all in io_dtype.
 * (kdafix-2026-10-02, "Fix 2": the decode read uses the same folded scale.)
 */
int kda_recurrent_step(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                       const void* v, const void* z, const void* beta, const float* A_log,
                       const float* dt_bias, float scale, float* state, void* out,
                       kda_stream_t stream);

/*
 * kda_fused_recurrent -- dims->T >= 0 consecutive tokens per (b, h) applied token by token
 * (the step of kda_recurrent_step, T times), with the state kept on chip between tokens:
 * `state` (B,H,K,V) float32 is read once and written once, in place.  q, k, z are
 * (B,H,T,K), v and out (B,H,T,V), beta (B,H,T), all in io_dtype (the chunked layouts).
 * For short sequences (multi-token decode, small prefills) it moves far fewer bytes
 * than T calls of kda_recurrent_step; kda_recurrent_step is the T = 1 case.
 */
int kda_fused_recurrent(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                        const void* v, const void* z, const void* beta, const float* A_log,
                        const float* dt_bias, float scale, float* state, void* out,
                        kda_stream_t stream);

/*
 * kda_chunk_backward -- the gradients of the chunked forward (kda_chunk_forward with the same
 * q, k, v, z, beta, A_log, dt_bias, scale and h0) with respect to all of its inputs, given
 * the gradients of a loss with respect to its outputs: d_o = dL/do (B,H,T,V) in io_dtype and
 * dhT = dL/dhT (B,H,K,V) float32 (NULL = 0).  The kda-adjoint-2026-10-01 page names this
 * backward and its gradients (dq, dk, dv, dg, dbeta and the state gradient); the gate's own
 * derivative carries dg on to z, A_log and dt_bias.
 *
 * Outputs, all float32, caller-owned, fully overwritten:
 *   dq, dk, dz (B,H,T,K)   dv (B,H,T,V)   dbeta (B,H,T)
 *   dA_log (H) and ddt_bias (H,K), summed over the batch
 *   dh0 (B,H,K,V): the gradient with respect to the initial state (a zero state when h0 is
 *   NULL); NULL skips it.
 * Inputs in io_dtype and float32 as for kda_chunk_forward; K, V as there.  The pass runs in
 * chunks of 16 tokens whatever the forward's chunk size (the gradient does not depend on it),
 * to float32 accuracy: for K = V = 128 the contractions with the state run on the tensor
 * cores, each float32 operand split into two bf16 halves and all four half products
 * accumulated in float32 (about 2^-15 relative per product term), the state and its gradient
 * kept in float32; other sizes run in float32 on the CUDA cores.  For K = V = 128 the pass is
 * one persistent kernel (at most one CTA per SM) that takes each sequence's forward and
 * reverse walks as work items, split into up to 8 segments per walk when the sequences
 * outnumber the SMs, the state handed between segments in scratch.  Scratch:
 * (B*H*ceil(T/16)*(K*V + R) + B*H*S*(K+1)) float32, R = 2*16*V + 3*16*16 + 16*K for
 * K = V = 128 and 2*16*V otherwise (the state entering every 16-token chunk and the chunk's
 * R, Delta and, for K = V = 128, A', T, M and the log decay g), S the segments per walk, plus
 * for K = V = 128 (1 + 2*B*H) uint32 (the schedule's counter and flags, cleared on `stream`)
 * and, with more than one segment, 2*B*H*K*V float32 (the handoffs); from the scratch pool on
 * `stream`, returned on it; KDA_ERR_NO_MEMORY if that fails.  A bounded wait of the tensor-core form that gives up is reported by
 * kda_device_status.  Alignment: q, k, v, z, d_o, dq,
 * dk, dv, dz, h0, dhT, dh0 16 bytes; beta, dbeta, dA_log, ddt_bias, A_log, dt_bias their
 * element size.  Two kernels per call (the pass, then the batch sum of dA_log / ddt_bias).
 */
int kda_chunk_backward(const kda_dims* dims, kda_dtype io_dtype, const void* q, const void* k,
                       const void* v, const void* z, const void* beta, const float* A_log,
                       const float* dt_bias, float scale, const float* h0, const void* d_o,
                       const float* dhT, float* dq, float* dk, float* dv, float* dz,
                       float* dbeta, float* dA_log, float* ddt_bias, float* dh0,
                       kda_stream_t stream);

/*
 * kda_release_scratch -- wait for the current device to finish its work, then hand the blocks
 * the library's scratch pool holds for later calls back to the system (the pool is described
 * at the top of this header; a later call takes its scratch anew).  KDA_ERR_CUDA if a CUDA
 * call fails.
 */
int kda_release_scratch(void);

/* A static, human-readable name for a status code. */
const char* kda_status_string(int status);

/*
 * kda_device_status -- waits for `stream` to drain, then reports whether any kernel of this
 * library gave up on one of its bounded waits since the last call (KDA_ERR_TIMEOUT; the
 * outputs of that call are not valid) and clears the report.  Every wait on a tensor-core or
 * copy completion inside the kernels is bounded (about two seconds), so a lost completion
 * ends the kernel with this report instead of hanging the GPU.  Returns KDA_OK, or
 * KDA_ERR_CUDA if the stream itself failed.
 */
int kda_device_status(kda_stream_t stream);

/*
 * kda_selftest_bounded_wait -- launches one tiny kernel whose wait can never be satisfied
 * (an mbarrier nobody arrives on) with the given limit in nanoseconds (1 .. 1e10).  It ends
 * after the limit and leaves a KDA_ERR_TIMEOUT report for kda_device_status: a way to
 * exercise the failure path without faulting the GPU.
 */
int kda_selftest_bounded_wait(unsigned long long limit_ns, kda_stream_t stream);

/*
 * Diagnostic: the number of CUDA kernels this library has launched in this
 * process so far (all devices, all threads; a relaxed atomic counter).
 * Benchmarks read it before and after a timed region to count launches.
 */
unsigned long long kda_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
