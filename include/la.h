/*
 * la.h -- causal linear attention, retention and gated linear attention on one
 * NVIDIA GB300 (sm_103a): the chunkwise-parallel forward pass and the
 * single-token recurrent decode step.
 *
 * The operation (one (b, h) sequence; every (b, h) is independent):
 *
 *   S_t = diag(A_t) S_{t-1} + phi(k_t) v_t^T        S: d_k x d_v, S_0 = 0
 *   z_t = A_t * z_{t-1} + phi(k_t)                  only with LA_NORMALIZE
 *   out_t = phi(q_t)^T S_t                          read after the update
 *   out_t = phi(q_t)^T S_t / (phi(q_t) . z_t)       with LA_NORMALIZE
 *
 * Sources: learnllm m22 "Linear & Recurrent Attention" -- "The Math: Linear
 * Attention" (phi = elu + 1, S_i, Z_i, y_i), "Retention: Add a Decay to the
 * State" (S_n = gamma S_{n-1} + k_n^T v_n), "The Three Faces of Retention"
 * (chunkwise form) and "Interactive Exploration" (the gate A_t: 1 for linear
 * attention, gamma for retention, input-dependent for gated linear attention);
 * linear_sparse_attention.py, linear_attn_recurrent and linear_attn_chunkwise
 * (self-inclusive read, ragged last chunk); "causal linear attention as an RNN"
 * (S_0 = Z_0 = 0). The per-channel gate alpha = exp(logsigmoid(g) / 16) is the
 * gated-linear-attention gate (Yang et al. 2023, named on the troisinh and
 * learnllm pages) with temperature 16.
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers to row-major, contiguous arrays, each
 *    16-byte aligned (LA_ERR_MISALIGNED otherwise). The caller owns every
 *    buffer; outputs must not alias inputs.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *    The return value reports argument validation (done before any launch)
 *    and launch errors; errors during execution surface at the caller's next
 *    synchronisation.
 *  - State block: per (b, h), S as fp32 [d_k][d_v], followed by z as fp32
 *    [d_k] when LA_NORMALIZE is set. A state array is [B][H][block].
 *  - Element type of q, k, v, out and the per-channel gate g: bf16 by default,
 *    fp32 with LA_DTYPE_F32. Accumulation and the state are always fp32.
 *  - d_k, d_v in {16, 32, 64, 128}.
 */
#ifndef RETENTION_GB300_LA_H
#define RETENTION_GB300_LA_H

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = -1, /* null pointer, bad size, bad mode combination */
    LA_ERR_UNSUPPORTED = -2, /* valid request the library does not run (e.g. d_k = 48) */
    LA_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned */
    LA_ERR_CUDA = -4,        /* a CUDA call or kernel launch failed */
    LA_ERR_TIMEOUT = -5,     /* a bounded device-side wait ran out */
    LA_ERR_INTERNAL = -6     /* an internal consistency check failed */
} la_status;

/* mode bits */
#define LA_PHI_IDENTITY 0x0  /* phi(x) = x */
#define LA_PHI_ELU1 0x1      /* phi(x) = elu(x) + 1 on q and k */
#define LA_NORMALIZE 0x2     /* out = phi(q)S / phi(q).z; the state carries z */
#define LA_GATE_NONE 0x0     /* A_t = 1 (linear attention) */
#define LA_GATE_HEAD 0x4     /* retention: gate = const float gamma[H], A_t = gamma_h */
#define LA_GATE_CHANNEL 0x8  /* gated: gate = g [B][H][L][d_k] (decode: [B][H][d_k]),
                                same type as q; A_t = diag(exp(logsigmoid(g_t) / 16)) */
#define LA_DTYPE_F32 0x10    /* q, k, v, g, out are fp32 instead of bf16 */
#define LA_KERNEL_SIMT 0x20  /* la_chunk_fwd: force the general CUDA-core kernel */
#define LA_REVERSE 0x40      /* la_chunk_fwd: the anti-causal form (each token reads itself
                                and every later token; see la_chunk_fwd) */

/*
 * la_chunk_fwd -- the chunkwise-parallel forward pass over whole sequences,
 * starting from S_0 = 0 (and z_0 = 0) (ajkdrag zettel "causal linear
 * attention as an RNN": the recurrence starts from an empty state).
 *
 * Chunkwise form (learnllm m22 "The Three Faces of Retention";
 * linear_sparse_attention.py linear_attn_chunkwise): the L tokens are cut into
 * chunks of `chunk` tokens, the last one ragged. Inside a chunk the output is
 * the causally masked (diagonal included) product (Q K^T (.) D) V with the
 * decay D_ij = prod_{r=j+1..i} A_r; across chunks a fixed d_k x d_v state is
 * carried, read by each query with the decay since the chunk start and
 * advanced as S <- (decay over the chunk) S + sum_s (decay s -> chunk end)
 * k_s^T v_s. The result equals the recurrence above up to rounding.
 *
 *   q, k   [B][H][L][d_k]     v, out [B][H][L][d_v]
 *   gate   NULL (LA_GATE_NONE), const float gamma[H] (LA_GATE_HEAD, each in
 *          [0, 1]) or g [B][H][L][d_k] (LA_GATE_CHANNEL)
 *   final_state  NULL, or [B][H][block] fp32: the state after the last token
 *   B, H >= 0; L >= 0 (L = 0 writes a zero final state and no output)
 *   chunk  1..128. The tensor-core kernel (bf16, d_k = d_v = 128, chunk 64)
 *          is chosen automatically; other cases run the general kernel, which
 *          returns LA_ERR_UNSUPPORTED when its tiles do not fit on chip.
 *   mode   LA_PHI_* | LA_NORMALIZE | LA_GATE_* | LA_DTYPE_F32 | LA_KERNEL_SIMT |
 *          LA_REVERSE
 *
 * LA_REVERSE: the anti-causal form, the same sums taken over the token and every
 * LATER one, out_s = sum_{t >= s} A^{t-s} (q_s . k_t) v_t, with the state carried
 * from the end of the sequence towards its start (final_state is then the state
 * before token 0; an initial state of la_chunk_fwd_from_state sits after the
 * last token). It equals the causal forward of the token-reversed sequence. The
 * backward pass is built from such sums. With LA_GATE_CHANNEL the decay from s
 * to t is prod_{j=s+1..t} alpha_j, so token s is decayed by the gate of token
 * s + 1 (the last token by none): out_s = sum_{t >= s} (prod_{j=s+1..t}
 * diag(alpha_j)) applied to phi(k_t)^T v_t, read by phi(q_s), and the final state
 * is sum_t (prod_{j=1..t} diag(alpha_j)) phi(k_t)^T v_t. Tensor-core kernel only:
 * bf16, d_k = d_v = 128, chunk 64, no normaliser, and no gate or the
 * per-channel gate (either feature map) or the head gate (identity feature
 * map); anything else returns LA_ERR_UNSUPPORTED.
 *
 * Scratch: when the batch has too few (b, h) sequences to fill the GPU (2 B H
 * at most the number of SMs), the tensor-core path splits each sequence into
 * segments and takes stream-ordered scratch (cudaMallocAsync / cudaFreeAsync
 * on `stream`) for the per-segment states; a failed allocation returns
 * LA_ERR_CUDA. All stream-ordered scratch of this library comes from a memory
 * pool of its own, created on a device (in each context, found by its unique
 * id, so a context made again after cudaDeviceReset gets a new pool) the first
 * time the library allocates there (cudaMemPoolCreate); its release threshold
 * keeps freed scratch mapped for the next call instead of unmapping it at every
 * synchronisation, so the pool holds up to the largest scratch any call used
 * until its context ends. The device's default memory pool is neither used nor
 * changed. The first call that takes scratch in a context creates the pool and
 * should come before any stream capture.
 * la_chunk_fwd_noalloc is the same call without any allocation.
 * A split call issues three kernels on `stream`: the segment end states (of
 * every segment but each sequence's last), a scan over them, and the full pass
 * (which writes final_state from its last segments). The full pass goes out as a programmatic
 * dependent launch behind the scan. Its CTAs may start before the scan ends,
 * but they wait for it before reading what it wrote, and the call's work is
 * complete, for later work on `stream`, only when all three have finished.
 *
 * Range of the tensor-core kernel: it factors the decay inside a chunk as
 * exp(b_t) * exp(-b_s), b the log decay from the chunk start, which is exact
 * in real arithmetic and stays in fp32/bf16 range while the log-decay over one
 * chunk, per channel, is above about -87 (retention: gamma^chunk > 1.6e-38);
 * the general kernel (LA_KERNEL_SIMT) has no such limit.
 */
int la_chunk_fwd(const void *q, const void *k, const void *v, const void *gate,
                 void *out, float *final_state, int B, int H, int L, int dk,
                 int dv, int mode, int chunk, la_stream_t stream);

/*
 * la_chunk_fwd_from_state -- la_chunk_fwd starting from a given state instead
 * of zero: the continuation of a sequence whose first part is summarised by
 * that state (learnllm m22 "Code: The Two Faces": the state is all a sequence
 * needs to go on; a prefill's final_state continues here, or in
 * la_decode_step, and this call's final_state continues in either).
 *
 *   initial_state  NULL (then exactly la_chunk_fwd), or [B][H][block] fp32,
 *                  the state S (then z when LA_NORMALIZE) before the first
 *                  token of each sequence; 16-byte aligned; read only, and it
 *                  must not overlap final_state or out
 *   every other argument, the results and the errors as in la_chunk_fwd; with
 *   L = 0 the final state is a copy of the initial state.
 */
int la_chunk_fwd_from_state(const void *q, const void *k, const void *v, const void *gate,
                            const float *initial_state, void *out, float *final_state, int B,
                            int H, int L, int dk, int dv, int mode, int chunk,
                            la_stream_t stream);

/*
 * la_delta_fwd -- the delta rule (DeltaNet) over whole sequences, recurrent
 * form, from S_0 = 0 (linear_sparse_attention.py, "delta_rule_recurrent"):
 *
 *   S <- S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T ;  out_t = S q_t
 *
 * Each token first erases what S returns for its key, then writes its value
 * there; the output is read after the update. S is d_v x d_k (the v k^T
 * orientation of that function). Keys are used as given: the rule expects
 * unit-norm keys and the caller normalises them (as that page does).
 *
 *   q, k   [B][H][L][d_k]     v, out [B][H][L][d_v]   (bf16, or fp32 with LA_DTYPE_F32)
 *   beta   [B][H][L], the same type; usually in (0, 1]
 *   final_state  NULL, or [B][H][d_v][d_k] fp32: S after the last token
 *   mode   0 or LA_DTYPE_F32 (no feature map, normaliser or gate), optionally
 *          | LA_KERNEL_SIMT to force the recurrent kernel
 *   d_k, d_v in {16, 32, 64, 128}; B, H, L >= 0 (L = 0 writes a zero state)
 *
 * bf16 with d_k = d_v = 128 runs in chunks of 64 tokens on the tensor cores:
 * each step is S_t = S_{t-1} + u_t k_t^T with u_t = beta_t (v_t - S_{t-1} k_t),
 * and inside a chunk the u_t solve a unit lower-triangular system (I + A) U =
 * diag(beta) (V - K S0^T), A[t][s] = beta_t k_t . k_s for s < t, so a chunk
 * is a triangular inverse and a few matrix products (the recurrence
 * rearranged; no page gives this form). T = (I + A)^-1 diag(beta) does not
 * depend on the state, so one kernel (a CTA per sequence) makes T of the next
 * chunk while the state runs through the current one; it allocates nothing.
 * Every other case runs the recurrence token by token on the CUDA cores in
 * fp32 (6 d_k d_v flops a token).
 * Errors as la_chunk_fwd; beta needs only element alignment.
 */
int la_delta_fwd(const void *q, const void *k, const void *v, const void *beta,
                 void *out, float *final_state, int B, int H, int L, int dk,
                 int dv, int mode, la_stream_t stream);

/*
 * la_group_norm_swish -- the RetNet output epilogue (learnllm m22,
 * "Retention": retention has no normaliser; RetNet steadies its output with a
 * GroupNorm and a swish gate instead). One group per head: each (b, h, t) row
 * of d_v values is normalised on its own,
 *
 *   y   = (x - mean) / sqrt(var + eps) * weight[h] + bias[h]   (var biased, over the d_v values)
 *   out = swish(ogate) * y,   swish(u) = u sigmoid(u)
 *
 * ogate is the output gate, the caller's projection of the layer input (X W_G
 * in RetNet); the output projection after it is the caller's too.
 *
 *   x, ogate, out  [B][H][L][d_v] (bf16, or fp32 with LA_DTYPE_F32); out may
 *                  be x (in place), otherwise no overlap
 *   weight, bias   NULL (1 and 0) or fp32 [H][d_v], 16-byte aligned
 *   eps            >= 0 and finite (LA_ERR_INVALID_ARG otherwise)
 *   mode           0 or LA_DTYPE_F32
 * Decode outputs ([B][H][d_v]) are the case L = 1. Errors as la_chunk_fwd.
 */
int la_group_norm_swish(const void *x, const void *ogate, const float *gn_weight,
                        const float *gn_bias, float gn_eps, void *out, int B, int H,
                        int L, int dv, int mode, la_stream_t stream);

/*
 * la_chunk_fwd_gn_swish -- la_chunk_fwd_from_state followed by the RetNet
 * output epilogue of la_group_norm_swish on its output: out is
 * swish(ogate) * GroupNorm_h(o), o the attention output (after the division by
 * the normaliser when LA_NORMALIZE is set). On the tensor-core kernel without
 * the normaliser and with no gate or the head gate (RetNet's retention among
 * them) the epilogue runs in the kernel's store: each token row is normalised
 * from the fp32 accumulator, and the output gate tile is read by TMA beside it,
 * so o never goes to memory. Otherwise it is a second kernel on the same
 * stream, in place on out. The swish in the store is formed in bf16 arithmetic
 * with the hardware tanh approximation (u sigmoid(u) = h + h tanh(h),
 * h = u / 2).
 *
 *   ogate          [B][H][L][d_v], the type of q; required
 *   gn_weight, gn_bias, gn_eps   as la_group_norm_swish
 *   every other argument, the results and the errors as la_chunk_fwd_from_state
 *   (initial_state may be NULL); the final state is that of the attention,
 *   untouched by the epilogue.
 */
int la_chunk_fwd_gn_swish(const void *q, const void *k, const void *v, const void *gate,
                          const float *initial_state, const void *ogate,
                          const float *gn_weight, const float *gn_bias, float gn_eps,
                          void *out, float *final_state, int B, int H, int L, int dk,
                          int dv, int mode, int chunk, la_stream_t stream);

/*
 * la_chunk_bwd -- the backward pass of la_chunk_fwd (from S_0 = 0): given the
 * gradient dout of the output, the gradients of q, k, v and of the per-channel
 * gate g. The pages give no gradient (learnllm m22 "The Three Faces of
 * Retention" motivates the chunkwise form for training); this is the chain
 * rule on the recurrence:
 *
 *   forward sweep   dQ_t = S_t w_t + z_t e_t
 *   reverse sweep   dS_t = diag(A_{t+1}) dS_{t+1} + phi(q_t) w_t^T  (dz_t with e_t)
 *                   dK_t = dS_t v_t + dz_t,   dv_t = dS_t^T phi(k_t)
 *   dq = dQ * phi'(q),  dk = dK * phi'(k)
 *   dg_r = sigmoid(-g_r) / 16 * sum_{t >= r} (phi(q_t) dQ_t - phi(k_t) dK_t)
 *
 * with w_t = dout_t, e_t = 0 without the normaliser, and w_t = dout_t / den_t,
 * e_t = -(dout_t . out_t) / den_t with it (formed inside from S_t w_t, so the
 * forward's output is not needed).
 *
 *   q, k, v, gate, B, H, L, dk, dv, mode   as given to la_chunk_fwd (the chunk
 *          size does not enter the gradient)
 *
 * Two routes. bf16 with d_k = d_v = 128 runs on the tensor-core forward kernel
 * (except the per-channel gate together with the normaliser): each gradient
 * term is a linear-attention forward with its roles permuted, causal for dQ and
 * anti-causal (the LA_REVERSE form, over later tokens) for dK and dv; with the
 * normaliser also w_t = dout_t / den_t and e_t = -(dout_t . num_t) / den_t^2 on
 * the scores and a carried sum (the cancelling terms in fp32); with the
 * per-channel gate dv is an anti-causal gated forward and dQ, dK are forwards
 * whose decay falls on the value channel, and dg comes from a segmented
 * reverse scan. Every other case (and LA_KERNEL_SIMT) runs three sweeps over
 * the sequence on the CUDA cores.
 *   dout   [B][H][L][d_v]; dq, dk [B][H][L][d_k] and dv [B][H][L][d_v] are
 *          written, in the type of q
 *   dgate  with LA_GATE_CHANNEL: NULL (not computed) or [B][H][L][d_k] in the
 *          type of q; ignored otherwise (no gradient is formed for gamma)
 * No gradient flows into a final state or out of an initial one. Scratch,
 * taken stream-ordered from the library's pool on `stream` (LA_ERR_CUDA if that
 * fails): on the tensor-core route none with the identity feature map (beyond
 * the per-segment states of batches too small to fill the GPU), four bf16
 * [B][H][L][128] arrays with LA_PHI_ELU1; with LA_NORMALIZE one bf16 array and
 * one fp32 [B][H][L] one without a gate (plus the per-segment states), five
 * bf16 and five fp32 arrays with the head gate; with LA_GATE_CHANNEL two bf16 arrays and
 * one fp32 one plus per-chunk sums; on the other route one fp32 [B][H][L][d_k]
 * array (two, plus three [B][H][L], with LA_NORMALIZE).
 * Errors as la_chunk_fwd; no output may overlap an input.
 */
int la_chunk_bwd(const void *q, const void *k, const void *v, const void *gate,
                 const void *dout, void *dq, void *dk, void *dv, void *dgate, int B,
                 int H, int L, int dk_, int dv_, int mode, la_stream_t stream);

/*
 * la_decode_step -- one recurrent step for every (b, h), in place on `state`
 * (learnllm m22 "Code: The Two Faces", the LinearAttentionState.step object;
 * insideout lesson 16: S <- S + k v^T, z <- z + k, out = q^T S / (q . z)):
 *
 *   S <- diag(A) S + phi(k) v^T ; z <- A * z + phi(k) ; out = phi(q)^T S [/ phi(q).z]
 *
 *   q, k   [B][H][d_k]   v, out [B][H][d_v]   (bf16, or fp32 with LA_DTYPE_F32)
 *   gate   NULL, const float gamma[H], or g [B][H][d_k]
 *   state  [B][H][block] fp32, read and written in place (S, then z when
 *          LA_NORMALIZE). A final_state of la_chunk_fwd continues here.
 *   mode   LA_PHI_* | LA_NORMALIZE | LA_GATE_* | LA_DTYPE_F32
 */
int la_decode_step(const void *q, const void *k, const void *v, const void *gate,
                   float *state, void *out, int B, int H, int dk, int dv, int mode,
                   la_stream_t stream);

/*
 * la_chunk_fwd_noalloc -- la_chunk_fwd without any device allocation. No page
 * of the method has a counterpart to this call; it exists for callers that
 * cannot let a library allocate device memory in the middle of their work,
 * such as servers that plan all device memory up front or code running while
 * another allocator owns the device's memory pool.
 *
 * Same arguments, results and errors as la_chunk_fwd. Where la_chunk_fwd would
 * take stream-ordered scratch (the tensor-core path splitting a short batch
 * into sequence segments), this call uses a fixed device array of
 * LA_NOALLOC_SCRATCH_BYTES bytes inside the library instead: every GPU that
 * loads the library holds that array until the process exits. A request that
 * would need more scratch returns LA_ERR_UNSUPPORTED. It never calls cudaMalloc,
 * cudaMallocAsync or cudaFree.
 *
 * - Each call that splits looks up the array's device address in the current
 *   device's context (a lookup, not an allocation). The array lives in the
 *   library's device code, which the CUDA driver loads lazily by default: the
 *   first such call in a context is when the driver maps the array's
 *   LA_NOALLOC_SCRATCH_BYTES on that device. A caller with a fixed memory plan
 *   should therefore make one call that splits (few sequences, e.g. B = H = 1,
 *   L = 64 * 152) on each device during set-up, and should make that first
 *   call before starting any stream capture.
 * - Every call on a device shares the one array and leaves its contents behind.
 *   Nothing in it has to start at zero: each call writes every scratch value
 *   before reading it. Calls whose work overlaps on the GPU (other streams,
 *   other host threads) race on the array; the caller must order them.
 */
#define LA_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)
int la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *gate,
                         void *out, float *final_state, int B, int H, int L, int dk,
                         int dv, int mode, int chunk, la_stream_t stream);

/*
 * la_chunk_fwd_path -- which kernel la_chunk_fwd would run for these sizes and
 * mode on the current device, without launching anything: 1 = tensor-core
 * kernel, 0 = general CUDA-core kernel, or a negative la_status for arguments
 * la_chunk_fwd would reject. Diagnostics only.
 */
int la_chunk_fwd_path(int B, int H, int L, int dk, int dv, int mode, int chunk);

/* A static, human-readable name for a la_status value. */
const char *la_status_string(int status);

/* Number of kernels this library has launched in this process (diagnostics). */
unsigned long long la_kernel_launches(void);

/*
 * la_device_status -- waits for the work queued on `stream`, then reports
 * whether any kernel of this library on the current device gave up a bounded
 * wait since the last call: LA_ERR_TIMEOUT if one did (its outputs are not
 * valid; the CUDA context stays usable), LA_OK if none did, LA_ERR_CUDA if the
 * synchronisation or the read failed. Reading clears the flags. In a library
 * built with LA_DEBUG (a test build that checks every shared-memory range, TMA
 * coordinate, TMEM address and global index of the tensor-core forward and the
 * decode step before using it, and skips an access that fails) it returns
 * LA_ERR_INTERNAL when a check failed. The kernels
 * with such waits are the tensor-core chunk forward (which the tensor-core
 * backward also runs) and the chunked delta rule; every wait gives up after
 * 2 s of wall time, far beyond any legitimate one.
 */
int la_device_status(la_stream_t stream);

/*
 * la_chunk_fwd_stall_test -- diagnostics: makes the bounded waits of the
 * tensor-core chunk forward run out on purpose, so that a caller (and this
 * library's tests) can check the time-out path on a GPU without faulting or
 * hanging it. The forward of la_chunk_fwd (d_k = d_v = 128, chunk 64, bf16,
 * no final state) is launched once, unsplit, with its TMA producer issuing no
 * tiles from chunk `stall_chunk` of each sequence on and every wait giving up
 * after `wait_ns` nanoseconds: the roles left waiting leave their loops, the
 * kernel drains what it issued, frees its tensor memory, sets the error word
 * that la_device_status reports as LA_ERR_TIMEOUT, and returns. The CUDA
 * context stays usable; `out` is not valid afterwards (chunks before
 * stall_chunk are written). No page of the method has a counterpart.
 *
 *   q, k, v, gate, out, B, H, L, mode   as la_chunk_fwd (d_k = d_v = 128)
 *   stall_chunk   >= 0; at or past the last chunk nothing stalls
 *   wait_ns       1e5 .. 2e9 (the ordinary calls use 2e9)
 * Returns LA_ERR_UNSUPPORTED where la_chunk_fwd would not take the
 * tensor-core kernel or would split the sequences (2 B H at most the number of
 * SMs); otherwise errors as la_chunk_fwd.
 */
int la_chunk_fwd_stall_test(const void *q, const void *k, const void *v, const void *gate,
                            void *out, int B, int H, int L, int mode, int stall_chunk,
                            long long wait_ns, la_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RETENTION_GB300_LA_H */
