// la_common.cuh -- device helpers and internal launch interfaces shared by the
// kernels of the library (never by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/la.h"

namespace la {

// ---------------------------------------------------------------- debug build
// Built with LA_DEBUG (a separate copy of the library, for tests): every
// shared-memory offset, TMA coordinate, TMEM column and global index the
// checked kernels compute is compared with its extent before the access. A
// failed check records its source line in the kernel's debug word (the first
// one wins) and the access is skipped; nothing traps. la_device_status reports
// a recorded failure as LA_ERR_INTERNAL. In the ordinary build a check is the
// constant true and its condition is not evaluated.
#ifdef LA_DEBUG
__device__ __forceinline__ bool debug_check(unsigned int *word, bool ok, int line) {
    if (!ok) atomicCAS(word, 0u, (unsigned int)line);
    return ok;
}
#define LA_CHECK(word, cond) ::la::debug_check(&(word), (cond), __LINE__)
#else
#define LA_CHECK(word, cond) true
#endif

// ---------------------------------------------------------------- elements
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// phi(x) = elu(x) + 1: x + 1 for x > 0, e^x otherwise (learnllm m22, "The Math:
// Linear Attention"); the identity when elu1 is false.
__device__ __forceinline__ float phi(float x, bool elu1) {
    if (!elu1) return x;
    return x > 0.f ? x + 1.f : expf(x);
}

// log(sigmoid(x)) without overflow in either tail.
__device__ __forceinline__ float log_sigmoid(float x) {
    return x >= 0.f ? -log1pf(expf(-x)) : x - log1pf(expf(x));
}

// Per-step log-decay of the per-channel gate: log alpha = logsigmoid(g) / 16.
__device__ __forceinline__ float channel_log_decay(float g) { return log_sigmoid(g) * 0.0625f; }

// ---------------------------------------------------------------- launches
struct ChunkArgs {
    const void *q, *k, *v, *gate;
    void *out;
    float *final_state;
    int B, H, L, dk, dv, mode, chunk;
    const float *initial_state;  // [B][H][block] state before the first token, or null (zero)
    int out_f32;                 // tensor-core path only: out is fp32 (identity phi, no normaliser)
    // tensor-core path only, with LA_GATE_CHANNEL: the gate g [B][H][L][dv] decays
    // the value channels (out_t[j] = sum_s (q_t . k_s) v_s[j] prod alpha[j]);
    // the kernel writes out_t / e^{b_t}, b_t the log decay since the chunk start
    int value_gate;
    // tensor-core path only, identity phi, no normaliser, no gate or the head gate:
    // the anti-causal form out_s = sum_{t >= s} gamma^{t-s} (q_s . k_t) v_t, the
    // chunks taken from the end; final_state is then the state before token 0
    int reverse;
    // tensor-core path only (chunk_tc_fuses_epilogue): the RetNet output epilogue
    // applied in the store, out = swish(og) * GroupNorm_h(o); null: none
    const void *gn_ogate;
    const float *gn_weight, *gn_bias;
    float gn_eps;
    // tensor-core path only, normalised causal form without a gate: the first step
    // of the normalised backward in the store. out receives w = dout / den (bf16)
    // and bp_e e_t = -(dout_t . num_t) / den_t^2 (fp32 [B][H][L]); null: none
    const void *bp_dout;
    float *bp_e;
    // tensor-core path only, no gate, normaliser, initial or final state: the score of every
    // (query, key) pair gets e_t added (1: e of the query token, causal; 2: e of
    // the key token, with reverse), bias_e [B][H][L] fp32; 0: none. With elu+1
    // the feature map applies to v alone, and every output row is multiplied by
    // phi'(x_t) = e^min(x_t, 0) of bias_x ([B][H][L][d] bf16, the map's input)
    int bias;
    const float *bias_e;
    const void *bias_x;
};

struct GnArgs {
    const void *x, *ogate;       // [B][H][L][dv]
    const float *weight, *bias;  // [H][dv] or null
    float eps;
    void *out;                   // may be x
    int B, H, L, dv, mode;
};

struct BwdArgs {
    const void *q, *k, *v, *gate, *dout;
    void *grad_q, *grad_k, *grad_v, *grad_g;    // grad_g: [B][H][L][dk] with the channel gate, or null
    int B, H, L, dk, dv, mode;
};

struct DecodeArgs {
    const void *q, *k, *v, *gate;
    float *state;
    void *out;
    int B, H, dk, dv, mode;
};

struct DeltaArgs {
    const void *q, *k, *v, *beta;
    void *out;
    float *final_state;
    int B, H, L, dk, dv, mode;
};

// Each returns LA_OK or an la_status; `launches` counts kernels launched.
int launch_chunk_simt(const ChunkArgs &a, cudaStream_t s, int *launches);
int launch_decode(const DecodeArgs &a, cudaStream_t s, int *launches);
int launch_delta(const DeltaArgs &a, cudaStream_t s, int *launches);
// the delta rule in chunks on the tensor cores (bf16, d_k = d_v = 128)
bool delta_tc_supports(const DeltaArgs &a);
// stream-ordered scratch from the library's own pool on the current device (kept mapped between calls)
int scratch_alloc(void **p, size_t bytes, cudaStream_t s);
// read and clear the device error words of the kernels with bounded waits
int tc_error_take(unsigned int *value);
int delta_tc_error_take(unsigned int *value);
// read and clear the debug words (LA_DEBUG builds: the line of a failed check)
int tc_debug_take(unsigned int *line);
int decode_debug_take(unsigned int *line);
int launch_delta_tc(const DeltaArgs &a, cudaStream_t s, int *launches);
int launch_gn_swish(const GnArgs &a, cudaStream_t s, int *launches);
int launch_bwd(const BwdArgs &a, cudaStream_t s, int *launches);
bool bwd_tc_supports(const BwdArgs &a);
int launch_bwd_tc(const BwdArgs &a, cudaStream_t s, int *launches);
size_t bwd_scratch_bytes(const BwdArgs &a);
int launch_chunk_tc(const ChunkArgs &a, cudaStream_t s, int *launches);
bool chunk_tc_supports(const ChunkArgs &a);
bool chunk_tc_fuses_epilogue(const ChunkArgs &a);
size_t chunk_tc_scratch_bytes(const ChunkArgs &a);
int launch_chunk_tc_into(const ChunkArgs &a, cudaStream_t s, int *launches, void *scratch, size_t scratch_bytes);
// diagnostics: the tensor-core forward (unsplit only) with its producer stopping
// before chunk stall_chunk and every bounded wait limited to wait_ns
int launch_chunk_tc_stalled(const ChunkArgs &a, cudaStream_t s, int *launches, int stall_chunk,
                            unsigned long long wait_ns);

}  // namespace la
