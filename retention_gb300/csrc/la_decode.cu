// la_decode.cu -- the single-token recurrent decode step, in place on the state.
//
// learnllm m22 "Code: The Two Faces" (LinearAttentionState.step: fold one
// token into the running state, constant work per token) and insideout lesson
// 16 (S <- S + k v^T, z <- z + k, out = q^T S / (q . z)), with the gate A of
// the unified recurrence:
//
//   S <- diag(A) S + phi(k) v^T,  z <- A * z + phi(k),
//   out = phi(q)^T S  [ / (phi(q) . z) ]          (read after the update)
//
// The step is bound by HBM traffic: every (b, h) reads and writes its fp32
// d_k x d_v state once (64 KiB at d = 128). One CTA per (b, h); each thread
// owns one 16-byte column group of the state across d_k / row_groups rows,
// issues all of its state loads before any arithmetic, updates the rows in
// registers, writes them back with streaming (evict-first) stores and keeps a
// partial phi(q)^T S; partials are summed across row groups in shared memory
// and phi(q) . z is a warp-shuffle reduction.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kDecThreads = 256;
// Three CTAs per SM (at most 85 registers a thread, no spills at d = 128):
// while one CTA updates and stores its state, the others have their loads in
// flight. Two CTAs per SM left the step at 85 % of the HBM copy rate, three
// reach 97 %.
constexpr int kDecCtasPerSm = 3;

__device__ unsigned int g_dec_debug;  // LA_DEBUG: source line of the first failed bounds check
#ifdef LA_DEBUG
#define DEC_CHECK(cond) LA_CHECK(g_dec_debug, cond)
#else
#define DEC_CHECK(cond) true
#endif

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm) decode_kernel(DecodeArgs a) {
    constexpr int C4 = DV / 4;                  // 16-byte column groups per row
    constexpr int RG = kDecThreads / C4;        // row groups
    constexpr int RPT = (DK + RG - 1) / RG;     // rows per thread
    __shared__ float qf[DK], kf[DK], ad[DK];
    __shared__ float4 red[RG][C4];
    __shared__ float den_s;

    const int tid = threadIdx.x;
    const int bh = blockIdx.x, h = bh % a.H;
    const bool elu1 = a.mode & LA_PHI_ELU1, norm = a.mode & LA_NORMALIZE;
    const bool ghead = a.mode & LA_GATE_HEAD, gchan = a.mode & LA_GATE_CHANNEL;
    const size_t blk = (size_t)DK * DV + (norm ? DK : 0);
    float *S = a.state + (size_t)bh * blk;
    const int c4 = tid % C4, rg = tid / C4;
    // (LA_DEBUG) this CTA's state block and token rows lie inside the arrays
    [[maybe_unused]] const size_t nbh = (size_t)a.B * a.H;
    const bool in = DEC_CHECK((size_t)bh < nbh && h < a.H && c4 * 4 + 3 < DV && rg < RG);

    // all state loads first: RPT independent 16-byte loads per thread
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = rg + r * RG;
        if (row < DK && in) s[r] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)row * DV) + c4);
    }

    const T *q = (const T *)a.q + (size_t)bh * DK;
    const T *k = (const T *)a.k + (size_t)bh * DK;
    const T *v = (const T *)a.v + (size_t)bh * DV;
    const float gamma = ghead && in ? ((const float *)a.gate)[h] : 1.f;
    for (int d = tid; d < DK && in; d += kDecThreads) {
        qf[d] = phi(to_f32(q[d]), elu1);
        kf[d] = phi(to_f32(k[d]), elu1);
        float aa = gamma;
        if (gchan) aa = expf(channel_log_decay(to_f32(((const T *)a.gate)[(size_t)bh * DK + d])));
        ad[d] = aa;
    }
    const float v0 = in ? to_f32(v[c4 * 4 + 0]) : 0.f, v1 = in ? to_f32(v[c4 * 4 + 1]) : 0.f;
    const float v2 = in ? to_f32(v[c4 * 4 + 2]) : 0.f, v3 = in ? to_f32(v[c4 * 4 + 3]) : 0.f;
    __syncthreads();

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int row = rg + r * RG;
        if (row < DK && in) {
            const float aa = ad[row], kk = kf[row], qq = qf[row];
            float4 x = s[r];
            x.x = aa * x.x + kk * v0;
            x.y = aa * x.y + kk * v1;
            x.z = aa * x.z + kk * v2;
            x.w = aa * x.w + kk * v3;
            __stcs(reinterpret_cast<float4 *>(S + (size_t)row * DV) + c4, x);
            acc.x += qq * x.x;
            acc.y += qq * x.y;
            acc.z += qq * x.z;
            acc.w += qq * x.w;
        }
    }
    red[rg][c4] = acc;

    if (norm && tid < 32 && in) {
        float part = 0.f;
        float *z = S + (size_t)DK * DV;
        for (int d = tid; d < DK; d += 32) {
            const float zz = ad[d] * z[d] + kf[d];
            z[d] = zz;
            part += qf[d] * zz;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (tid == 0) den_s = part;
    }
    __syncthreads();

    if (tid < DV) {
        const int cg = tid >> 2, comp = tid & 3;
        float sum = 0.f;
#pragma unroll 8
        for (int r = 0; r < RG; ++r) {
            const float4 p = red[r][cg];
            sum += comp == 0 ? p.x : comp == 1 ? p.y : comp == 2 ? p.z : p.w;
        }
        if (norm) sum = sum / den_s;
        if (in) ((T *)a.out)[(size_t)bh * DV + tid] = from_f32<T>(sum);
    }
}

template <typename T>
cudaError_t launch_t(const DecodeArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)((long)a.B * a.H));
#define LA_DEC_CASE(DKV, DVV)                                                   \
    if (a.dk == DKV && a.dv == DVV) {                                           \
        decode_kernel<DKV, DVV, T><<<grid, kDecThreads, 0, s>>>(a);            \
        return cudaGetLastError();                                              \
    }
#define LA_DEC_ROW(DKV) LA_DEC_CASE(DKV, 16) LA_DEC_CASE(DKV, 32) LA_DEC_CASE(DKV, 64) LA_DEC_CASE(DKV, 128)
    LA_DEC_ROW(16)
    LA_DEC_ROW(32)
    LA_DEC_ROW(64)
    LA_DEC_ROW(128)
#undef LA_DEC_ROW
#undef LA_DEC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

// The decode kernel's debug word (LA_DEBUG builds: the source line of the
// first failed bounds check; always 0 otherwise), read and cleared.
int decode_debug_take(unsigned int *line) {
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(line, g_dec_debug, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_dec_debug, &zero, sizeof(unsigned int)) != cudaSuccess)
        return LA_ERR_CUDA;
    return LA_OK;
}

int launch_decode(const DecodeArgs &a, cudaStream_t s, int *launches) {
    cudaError_t e = (a.mode & LA_DTYPE_F32) ? launch_t<float>(a, s) : launch_t<__nv_bfloat16>(a, s);
    if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    return LA_OK;
}

}  // namespace la
