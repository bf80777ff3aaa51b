// la_delta.cu -- the delta rule (DeltaNet), recurrent form, on the CUDA cores.
//
// linear_sparse_attention.py, "delta_rule_recurrent": the state S is d_v x d_k
// (the v k^T orientation of that function) and each token first erases what S
// returns for its key, then writes its value there:
//
//   S <- S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T  =  S - beta_t (S k_t - v_t) k_t^T
//   out_t = S q_t                                      (read after the update)
//
// Every token depends on the state the previous one left, so a sequence is a
// chain of L rank-1 updates; the work is 6 d_k d_v flops a token and the time
// is set by the FMA pipe. One CTA per (b, h); four threads per value row i,
// thread c of the row holding columns [c d_k/4, (c+1) d_k/4) of S in registers.
// Per token: u_i = (S k)_i and o_i = (S q)_i as partial dot products combined
// across the row's four lanes (two shuffles each), and the update
// S_ij -= beta (u_i - v_i) k_j. Tokens come in blocks of kTB: while a block is
// processed, the next one's q, k, v are already being loaded into registers,
// and they are converted to fp32 in shared memory between blocks.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kTB = 32;  // tokens per block

template <int DK, int DV, typename T>
struct DeltaCfg {
    static constexpr int NT = DV * 4;                 // threads
    static constexpr int CPT = DK / 4;                // state columns per thread
    static constexpr int EPC = 16 / sizeof(T);        // elements per 16-byte chunk
    static constexpr int CQ = kTB * DK / EPC;         // chunks of one block of q (or k)
    static constexpr int CV = kTB * DV / EPC;         // chunks of one block of v
    static constexpr int CH = 2 * CQ + CV;            // chunks of a block
    static constexpr int R = (CH + NT - 1) / NT;      // chunks per thread
    // shared memory: fp32 q, k [kTB][DK], v [kTB][DV], beta [kTB], out [kTB][DV]
    static constexpr size_t smem = sizeof(float) * ((size_t)kTB * (2 * DK + 2 * DV) + kTB);
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DV * 4) delta_kernel(DeltaArgs a) {
    using C = DeltaCfg<DK, DV, T>;
    extern __shared__ float dsm[];
    float *qs = dsm, *ks = qs + kTB * DK, *vs = ks + kTB * DK, *bs = vs + kTB * DV, *os = bs + kTB;
    const int tid = threadIdx.x, row = tid >> 2, c = tid & 3;
    const int bh = blockIdx.x, L = a.L;
    const size_t tq = (size_t)bh * L * DK, tv = (size_t)bh * L * DV;
    const T *q = (const T *)a.q + tq, *k = (const T *)a.k + tq, *v = (const T *)a.v + tv;
    const T *beta = (const T *)a.beta + (size_t)bh * L;
    T *out = (T *)a.out + tv;

    float S[C::CPT];
#pragma unroll
    for (int j = 0; j < C::CPT; ++j) S[j] = 0.f;

    // chunk ci of a block: q, then k, then v, each [kTB][d] contiguous in global
    uint4 pre[C::R];
    float bpre = 0.f;
    auto fetch = [&](int t0) {
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
            const int ci = tid + r * C::NT;
            pre[r] = make_uint4(0u, 0u, 0u, 0u);
            if (ci < C::CH) {
                const bool isv = ci >= 2 * C::CQ;
                const int cc = isv ? ci - 2 * C::CQ : ci % C::CQ, d = isv ? DV : DK;
                const int t = (cc * C::EPC) / d;
                if (t0 + t < L) {
                    const T *src = isv ? v + (size_t)t0 * DV : (ci < C::CQ ? q : k) + (size_t)t0 * DK;
                    pre[r] = __ldcs(reinterpret_cast<const uint4 *>(src) + cc);
                }
            }
        }
        if (tid < kTB) bpre = t0 + tid < L ? to_f32(beta[t0 + tid]) : 0.f;
    };
    auto stash = [&]() {
#pragma unroll
        for (int r = 0; r < C::R; ++r) {
            const int ci = tid + r * C::NT;
            if (ci < C::CH) {
                const bool isv = ci >= 2 * C::CQ;
                const int cc = isv ? ci - 2 * C::CQ : ci % C::CQ;
                float *dst = (isv ? vs : (ci < C::CQ ? qs : ks)) + cc * C::EPC;
                const T *e = reinterpret_cast<const T *>(&pre[r]);
#pragma unroll
                for (int x = 0; x < C::EPC; ++x) dst[x] = to_f32(e[x]);
            }
        }
        if (tid < kTB) bs[tid] = bpre;
    };

    fetch(0);
    for (int t0 = 0; t0 < L; t0 += kTB) {
        stash();
        __syncthreads();
        if (t0 + kTB < L) fetch(t0 + kTB);  // in flight while this block runs
        const int nt = min(kTB, L - t0);
        for (int t = 0; t < nt; ++t) {
            const float *kt = ks + t * DK + c * C::CPT, *qt = qs + t * DK + c * C::CPT;
            float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
            for (int j = 0; j < C::CPT; j += 4) {
                const float4 kk = *reinterpret_cast<const float4 *>(kt + j);
                u0 = fmaf(S[j], kk.x, u0);
                u1 = fmaf(S[j + 1], kk.y, u1);
                u2 = fmaf(S[j + 2], kk.z, u2);
                u3 = fmaf(S[j + 3], kk.w, u3);
            }
            float u = (u0 + u1) + (u2 + u3);
            u += __shfl_xor_sync(0xffffffffu, u, 1);
            u += __shfl_xor_sync(0xffffffffu, u, 2);
            const float coef = bs[t] * (u - vs[t * DV + row]);
            float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
            for (int j = 0; j < C::CPT; j += 4) {
                const float4 kk = *reinterpret_cast<const float4 *>(kt + j);
                const float4 qq = *reinterpret_cast<const float4 *>(qt + j);
                S[j] = fmaf(-coef, kk.x, S[j]);
                S[j + 1] = fmaf(-coef, kk.y, S[j + 1]);
                S[j + 2] = fmaf(-coef, kk.z, S[j + 2]);
                S[j + 3] = fmaf(-coef, kk.w, S[j + 3]);
                o0 = fmaf(S[j], qq.x, o0);
                o1 = fmaf(S[j + 1], qq.y, o1);
                o2 = fmaf(S[j + 2], qq.z, o2);
                o3 = fmaf(S[j + 3], qq.w, o3);
            }
            float o = (o0 + o1) + (o2 + o3);
            o += __shfl_xor_sync(0xffffffffu, o, 1);
            o += __shfl_xor_sync(0xffffffffu, o, 2);
            if (c == 0) os[t * DV + row] = o;
        }
        __syncthreads();
        // the block's outputs, coalesced
        for (int i = tid; i < nt * DV; i += C::NT) out[(size_t)t0 * DV + i] = from_f32<T>(os[i]);
    }
    if (a.final_state) {
        float *fs = a.final_state + (size_t)bh * DV * DK + (size_t)row * DK + c * C::CPT;
#pragma unroll
        for (int j = 0; j < C::CPT; j += 4)
            *reinterpret_cast<float4 *>(fs + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_dkdv(const DeltaArgs &a, cudaStream_t s) {
    using C = DeltaCfg<DK, DV, T>;
    auto kern = delta_kernel<DK, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((unsigned)((long)a.B * a.H)), C::NT, C::smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const DeltaArgs &a, cudaStream_t s) {
#define LA_DELTA_CASE(DKV, DVV) \
    if (a.dk == DKV && a.dv == DVV) return launch_dkdv<DKV, DVV, T>(a, s);
#define LA_DELTA_ROW(DKV) LA_DELTA_CASE(DKV, 16) LA_DELTA_CASE(DKV, 32) LA_DELTA_CASE(DKV, 64) LA_DELTA_CASE(DKV, 128)
    LA_DELTA_ROW(16)
    LA_DELTA_ROW(32)
    LA_DELTA_ROW(64)
    LA_DELTA_ROW(128)
#undef LA_DELTA_ROW
#undef LA_DELTA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

int launch_delta(const DeltaArgs &a, cudaStream_t s, int *launches) {
    cudaError_t e = (a.mode & LA_DTYPE_F32) ? launch_t<float>(a, s) : launch_t<__nv_bfloat16>(a, s);
    if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    return LA_OK;
}

}  // namespace la
