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
// is set by the FMA pipe. One CTA per (b, h). A thread holds a 2-row x 16-column
// tile of S in registers (rows = value dimensions); the d_k/16 threads of a row
// group are consecutive lanes. Per token: u = S k and o = S q as partial dot
// products combined across those lanes (shuffles), and the update
// S_ij -= beta (u_i - v_i) k_j. Each k and q value a thread loads serves its two
// rows, and the 16-column segments of the shared k and q rows are padded by
// four floats so that the lanes of a quarter warp read eight different bank
// groups. Tokens come in blocks of kTB: while a block is processed, the next
// one's q, k, v are already being loaded into registers, and they are converted
// to fp32 in shared memory between blocks.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kTB = 32;  // tokens per block

template <int DK, int DV, typename T>
struct DeltaCfg {
    static constexpr int RPT = 2, CPT = 16;           // rows and columns of S per thread
    static constexpr int NCG = DK / CPT;              // column groups (lanes per row group)
    static constexpr int NTC = (DV / RPT) * NCG;      // threads holding S
    static constexpr int NT = NTC > 256 ? NTC : 256;  // threads (the rest only load and store)
    static constexpr int SEG = CPT + 4;               // padded 16-column segment
    static constexpr int ROWP = NCG * SEG;            // padded q / k row
    static constexpr unsigned MASK = NTC >= 32 ? 0xffffffffu : ((1u << NTC) - 1u);
    static constexpr int EPC = 16 / sizeof(T);        // elements per 16-byte chunk
    static constexpr int CQ = kTB * DK / EPC;         // chunks of one block of q (or k)
    static constexpr int CV = kTB * DV / EPC;         // chunks of one block of v
    static constexpr int CH = 2 * CQ + CV;            // chunks of a block
    static constexpr int R = (CH + NT - 1) / NT;      // chunks per thread
    // shared memory: fp32 q, k [kTB][ROWP], v [kTB][DV], beta [kTB], out [kTB][DV]
    static constexpr size_t smem = sizeof(float) * ((size_t)kTB * (2 * ROWP + 2 * DV) + kTB);
};

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DeltaCfg<DK, DV, T>::NT) delta_kernel(DeltaArgs a) {
    using C = DeltaCfg<DK, DV, T>;
    extern __shared__ float dsm[];
    float *qs = dsm, *ks = qs + kTB * C::ROWP, *vs = ks + kTB * C::ROWP, *bs = vs + kTB * DV, *os = bs + kTB;
    const int tid = threadIdx.x, rg = tid / C::NCG, cg = tid % C::NCG;
    const int bh = blockIdx.x, L = a.L;
    const size_t tq = (size_t)bh * L * DK, tv = (size_t)bh * L * DV;
    const T *q = (const T *)a.q + tq, *k = (const T *)a.k + tq, *v = (const T *)a.v + tv;
    const T *beta = (const T *)a.beta + (size_t)bh * L;
    T *out = (T *)a.out + tv;

    float S[C::RPT][C::CPT];
#pragma unroll
    for (int r = 0; r < C::RPT; ++r)
#pragma unroll
        for (int j = 0; j < C::CPT; ++j) S[r][j] = 0.f;

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
                float *dst;
                if (isv) {
                    dst = vs + cc * C::EPC;
                } else {
                    // element e of token t sits at t ROWP + (e / 16) SEG + e % 16
                    const int e0 = cc * C::EPC, t = e0 / DK, e = e0 % DK;
                    dst = (ci < C::CQ ? qs : ks) + t * C::ROWP + (e / C::CPT) * C::SEG + e % C::CPT;
                }
                const T *el = reinterpret_cast<const T *>(&pre[r]);
#pragma unroll
                for (int x = 0; x < C::EPC; ++x) dst[x] = to_f32(el[x]);
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
        for (int t = 0; t < nt && tid < C::NTC; ++t) {
            float kk[C::CPT], qq[C::CPT];
            const float *kt = ks + t * C::ROWP + cg * C::SEG, *qt = qs + t * C::ROWP + cg * C::SEG;
#pragma unroll
            for (int j = 0; j < C::CPT; j += 4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kt + j);
                const float4 q4 = *reinterpret_cast<const float4 *>(qt + j);
                kk[j] = k4.x, kk[j + 1] = k4.y, kk[j + 2] = k4.z, kk[j + 3] = k4.w;
                qq[j] = q4.x, qq[j + 1] = q4.y, qq[j + 2] = q4.z, qq[j + 3] = q4.w;
            }
            float u[C::RPT];
#pragma unroll
            for (int r = 0; r < C::RPT; ++r) {
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < C::CPT; j += 2) {
                    a0 = fmaf(S[r][j], kk[j], a0);
                    a1 = fmaf(S[r][j + 1], kk[j + 1], a1);
                }
                u[r] = a0 + a1;
            }
#pragma unroll
            for (int off = 1; off < C::NCG; off <<= 1)
#pragma unroll
                for (int r = 0; r < C::RPT; ++r) u[r] += __shfl_xor_sync(C::MASK, u[r], off);
            float vr[C::RPT];
#pragma unroll
            for (int r = 0; r < C::RPT; ++r) vr[r] = vs[t * DV + rg * C::RPT + r];
            const float bt = bs[t];
            float o[C::RPT];
#pragma unroll
            for (int r = 0; r < C::RPT; ++r) {
                const float coef = bt * (u[r] - vr[r]);
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < C::CPT; j += 2) {
                    S[r][j] = fmaf(-coef, kk[j], S[r][j]);
                    S[r][j + 1] = fmaf(-coef, kk[j + 1], S[r][j + 1]);
                    a0 = fmaf(S[r][j], qq[j], a0);
                    a1 = fmaf(S[r][j + 1], qq[j + 1], a1);
                }
                o[r] = a0 + a1;
            }
#pragma unroll
            for (int off = 1; off < C::NCG; off <<= 1)
#pragma unroll
                for (int r = 0; r < C::RPT; ++r) o[r] += __shfl_xor_sync(C::MASK, o[r], off);
            if (cg == 0)
#pragma unroll
                for (int r = 0; r < C::RPT; ++r) os[t * DV + rg * C::RPT + r] = o[r];
        }
        __syncthreads();
        // the block's outputs, coalesced
        for (int i = tid; i < nt * DV; i += C::NT) out[(size_t)t0 * DV + i] = from_f32<T>(os[i]);
    }
    if (a.final_state && tid < C::NTC) {
#pragma unroll
        for (int r = 0; r < C::RPT; ++r) {
            float *fs = a.final_state + (size_t)bh * DV * DK + (size_t)(rg * C::RPT + r) * DK + cg * C::CPT;
#pragma unroll
            for (int j = 0; j < C::CPT; j += 4)
                *reinterpret_cast<float4 *>(fs + j) = make_float4(S[r][j], S[r][j + 1], S[r][j + 2], S[r][j + 3]);
        }
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
