// la_simt.cu -- the general chunkwise forward on CUDA cores (fp32 arithmetic).
//
// It runs every case the tensor-core kernel does not: fp32 inputs (whose
// tolerance rules out TF32 tensor cores), any chunk in 1..128 that fits on
// chip, any d_k, d_v in {16, 32, 64, 128}, and every mode. It follows the
// chunkwise form of learnllm m22 "The Three Faces of Retention" and
// linear_sparse_attention.py linear_attn_chunkwise, with the decay written
// exactly per element (no factoring), so it holds for any gate value:
//
//   P_ij   = sum_d phi(q_i)[d] phi(k_j)[d] D_ij[d],   j <= i inside the chunk,
//            D_ij[d] = exp(b_i[d] - b_j[d]) (gated), gamma^(i-j) (retention), 1
//   out_i  = sum_j P_ij v_j + (phi(q_i) * e^{b_i}) S          [/ den_i]
//   den_i  = sum_j P_ij + (phi(q_i) * e^{b_i}) . z
//   S      <- diag(e^{b_last}) S + sum_s (phi(k_s) * e^{b_last - b_s}) v_s^T
//   z      <- e^{b_last} * z + sum_s phi(k_s) * e^{b_last - b_s}
//
// with b_t the inclusive running sum of log A inside the chunk (for retention
// gamma^(t+1), gamma^(c-1-s) and gamma^c, c the chunk's actual length).
//
// One CTA per (b, h, d_v tile); the d_k x d_v-tile state stays in shared
// memory across the sequential loop over chunks.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kSimtThreads = 256;

struct SimtPlan {
    int dvt;        // d_v columns per CTA
    size_t smem;    // bytes of dynamic shared memory
};

__host__ __device__ inline size_t simt_smem_floats(int C, int dk, int dvt, bool gated_channel) {
    const size_t ld = (size_t)dk + 1;
    return 2 * C * ld + (gated_channel ? C * ld : 0) + (size_t)C * dvt + (size_t)C * C +
           (size_t)dk * dvt + 2 * (size_t)dk + (size_t)C;
}

template <typename T>
__global__ void __launch_bounds__(kSimtThreads) chunk_simt_kernel(ChunkArgs a, int dvt) {
    extern __shared__ float sm[];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh = blockIdx.x, h = bh % a.H;
    const int col0 = blockIdx.y * dvt;
    const int C = a.chunk, dk = a.dk, dv = a.dv, L = a.L;
    const int ld = dk + 1;
    const bool elu1 = a.mode & LA_PHI_ELU1, norm = a.mode & LA_NORMALIZE;
    const bool ghead = a.mode & LA_GATE_HEAD, gchan = a.mode & LA_GATE_CHANNEL;
    const bool gated = ghead || gchan;

    float *Qs = sm;                              // [C][ld]   phi(q), then phi(q) e^{b_t}
    float *Ks = Qs + (size_t)C * ld;             // [C][ld]   phi(k), then phi(k) e^{b_c - b_s}
    float *Bs = Ks + (size_t)C * ld;             // [C][ld]   b_t (gated channel only)
    float *Vs = Bs + (gchan ? (size_t)C * ld : 0);  // [C][dvt]
    float *Ps = Vs + (size_t)C * dvt;            // [C][C]
    float *Ss = Ps + (size_t)C * C;              // [dk][dvt]
    float *zs = Ss + (size_t)dk * dvt;           // [dk]
    float *Ad = zs + dk;                         // [dk] decay over the chunk
    float *dens = Ad + dk;                       // [C]

    const size_t qoff = (size_t)bh * L * dk;
    const T *q = (const T *)a.q + qoff;
    const T *k = (const T *)a.k + qoff;
    const T *v = (const T *)a.v + (size_t)bh * L * dv;
    const T *g = gchan ? (const T *)a.gate + qoff : nullptr;
    const float gamma = ghead ? ((const float *)a.gate)[h] : 1.f;
    T *out = (T *)a.out + (size_t)bh * L * dv;

    // the state before the first token: zero, or this CTA's columns of the given one
    const float *S0 = a.initial_state ? a.initial_state + (size_t)bh * ((size_t)dk * dv + (norm ? dk : 0)) : nullptr;
    for (int i = tid; i < dk * dvt; i += nt) Ss[i] = S0 ? S0[(size_t)(i / dvt) * dv + col0 + i % dvt] : 0.f;
    for (int i = tid; i < dk; i += nt) zs[i] = (S0 && norm) ? S0[(size_t)dk * dv + i] : 0.f;
    __syncthreads();

    for (int t0 = 0; t0 < L; t0 += C) {
        const int c = min(C, L - t0);
        // (1) load the chunk, applying the feature map
        for (int idx = tid; idx < c * dk; idx += nt) {
            const int t = idx / dk, d = idx - t * dk;
            const size_t gi = (size_t)(t0 + t) * dk + d;
            Qs[t * ld + d] = phi(to_f32(q[gi]), elu1);
            Ks[t * ld + d] = phi(to_f32(k[gi]), elu1);
        }
        for (int idx = tid; idx < c * dvt; idx += nt) {
            const int t = idx / dvt, j = idx - t * dvt;
            Vs[idx] = to_f32(v[(size_t)(t0 + t) * dv + col0 + j]);
        }
        if (gchan) {
            // inclusive running sum of log alpha along the chunk, per channel
            for (int d = tid; d < dk; d += nt) {
                float b = 0.f;
                for (int t = 0; t < c; ++t) {
                    b += channel_log_decay(to_f32(g[(size_t)(t0 + t) * dk + d]));
                    Bs[t * ld + d] = b;
                }
            }
        }
        __syncthreads();

        // (2) masked intra-chunk scores, diagonal included
        for (int idx = tid; idx < c * c; idx += nt) {
            const int i = idx / c, j = idx - i * c;
            float acc = 0.f;
            if (j <= i) {
                const float *qi = Qs + i * ld, *kj = Ks + j * ld;
                if (gchan) {
                    const float *bi = Bs + i * ld, *bj = Bs + j * ld;
                    for (int d = 0; d < dk; ++d) acc += qi[d] * kj[d] * expf(bi[d] - bj[d]);
                } else {
                    for (int d = 0; d < dk; ++d) acc += qi[d] * kj[d];
                    if (ghead) acc *= powf(gamma, (float)(i - j));
                }
            }
            Ps[i * C + j] = acc;
        }
        __syncthreads();

        // (3) decay the query rows from the chunk start and the key rows to
        // the chunk end; the decay over the whole chunk
        if (gated) {
            for (int idx = tid; idx < c * dk; idx += nt) {
                const int t = idx / dk, d = idx - t * dk;
                float fq, fk;
                if (gchan) {
                    const float bt = Bs[t * ld + d], bc = Bs[(c - 1) * ld + d];
                    fq = expf(bt);
                    fk = expf(bc - bt);
                } else {
                    fq = powf(gamma, (float)(t + 1));
                    fk = powf(gamma, (float)(c - 1 - t));
                }
                Qs[t * ld + d] *= fq;
                Ks[t * ld + d] *= fk;
            }
            for (int d = tid; d < dk; d += nt)
                Ad[d] = gchan ? expf(Bs[(c - 1) * ld + d]) : powf(gamma, (float)c);
        }
        __syncthreads();
        if (norm) {
            for (int i = tid; i < c; i += nt) {
                float s = 0.f;
                for (int j = 0; j <= i; ++j) s += Ps[i * C + j];
                for (int d = 0; d < dk; ++d) s += Qs[i * ld + d] * zs[d];
                dens[i] = s;
            }
            __syncthreads();
        }

        // (4) outputs: intra-chunk term plus the carried state
        for (int idx = tid; idx < c * dvt; idx += nt) {
            const int i = idx / dvt, j = idx - i * dvt;
            float acc = 0.f;
            for (int s = 0; s <= i; ++s) acc += Ps[i * C + s] * Vs[s * dvt + j];
            const float *qi = Qs + i * ld;
            for (int d = 0; d < dk; ++d) acc += qi[d] * Ss[d * dvt + j];
            if (norm) acc = acc / dens[i];
            out[(size_t)(t0 + i) * dv + col0 + j] = from_f32<T>(acc);
        }
        __syncthreads();

        // (5) advance the state over the chunk
        for (int idx = tid; idx < dk * dvt; idx += nt) {
            const int d = idx / dvt, j = idx - d * dvt;
            float acc = gated ? Ad[d] * Ss[idx] : Ss[idx];
            for (int s = 0; s < c; ++s) acc += Ks[s * ld + d] * Vs[s * dvt + j];
            Ss[idx] = acc;
        }
        if (norm) {
            for (int d = tid; d < dk; d += nt) {
                float zz = gated ? Ad[d] * zs[d] : zs[d];
                for (int s = 0; s < c; ++s) zz += Ks[s * ld + d];
                zs[d] = zz;
            }
        }
        __syncthreads();
    }

    if (a.final_state) {
        const size_t blk = (size_t)dk * dv + (norm ? dk : 0);
        float *fs = a.final_state + (size_t)bh * blk;
        for (int idx = tid; idx < dk * dvt; idx += nt) {
            const int d = idx / dvt, j = idx - d * dvt;
            fs[(size_t)d * dv + col0 + j] = Ss[idx];
        }
        if (norm && blockIdx.y == 0)
            for (int d = tid; d < dk; d += nt) fs[(size_t)dk * dv + d] = zs[d];
    }
}

int plan_simt(const ChunkArgs &a, SimtPlan *p) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return LA_ERR_CUDA;
    const bool gchan = a.mode & LA_GATE_CHANNEL;
    for (int dvt = a.dv < 64 ? a.dv : 64; dvt >= 16; dvt /= 2) {
        const size_t bytes = simt_smem_floats(a.chunk, a.dk, dvt, gchan) * sizeof(float);
        if (bytes <= (size_t)optin) {
            p->dvt = dvt;
            p->smem = bytes;
            return LA_OK;
        }
    }
    return LA_ERR_UNSUPPORTED;
}

}  // namespace

int launch_chunk_simt(const ChunkArgs &a, cudaStream_t s, int *launches) {
    SimtPlan p;
    int rc = plan_simt(a, &p);
    if (rc != LA_OK) return rc;
    dim3 grid((unsigned)((long)a.B * a.H), (unsigned)(a.dv / p.dvt));
    cudaError_t e;
    if (a.mode & LA_DTYPE_F32) {
        e = cudaFuncSetAttribute(chunk_simt_kernel<float>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return LA_ERR_CUDA;
        chunk_simt_kernel<float><<<grid, kSimtThreads, p.smem, s>>>(a, p.dvt);
    } else {
        e = cudaFuncSetAttribute(chunk_simt_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return LA_ERR_CUDA;
        chunk_simt_kernel<__nv_bfloat16><<<grid, kSimtThreads, p.smem, s>>>(a, p.dvt);
    }
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    return LA_OK;
}

}  // namespace la
