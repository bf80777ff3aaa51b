// la_bwd.cu -- gradients of the forward pass (from S_0 = 0) with respect to q,
// k, v and the per-channel gate, on the CUDA cores in fp32.
//
// The pages motivate the chunkwise form "for training" (learnllm m22, "The
// Three Faces of Retention") but give no gradient; this is the chain rule on
// the recurrence S_t = diag(a_t) S_{t-1} + K_t v_t^T, out_t = S_t^T Q_t
// (Q = phi(q), K = phi(k); with the normaliser, out = num / den and the
// value is widened by a column of ones whose state is z):
//
//   w_t  = dout_t                      e_t = 0                      (no normaliser)
//   w_t  = dout_t / den_t              e_t = -(dout_t . out_t) / den_t
//                                          = -(Q_t . S_t w_t) / den_t
//   dQ_t = S_t w_t + z_t e_t                                    forward sweep
//   dS_t = diag(a_{t+1}) dS_{t+1} + Q_t w_t^T,  dz_t likewise with e_t   reverse
//   dK_t = dS_t v_t + dz_t,   dv_t = dS_t^T K_t
//   dq = dQ * phi'(q),  dk = dK * phi'(k)
//   dg_r = sigmoid(-g_r) / 16 * sum_{t >= r} (Q_t * dQ_t - K_t * dK_t)
//
// (the last line: every term of the output carries e^{B_t - B_s} with
// B_t = sum_{r<=t} log a_r, so dl/dB_t = Q_t dQ_t - K_t dK_t, and log a_r
// enters every B_t with t >= r).
//
// e_t is formed from S_t w_t (the dQ sweep's own product) rather than from the
// forward's stored output, whose rounding the difference S_t w_t + z_t e_t
// would magnify.
//
// Kernels, in stream order: the normaliser's den_t (only with it); three
// sweeps that each carry one matrix in registers through the sequence, one
// rank-1 update and one matrix-vector product per token, so that every
// reduction stays inside a thread's row group:
//   dQ sweep  rows = key channels (16 per CTA), columns = value channels, forward
//   (e_t, one warp per token, with the normaliser)
//   dK sweep  rows = key channels, columns = value channels, reverse
//   dV sweep  rows = value channels, columns = key channels (dS transposed), reverse
// and a last pass that adds z_t e_t, applies phi' and forms the gate gradient.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kTB = 16;        // tokens per staged block
constexpr int kRows = 16;      // matrix rows per CTA
constexpr int kFinThreads = 128;

struct BwdParams {
    const void *q, *k, *v, *gate, *dout;
    void *grad_q, *grad_k, *grad_v, *grad_g;
    float *gq, *gk;            // [BH][L][dk] fp32: gradients with respect to Q = phi(q), K = phi(k)
    float *den_inv, *ecol;     // [BH][L]: 1 / den_t and e_t (normaliser only)
    int B, H, L, dk, dv, mode;
};

__device__ __forceinline__ float dphi(float x, bool elu1) { return (elu1 && x <= 0.f) ? __expf(x) : 1.f; }

// gate value of key channel d at token t of sequence bh (1 without a gate)
template <typename T>
__device__ __forceinline__ float gate_value(const BwdParams &p, int bh, int t, int d) {
    if (p.mode & LA_GATE_CHANNEL)
        return __expf(channel_log_decay(to_f32(static_cast<const T *>(p.gate)[((size_t)bh * p.L + t) * p.dk + d])));
    if (p.mode & LA_GATE_HEAD) return static_cast<const float *>(p.gate)[bh % p.H];
    return 1.f;
}

// ---------------------------------------------------------------- normaliser
// den_t = Q_t . z_t with z_t = a_t * z_{t-1} + K_t. One CTA per sequence, one
// thread per key channel; tokens in blocks of kTB, the per-channel products
// reduced per token through shared memory.
template <typename T>
__global__ void __launch_bounds__(128) bwd_den_kernel(BwdParams p) {
    __shared__ float prod[kTB][129];
    const int bh = blockIdx.x, i = threadIdx.x, dk = p.dk, L = p.L;
    const bool elu1 = p.mode & LA_PHI_ELU1;
    const T *q = static_cast<const T *>(p.q) + (size_t)bh * L * dk;
    const T *k = static_cast<const T *>(p.k) + (size_t)bh * L * dk;
    float z = 0.f;
    for (int t0 = 0; t0 < L; t0 += kTB) {
        const int nt = min(kTB, L - t0);
        if (i < dk)
            for (int tt = 0; tt < nt; ++tt) {
                const int t = t0 + tt;
                z = gate_value<T>(p, bh, t, i) * z + phi(to_f32(k[(size_t)t * dk + i]), elu1);
                prod[tt][i] = phi(to_f32(q[(size_t)t * dk + i]), elu1) * z;
            }
        __syncthreads();
        // warp w reduces tokens w, w + 4, ...
        const int warp = i >> 5, lane = i & 31;
        for (int tt = warp; tt < nt; tt += 4) {
            float den = 0.f;
            for (int c = lane; c < dk; c += 32) den += prod[tt][c];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
            if (lane == 0) p.den_inv[(size_t)bh * L + t0 + tt] = 1.f / den;
        }
        __syncthreads();
    }
}

// e_t = -(Q_t . gq_t) / den_t, gq_t = S_t w_t from the dQ sweep: one warp per
// token.
template <typename T>
__global__ void __launch_bounds__(256) bwd_ecol_kernel(BwdParams p) {
    const long w = ((long)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, dk = p.dk;
    if (w >= (long)p.B * p.H * p.L) return;
    const bool elu1 = p.mode & LA_PHI_ELU1;
    const T *q = static_cast<const T *>(p.q) + (size_t)w * dk;
    const float *gq = p.gq + (size_t)w * dk;
    float s = 0.f;
    for (int c = lane; c < dk; c += 32) s += phi(to_f32(q[c]), elu1) * gq[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) p.ecol[w] = -s * p.den_inv[w];
}

// ---------------------------------------------------------------- sweeps
enum { kSweepDQ = 0, kSweepDK = 1, kSweepDV = 2 };

// C columns per row (dv for the dQ and dK sweeps, dk for the dV sweep). A
// compute thread holds rows 2 rg, 2 rg + 1 of the CTA's 16 and columns
// 16 cg .. 16 cg + 15; the C / 16 threads of a row group are consecutive lanes.
template <int SW, int C>
struct SweepCfg {
    static constexpr int NCG = C / 16;
    static constexpr int NTC = (kRows / 2) * NCG;
    static constexpr int NT = NTC < 64 ? 64 : NTC;
    static constexpr int SEG = 20;                 // padded 16-column segment
    static constexpr int ROWP = NCG * SEG;
    static constexpr unsigned MASK = NTC >= 32 ? 0xffffffffu : ((1u << NTC) - 1u);
};

template <int SW, int C, typename T>
__global__ void __launch_bounds__(SweepCfg<SW, C>::NT) bwd_sweep_kernel(BwdParams p) {
    using G = SweepCfg<SW, C>;
    constexpr bool REV = SW != kSweepDQ;
    __shared__ float xs[kTB][kRows];        // row-side factor of the rank-1 update
    __shared__ float dr[kTB][kRows];        // per-row decay (dQ, dK sweeps)
    __shared__ __align__(16) float ys[kTB][G::ROWP];   // column-side factor
    __shared__ __align__(16) float us[kTB][G::ROWP];   // contracted vector
    __shared__ __align__(16) float dc[kTB][SW == kSweepDV ? G::ROWP : 4];  // per-column decay (dV sweep)
    __shared__ float es[kTB];
    __shared__ float os[kTB][kRows];
    const int tid = threadIdx.x, rg = tid / G::NCG, cg = tid % G::NCG;
    const bool compute = tid < G::NTC;
    const int bh = blockIdx.x, row0 = blockIdx.y * kRows;
    const int L = p.L, dk = p.dk, dv = p.dv;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE;
    const bool gchan = p.mode & LA_GATE_CHANNEL, ghead = p.mode & LA_GATE_HEAD;
    const float gamma = ghead ? static_cast<const float *>(p.gate)[bh % p.H] : 1.f;
    const T *q = static_cast<const T *>(p.q) + (size_t)bh * L * dk;
    const T *k = static_cast<const T *>(p.k) + (size_t)bh * L * dk;
    const T *v = static_cast<const T *>(p.v) + (size_t)bh * L * dv;
    const T *d = static_cast<const T *>(p.dout) + (size_t)bh * L * dv;
    const float *dinv = norm ? p.den_inv + (size_t)bh * L : nullptr;
    const float *ec = norm ? p.ecol + (size_t)bh * L : nullptr;
    auto colp = [](int c) { return (c >> 4) * G::SEG + (c & 15); };

    float M[2][16], zr[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < 16; ++j) M[r][j] = 0.f;

    const int nblk = (L + kTB - 1) / kTB;
    for (int bi = 0; bi < nblk; ++bi) {
        const int blk = REV ? nblk - 1 - bi : bi, t0 = blk * kTB, nt = min(kTB, L - t0);
        __syncthreads();  // the previous block's shared rows are consumed
        // stage the block: decays of token t (dQ sweep) or t + 1 (reverse sweeps)
        for (int x = tid; x < nt * kRows; x += G::NT) {
            const int tt = x / kRows, r = x % kRows, t = t0 + tt, row = row0 + r;
            float xv;
            if (SW == kSweepDQ) xv = phi(to_f32(k[(size_t)t * dk + row]), elu1);
            else if (SW == kSweepDK) xv = phi(to_f32(q[(size_t)t * dk + row]), elu1);
            else xv = to_f32(d[(size_t)t * dv + row]) * (norm ? dinv[t] : 1.f);
            xs[tt][r] = xv;
            if (SW != kSweepDV && gchan) {
                const int tg = SW == kSweepDQ ? t : t + 1;
                dr[tt][r] = tg < L ? gate_value<T>(p, bh, tg, row) : 1.f;
            }
        }
        for (int x = tid; x < nt * C; x += G::NT) {
            const int tt = x / C, c = x % C, t = t0 + tt;
            float yv, uv;
            if (SW == kSweepDQ) {
                yv = to_f32(v[(size_t)t * dv + c]);
                uv = to_f32(d[(size_t)t * dv + c]) * (norm ? dinv[t] : 1.f);
            } else if (SW == kSweepDK) {
                yv = to_f32(d[(size_t)t * dv + c]) * (norm ? dinv[t] : 1.f);
                uv = to_f32(v[(size_t)t * dv + c]);
            } else {
                yv = phi(to_f32(q[(size_t)t * dk + c]), elu1);
                uv = phi(to_f32(k[(size_t)t * dk + c]), elu1);
                if (gchan) dc[tt][colp(c)] = t + 1 < L ? gate_value<T>(p, bh, t + 1, c) : 1.f;
            }
            ys[tt][colp(c)] = yv;
            us[tt][colp(c)] = uv;
        }
        if (norm && SW == kSweepDK)
            for (int x = tid; x < nt; x += G::NT) es[x] = ec[t0 + x];
        __syncthreads();
        if (compute) {
            for (int s = 0; s < nt; ++s) {
                const int tt = REV ? nt - 1 - s : s;
                float yy[16], uu[16], dd[16];
                const float *yp = &ys[tt][cg * G::SEG], *up = &us[tt][cg * G::SEG];
#pragma unroll
                for (int j = 0; j < 16; j += 4) {
                    const float4 y4 = *reinterpret_cast<const float4 *>(yp + j);
                    const float4 u4 = *reinterpret_cast<const float4 *>(up + j);
                    yy[j] = y4.x, yy[j + 1] = y4.y, yy[j + 2] = y4.z, yy[j + 3] = y4.w;
                    uu[j] = u4.x, uu[j + 1] = u4.y, uu[j + 2] = u4.z, uu[j + 3] = u4.w;
                }
                // decay of this step: per row (dQ, dK sweeps) or per column (dV sweep)
                float drow[2] = {gamma, gamma};
                if (SW != kSweepDV) {
                    if (gchan) drow[0] = dr[tt][2 * rg], drow[1] = dr[tt][2 * rg + 1];
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) dd[j] = gamma;
                    if (gchan) {
                        const float *dp = &dc[tt][cg * G::SEG];
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float4 d4 = *reinterpret_cast<const float4 *>(dp + j);
                            dd[j] = d4.x, dd[j + 1] = d4.y, dd[j + 2] = d4.z, dd[j + 3] = d4.w;
                        }
                    }
                }
                float acc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float xr = xs[tt][2 * rg + r];
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float d0 = SW == kSweepDV ? dd[j] : drow[r];
                        const float d1 = SW == kSweepDV ? dd[j + 1] : drow[r];
                        M[r][j] = fmaf(xr, yy[j], d0 * M[r][j]);
                        M[r][j + 1] = fmaf(xr, yy[j + 1], d1 * M[r][j + 1]);
                        a0 = fmaf(M[r][j], uu[j], a0);
                        a1 = fmaf(M[r][j + 1], uu[j + 1], a1);
                    }
                    acc[r] = a0 + a1;
                }
#pragma unroll
                for (int off = 1; off < G::NCG; off <<= 1)
#pragma unroll
                    for (int r = 0; r < 2; ++r) acc[r] += __shfl_xor_sync(G::MASK, acc[r], off);
                if (cg == 0) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float o = acc[r];
                        if (norm && SW == kSweepDK) {
                            // dz_t = a_{t+1} dz_{t+1} + Q_t e_t; dK_t += dz_t
                            zr[r] = fmaf(drow[r], zr[r], xs[tt][2 * rg + r] * es[tt]);
                            o += zr[r];
                        }
                        os[tt][2 * rg + r] = o;
                    }
                }
            }
        }
        __syncthreads();
        // the block's outputs, one row of 16 values per token
        for (int x = tid; x < nt * kRows; x += G::NT) {
            const int tt = x / kRows, r = x % kRows, t = t0 + tt;
            if (SW == kSweepDQ) p.gq[((size_t)bh * L + t) * dk + row0 + r] = os[tt][r];
            else if (SW == kSweepDK) p.gk[((size_t)bh * L + t) * dk + row0 + r] = os[tt][r];
            else static_cast<T *>(p.grad_v)[((size_t)bh * L + t) * dv + row0 + r] = from_f32<T>(os[tt][r]);
        }
    }
}

// ---------------------------------------------------------------- finish
// dQ = gq + z e (normaliser), dq = dQ phi'(q), dk = dK phi'(k), and with the
// per-channel gate the running sum for dg. Without either, an elementwise
// pass; otherwise one thread per (sequence, key channel) walks the tokens:
// forwards for z (normaliser), backwards for the running sum (channel gate).
template <typename T>
__global__ void __launch_bounds__(kFinThreads) bwd_finish_kernel(BwdParams p) {
    const int dk = p.dk, L = p.L;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE, gchan = p.mode & LA_GATE_CHANNEL;
    const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k);
    T *dq = static_cast<T *>(p.grad_q), *dkk = static_cast<T *>(p.grad_k);
    if (!norm && !gchan) {
        const size_t n = (size_t)p.B * p.H * L * dk;
        for (size_t x = (size_t)blockIdx.x * kFinThreads + threadIdx.x; x < n; x += (size_t)gridDim.x * kFinThreads) {
            dq[x] = from_f32<T>(p.gq[x] * dphi(to_f32(q[x]), elu1));
            dkk[x] = from_f32<T>(p.gk[x] * dphi(to_f32(k[x]), elu1));
        }
        return;
    }
    const long lane = (long)blockIdx.x * kFinThreads + threadIdx.x;
    if (lane >= (long)p.B * p.H * dk) return;
    const int bh = (int)(lane / dk), i = (int)(lane % dk);
    const size_t base = (size_t)bh * L * dk + i;
    if (norm) {
        float z = 0.f;
#pragma unroll 4
        for (int t = 0; t < L; ++t) {
            const size_t x = base + (size_t)t * dk;
            z = gate_value<T>(p, bh, t, i) * z + phi(to_f32(k[x]), elu1);
            const float gq = fmaf(z, p.ecol[(size_t)bh * L + t], p.gq[x]);
            if (gchan) {
                p.gq[x] = gq;  // the running sum below reads the completed dQ
            } else {
                dq[x] = from_f32<T>(gq * dphi(to_f32(q[x]), elu1));
                dkk[x] = from_f32<T>(p.gk[x] * dphi(to_f32(k[x]), elu1));
            }
        }
        if (!gchan) return;
    }
    const T *g = static_cast<const T *>(p.gate);
    T *dg = static_cast<T *>(p.grad_g);
    float c = 0.f;
#pragma unroll 4
    for (int t = L - 1; t >= 0; --t) {
        const size_t x = base + (size_t)t * dk;
        const float qx = to_f32(q[x]), kx = to_f32(k[x]), gq = p.gq[x], gk = p.gk[x];
        dq[x] = from_f32<T>(gq * dphi(qx, elu1));
        dkk[x] = from_f32<T>(gk * dphi(kx, elu1));
        c += phi(qx, elu1) * gq - phi(kx, elu1) * gk;
        if (dg) {
            const float gx = to_f32(g[x]);
            const float sm = 1.f / (1.f + __expf(fminf(gx, 80.f)));  // sigmoid(-g)
            dg[x] = from_f32<T>(c * sm * 0.0625f);
        }
    }
}

template <int SW, typename T>
cudaError_t launch_sweep(const BwdParams &p, cudaStream_t s) {
    const int cols = SW == kSweepDV ? p.dk : p.dv, rows = SW == kSweepDV ? p.dv : p.dk;
    const dim3 grid((unsigned)(p.B * p.H), (unsigned)(rows / kRows));
#define LA_BWD_SWEEP(CC) \
    if (cols == CC) { bwd_sweep_kernel<SW, CC, T><<<grid, SweepCfg<SW, CC>::NT, 0, s>>>(p); return cudaGetLastError(); }
    LA_BWD_SWEEP(16)
    LA_BWD_SWEEP(32)
    LA_BWD_SWEEP(64)
    LA_BWD_SWEEP(128)
#undef LA_BWD_SWEEP
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t launch_all(const BwdParams &p, cudaStream_t s, int *launches) {
    cudaError_t e = cudaSuccess;
    if (p.mode & LA_NORMALIZE) {
        bwd_den_kernel<T><<<(unsigned)(p.B * p.H), 128, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        ++*launches;
    }
    if ((e = launch_sweep<kSweepDQ, T>(p, s)) != cudaSuccess) return e;
    ++*launches;
    if (p.mode & LA_NORMALIZE) {
        const long warps = (long)p.B * p.H * p.L;
        bwd_ecol_kernel<T><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        ++*launches;
    }
    if ((e = launch_sweep<kSweepDK, T>(p, s)) != cudaSuccess) return e;
    ++*launches;
    if ((e = launch_sweep<kSweepDV, T>(p, s)) != cudaSuccess) return e;
    ++*launches;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const bool per_channel = p.mode & (LA_GATE_CHANNEL | LA_NORMALIZE);
    const long n = per_channel ? (long)p.B * p.H * p.dk : (long)p.B * p.H * p.L * p.dk;
    long blocks = (n + kFinThreads - 1) / kFinThreads;
    if (!per_channel && blocks > (long)sms * 16) blocks = (long)sms * 16;
    bwd_finish_kernel<T><<<(unsigned)blocks, kFinThreads, 0, s>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*launches;
    return cudaSuccess;
}

}  // namespace

size_t bwd_scratch_bytes(const BwdArgs &a) {
    const size_t n = (size_t)a.B * a.H * a.L;
    return (2 * n * a.dk + ((a.mode & LA_NORMALIZE) ? 2 * n : 0)) * sizeof(float);
}

int launch_bwd(const BwdArgs &a, cudaStream_t s, int *launches) {
    const size_t bytes = bwd_scratch_bytes(a);
    void *scratch = nullptr;
    if (cudaMallocAsync(&scratch, bytes, s) != cudaSuccess) return LA_ERR_CUDA;
    const size_t n = (size_t)a.B * a.H * a.L;
    BwdParams p{a.q, a.k, a.v, a.gate, a.dout, a.grad_q, a.grad_k, a.grad_v, a.grad_g,
                static_cast<float *>(scratch), static_cast<float *>(scratch) + n * a.dk, nullptr, nullptr,
                a.B, a.H, a.L, a.dk, a.dv, a.mode};
    if (a.mode & LA_NORMALIZE) {
        p.den_inv = p.gk + n * a.dk;
        p.ecol = p.den_inv + n;
    }
    const cudaError_t e = (a.mode & LA_DTYPE_F32) ? launch_all<float>(p, s, launches)
                                                  : launch_all<__nv_bfloat16>(p, s, launches);
    int rc = e == cudaSuccess ? LA_OK : (e == cudaErrorInvalidValue ? LA_ERR_UNSUPPORTED : LA_ERR_CUDA);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

}  // namespace la
