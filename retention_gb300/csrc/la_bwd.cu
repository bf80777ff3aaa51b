// la_bwd.cu -- gradients of the forward pass (from S_0 = 0) with respect to q,
// k, v and the per-channel gate, on the CUDA cores in fp32.
//
// The pages motivate the chunkwise form "for training" (learnllm m22, "The
// Three Faces of Retention") but give no gradient; this is the chain rule on
// the recurrence S_t = diag(a_t) S_{t-1} + K_t v_t^T, out_t = S_t^T Q_t
// (Q = phi(q), K = phi(k); with the normaliser, out = num / den and the value
// is widened by a column of ones whose state is z):
//
//   w_t  = dout_t                      e_t = 0                    (no normaliser)
//   w_t  = dout_t / den_t              e_t = -(dout_t . out_t) / den_t
//                                          = -(Q_t . S_t dout_t) / den_t^2
//   dQ_t = S_t w_t + z_t e_t                                   forward sweep
//   dS_t = diag(a_{t+1}) dS_{t+1} + Q_t w_t^T,  dz_t likewise with e_t   reverse
//   dK_t = dS_t v_t + dz_t,   dv_t = dS_t^T K_t
//   dq = dQ * phi'(q),  dk = dK * phi'(k)
//   dg_r = sigmoid(-g_r) / 16 * sum_{t >= r} (Q_t * dQ_t - K_t * dK_t)
//
// (the last line: every term of the output carries e^{B_t - B_s} with
// B_t = sum_{r<=t} log a_r, so dl/dB_t = Q_t dQ_t - K_t dK_t, and log a_r
// enters every B_t with t >= r). e_t is formed from S_t dout_t, the dQ
// sweep's own product, not from the forward's stored output, whose rounding
// the difference S_t w_t + z_t e_t would magnify.
//
// Three sweeps, each carrying one matrix in registers through the sequence
// with one rank-1 update and one matrix-vector product per token, laid out so
// that every reduction stays inside a thread's row group:
//   dQ sweep  rows = key channels (16 per CTA), columns = value channels,
//             forward; with the normaliser it also carries z and adds each
//             CTA's share of den_t atomically
//   (normaliser only: e_t, 1/den_t and the finished dQ_t, one warp per token)
//   dK sweep  rows = key channels, columns = value channels, reverse; it
//             finishes dq, dk (phi') and the gate gradient (the running sum
//             runs backwards with it)
//   dV sweep  rows = value channels, columns = key channels (dS transposed),
//             reverse
// Each sweep stages blocks of kTB tokens in shared memory; the next block's
// 16-byte loads are in flight in registers while a block is processed.
//
// bf16 at head dim 128 (every form but the per-channel gate with the
// normaliser) takes the tensor-core route of la_bwd_tc.cu instead.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kTB = 16;    // tokens per staged block
constexpr int kRows = 16;  // matrix rows per CTA

struct BwdParams {
    const void *q, *k, *v, *gate, *dout;
    void *grad_q, *grad_k, *grad_v, *grad_g;
    float *gq;                     // [BH][L][dk]: dQ (pre phi'); S_t dout_t before the normaliser's finish
    float *zb;                     // [BH][L][dk]: z_t (normaliser)
    float *den, *dinv, *ecol;      // [BH][L] (normaliser)
    int B, H, L, dk, dv, mode;
};

__device__ __forceinline__ float dphi(float x, bool elu1) { return (elu1 && x <= 0.f) ? __expf(x) : 1.f; }
__device__ __forceinline__ float chan_gate(float g) { return __expf(channel_log_decay(g)); }

// A staged stream: per token, NE consecutive elements of a [BH][L][ld] array
// starting at column col0, from token t + off, moved as 16-byte chunks; the
// threads of the CTA take chunks tid, tid + NT, ...
template <typename E, int NE, int NT>
struct Stream {
    static constexpr int EPC = 16 / (int)sizeof(E);
    static constexpr int CPT = NE / EPC;            // chunks per token
    static constexpr int N = kTB * CPT;             // chunks per block
    static constexpr int R = (N + NT - 1) / NT;     // chunks per thread
    uint4 r[R];
    __device__ __forceinline__ void fetch(const E *base, int ld, int col0, int t0, int off, int L, int tid) {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int ci = tid + i * NT;
            r[i] = make_uint4(0u, 0u, 0u, 0u);
            if (ci < N) {
                const int t = t0 + ci / CPT + off;
                if (t < L) r[i] = __ldcs(reinterpret_cast<const uint4 *>(base + (size_t)t * ld + col0) + ci % CPT);
            }
        }
    }
    // element e of token tt goes to dst[tt * ldd + pos(e)], as f(value, in range)
    template <typename Pos, typename F>
    __device__ __forceinline__ void stash(float *dst, int ldd, Pos pos, F f, int t0, int off, int L, int tid) const {
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int ci = tid + i * NT;
            if (ci < N) {
                const int tt = ci / CPT, e0 = (ci % CPT) * EPC;
                const bool in = t0 + tt + off < L;
                const E *el = reinterpret_cast<const E *>(&r[i]);
#pragma unroll
                for (int x = 0; x < EPC; ++x) dst[tt * ldd + pos(e0 + x)] = f(to_f32(el[x]), in);
            }
        }
    }
};

template <int C>
struct SweepCfg {
    static constexpr int NCG = C / 16;              // column groups (lanes of a row group)
    static constexpr int NRG = kRows / 2;           // row groups (two rows each)
    static constexpr int NTC = NRG * NCG;           // compute threads
    static constexpr int NT = NTC < 64 ? 64 : NTC;
    static constexpr int ROWP = NCG * 20;           // padded row: 16-column segments of 20
    static constexpr unsigned MASK = NTC >= 32 ? 0xffffffffu : ((1u << NTC) - 1u);
};

// positions in a staged row: padded 16-column segments, or plain
struct ColPos {
    __device__ __forceinline__ int operator()(int c) const { return (c >> 4) * 20 + (c & 15); }
};
struct RowPos {
    __device__ __forceinline__ int operator()(int r) const { return r; }
};
struct Raw {
    __device__ __forceinline__ float operator()(float x, bool) const { return x; }
};
struct Phi {
    bool elu1;
    __device__ __forceinline__ float operator()(float x, bool) const { return phi(x, elu1); }
};
struct Gate {  // a = exp(logsigmoid(g) / 16); 1 beyond the sequence
    __device__ __forceinline__ float operator()(float x, bool in) const { return in ? chan_gate(x) : 1.f; }
};

// the 16 columns of column group cg of a padded staged row
__device__ __forceinline__ void load16(const float *row, int cg, float (&x)[16]) {
    const float *p = row + cg * 20;
#pragma unroll
    for (int j = 0; j < 16; j += 4) {
        const float4 v4 = *reinterpret_cast<const float4 *>(p + j);
        x[j] = v4.x, x[j + 1] = v4.y, x[j + 2] = v4.z, x[j + 3] = v4.w;
    }
}

// ---------------------------------------------------------------- dQ sweep
template <int C, typename T>
__global__ void __launch_bounds__(SweepCfg<C>::NT) bwd_dq_kernel(BwdParams p) {
    using G = SweepCfg<C>;
    constexpr int NT = G::NT;
    __shared__ float xk[kTB][kRows], xq[kTB][kRows], ar[kTB][kRows], os[kTB][kRows], oz[kTB][kRows];
    __shared__ float pden[kTB][G::NRG];
    __shared__ __align__(16) float ys[kTB][G::ROWP], us[kTB][G::ROWP];
    const int tid = threadIdx.x, rg = tid / G::NCG, cg = tid % G::NCG;
    const int bh = blockIdx.x, row0 = blockIdx.y * kRows, L = p.L, dk = p.dk, dv = p.dv;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE, gchan = p.mode & LA_GATE_CHANNEL;
    const float gamma = (p.mode & LA_GATE_HEAD) ? static_cast<const float *>(p.gate)[bh % p.H] : 1.f;
    const T *k = static_cast<const T *>(p.k) + (size_t)bh * L * dk, *q = static_cast<const T *>(p.q) + (size_t)bh * L * dk;
    const T *g = gchan ? static_cast<const T *>(p.gate) + (size_t)bh * L * dk : nullptr;
    const T *v = static_cast<const T *>(p.v) + (size_t)bh * L * dv, *d = static_cast<const T *>(p.dout) + (size_t)bh * L * dv;
    Stream<T, kRows, NT> sk, sq, sg;
    Stream<T, C, NT> sv, sd;
    auto fetch = [&](int t0) {
        sk.fetch(k, dk, row0, t0, 0, L, tid);
        if (norm) sq.fetch(q, dk, row0, t0, 0, L, tid);
        if (gchan) sg.fetch(g, dk, row0, t0, 0, L, tid);
        sv.fetch(v, dv, 0, t0, 0, L, tid);
        sd.fetch(d, dv, 0, t0, 0, L, tid);
    };

    float M[2][16], zr[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < 16; ++j) M[r][j] = 0.f;
    fetch(0);
    for (int t0 = 0; t0 < L; t0 += kTB) {
        const int nt = min(kTB, L - t0);
        sk.stash(&xk[0][0], kRows, RowPos(), Phi{elu1}, t0, 0, L, tid);
        if (norm) sq.stash(&xq[0][0], kRows, RowPos(), Phi{elu1}, t0, 0, L, tid);
        if (gchan) sg.stash(&ar[0][0], kRows, RowPos(), Gate(), t0, 0, L, tid);
        sv.stash(&ys[0][0], G::ROWP, ColPos(), Raw(), t0, 0, L, tid);
        sd.stash(&us[0][0], G::ROWP, ColPos(), Raw(), t0, 0, L, tid);
        __syncthreads();
        if (t0 + kTB < L) fetch(t0 + kTB);  // in flight while this block runs
        if (tid < G::NTC) {
            for (int tt = 0; tt < nt; ++tt) {
                float yy[16], uu[16];
                load16(ys[tt], cg, yy);
                load16(us[tt], cg, uu);
                float a[2] = {gamma, gamma};
                if (gchan) a[0] = ar[tt][2 * rg], a[1] = ar[tt][2 * rg + 1];
                float acc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float xr = xk[tt][2 * rg + r];
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        M[r][j] = fmaf(xr, yy[j], a[r] * M[r][j]);
                        M[r][j + 1] = fmaf(xr, yy[j + 1], a[r] * M[r][j + 1]);
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
                    float pd = 0.f;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        os[tt][2 * rg + r] = acc[r];
                        if (norm) {
                            zr[r] = fmaf(a[r], zr[r], xk[tt][2 * rg + r]);
                            oz[tt][2 * rg + r] = zr[r];
                            pd = fmaf(xq[tt][2 * rg + r], zr[r], pd);
                        }
                    }
                    if (norm) pden[tt][rg] = pd;
                }
            }
        }
        __syncthreads();
        for (int x = tid; x < nt * kRows; x += NT) {
            const int tt = x / kRows, r = x % kRows;
            const size_t o = ((size_t)bh * L + t0 + tt) * dk + row0 + r;
            p.gq[o] = os[tt][r];
            if (norm) p.zb[o] = oz[tt][r];
        }
        if (norm)
            for (int tt = tid; tt < nt; tt += NT) {
                float s = 0.f;
#pragma unroll
                for (int x = 0; x < G::NRG; ++x) s += pden[tt][x];
                atomicAdd(p.den + (size_t)bh * L + t0 + tt, s);
            }
        __syncthreads();  // the staged rows are free for the next block
    }
}

// ---------------------------------------------------------------- normaliser
// Per token (one warp): den_t complete, e_t = -(Q_t . S_t dout_t) / den_t^2,
// dQ_t = S_t dout_t / den_t + z_t e_t.
template <typename T>
__global__ void __launch_bounds__(256) bwd_norm_kernel(BwdParams p) {
    const long w = ((long)blockIdx.x * 256 + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, dk = p.dk;
    if (w >= (long)p.B * p.H * p.L) return;
    const bool elu1 = p.mode & LA_PHI_ELU1;
    const T *q = static_cast<const T *>(p.q) + (size_t)w * dk;
    float *gq = p.gq + (size_t)w * dk;
    const float *z = p.zb + (size_t)w * dk;
    float s = 0.f;
    for (int c = lane; c < dk; c += 32) s += phi(to_f32(q[c]), elu1) * gq[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    const float di = 1.f / p.den[w], e = -s * di * di;
    for (int c = lane; c < dk; c += 32) gq[c] = fmaf(gq[c], di, z[c] * e);
    if (lane == 0) {
        p.dinv[w] = di;
        p.ecol[w] = e;
    }
}

// ---------------------------------------------------------------- dK sweep
template <int C, typename T>
__global__ void __launch_bounds__(SweepCfg<C>::NT) bwd_dk_kernel(BwdParams p) {
    using G = SweepCfg<C>;
    constexpr int NT = G::NT;
    __shared__ float xq[kTB][kRows], xk[kTB][kRows], xg[kTB][kRows], an[kTB][kRows], gr[kTB][kRows];
    __shared__ float odq[kTB][kRows], odk[kTB][kRows], odg[kTB][kRows];
    __shared__ float dis[kTB], es[kTB];
    __shared__ __align__(16) float ys[kTB][G::ROWP], us[kTB][G::ROWP];
    const int tid = threadIdx.x, rg = tid / G::NCG, cg = tid % G::NCG;
    const int bh = blockIdx.x, row0 = blockIdx.y * kRows, L = p.L, dk = p.dk, dv = p.dv;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE, gchan = p.mode & LA_GATE_CHANNEL;
    const bool want_dg = gchan && p.grad_g != nullptr;
    const float gamma = (p.mode & LA_GATE_HEAD) ? static_cast<const float *>(p.gate)[bh % p.H] : 1.f;
    const T *q = static_cast<const T *>(p.q) + (size_t)bh * L * dk, *k = static_cast<const T *>(p.k) + (size_t)bh * L * dk;
    const T *g = gchan ? static_cast<const T *>(p.gate) + (size_t)bh * L * dk : nullptr;
    const T *v = static_cast<const T *>(p.v) + (size_t)bh * L * dv, *d = static_cast<const T *>(p.dout) + (size_t)bh * L * dv;
    const float *gqb = p.gq + (size_t)bh * L * dk;
    Stream<T, kRows, NT> sq, sk, sgn, sgc;
    Stream<float, kRows, NT> sdq;
    Stream<T, C, NT> sd, sv;
    float pdi = 1.f, pe = 0.f;
    auto fetch = [&](int t0) {
        sq.fetch(q, dk, row0, t0, 0, L, tid);
        sk.fetch(k, dk, row0, t0, 0, L, tid);
        sdq.fetch(gqb, dk, row0, t0, 0, L, tid);
        if (gchan) sgn.fetch(g, dk, row0, t0, 1, L, tid);
        if (want_dg) sgc.fetch(g, dk, row0, t0, 0, L, tid);
        sd.fetch(d, dv, 0, t0, 0, L, tid);
        sv.fetch(v, dv, 0, t0, 0, L, tid);
        if (norm && tid < kTB && t0 + tid < L) {
            pdi = p.dinv[(size_t)bh * L + t0 + tid];
            pe = p.ecol[(size_t)bh * L + t0 + tid];
        }
    };

    float M[2][16], dz[2] = {0.f, 0.f}, cs[2] = {0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < 16; ++j) M[r][j] = 0.f;
    const int nblk = (L + kTB - 1) / kTB;
    fetch((nblk - 1) * kTB);
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * kTB, nt = min(kTB, L - t0);
        sq.stash(&xq[0][0], kRows, RowPos(), Raw(), t0, 0, L, tid);
        sk.stash(&xk[0][0], kRows, RowPos(), Raw(), t0, 0, L, tid);
        sdq.stash(&xg[0][0], kRows, RowPos(), Raw(), t0, 0, L, tid);
        if (gchan) sgn.stash(&an[0][0], kRows, RowPos(), Gate(), t0, 1, L, tid);
        if (want_dg) sgc.stash(&gr[0][0], kRows, RowPos(), Raw(), t0, 0, L, tid);
        sd.stash(&ys[0][0], G::ROWP, ColPos(), Raw(), t0, 0, L, tid);
        sv.stash(&us[0][0], G::ROWP, ColPos(), Raw(), t0, 0, L, tid);
        if (tid < kTB) dis[tid] = pdi, es[tid] = pe;
        __syncthreads();
        if (bi > 0) fetch(t0 - kTB);  // in flight while this block runs
        if (tid < G::NTC) {
            for (int tt = nt - 1; tt >= 0; --tt) {
                float yy[16], uu[16];
                load16(ys[tt], cg, yy);
                load16(us[tt], cg, uu);
                float a[2] = {gamma, gamma};
                if (gchan) a[0] = an[tt][2 * rg], a[1] = an[tt][2 * rg + 1];
                const float di = norm ? dis[tt] : 1.f;
                float Qf[2], acc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    Qf[r] = phi(xq[tt][2 * rg + r], elu1);
                    const float xr = Qf[r] * di;  // Q_t w_t^T with w_t = dout_t / den_t
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        M[r][j] = fmaf(xr, yy[j], a[r] * M[r][j]);
                        M[r][j + 1] = fmaf(xr, yy[j + 1], a[r] * M[r][j + 1]);
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
                        const int rr = 2 * rg + r;
                        float dK = acc[r];
                        if (norm) {
                            dz[r] = fmaf(a[r], dz[r], Qf[r] * es[tt]);
                            dK += dz[r];
                        }
                        const float kx = xk[tt][rr], qx = xq[tt][rr], dQ = xg[tt][rr];
                        odk[tt][rr] = dK * dphi(kx, elu1);
                        odq[tt][rr] = dQ * dphi(qx, elu1);
                        if (want_dg) {
                            cs[r] += Qf[r] * dQ - phi(kx, elu1) * dK;
                            // times sigmoid(-g) / 16, with e^g capped so that it stays finite
                            odg[tt][rr] = cs[r] * 0.0625f / (1.f + __expf(fminf(gr[tt][rr], 80.f)));
                        }
                    }
                }
            }
        }
        __syncthreads();
        T *dq = static_cast<T *>(p.grad_q), *dkk = static_cast<T *>(p.grad_k), *dg = static_cast<T *>(p.grad_g);
        for (int x = tid; x < nt * kRows; x += NT) {
            const int tt = x / kRows, r = x % kRows;
            const size_t o = ((size_t)bh * L + t0 + tt) * dk + row0 + r;
            dq[o] = from_f32<T>(odq[tt][r]);
            dkk[o] = from_f32<T>(odk[tt][r]);
            if (want_dg) dg[o] = from_f32<T>(odg[tt][r]);
        }
        __syncthreads();  // the staged rows are free for the next block
    }
}

// ---------------------------------------------------------------- dV sweep
template <int C, typename T>
__global__ void __launch_bounds__(SweepCfg<C>::NT) bwd_dv_kernel(BwdParams p) {
    using G = SweepCfg<C>;
    constexpr int NT = G::NT;
    __shared__ float xd[kTB][kRows], os[kTB][kRows], dis[kTB];
    __shared__ __align__(16) float ys[kTB][G::ROWP], us[kTB][G::ROWP], dc[kTB][G::ROWP];
    const int tid = threadIdx.x, rg = tid / G::NCG, cg = tid % G::NCG;
    const int bh = blockIdx.x, row0 = blockIdx.y * kRows, L = p.L, dk = p.dk, dv = p.dv;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE, gchan = p.mode & LA_GATE_CHANNEL;
    const float gamma = (p.mode & LA_GATE_HEAD) ? static_cast<const float *>(p.gate)[bh % p.H] : 1.f;
    const T *q = static_cast<const T *>(p.q) + (size_t)bh * L * dk, *k = static_cast<const T *>(p.k) + (size_t)bh * L * dk;
    const T *g = gchan ? static_cast<const T *>(p.gate) + (size_t)bh * L * dk : nullptr;
    const T *d = static_cast<const T *>(p.dout) + (size_t)bh * L * dv;
    Stream<T, kRows, NT> sd;
    Stream<T, C, NT> sq, sk, sg;
    float pdi = 1.f;
    auto fetch = [&](int t0) {
        sd.fetch(d, dv, row0, t0, 0, L, tid);
        sq.fetch(q, dk, 0, t0, 0, L, tid);
        sk.fetch(k, dk, 0, t0, 0, L, tid);
        if (gchan) sg.fetch(g, dk, 0, t0, 1, L, tid);
        if (norm && tid < kTB && t0 + tid < L) pdi = p.dinv[(size_t)bh * L + t0 + tid];
    };

    float M[2][16];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < 16; ++j) M[r][j] = 0.f;
    const int nblk = (L + kTB - 1) / kTB;
    fetch((nblk - 1) * kTB);
    for (int bi = nblk - 1; bi >= 0; --bi) {
        const int t0 = bi * kTB, nt = min(kTB, L - t0);
        sd.stash(&xd[0][0], kRows, RowPos(), Raw(), t0, 0, L, tid);
        sq.stash(&ys[0][0], G::ROWP, ColPos(), Phi{elu1}, t0, 0, L, tid);
        sk.stash(&us[0][0], G::ROWP, ColPos(), Phi{elu1}, t0, 0, L, tid);
        if (gchan) sg.stash(&dc[0][0], G::ROWP, ColPos(), Gate(), t0, 1, L, tid);
        if (tid < kTB) dis[tid] = pdi;
        __syncthreads();
        if (bi > 0) fetch(t0 - kTB);
        if (tid < G::NTC) {
            for (int tt = nt - 1; tt >= 0; --tt) {
                float yy[16], uu[16], aa[16];
                load16(ys[tt], cg, yy);
                load16(us[tt], cg, uu);
                if (gchan) {
                    load16(dc[tt], cg, aa);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) aa[j] = gamma;
                }
                const float di = norm ? dis[tt] : 1.f;
                float acc[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float xr = xd[tt][2 * rg + r] * di;
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        M[r][j] = fmaf(xr, yy[j], aa[j] * M[r][j]);
                        M[r][j + 1] = fmaf(xr, yy[j + 1], aa[j + 1] * M[r][j + 1]);
                        a0 = fmaf(M[r][j], uu[j], a0);
                        a1 = fmaf(M[r][j + 1], uu[j + 1], a1);
                    }
                    acc[r] = a0 + a1;
                }
#pragma unroll
                for (int off = 1; off < G::NCG; off <<= 1)
#pragma unroll
                    for (int r = 0; r < 2; ++r) acc[r] += __shfl_xor_sync(G::MASK, acc[r], off);
                if (cg == 0) os[tt][2 * rg] = acc[0], os[tt][2 * rg + 1] = acc[1];
            }
        }
        __syncthreads();
        T *dvo = static_cast<T *>(p.grad_v);
        for (int x = tid; x < nt * kRows; x += NT) {
            const int tt = x / kRows, r = x % kRows;
            dvo[((size_t)bh * L + t0 + tt) * dv + row0 + r] = from_f32<T>(os[tt][r]);
        }
        __syncthreads();  // the staged rows are free for the next block
    }
}

#define LA_BWD_DISPATCH(NAME)                                                                   \
    template <typename T>                                                                       \
    cudaError_t launch_##NAME(const BwdParams &p, int cols, int rows, cudaStream_t s) {         \
        const dim3 grid((unsigned)(p.B * p.H), (unsigned)(rows / kRows));                       \
        switch (cols) {                                                                         \
            case 16: bwd_##NAME##_kernel<16, T><<<grid, SweepCfg<16>::NT, 0, s>>>(p); break;    \
            case 32: bwd_##NAME##_kernel<32, T><<<grid, SweepCfg<32>::NT, 0, s>>>(p); break;    \
            case 64: bwd_##NAME##_kernel<64, T><<<grid, SweepCfg<64>::NT, 0, s>>>(p); break;    \
            case 128: bwd_##NAME##_kernel<128, T><<<grid, SweepCfg<128>::NT, 0, s>>>(p); break; \
            default: return cudaErrorInvalidValue;                                              \
        }                                                                                       \
        return cudaGetLastError();                                                              \
    }
LA_BWD_DISPATCH(dq)
LA_BWD_DISPATCH(dk)
LA_BWD_DISPATCH(dv)
#undef LA_BWD_DISPATCH

template <typename T>
cudaError_t launch_all(const BwdParams &p, cudaStream_t s, int *launches) {
    cudaError_t e = cudaSuccess;
    const bool norm = p.mode & LA_NORMALIZE;
    if (norm && (e = cudaMemsetAsync(p.den, 0, sizeof(float) * (size_t)p.B * p.H * p.L, s)) != cudaSuccess) return e;
    if ((e = launch_dq<T>(p, p.dv, p.dk, s)) != cudaSuccess) return e;
    ++*launches;
    if (norm) {
        const long warps = (long)p.B * p.H * p.L;
        bwd_norm_kernel<T><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        ++*launches;
    }
    if ((e = launch_dk<T>(p, p.dv, p.dk, s)) != cudaSuccess) return e;
    ++*launches;
    if ((e = launch_dv<T>(p, p.dk, p.dv, s)) != cudaSuccess) return e;
    ++*launches;
    return cudaSuccess;
}

}  // namespace

size_t bwd_scratch_bytes(const BwdArgs &a) {
    const size_t n = (size_t)a.B * a.H * a.L;
    return (n * a.dk + ((a.mode & LA_NORMALIZE) ? n * a.dk + 3 * n : 0)) * sizeof(float);
}

int launch_bwd(const BwdArgs &a, cudaStream_t s, int *launches) {
    const size_t bytes = bwd_scratch_bytes(a);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, bytes, s) != LA_OK) return LA_ERR_CUDA;
    const size_t n = (size_t)a.B * a.H * a.L;
    float *f = static_cast<float *>(scratch);
    BwdParams p{a.q, a.k, a.v, a.gate, a.dout, a.grad_q, a.grad_k, a.grad_v, a.grad_g,
                f, nullptr, nullptr, nullptr, nullptr, a.B, a.H, a.L, a.dk, a.dv, a.mode};
    if (a.mode & LA_NORMALIZE) {
        p.zb = f + n * a.dk;
        p.den = p.zb + n * a.dk;
        p.dinv = p.den + n;
        p.ecol = p.dinv + n;
    }
    const cudaError_t e = (a.mode & LA_DTYPE_F32) ? launch_all<float>(p, s, launches)
                                                  : launch_all<__nv_bfloat16>(p, s, launches);
    int rc = e == cudaSuccess ? LA_OK : (e == cudaErrorInvalidValue ? LA_ERR_UNSUPPORTED : LA_ERR_CUDA);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

}  // namespace la
