// la_bwd_tc.cu -- the backward pass on the tensor cores: each gradient term as
// a causal linear-attention forward with its roles permuted, run on the
// tensor-core forward kernel (bf16, d_k = d_v = 128).
//
// The gradients themselves are those of la_bwd.cu (the chain rule on the
// recurrence; the pages give no gradient). With a decay that does not depend on
// the channel (A_t = 1 or gamma_h), (Q_t . K_s) gamma^{t-s} is symmetric in the
// roles, so
//   dQ_t = sum_{s<=t} gamma^{t-s} (dout_t . v_s) K_s        = fwd(dout, v, K)
//   dK_s = sum_{t>=s} gamma^{t-s} (v_s . dout_t) Q_t        = afwd(v, dout, Q)
//   dv_s = sum_{t>=s} gamma^{t-s} (K_s . Q_t) dout_t        = afwd(K, Q, dout)
// where afwd is the anti-causal instance of the forward kernel (the sum over the
// token and every later one, chunks taken from the end), run on the arrays in
// their own order. The normaliser and the per-channel gate add the terms
// described above their routes below.
#include "la_common.cuh"

namespace la {
namespace {

// The hardware base-2 exponential and logarithm (denormals flushed), for the
// elementwise passes around the forwards (the gated pass works in log2 units,
// as the forward kernel's gate arithmetic does).
__device__ __forceinline__ float hw_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float hw_lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;
// log2 alpha = log2(sigmoid(g)) / 16 = (min(g, 0) log2 e - log2(1 + 2^(-|g| log2 e))) / 16
__device__ __forceinline__ float log2_alpha(float g) {
    return (fminf(g, 0.f) * kLog2e - hw_lg2(1.f + hw_ex2(-fabsf(g) * kLog2e))) * 0.0625f;
}

// ---------------------------------------------------------------- scalar gate, no normaliser
// With the identity feature map the three forwards read the caller's arrays and
// write the gradients directly. With phi = elu + 1 a first pass writes phi(q)
// and phi(k) in order, and a last pass applies phi' to dQ and dK.
constexpr int kEw = 256;  // threads of the elementwise passes
constexpr int kD = 128;   // the tensor-core kernel's head dim

__device__ __forceinline__ uint4 phi8(uint4 x, bool elu1) {
    if (!elu1) return x;
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xffff0000u);
        const float lo = x0 > 0.f ? x0 + 1.f : hw_ex2(x0 * kLog2e), hi = x1 > 0.f ? x1 + 1.f : hw_ex2(x1 * kLog2e);
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// g * phi'(x) on eight bf16 values (elu + 1: 1 for x > 0, e^x otherwise)
__device__ __forceinline__ uint4 dphi8(uint4 g, uint4 x) {
    uint32_t gw[4] = {g.x, g.y, g.z, g.w}, xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = __uint_as_float(xw[i] << 16), x1 = __uint_as_float(xw[i] & 0xffff0000u);
        const float g0 = __uint_as_float(gw[i] << 16), g1 = __uint_as_float(gw[i] & 0xffff0000u);
        __nv_bfloat162 h = __floats2bfloat162_rn(x0 > 0.f ? g0 : g0 * __expf(x0), x1 > 0.f ? g1 : g1 * __expf(x1));
        gw[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(gw[0], gw[1], gw[2], gw[3]);
}

// Qf = phi(q), Kf = phi(k), in order; one uint4 (8 bf16) per step
__global__ void __launch_bounds__(kEw) bwd_phi_kernel(const uint4 *q, const uint4 *k, uint4 *Qf, uint4 *Kf, long n) {
    for (long x = (long)blockIdx.x * kEw + threadIdx.x; x < n; x += (long)gridDim.x * kEw) {
        Qf[x] = phi8(__ldcs(q + x), true);
        Kf[x] = phi8(__ldcs(k + x), true);
    }
}

// dq = dQ phi'(q), dk = dK phi'(k), in order
__global__ void __launch_bounds__(kEw) bwd_dphi_kernel(const uint4 *q, const uint4 *k, const uint4 *dQ, const uint4 *dK,
                                                       uint4 *dq, uint4 *dk, long n) {
    for (long x = (long)blockIdx.x * kEw + threadIdx.x; x < n; x += (long)gridDim.x * kEw) {
        dq[x] = dphi8(__ldcs(dQ + x), __ldg(q + x));
        dk[x] = dphi8(__ldcs(dK + x), __ldg(k + x));
    }
}

// ---------------------------------------------------------------- tensor-core route, normalised
// With the normaliser (w_t = dout_t / den_t, e_t = -(Q_t . S_t w_t) / den_t):
//   den_t = Q_t . z_t                   = fwd(Q, K, J)            (columns 0 and 1)
//   U_t   = S_t w_t                     = fwd(w, v, K)
//   z_t e_t                             = fwd(E, J, K)            E_t = (e_t hi, e_t lo, 0 ..), J_s = (1, 1, 0 ..)
//   dK_s  = sum_{t>=s} Q_t (v_s . w_t) + sum_{t>=s} Q_t e_t
//         = afwd(v, w, Q) + afwd(J, E, Q)
//   dv_s  = afwd(K, Q, w)
//   dQ_t  = U_t + z_t e_t
// dQ and dK are differences of nearly equal terms, so those forwards write
// fp32 and e_t travels as two bf16 parts (hi + lo).
constexpr int CPR = kD / 8;  // 16-byte chunks per row

// Q = phi(q), K = phi(k) in order; the constant J
__global__ void __launch_bounds__(kEw) bwdn_prep1_kernel(const uint4 *q, const uint4 *k, uint4 *Qf, uint4 *Kf,
                                                         uint4 *J, long rows, bool elu1) {
    const long n = rows * CPR;
    const uint32_t one2 = 0x3F803F80u;  // bf16 1.0 twice
    for (long x = (long)blockIdx.x * kEw + threadIdx.x; x < n; x += (long)gridDim.x * kEw) {
        Qf[x] = phi8(__ldcs(q + x), elu1);
        Kf[x] = phi8(__ldcs(k + x), elu1);
        J[x] = (x % CPR) == 0 ? make_uint4(one2, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// w = dout / den (den from column 0 of the fp32 forward with values J)
__global__ void __launch_bounds__(kEw) bwdn_prep2_kernel(const uint4 *d, const float *den_full, uint4 *w, float *den,
                                                         long rows) {
    const long n = rows * CPR;
    for (long x = (long)blockIdx.x * kEw + threadIdx.x; x < n; x += (long)gridDim.x * kEw) {
        const long row = x / CPR;
        const float dn = den_full[row * kD];
        if (x % CPR == 0) den[row] = dn;
        const float r = 1.f / dn;
        const uint4 g = __ldcs(d + x);
        uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(gw[i] << 16) * r, __uint_as_float(gw[i] & 0xffff0000u) * r);
            gw[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        w[x] = make_uint4(gw[0], gw[1], gw[2], gw[3]);
    }
}

// e_t = -(Q_t . U_t) / den_t, one warp per token; E_t = (hi, lo, 0 ..)
__global__ void __launch_bounds__(kEw) bwdn_prep3_kernel(const uint4 *Qf, const float *U, const float *den, uint4 *E,
                                                         long rows) {
    const long row = ((long)blockIdx.x * kEw + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    // lane covers columns 4 lane .. 4 lane + 3
    const uint2 qq = reinterpret_cast<const uint2 *>(Qf + row * CPR)[lane];
    const float4 uu = reinterpret_cast<const float4 *>(U + row * kD)[lane];
    float sdot = __uint_as_float(qq.x << 16) * uu.x + __uint_as_float(qq.x & 0xffff0000u) * uu.y +
                 __uint_as_float(qq.y << 16) * uu.z + __uint_as_float(qq.y & 0xffff0000u) * uu.w;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
    const float e = -sdot / den[row];
    if (lane < CPR) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (lane == 0) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(e);
            const __nv_bfloat16 lo = __float2bfloat16_rn(e - __bfloat162float(hi));
            __nv_bfloat162 h2;
            h2.x = hi;
            h2.y = lo;
            o.x = *reinterpret_cast<uint32_t *>(&h2);
        }
        E[row * CPR + lane] = o;
    }
}

// dq = (U + ZE) phi'(q), dk = (dKm + dz) phi'(k), in order
__global__ void __launch_bounds__(kEw) bwdn_post_kernel(const uint4 *q, const uint4 *k, const float4 *U,
                                                        const float4 *ZE, const float4 *dkm, const float4 *dz,
                                                        uint4 *dq, uint4 *dk, long rows, bool elu1) {
    const long n = rows * CPR;
    auto combine = [elu1](float4 a0, float4 a1, float4 b0, float4 b1, uint4 x) {
        const float g[8] = {a0.x + b0.x, a0.y + b0.y, a0.z + b0.z, a0.w + b0.w,
                            a1.x + b1.x, a1.y + b1.y, a1.z + b1.z, a1.w + b1.w};
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(xw[i] << 16), x1 = __uint_as_float(xw[i] & 0xffff0000u);
            const float g0 = (elu1 && x0 <= 0.f) ? g[2 * i] * __expf(x0) : g[2 * i];
            const float g1 = (elu1 && x1 <= 0.f) ? g[2 * i + 1] * __expf(x1) : g[2 * i + 1];
            __nv_bfloat162 h = __floats2bfloat162_rn(g0, g1);
            o[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    };
    for (long x = (long)blockIdx.x * kEw + threadIdx.x; x < n; x += (long)gridDim.x * kEw) {
        dq[x] = combine(__ldcs(U + 2 * x), __ldcs(U + 2 * x + 1), __ldcs(ZE + 2 * x), __ldcs(ZE + 2 * x + 1), __ldg(q + x));
        dk[x] = combine(__ldcs(dkm + 2 * x), __ldcs(dkm + 2 * x + 1), __ldcs(dz + 2 * x), __ldcs(dz + 2 * x + 1),
                        __ldg(k + x));
    }
}

// ---------------------------------------------------------------- tensor-core route, per-channel gate
// With the gate diag(alpha_t) on the key channels (B_t = sum_{r<=t} log alpha_r):
//   dv_s    = sum_{t>=s} (Q_t . K_s e^{B_t - B_s}) dout_t        = afwd_key(K, Q, dout)
//   dQ_t[i] = sum_{s<=t} e^{B_t[i] - B_s[i]} K_s[i] (dout_t . v_s)  = fwd_value(dout, v, K)
//   dK_s[i] = sum_{t>=s} e^{B_t[i] - B_s[i]} Q_t[i] (v_s . dout_t)  = afwd_value(v, dout, Q)
// fwd_value is the forward with the decay on the value channels (the kernel
// writes it without the factor e^{b_t}, b the log decay since the chunk start,
// which the passes after apply); afwd is the anti-causal instance, whose
// mirrored sequence decays token t by the gate of token t + 1, so its products
// are the same gate products. With elu+1 each forward applies the feature map
// itself (the value-side ones to their value tile). Then dg_r = sigmoid(-g_r) / 16 sum_{t>=r} (Q dQ -
// K dK)_t by a segmented reverse scan over chunks of 64 tokens.

// The passes below take one thread per (sequence, chunk of 64 tokens, group
// of 8 channels) and walk the chunk's tokens: 16-byte loads of bf16 rows
// (two of fp32), consecutive threads on consecutive channel groups.
struct Grp {
    long bh;
    int c, i0;  // chunk, first channel
};
__device__ __forceinline__ bool grp_of(long x, long nbh, int L, Grp &g) {
    const int nch = (L + 63) / 64;
    if (x >= nbh * nch * CPR) return false;
    g.i0 = 8 * (int)(x % CPR);
    g.c = (int)((x / CPR) % nch);
    g.bh = x / CPR / nch;
    return true;
}
__device__ __forceinline__ void unpack8(uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[2 * i] = __uint_as_float(u[i] << 16), f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        u[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}
__device__ __forceinline__ void ld8f(const float *p, float (&f)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(p)), b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}
__device__ __forceinline__ void st8f(float *p, const float (&f)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// One pass over the two brackets, a thread per (sequence, chunk of 64 tokens,
// group of 8 channels). With P_t the sum of log alpha(g_t') over t' = chunk
// start .. t (the causal decay since the chunk start) and A the same sum up to
// the chunk's last token's successor (the sequence's last token decays
// nothing), the anti-causal decay to the chunk's end is A - P_t, so:
//   dQ_t = e^{P_t} bracket_q,t      dK_t = e^{A - P_t} bracket_k,t
//   dq = dQ phi'(q), dk = dK phi'(k), r_t = phi(q) dQ - phi(k) dK (fp32)
// and the chunk's total of r (r and the totals only when `r` is given). The
// first walk sums A over the chunk's gates (the second finds them in L2).
__global__ void __launch_bounds__(kEw) bwdg_post_kernel(const uint4 *q, const uint4 *k, const uint4 *g,
                                                        const uint4 *brq, const uint4 *brk, uint4 *dq, uint4 *dk,
                                                        float *r, float *tot, long nbh, int L, bool elu1) {
    Grp G;
    const long x = (long)blockIdx.x * kEw + threadIdx.x;
    if (!grp_of(x, nbh, L, G)) return;
    const int t0 = 64 * G.c, t1 = min(L, t0 + 64), umax = min(t1, L - 1);
    const size_t base = ((size_t)G.bh * L) * kD + G.i0;
    // (log2 units throughout)
    float A[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int t = t0; t <= umax; ++t) {
        float gv[8];
        unpack8(__ldg(g + (base + (size_t)t * kD) / 8), gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) A[e] += log2_alpha(gv[e]);
    }
    float P[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int t = t0; t < t1; ++t) {
        const size_t o = base + (size_t)t * kD;
        float gv[8], bq[8], bk[8], qv[8], kv[8], rv[8], oq[8], ok[8];
        unpack8(__ldcs(g + o / 8), gv);
        unpack8(__ldcs(brq + o / 8), bq);
        unpack8(__ldcs(brk + o / 8), bk);
        unpack8(__ldg(q + o / 8), qv);
        unpack8(__ldg(k + o / 8), kv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            P[e] += log2_alpha(gv[e]);
            const float dQ = hw_ex2(P[e]) * bq[e], dK = hw_ex2(A[e] - P[e]) * bk[e];
            // phi and phi' from one exponential each: e^min(x, 0)
            float pq = qv[e], dpq = 1.f, pk = kv[e], dpk = 1.f;
            if (elu1) {
                const float eq = hw_ex2(fminf(qv[e], 0.f) * kLog2e), ek = hw_ex2(fminf(kv[e], 0.f) * kLog2e);
                pq = qv[e] > 0.f ? qv[e] + 1.f : eq;
                dpq = qv[e] > 0.f ? 1.f : eq;
                pk = kv[e] > 0.f ? kv[e] + 1.f : ek;
                dpk = kv[e] > 0.f ? 1.f : ek;
            }
            oq[e] = dQ * dpq;
            ok[e] = dK * dpk;
            rv[e] = pq * dQ - pk * dK;
            rs[e] += rv[e];
        }
        dq[o / 8] = pack8(oq);
        dk[o / 8] = pack8(ok);
        if (r) st8f(r + o, rv);
    }
    if (tot) st8f(tot + (size_t)x * 8, rs);
}

// The chunk totals of r (from the pass above), then (one CTA per sequence and
// channel group) the sums over all later chunks, then dg = sigmoid(-g) / 16
// (later chunks + the chunk's tail).
// One CTA per (sequence, group of 8 channels): thread j takes a run of
// consecutive chunks, the runs' totals are summed over the later runs (a suffix
// scan across the warp by shuffles, then across the warps through shared
// memory), and each thread walks its run from the last chunk, writing the sum
// over all later chunks in place of each chunk's total.
__global__ void __launch_bounds__(kEw) bwdg_carry_kernel(float *tot, int L) {
    __shared__ float wt[kEw / 32][8];
    const int nch = (L + 63) / 64;
    const long bh = blockIdx.x / CPR;
    const int i0 = 8 * (int)(blockIdx.x % CPR), j = threadIdx.x, lane = j & 31, w = j >> 5;
    const int per = (nch + kEw - 1) / kEw, c0 = min(nch, j * per), c1 = min(nch, c0 + per);
    float run[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c = c0; c < c1; ++c) {
        float v[8];
        ld8f(tot + ((size_t)bh * nch + c) * kD + i0, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) run[e] += v[e];
    }
    // inclusive suffix sums of the runs within the warp
    float suf[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) suf[e] = run[e];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float o = __shfl_down_sync(0xffffffffu, suf[e], off);
            if (lane + off < 32) suf[e] += o;
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) wt[w][e] = suf[e];
    }
    __syncthreads();
    // the sum over every later run: later lanes of this warp, then later warps
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        acc[e] = suf[e] - run[e];
        for (int w2 = w + 1; w2 < kEw / 32; ++w2) acc[e] += wt[w2][e];
    }
    for (int c = c1 - 1; c >= c0; --c) {
        float *p = tot + ((size_t)bh * nch + c) * kD + i0;
        float v[8];
        ld8f(p, v);
        st8f(p, acc);  // the sum over later chunks
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += v[e];
    }
}
__global__ void __launch_bounds__(kEw) bwdg_dg_kernel(const float *r, const float *carry, const uint4 *g, uint4 *dg,
                                                      long nbh, int L) {
    Grp G;
    const long x = (long)blockIdx.x * kEw + threadIdx.x;
    if (!grp_of(x, nbh, L, G)) return;
    float acc[8];
    ld8f(carry + (size_t)x * 8, acc);
#pragma unroll 2
    for (int t = min(L, 64 * G.c + 64) - 1; t >= 64 * G.c; --t) {
        const size_t o = ((size_t)G.bh * L + t) * kD + G.i0;
        float v[8], gv[8], out[8];
        ld8f(r + o, v);
        unpack8(__ldcs(g + o / 8), gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc[e] += v[e];
            out[e] = acc[e] * 0.0625f / (1.f + __expf(fminf(gv[e], 80.f)));
        }
        dg[o / 8] = pack8(out);
    }
}

int ew_blocks(long n) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        sms = 132;
    const long need = (n + kEw - 1) / kEw, cap = (long)sms * 8;
    return (int)(need < cap ? need : cap);
}

}  // namespace

bool bwd_tc_supports(const BwdArgs &a) {
    if (a.mode & LA_DTYPE_F32) return false;
    if ((a.mode & LA_GATE_CHANNEL) && (a.mode & LA_NORMALIZE)) return false;
    if (a.dk != kD || a.dv != kD || a.L < 1) return false;
    ChunkArgs c{a.q, a.k, a.v, a.gate, nullptr, nullptr, a.B, a.H, a.L, kD, kD, a.mode & LA_GATE_HEAD, 64, nullptr};
    return chunk_tc_supports(c);
}

static int launch_bwd_tc_gated(const BwdArgs &a, cudaStream_t s, int *launches) {
    const long nbh = (long)a.B * a.H, rows = nbh * a.L;
    const int nch = (a.L + 63) / 64;
    const size_t hb = (size_t)rows * kD * sizeof(__nv_bfloat16);
    const bool elu1 = a.mode & LA_PHI_ELU1;
    // bf16: bracket_q bracket_k; fp32: r; chunk totals
    const size_t bytes = 2 * hb + 2 * hb + (size_t)nbh * nch * kD * sizeof(float);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, bytes, s) != LA_OK) return LA_ERR_CUDA;
    char *b = static_cast<char *>(scratch);
    uint4 *brq = reinterpret_cast<uint4 *>(b), *brk = reinterpret_cast<uint4 *>(b + hb);
    float *rf = reinterpret_cast<float *>(b + 2 * hb), *tot = reinterpret_cast<float *>(b + 4 * hb);
    int rc = LA_OK;
    auto ok = [&]() {
        if (rc == LA_OK && cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
        if (rc == LA_OK) ++*launches;
    };
    // the feature map runs inside each forward: on the value tile (value side)
    // or on q and k
    auto fwd = [&](const void *q, const void *k, const void *v, void *out, bool value_side, bool anti) {
        if (rc != LA_OK) return;
        ChunkArgs c{q, k, v, a.gate, out, nullptr, a.B, a.H, a.L, kD, kD, LA_GATE_CHANNEL | (elu1 ? LA_PHI_ELU1 : 0),
                    64, nullptr, 0, value_side ? 1 : 0, anti ? 1 : 0};
        rc = launch_chunk_tc(c, s, launches);
    };
    fwd(a.dout, a.v, a.k, brq, true, false);  // dQ without e^{b_t}; values phi(k)
    fwd(a.v, a.dout, a.q, brk, true, true);   // dK without e^{b_t}; values phi(q)
    fwd(a.k, a.q, a.dout, a.grad_v, false, true);  // dv: phi(k) . phi(q)
    const long nt = nbh * nch * CPR;  // (sequence, chunk, channel group) threads
    const unsigned nbk = (unsigned)((nt + kEw - 1) / kEw);
    if (rc == LA_OK) {
        // (r and the chunk totals only when the gate gradient is wanted)
        const bool want_dg = a.grad_g != nullptr;
        bwdg_post_kernel<<<nbk, kEw, 0, s>>>(static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.k),
                                             static_cast<const uint4 *>(a.gate), brq, brk,
                                             static_cast<uint4 *>(a.grad_q), static_cast<uint4 *>(a.grad_k),
                                             want_dg ? rf : nullptr, want_dg ? tot : nullptr, nbh, a.L, elu1);
        ok();
    }
    if (rc == LA_OK && a.grad_g) {
        bwdg_carry_kernel<<<(unsigned)(nbh * CPR), kEw, 0, s>>>(tot, a.L);
        ok();
        if (rc == LA_OK) {
            bwdg_dg_kernel<<<nbk, kEw, 0, s>>>(rf, tot, static_cast<const uint4 *>(a.gate),
                                               static_cast<uint4 *>(a.grad_g), nbh, a.L);
            ok();
        }
    }
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

// The normalised form without a gate: four forwards (four launches, or twelve
// when short batches split each sequence into segments). With
// num_t = Q_t S_t and den_t = Q_t . z_t of the forward, w_t = dout_t / den_t and
// e_t = -(dout_t . num_t) / den_t^2:
//   dQ_t = sum_{s<=t} K_s (v_s . w_t + e_t)     causal, e on the query row
//   dK_s = sum_{t>=s} Q_t (v_s . w_t + e_t)     anti-causal, e on the key column
//   dv_s = sum_{t>=s} (K_s . Q_t) w_t           anti-causal
// The forward kernel's backward-prep instance gives w and e in one pass (num_t
// stays in its fp32 accumulator), and its bias instances add the e terms
// inside the chunk (on the scores, before the mask) and across chunks (a
// carried sum of value rows), so the cancelling sums are formed in fp32 and
// leave as the bf16 gradients. With elu+1 the bias instances also take phi'
// of q (dQ) or k (dK) in their store, so the gradients leave finished.
static int launch_bwd_tc_norm_fused(const BwdArgs &a, cudaStream_t s, int *launches) {
    const long rows = (long)a.B * a.H * a.L;
    const size_t hb = (size_t)rows * kD * sizeof(__nv_bfloat16);
    const bool elu1 = a.mode & LA_PHI_ELU1;
    // bf16 w; fp32 e [rows]
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, hb + (size_t)rows * sizeof(float), s) != LA_OK) return LA_ERR_CUDA;
    char *b = static_cast<char *>(scratch);
    uint4 *w = reinterpret_cast<uint4 *>(b);
    float *e = reinterpret_cast<float *>(b + hb);
    const int phi = elu1 ? LA_PHI_ELU1 : 0;
    int rc = LA_OK;
    // the feature map runs inside each forward: on q and k (the prep, dv) or on
    // the value tile (the bias instances, which take phi' of x in the store)
    auto fwd = [&](const void *q, const void *k, const void *v, void *out, bool anti, int bias, const void *x) {
        if (rc != LA_OK) return;
        ChunkArgs c{q, k, v, nullptr, out, nullptr, a.B, a.H, a.L, kD, kD, phi, 64, nullptr, 0, 0, anti ? 1 : 0};
        c.bias = bias;
        c.bias_e = bias ? e : nullptr;
        c.bias_x = x;
        rc = launch_chunk_tc(c, s, launches);
    };
    {
        // w and e from the normalised forward
        ChunkArgs c{a.q, a.k, a.v, nullptr, w, nullptr, a.B, a.H, a.L, kD, kD, LA_NORMALIZE | phi, 64, nullptr};
        c.bp_dout = a.dout;
        c.bp_e = e;
        rc = launch_chunk_tc(c, s, launches);
    }
    fwd(w, a.v, a.k, a.grad_q, false, 1, a.q);  // values phi(k); rows phi'(q)
    fwd(a.v, w, a.q, a.grad_k, true, 2, a.k);   // values phi(q); rows phi'(k)
    fwd(a.k, a.q, w, a.grad_v, true, 0, nullptr);  // phi(k) . phi(q)
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

static int launch_bwd_tc_norm(const BwdArgs &a, cudaStream_t s, int *launches) {
    if (!(a.mode & LA_GATE_HEAD)) return launch_bwd_tc_norm_fused(a, s, launches);
    const long rows = (long)a.B * a.H * a.L;
    const size_t hb = (size_t)rows * kD * sizeof(__nv_bfloat16), fb = 2 * hb;
    // bf16: Q K J w E; fp32: den_full U ZE dKm dz; den [rows]
    const size_t bytes = 5 * hb + 5 * fb + (size_t)rows * sizeof(float);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, bytes, s) != LA_OK) return LA_ERR_CUDA;
    char *b = static_cast<char *>(scratch);
    uint4 *h[5];
    for (int i = 0; i < 5; ++i) h[i] = reinterpret_cast<uint4 *>(b + i * hb);
    uint4 *Qf = h[0], *Kf = h[1], *J = h[2], *w = h[3], *E = h[4];
    float *f[5];
    for (int i = 0; i < 5; ++i) f[i] = reinterpret_cast<float *>(b + 5 * hb + i * fb);
    float *den_full = f[0], *U = f[1], *ZE = f[2], *dkm = f[3], *dz = f[4];
    float *den = reinterpret_cast<float *>(b + 5 * hb + 5 * fb);
    const bool elu1 = a.mode & LA_PHI_ELU1;
    const int mode = a.mode & LA_GATE_HEAD;  // identity feature map, bf16, no normaliser
    const int nb = ew_blocks(rows * CPR);
    int rc = LA_OK;
    auto ok = [&]() {
        if (rc == LA_OK && cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
        if (rc == LA_OK) ++*launches;
    };
    auto fwd = [&](const void *q, const void *k, const void *v, void *out, bool f32, bool anti) {
        if (rc != LA_OK) return;
        ChunkArgs c{q, k, v, a.gate, out, nullptr, a.B, a.H, a.L, kD, kD, mode, 64, nullptr, f32 ? 1 : 0, 0,
                    anti ? 1 : 0};
        rc = launch_chunk_tc(c, s, launches);
    };
    bwdn_prep1_kernel<<<nb, kEw, 0, s>>>(static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.k), Qf, Kf, J,
                                         rows, elu1);
    ok();
    fwd(Qf, Kf, J, den_full, true, false);  // den_t in columns 0 and 1
    if (rc == LA_OK) {
        bwdn_prep2_kernel<<<nb, kEw, 0, s>>>(static_cast<const uint4 *>(a.dout), den_full, w, den, rows);
        ok();
    }
    fwd(w, a.v, Kf, U, true, false);  // U_t = S_t w_t
    if (rc == LA_OK) {
        bwdn_prep3_kernel<<<(unsigned)((rows + kEw / 32 - 1) / (kEw / 32)), kEw, 0, s>>>(Qf, U, den, E, rows);
        ok();
    }
    fwd(E, J, Kf, ZE, true, false);   // z_t e_t
    fwd(a.v, w, Qf, dkm, true, true);  // sum_{t>=s} (v_s . w_t) Q_t
    fwd(J, E, Qf, dz, true, true);     // sum_{t>=s} e_t Q_t
    fwd(Kf, Qf, w, a.grad_v, false, true);
    if (rc == LA_OK) {
        bwdn_post_kernel<<<nb, kEw, 0, s>>>(static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.k),
                                            reinterpret_cast<const float4 *>(U), reinterpret_cast<const float4 *>(ZE),
                                            reinterpret_cast<const float4 *>(dkm), reinterpret_cast<const float4 *>(dz),
                                            static_cast<uint4 *>(a.grad_q), static_cast<uint4 *>(a.grad_k), rows, elu1);
        ok();
    }
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

int launch_bwd_tc(const BwdArgs &a, cudaStream_t s, int *launches) {
    if (a.mode & LA_GATE_CHANNEL) return launch_bwd_tc_gated(a, s, launches);
    if (a.mode & LA_NORMALIZE) return launch_bwd_tc_norm(a, s, launches);
    const long rows = (long)a.B * a.H * a.L;
    const bool elu1 = a.mode & LA_PHI_ELU1;
    const int mode = a.mode & LA_GATE_HEAD;  // identity feature map, bf16, no normaliser
    int rc = LA_OK;
    auto fwd = [&](const void *q, const void *k, const void *v, void *out, bool anti) {
        if (rc != LA_OK) return;
        ChunkArgs c{q, k, v, a.gate, out, nullptr, a.B, a.H, a.L, kD, kD, mode, 64, nullptr, 0, 0, anti ? 1 : 0};
        rc = launch_chunk_tc(c, s, launches);
    };
    if (!elu1) {
        // three forwards on the caller's arrays, straight into the gradients
        fwd(a.dout, a.v, a.k, a.grad_q, false);
        fwd(a.v, a.dout, a.q, a.grad_k, true);
        fwd(a.k, a.q, a.dout, a.grad_v, true);
        return rc;
    }
    // phi(q), phi(k), dQ and dK (before phi') in scratch
    const size_t arr = (size_t)rows * kD * sizeof(__nv_bfloat16);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, 4 * arr, s) != LA_OK) return LA_ERR_CUDA;
    char *b = static_cast<char *>(scratch);
    uint4 *Qf = reinterpret_cast<uint4 *>(b), *Kf = reinterpret_cast<uint4 *>(b + arr);
    uint4 *dQ = reinterpret_cast<uint4 *>(b + 2 * arr), *dK = reinterpret_cast<uint4 *>(b + 3 * arr);
    const long n = rows * CPR;
    const int nb = ew_blocks(n);
    bwd_phi_kernel<<<nb, kEw, 0, s>>>(static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.k), Qf, Kf, n);
    if (cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
    else ++*launches;
    fwd(a.dout, a.v, Kf, dQ, false);
    fwd(a.v, a.dout, Qf, dK, true);
    fwd(Kf, Qf, a.dout, a.grad_v, true);
    if (rc == LA_OK) {
        bwd_dphi_kernel<<<nb, kEw, 0, s>>>(static_cast<const uint4 *>(a.q), static_cast<const uint4 *>(a.k), dQ, dK,
                                           static_cast<uint4 *>(a.grad_q), static_cast<uint4 *>(a.grad_k), n);
        if (cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
        else ++*launches;
    }
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}


}  // namespace la
