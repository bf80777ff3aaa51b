// la_epilogue.cu -- the RetNet output epilogue as a kernel of its own.
//
// learnllm m22, "Retention": retention drops the normaliser of linear attention
// and RetNet steadies the output with a GroupNorm and a swish gate instead. One
// group per head, so each (b, h, t) row of d_v outputs is normalised on its own
// (biased variance, eps inside the root), scaled and shifted per head channel,
// and multiplied by swish(og), og being the output gate the caller projected
// from the layer input:
//
//   out = swish(og) * ((x - mean) / sqrt(var + eps) * weight[h] + bias[h])
//
// It runs after the chunk forward (in place on its output) and on decode
// outputs. Applying it in the tensor-core kernel's store was slower: only the
// two output warps can read the accumulator rows there, and the extra
// arithmetic on them set the pace of the whole kernel. It is a streaming pass
// (read x and og, write out), bound by HBM: a row is spread over lanes 16 bytes each, with
// the two reductions (mean, then the squared deviations) done by shuffles
// inside the lane group; warps stride over rows with two row groups in flight.
#include "la_common.cuh"

namespace la {
namespace {

constexpr int kGnThreads = 256;
constexpr int kGnUnroll = 2;  // row groups a warp has in flight at once

// 16 bytes of a row: 8 bf16 or 4 fp32 values
template <typename T> struct Pack16;
template <> struct Pack16<float> {
    static constexpr int N = 4;
    static __device__ __forceinline__ void get(const uint4 &r, float (&x)[N]) {
        x[0] = __uint_as_float(r.x), x[1] = __uint_as_float(r.y), x[2] = __uint_as_float(r.z),
        x[3] = __uint_as_float(r.w);
    }
    static __device__ __forceinline__ uint4 put(const float (&x)[N]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
};
template <> struct Pack16<__nv_bfloat16> {
    static constexpr int N = 8;
    static __device__ __forceinline__ void get(const uint4 &r, float (&x)[N]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) x[2 * i] = __uint_as_float(w[i] << 16), x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    static __device__ __forceinline__ uint4 put(const float (&x)[N]) {
        return make_uint4(pack(x[0], x[1]), pack(x[2], x[3]), pack(x[4], x[5]), pack(x[6], x[7]));
    }
};

// swish(u) = u / (1 + e^-u) with the fast exponential and division; e^-u is
// capped at e^80 so that the fast division stays in its range (for u < -80
// the result is below 1e-33 in magnitude either way).
__device__ __forceinline__ float swish_fast(float u) { return __fdividef(u, 1.f + __expf(fminf(-u, 80.f))); }

// A row is spread over DV / N lanes, N values (16 bytes) each; a warp holds
// 32 / (DV / N) rows at a time and kGnUnroll such groups in flight.
template <typename T, int DV>
__global__ void __launch_bounds__(kGnThreads, 4) gn_swish_kernel(const GnArgs a, long rows) {
    using P = Pack16<T>;
    constexpr int N = P::N;
    constexpr int LPR = DV / N;    // lanes per row
    constexpr int RPW = 32 / LPR;  // rows per warp
    const int lane = threadIdx.x & 31, li = lane % LPR;
    const long warp = ((long)blockIdx.x * kGnThreads + threadIdx.x) >> 5;
    const long nwarps = ((long)gridDim.x * kGnThreads) >> 5;
    const uint4 *x = reinterpret_cast<const uint4 *>(a.x);
    const uint4 *og = reinterpret_cast<const uint4 *>(a.ogate);
    uint4 *out = reinterpret_cast<uint4 *>(a.out);
    for (long r0 = warp * RPW * kGnUnroll; r0 < rows; r0 += nwarps * RPW * kGnUnroll) {
        uint4 xr[kGnUnroll], gr[kGnUnroll];
#pragma unroll
        for (int u = 0; u < kGnUnroll; ++u) {
            const long r = r0 + u * RPW + lane / LPR;
            xr[u] = gr[u] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows) {
                xr[u] = __ldcs(x + r * LPR + li);
                gr[u] = __ldcs(og + r * LPR + li);
            }
        }
#pragma unroll
        for (int u = 0; u < kGnUnroll; ++u) {
            const long r = r0 + u * RPW + lane / LPR;
            float xv[N], gv[N];
            P::get(xr[u], xv);
            P::get(gr[u], gv);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < N; ++i) s += xv[i];
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            const float mean = s * (1.f / DV);
            float s2 = 0.f;
#pragma unroll
            for (int i = 0; i < N; ++i) {
                xv[i] -= mean;
                s2 = fmaf(xv[i], xv[i], s2);
            }
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
            const float rstd = rsqrtf(fmaf(s2, 1.f / DV, a.eps));
            if (r < rows) {
                // rows < 2^31 (checked by the launcher): 32-bit division
                const int h = (int)(((uint32_t)r / (uint32_t)a.L) % (uint32_t)a.H);
                float w[N], b[N];
#pragma unroll
                for (int i = 0; i < N; i += 4) {
                    const float4 w4 = a.weight ? __ldg(reinterpret_cast<const float4 *>(a.weight + (size_t)h * DV + li * N + i))
                                               : make_float4(1.f, 1.f, 1.f, 1.f);
                    const float4 b4 = a.bias ? __ldg(reinterpret_cast<const float4 *>(a.bias + (size_t)h * DV + li * N + i))
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    w[i] = w4.x, w[i + 1] = w4.y, w[i + 2] = w4.z, w[i + 3] = w4.w;
                    b[i] = b4.x, b[i + 1] = b4.y, b[i + 2] = b4.z, b[i + 3] = b4.w;
                }
                float o[N];
#pragma unroll
                for (int i = 0; i < N; ++i) o[i] = swish_fast(gv[i]) * fmaf(xv[i] * rstd, w[i], b[i]);
                __stcs(out + r * LPR + li, P::put(o));
            }
        }
    }
}

template <typename T, int DV>
cudaError_t launch_dv(const GnArgs &a, cudaStream_t s) {
    const long rows = (long)a.B * a.H * a.L;
    constexpr long rows_per_cta = (kGnThreads / 32) * (32 / (DV / Pack16<T>::N)) * kGnUnroll;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // one wave: four resident CTAs per SM, no more
    const long need = (rows + rows_per_cta - 1) / rows_per_cta;
    const long cap = (long)sms * 4;
    gn_swish_kernel<T, DV><<<(unsigned)(need < cap ? need : cap), kGnThreads, 0, s>>>(a, rows);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const GnArgs &a, cudaStream_t s) {
    switch (a.dv) {
        case 16: return launch_dv<T, 16>(a, s);
        case 32: return launch_dv<T, 32>(a, s);
        case 64: return launch_dv<T, 64>(a, s);
        case 128: return launch_dv<T, 128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int launch_gn_swish(const GnArgs &a, cudaStream_t s, int *launches) {
    const long rows = (long)a.B * a.H * a.L;
    if (rows == 0) return LA_OK;
    if (rows > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    const cudaError_t e = (a.mode & LA_DTYPE_F32) ? launch_t<float>(a, s) : launch_t<__nv_bfloat16>(a, s);
    if (e == cudaErrorInvalidValue) return LA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    return LA_OK;
}

}  // namespace la
