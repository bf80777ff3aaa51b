// la_delta_tc.cu -- the delta rule (DeltaNet) in chunks of 64 tokens on the
// 5th-generation tensor cores (tcgen05, TMEM), bf16 operands, fp32 state.
//
// The recurrence (linear_sparse_attention.py, "delta_rule_recurrent"),
// S_t = S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with S d_v x d_k and
// out_t = S_t q_t, written per step as S_t = S_{t-1} + u_t k_t^T with the
// pseudo-value u_t = beta_t (v_t - S_{t-1} k_t). Inside a chunk that starts
// from S0, S_{t-1} = S0 + sum_{s<t} u_s k_s^T, so the pseudo-values solve the
// unit lower-triangular system
//   (I + A) Ut = diag(beta) (V - K S0^T),   A[t, s] = beta_t k_t . k_s  (s < t)
// and with L = I + A, T = L^-1 diag(beta), W = T K, U = T V (free of the state):
//   Ut  = U - W S0^T
//   out = Q S0^T + tril(Q K^T) Ut      (diagonal included)
//   S   = S0 + Ut^T K
// No page gives this form; it is the recurrence rearranged (the oracle's numpy
// restatement pins it to the recurrence).
//
// One CTA of 128 threads per (b, h), chunks in order. The state is kept
// transposed in TMEM (S^T: lane = key channel i, column = value channel j,
// fp32) with a bf16 copy in shared memory for the products that read it. Per
// chunk, four rounds of MMAs (one thread issues them, all wait on one
// mbarrier), each followed by the threads' work on the results:
//   1  K K^T and Q K^T                -> L (fp32, shared) and the masked P (bf16)
//      L^-1 by blocks of 16 (diagonal blocks by substitution, then block rows)
//      -> T (bf16)
//   2  W = T K, U = T V               -> W (bf16)
//   3  X = W S0^T                     -> Ut = U - X (bf16)
//   4  O = Q S0^T + P Ut, S^T += K^T Ut -> out (bf16), the new bf16 copy of S^T
// Accumulators with 64 valid rows are M = 128 products whose rows 64..127 are
// not read; warps 0 and 1 (TMEM lanes 0..63) own those rows.
#include <cstring>

#include "la_common.cuh"
#include "sm100.cuh"

namespace la {
namespace {
using namespace sm100;

constexpr int kC = 64, kD = 128, kThreads = 128;
constexpr uint64_t kWaitNs = 2000000000ull;  // far beyond any legitimate wait

// shared memory (offsets from a 1024-byte aligned base). A operands of M = 128
// products read 64 rows past their 64-row tiles; every such tile is followed
// by at least 8 KiB of other tiles. q, k, v come in two sets: chunk n + 1's
// tiles are copied in (cp.async) while chunk n is processed.
constexpr uint32_t kSet = 49152;                    // one set: q, k, v
constexpr uint32_t kQ = 0, kK = 16384, kV = 32768;  // [64 x 128] bf16 tiles in a set, two 8 KiB halves
constexpr uint32_t kW = 2 * kSet;                   // W, K-major, two halves
constexpr uint32_t kT = kW + 16384;                 // T, K-major [64 x 64]
constexpr uint32_t kP = kT + 8192;                  // P, K-major [64 x 64]
constexpr uint32_t kU = kP + 8192;                  // Ut, MN-major [64 tokens x 128], two halves
constexpr uint32_t kS = kU + 16384;                 // S^T copy, MN-major: 128 lines x 128 values, two 16 KiB halves
constexpr int kLd = 68;                             // fp32 row: 16-byte aligned, rows 4 banks apart
constexpr uint32_t kL = kS + 32768;                 // L = I + A, fp32 [64][kLd]
constexpr uint32_t kLi = kL + 64 * kLd * 4;         // L^-1, fp32 [64][kLd]
constexpr int kYd = 20;                             // Y row: 16 + 4, 16-byte aligned
constexpr uint32_t kY = kLi + 64 * kLd * 4;         // block-row partial products, fp32 [3][16][kYd]
constexpr uint32_t kB = kY + 3 * 16 * kYd * 4;      // beta [64]
constexpr uint32_t kBar = kB + 64 * 4;              // mbarrier, TMEM address
constexpr uint32_t kSmem = kBar + 16 + 1024;        // + alignment slack
// TMEM columns
constexpr uint32_t cS = 0, cA = 128, cP = 192, cX = 256, cU = 384, kTmemCols = 512;

__device__ unsigned int g_delta_tc_error;

// 16-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// byte offset of 16-byte chunk c8 (8 bf16) of row r in a tile of 64-wide
// swizzled halves that are `half` bytes apart
__device__ __forceinline__ uint32_t chunk_off(int r, int c8, uint32_t half) {
    return (uint32_t)(c8 >> 3) * half + (uint32_t)r * 128u + ((((uint32_t)c8 & 7u) ^ ((uint32_t)r & 7u)) << 4);
}

using bf16 = __nv_bfloat16;

__global__ void __launch_bounds__(kThreads, 1) delta_tc_kernel(const DeltaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x, L = a.L;
    float *Lm = reinterpret_cast<float *>(sm + kL), *Li = reinterpret_cast<float *>(sm + kLi);
    float *Yb = reinterpret_cast<float *>(sm + kY), *bs = reinterpret_cast<float *>(sm + kB);
    uint64_t *mb = reinterpret_cast<uint64_t *>(sm + kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kBar + 8);
    const bf16 *q = static_cast<const bf16 *>(a.q) + (size_t)bh * L * kD;
    const bf16 *k = static_cast<const bf16 *>(a.k) + (size_t)bh * L * kD;
    const bf16 *v = static_cast<const bf16 *>(a.v) + (size_t)bh * L * kD;
    const bf16 *beta = static_cast<const bf16 *>(a.beta) + (size_t)bh * L;
    bf16 *out = static_cast<bf16 *>(a.out) + (size_t)bh * L * kD;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(mb, 1);
        fence_mbar_init();
    }
    // S0 = 0: the bf16 copy starts at zero
    for (int i = tid; i < 32768 / 16; i += kThreads)
        reinterpret_cast<uint4 *>(sm + kS)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t sm0 = smem_u32(sm);
    int bad = 0;
    uint32_t phase = 0;

    constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);    // K-major A and B
    constexpr uint32_t idKM = idesc_bf16(128, 128, false, true);    // K-major A, MN-major B
    constexpr uint32_t idMM = idesc_bf16(128, 128, true, true);     // MN-major A and B
    // descriptors: K-major tile of two halves (K = 128), K-major block (K = 64),
    // MN-major operand (K rows of 128 bytes, N atoms `lbo` apart)
    auto kmaj2 = [&](uint32_t off, int ks) {
        return sdesc_sw128(sm0 + off + (ks >= 4 ? 8192u : 0u), 16, 1024) + (uint64_t)((ks & 3) * 2);
    };
    auto kmaj1 = [&](uint32_t off, int ks) { return sdesc_sw128(sm0 + off, 16, 1024) + (uint64_t)(ks * 2); };
    auto mnmaj = [&](uint32_t off, uint32_t lbo, int ks) {
        return sdesc_sw128(sm0 + off, lbo, 1024) + (uint64_t)(ks * 128);
    };
    // every thread waits for the MMAs committed last; false on time-out
    auto wait_mma = [&]() -> bool {
        const bool ok = mbar_wait(mb, phase & 1u, kWaitNs);
        ++phase;
        tc_fence_after();
        return ok;
    };

    const int nchunks = (L + kC - 1) / kC;
    // chunk m's q, k, v into tile set m % 2: 3 x 64 rows x 16 chunks of 16
    // bytes, 24 per thread; rows past the sequence are zero-filled
    auto fetch = [&](int m) {
        const int f0 = m * kC, fn = min(kC, L - f0);
        const uint32_t set = sm0 + (uint32_t)(m & 1) * kSet;
#pragma unroll
        for (int u = 0; u < 24; ++u) {
            const int x = tid + u * kThreads;
            const int mm = x / (kC * 16), r = (x / 16) % kC, c8 = x % 16;
            const bf16 *src = mm == 0 ? q : mm == 1 ? k : v;
            const bool in = r < fn;
            cp_async16(set + (mm == 0 ? kQ : mm == 1 ? kK : kV) + chunk_off(r, c8, 8192),
                       src + (size_t)(f0 + (in ? r : 0)) * kD + c8 * 8, in ? 16u : 0u);
        }
        cp_async_commit();
    };
    fetch(0);
    float bpre = (tid < kC && tid < L) ? to_f32(beta[tid]) : 0.f;
    for (int n = 0; n < nchunks; ++n) {
        const int t0 = n * kC, nt = min(kC, L - t0);
        const uint32_t set = (uint32_t)(n & 1) * kSet;
        const uint32_t sQ = set + kQ, sK = set + kK, sV = set + kV;
        // ---------------------------------------------------------------- this chunk's tiles
        if (tid < kC) bs[tid] = bpre;
        cp_async_wait_all();
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------------------------- round 1: K K^T, Q K^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + cA, kmaj2(sK, ks), kmaj2(sK, ks), id64, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + cP, kmaj2(sQ, ks), kmaj2(sK, ks), id64, ks > 0);
            umma_commit(mb);
        }
        if (n + 1 < nchunks) {
            // the next chunk's tiles and beta, in flight while this chunk runs
            // (its tile set was last read by chunk n - 1's MMAs, which are done)
            fetch(n + 1);
            const int nb = t0 + kC + tid;
            bpre = (tid < kC && nb < L) ? to_f32(beta[nb]) : 0.f;
        }
        if (__syncthreads_or(!wait_mma())) {
            bad = 1;
            break;
        }
        if (tid < kC) {
            // row t: L[t][s] = beta_t k_t . k_s (s < t), 1 (s = t), 0 (s > t);
            // P[t][s] = q_t . k_s (s <= t), 0 (s > t), bf16 K-major
            const int t = tid;
            const float bt = bs[t];
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + cA, r0);
            tmem_ld32(tmem + lane_base + cA + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int s4 = 0; s4 < 64; s4 += 4) {
                float l4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = s4 + e;
                    const float x = __uint_as_float(s < 32 ? r0[s] : r1[s - 32]);
                    l4[e] = s < t ? bt * x : (s == t ? 1.f : 0.f);
                }
                *reinterpret_cast<float4 *>(Lm + t * kLd + s4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
            }
            tmem_ld32(tmem + lane_base + cP, r0);
            tmem_ld32(tmem + lane_base + cP + 32, r1);
            tmem_ld_wait();
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = c8 * 8 + 2 * e;
                    const float x0 = __uint_as_float(s < 32 ? r0[s] : r1[s - 32]);
                    const float x1 = __uint_as_float(s + 1 < 32 ? r0[s + 1] : r1[s - 31]);
                    w[e] = pack2(s <= t ? x0 : 0.f, s + 1 <= t ? x1 : 0.f);
                }
                *reinterpret_cast<uint4 *>(sm + kP + chunk_off(t, c8, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        tc_fence_before();
        __syncthreads();
        // ---------------------------------------------------------------- L^-1 by 16 x 16 blocks
        if (tid < kC) {
            // diagonal block b, column c: forward substitution of a unit lower-triangular system
            const int b = tid >> 4, c = tid & 15, o = 16 * b;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = r == c ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < r; ++s) acc = fmaf(-Lm[(o + r) * kLd + o + s], x[s], acc);
                x[r] = r < c ? 0.f : acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Li[(o + r) * kLd + o + c] = x[r];
        }
        __syncthreads();
#pragma unroll
        for (int bi = 1; bi < 4; ++bi) {
            // block row bi: Y_bj = sum_{m=j}^{bi-1} L_bi,m Li_m,j, then Li_bi,j = -Li_bi,bi Y_bj.
            // A thread takes four adjacent columns of one row (float4 loads of
            // Li and Y rows, one L value per four products); the zeros above
            // the diagonal of Li_bi,bi make the second product a full 16 terms.
#pragma unroll
            for (int e0 = 0; e0 < bi * 64; e0 += kThreads) {
                const int e = e0 + tid;
                if (e < bi * 64) {
                    const int j = e >> 6, r = (e >> 2) & 15, c0 = 4 * (e & 3);
                    const float *lrow = Lm + (16 * bi + r) * kLd;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int kb = j; kb < bi; ++kb) {
                        float lv[16];
                        float4 iv[16];
#pragma unroll
                        for (int m = 0; m < 16; m += 4) {
                            const float4 l4 = *reinterpret_cast<const float4 *>(lrow + 16 * kb + m);
                            lv[m] = l4.x, lv[m + 1] = l4.y, lv[m + 2] = l4.z, lv[m + 3] = l4.w;
                        }
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            iv[m] = *reinterpret_cast<const float4 *>(Li + (16 * kb + m) * kLd + 16 * j + c0);
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            acc.x = fmaf(lv[m], iv[m].x, acc.x);
                            acc.y = fmaf(lv[m], iv[m].y, acc.y);
                            acc.z = fmaf(lv[m], iv[m].z, acc.z);
                            acc.w = fmaf(lv[m], iv[m].w, acc.w);
                        }
                    }
                    *reinterpret_cast<float4 *>(Yb + (j * 16 + r) * kYd + c0) = acc;
                }
            }
            __syncthreads();
#pragma unroll
            for (int e0 = 0; e0 < bi * 64; e0 += kThreads) {
                const int e = e0 + tid;
                if (e < bi * 64) {
                    const int j = e >> 6, r = (e >> 2) & 15, c0 = 4 * (e & 3);
                    const float *irow = Li + (16 * bi + r) * kLd + 16 * bi;
                    float lv[16];
                    float4 yv[16];
#pragma unroll
                    for (int m = 0; m < 16; m += 4) {
                        const float4 l4 = *reinterpret_cast<const float4 *>(irow + m);
                        lv[m] = l4.x, lv[m + 1] = l4.y, lv[m + 2] = l4.z, lv[m + 3] = l4.w;
                    }
#pragma unroll
                    for (int m = 0; m < 16; ++m) yv[m] = *reinterpret_cast<const float4 *>(Yb + (j * 16 + m) * kYd + c0);
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        acc.x = fmaf(lv[m], yv[m].x, acc.x);
                        acc.y = fmaf(lv[m], yv[m].y, acc.y);
                        acc.z = fmaf(lv[m], yv[m].z, acc.z);
                        acc.w = fmaf(lv[m], yv[m].w, acc.w);
                    }
                    *reinterpret_cast<float4 *>(Li + (16 * bi + r) * kLd + 16 * j + c0) =
                        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
            }
            __syncthreads();
        }
        // T = L^-1 diag(beta), lower triangular, bf16 K-major
#pragma unroll
        for (int x0 = 0; x0 < kC * 8; x0 += kThreads) {
            const int x = x0 + tid, t = x >> 3, c8 = x & 7;
            const float4 l0 = *reinterpret_cast<const float4 *>(Li + t * kLd + 8 * c8);
            const float4 l1 = *reinterpret_cast<const float4 *>(Li + t * kLd + 8 * c8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(bs + 8 * c8);
            const float4 b1 = *reinterpret_cast<const float4 *>(bs + 8 * c8 + 4);
            const float lv[8] = {l0.x * b0.x, l0.y * b0.y, l0.z * b0.z, l0.w * b0.w,
                                 l1.x * b1.x, l1.y * b1.y, l1.z * b1.z, l1.w * b1.w};
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int s = c8 * 8 + 2 * e;
                w[e] = pack2(s <= t ? lv[2 * e] : 0.f, s + 1 <= t ? lv[2 * e + 1] : 0.f);
            }
            *reinterpret_cast<uint4 *>(sm + kT + chunk_off(t, c8, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---------------------------------------------------------------- round 2: W = T K, U = T V
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + cX, kmaj1(kT, ks), mnmaj(sK, 8192, ks), idKM, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + cU, kmaj1(kT, ks), mnmaj(sV, 8192, ks), idKM, ks > 0);
            umma_commit(mb);
        }
        if (__syncthreads_or(!wait_mma())) {
            bad = 1;
            break;
        }
        if (tid < kC) {
            // W row t -> bf16, K-major A operand of round 3
            const int t = tid;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + cX + 32 * j, r);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 4 * j + c4;
                    *reinterpret_cast<uint4 *>(sm + kW + chunk_off(t, c8, 8192)) =
                        make_uint4(pack2(__uint_as_float(r[8 * c4]), __uint_as_float(r[8 * c4 + 1])),
                                   pack2(__uint_as_float(r[8 * c4 + 2]), __uint_as_float(r[8 * c4 + 3])),
                                   pack2(__uint_as_float(r[8 * c4 + 4]), __uint_as_float(r[8 * c4 + 5])),
                                   pack2(__uint_as_float(r[8 * c4 + 6]), __uint_as_float(r[8 * c4 + 7])));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---------------------------------------------------------------- round 3: X = W S0^T
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + cX, kmaj2(kW, ks), mnmaj(kS, 16384, ks), idKM, ks > 0);
            umma_commit(mb);
        }
        if (__syncthreads_or(!wait_mma())) {
            bad = 1;
            break;
        }
        if (tid < kC) {
            // Ut row t = U - X -> bf16, MN-major (tokens x value channels)
            const int t = tid;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t ru[32], rx[32];
                tmem_ld32(tmem + lane_base + cU + 32 * j, ru);
                tmem_ld32(tmem + lane_base + cX + 32 * j, rx);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 4 * j + c4;
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i0 = 8 * c4 + 2 * e;
                        w[e] = pack2(__uint_as_float(ru[i0]) - __uint_as_float(rx[i0]),
                                     __uint_as_float(ru[i0 + 1]) - __uint_as_float(rx[i0 + 1]));
                    }
                    *reinterpret_cast<uint4 *>(sm + kU + chunk_off(t, c8, 8192)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---------------------------------------------------------------- round 4: outputs and state
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + cX, kmaj2(sQ, ks), mnmaj(kS, 16384, ks), idKM, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + cX, kmaj1(kP, ks), mnmaj(kU, 8192, ks), idKM, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(tmem + cS, mnmaj(sK, 8192, ks), mnmaj(kU, 8192, ks), idMM, (n > 0 || ks > 0));
            umma_commit(mb);
        }
        if (__syncthreads_or(!wait_mma())) {
            bad = 1;
            break;
        }
        if (tid < kC) {
            // out row t (warps 0 and 1 read together: tcgen05.ld is collective;
            // rows past a ragged chunk are read and dropped)
            const int t = tid;
            uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)(t0 + t) * kD);
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + cX + 32 * j, r);
                tmem_ld_wait();
                if (t < nt) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        __stcs(dst + 4 * j + c4,
                               make_uint4(pack2(__uint_as_float(r[8 * c4]), __uint_as_float(r[8 * c4 + 1])),
                                          pack2(__uint_as_float(r[8 * c4 + 2]), __uint_as_float(r[8 * c4 + 3])),
                                          pack2(__uint_as_float(r[8 * c4 + 4]), __uint_as_float(r[8 * c4 + 5])),
                                          pack2(__uint_as_float(r[8 * c4 + 6]), __uint_as_float(r[8 * c4 + 7]))));
                }
            }
        }
        {
            // S^T row i (TMEM lane i) -> bf16 copy, MN-major line i
            const int i = tid;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + cS + 32 * j, r);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 4 * j + c4;
                    *reinterpret_cast<uint4 *>(sm + kS + chunk_off(i, c8, 16384)) =
                        make_uint4(pack2(__uint_as_float(r[8 * c4]), __uint_as_float(r[8 * c4 + 1])),
                                   pack2(__uint_as_float(r[8 * c4 + 2]), __uint_as_float(r[8 * c4 + 3])),
                                   pack2(__uint_as_float(r[8 * c4 + 4]), __uint_as_float(r[8 * c4 + 5])),
                                   pack2(__uint_as_float(r[8 * c4 + 6]), __uint_as_float(r[8 * c4 + 7])));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    }
    if (!bad && a.final_state) {
        // S = (S^T)^T: state block [d_v][d_k], thread i writes column i
        const int i = tid;
        float *fs = a.final_state + (size_t)bh * kD * kD;
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + cS + 32 * j, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) fs[(size_t)(32 * j + e) * kD + i] = __uint_as_float(r[e]);
        }
    }
    // teardown: no copy may still be landing in shared memory, and every MMA
    // issued has completed (the last wait saw it, or on a time-out a final
    // commit is waited for, bounded)
    cp_async_wait_all();
    if (bad) {
        if (tid == 0) {
            atomicOr(&g_delta_tc_error, 1u);
            umma_commit(mb);
        }
        __syncthreads();
        mbar_wait(mb, phase & 1u, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool delta_tc_supports(const DeltaArgs &a) {
    if ((a.mode & LA_DTYPE_F32) || a.dk != kD || a.dv != kD || a.L < 1) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10;
}

int launch_delta_tc(const DeltaArgs &a, cudaStream_t s, int *launches) {
    auto kern = delta_tc_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
        return LA_ERR_CUDA;
    kern<<<(unsigned)(a.B * a.H), kThreads, kSmem, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    return LA_OK;
}

}  // namespace la
