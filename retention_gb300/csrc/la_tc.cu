// la_tc.cu -- the chunkwise forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 operands, fp32 accumulation and state.
//
// Method (learnllm m22 "The Three Faces of Retention"; linear_sparse_attention.py
// linear_attn_chunkwise; the gate A_t of learnllm m22 "Interactive Exploration").
// Inside chunk n (c <= 64 tokens, local index t), with b_t[d] the inclusive
// running sum of log A over the chunk and beta[d] = b at the chunk's middle:
//
//   q~_t = phi(q_t) e^{b_t - beta}        k~_s = phi(k_s) e^{beta - b_s}
//   P    = causal_mask(q~ k~^T)           (= sum_d phi(q)phi(k) e^{b_t - b_s})
//   O^T  = V^T P^T + (diag(e^beta) S_{n-1})^T q~^T
//   T_n  = diag(e^beta) S_{n-1} + k~^T V,  S_n = diag(e^{b_last - beta}) T_n
//
// which is the chunkwise form with the decay factored around the chunk middle
// (exact in real arithmetic; every factor stays within e^{+-|b_last|/2}). For
// linear attention b = 0 and all factors are 1; for retention b_t = (t+1) ln
// gamma. With the normaliser, z is carried the same way and
// den_t = rowsum(P)_t + q~_t . (e^beta z_{n-1}).
//
// Tensor-core mapping (all M = 128, accumulators in TMEM, fp32):
//   QK    D_P [128 x 64]   = q~ (K-major, rows 64..127 unused) . k~^T
//   inter D_O [128 x 64]  += S'^T (MN-major bf16 copy of S') . q~^T
//   S     D_S [128 x 128] += k~^T (MN-major) . V (MN-major)
//   intra D_O             += V^T (MN-major) . P^T (K-major bf16 P)
// O is produced transposed (lane = value channel), so every operand comes
// straight from the TMA-written tiles with the 128-byte swizzle, except the
// bf16 copies of P and S' which the threads write in the same layout.
//
// One CTA per (b, h): 4 warps. The S' copy, P masking and the epilogues run on
// all threads between tcgen05 phases; q, k, v (and g) tiles stream through a
// multi-stage TMA ring so the next chunks' loads overlap the current chunk.
#include <cudaTypedefs.h>
#include <cstring>
#include <mutex>

#include "la_common.cuh"
#include "sm100.cuh"

namespace la {
namespace {
using namespace sm100;

constexpr int kC = 64;                 // chunk length
constexpr int kD = 128;                // d_k = d_v
constexpr int kThreads = 128;
constexpr uint32_t kTile = kC * kD * 2;  // one bf16 [64 x 128] tile: 16 KiB (two 8 KiB swizzle blocks)
constexpr uint32_t kHalf = 8192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColO = 128, kColP = 192;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

__device__ unsigned int g_tc_error;

struct TcParams {
    CUtensorMap tq, tk, tv, tg, to;
    const float *gamma;
    float *final_state;
    int H, L, mode;
};

template <int NS, int GATE>
struct Layout {
    static constexpr uint32_t stage = (GATE == 2 ? 4 : 3) * kTile;
    static constexpr uint32_t P = NS * stage;            // bf16 P tile, 8 KiB
    static constexpr uint32_t S = P + 8192;              // bf16 S' copy, 32 KiB
    static constexpr uint32_t O = S + 32768;             // bf16 O staging, 16 KiB
    static constexpr uint32_t Bt = O + 16384;            // fp32 b_t [64][128] (gated), 32 KiB
    static constexpr uint32_t F = Bt + (GATE == 2 ? 32768 : 0);  // float scratch
    // float scratch: zT, zU, zsum, beta, bc, beta_prev, bc_prev (128 each), dens, fq, fk (64 each)
    static constexpr uint32_t nfloat = 7 * 128 + 3 * 64;
    static constexpr uint32_t Bar = F + nfloat * 4;      // mbarriers
    static constexpr uint32_t Misc = Bar + (NS + 2) * 8;  // tmem slot, abort flag
    static constexpr uint32_t bytes = Misc + 16 + 1024;  // + alignment slack
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float load_bf16(const uint8_t *p) {
    return __uint_as_float(((uint32_t) * reinterpret_cast<const uint16_t *>(p)) << 16);
}
// log alpha = logsigmoid(g) / 16 with the hardware exp/log (absolute error
// ~1e-7 before the / 16).
__device__ __forceinline__ float log_decay_fast(float g) {
    return (fminf(g, 0.f) - __logf(1.f + __expf(-fabsf(g)))) * 0.0625f;
}
__device__ __forceinline__ float phi_fast(float x, bool elu1) {
    return elu1 ? fmaxf(x, 0.f) + __expf(fminf(x, 0.f)) : x;
}

template <int NS, int GATE>
__global__ void __launch_bounds__(kThreads, 1) la_chunk_tc_kernel(const __grid_constant__ TcParams p) {
    using LY = Layout<NS, GATE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x, h = bh % p.H, L = p.L;
    const bool elu1 = p.mode & LA_PHI_ELU1, norm = p.mode & LA_NORMALIZE;
    const int nchunks = (L + kC - 1) / kC;

    float *F = reinterpret_cast<float *>(sm + LY::F);
    float *zT = F, *zU = F + 128, *zsum = F + 256, *beta = F + 384, *bc = F + 512;
    float *beta_prev = F + 640, *bc_prev = F + 768, *dens = F + 896, *fq = F + 960, *fk = F + 1024;
    float *Bt = reinterpret_cast<float *>(sm + LY::Bt);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + LY::Bar);
    uint64_t *bar_qk = full + NS, *bar_o = full + NS + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::Misc);
    int bad = 0;  // this thread saw a bounded wait run out (block-wide OR at barriers)
    uint8_t *sP = sm + LY::P, *sS = sm + LY::S, *sO = sm + LY::O;

    if (warp == 0) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
        mbar_init(bar_qk, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.to);
        if (GATE == 2) tma_prefetch_desc(&p.tg);
    }
    zT[tid] = 0.f;
    float ln_gamma = 0.f;
    if (GATE == 1) ln_gamma = __logf(p.gamma[h]);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    auto issue_load = [&](int stage, int chunk) {
        uint8_t *base = sm + stage * LY::stage;
        const int t0 = chunk * kC;
        mbar_arrive_expect_tx(&full[stage], LY::stage);
        tma_load_3d(base, &p.tq, &full[stage], 0, t0, bh);
        tma_load_3d(base + kHalf, &p.tq, &full[stage], 64, t0, bh);
        tma_load_3d(base + kTile, &p.tk, &full[stage], 0, t0, bh);
        tma_load_3d(base + kTile + kHalf, &p.tk, &full[stage], 64, t0, bh);
        tma_load_3d(base + 2 * kTile, &p.tv, &full[stage], 0, t0, bh);
        tma_load_3d(base + 2 * kTile + kHalf, &p.tv, &full[stage], 64, t0, bh);
        if (GATE == 2) {
            tma_load_3d(base + 3 * kTile, &p.tg, &full[stage], 0, t0, bh);
            tma_load_3d(base + 3 * kTile + kHalf, &p.tg, &full[stage], 64, t0, bh);
        }
    };
    if (tid == 0)
        for (int s = 0; s < NS && s < nchunks; ++s) issue_load(s, s);

    constexpr uint32_t id_qk = idesc_bf16(128, 64, false, false);
    constexpr uint32_t id_o = idesc_bf16(128, 64, true, false);
    constexpr uint32_t id_s = idesc_bf16(128, 128, true, true);

    int n = 0;
    for (; n < nchunks; ++n) {
        const int s = n % NS;
        const uint32_t ph = (uint32_t)(n / NS) & 1u;
        const int t0 = n * kC, c = min(kC, L - t0);
        uint8_t *sQ = sm + s * LY::stage, *sK = sQ + kTile, *sV = sK + kTile, *sG = sV + kTile;
        if (!mbar_wait(&full[s], ph, kWaitNs)) bad = 1;

        // ------------------------------------------------ prologue: phi, decay factors
        const int mid = (c - 1) >> 1;
        if (GATE == 2) {
            const int d = tid;
            const uint8_t *gcol = sG + (d >> 6) * kHalf;
            float b = 0.f, bm = 0.f;
            for (int t = 0; t < c; ++t) {
                b += log_decay_fast(load_bf16(gcol + sw128_offset(t, d & 63)));
                Bt[t * 128 + d] = b;
                if (t == mid) bm = b;
            }
            beta[d] = bm;
            bc[d] = b;
        } else if (GATE == 1) {
            if (tid < 64) {
                fq[tid] = __expf((float)(tid - mid) * ln_gamma);
                fk[tid] = __expf((float)(mid - tid) * ln_gamma);
            }
            if (tid == 0) {
                beta[0] = (float)(mid + 1) * ln_gamma;
                bc[0] = (float)c * ln_gamma;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
            const int pidx = it * kThreads + tid;
            const int isk = pidx >> 10, pp = pidx & 1023;
            const int kb = pp >> 9, row = (pp >> 3) & 63, pc = pp & 7;
            const int col = kb * 64 + ((pc ^ row) & 7) * 8;
            uint4 *addr = reinterpret_cast<uint4 *>((isk ? sK : sQ) + kb * kHalf + row * 128 + pc * 16);
            uint4 w = *addr;
            uint32_t u[4] = {w.x, w.y, w.z, w.w};
            if (isk && row >= c) {
                u[0] = u[1] = u[2] = u[3] = 0u;
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x0 = phi_fast(bf16lo(u[e]), elu1), x1 = phi_fast(bf16hi(u[e]), elu1);
                    if (GATE == 2) {
                        const int d0 = col + 2 * e;
                        const float e0 = Bt[row * 128 + d0] - beta[d0];
                        const float e1 = Bt[row * 128 + d0 + 1] - beta[d0 + 1];
                        x0 *= __expf(isk ? -e0 : e0);
                        x1 *= __expf(isk ? -e1 : e1);
                    } else if (GATE == 1) {
                        const float f = isk ? fk[row] : fq[row];
                        x0 *= f;
                        x1 *= f;
                    }
                    u[e] = pack_bf16(x0, x1);
                }
            }
            *addr = make_uint4(u[0], u[1], u[2], u[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ------------------------------------------------ z increment and S' = diag(f) T
        if (norm) {
            const int d = tid;
            const uint8_t *kcol = sK + (d >> 6) * kHalf;
            float zs = 0.f;
            for (int t = 0; t < c; ++t) zs += load_bf16(kcol + sw128_offset(t, d & 63));
            zsum[d] = zs;
        }
        if (n > 0) {
            const int i = tid;  // TMEM lane = state row (key channel)
            float f = 1.f;
            if (GATE == 2) f = __expf(bc_prev[i] - beta_prev[i] + beta[i]);
            if (GATE == 1) f = __expf(bc_prev[0] - beta_prev[0] + beta[0]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                const uint32_t ta = tmem + lane_base + kColS + 32 * j;
                tmem_ld32(ta, r);
                tmem_ld_wait();
                if (GATE != 0) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
                    tmem_st32(ta, r);
                }
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int lc = 4 * (j & 1) + q4;
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(r[8 * q4 + 0]), __uint_as_float(r[8 * q4 + 1]));
                    w.y = pack_bf16(__uint_as_float(r[8 * q4 + 2]), __uint_as_float(r[8 * q4 + 3]));
                    w.z = pack_bf16(__uint_as_float(r[8 * q4 + 4]), __uint_as_float(r[8 * q4 + 5]));
                    w.w = pack_bf16(__uint_as_float(r[8 * q4 + 6]), __uint_as_float(r[8 * q4 + 7]));
                    *reinterpret_cast<uint4 *>(sS + (j >> 1) * 16384 + i * 128 + ((lc ^ (i & 7)) << 4)) = w;
                }
            }
            if (GATE != 0) tmem_st_wait();
            if (norm) zU[i] = f * zT[i];
        } else if (norm) {
            zU[tid] = 0.f;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) {
            bad = 1;
            break;
        }

        // ------------------------------------------------ MMA group 1: QK, inter, state
        if (tid == 0) {
            tc_fence_after();
            const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), v0 = smem_u32(sV);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t off = (ks >> 2) * kHalf + (ks & 3) * 32;
                umma_bf16(tmem + kColP, sdesc_sw128(q0 + off, 16, 1024), sdesc_sw128(k0 + off, 16, 1024),
                          id_qk, ks > 0);
            }
            umma_commit(bar_qk);
            if (n > 0) {
                const uint32_t s0 = smem_u32(sS);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t offb = (ks >> 2) * kHalf + (ks & 3) * 32;
                    umma_bf16(tmem + kColO, sdesc_sw128(s0 + ks * 2048, 16384, 1024),
                              sdesc_sw128(q0 + offb, 16, 1024), id_o, ks > 0);
                }
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(tmem + kColS, sdesc_sw128(k0 + ks * 2048, kHalf, 1024),
                          sdesc_sw128(v0 + ks * 2048, kHalf, 1024), id_s, (n > 0 || ks > 0));
        }

        // ------------------------------------------------ P: mask, bf16, row sums
        if (!mbar_wait(bar_qk, (uint32_t)n & 1u, kWaitNs)) bad = 1;
        tc_fence_after();
        if (warp < 2) {
            const int t = tid;
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + kColP, r0);
            tmem_ld32(tmem + lane_base + kColP + 32, r1);
            tmem_ld_wait();
            float rs = 0.f;
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint32_t u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j0 = q8 * 8 + 2 * e;
                    const uint32_t a0 = q8 < 4 ? r0[j0] : r1[j0 - 32];
                    const uint32_t a1 = q8 < 4 ? r0[j0 + 1] : r1[j0 + 1 - 32];
                    const float x0 = j0 <= t ? __uint_as_float(a0) : 0.f;
                    const float x1 = j0 + 1 <= t ? __uint_as_float(a1) : 0.f;
                    u[e] = pack_bf16(x0, x1);
                    rs += bf16lo(u[e]) + bf16hi(u[e]);
                }
                *reinterpret_cast<uint4 *>(sP + t * 128 + (((q8 ^ t) & 7) << 4)) =
                    make_uint4(u[0], u[1], u[2], u[3]);
            }
            if (norm) {
                float den = rs;
#pragma unroll 4
                for (int c16 = 0; c16 < 16; ++c16) {
                    const int kb = c16 >> 3, lc = c16 & 7;
                    const uint4 w = *reinterpret_cast<const uint4 *>(sQ + kb * kHalf + t * 128 + (((lc ^ t) & 7) << 4));
                    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
                    const float *z8 = zU + kb * 64 + lc * 8;
#pragma unroll
                    for (int e = 0; e < 4; ++e) den += bf16lo(u[e]) * z8[2 * e] + bf16hi(u[e]) * z8[2 * e + 1];
                }
                dens[t] = den;
            }
        }
        fence_proxy_async_smem();
        if (tid == 0) bulk_wait_read<0>();  // the previous O tile has left the staging buffer
        tc_fence_before();
        __syncthreads();

        // ------------------------------------------------ MMA group 2: intra
        if (tid == 0) {
            tc_fence_after();
            const uint32_t v0 = smem_u32(sV), p0 = smem_u32(sP);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(tmem + kColO, sdesc_sw128(v0 + ks * 2048, kHalf, 1024),
                          sdesc_sw128(p0 + ks * 32, 16, 1024), id_o, (n > 0 || ks > 0));
            umma_commit(bar_o);
        }
        if (!mbar_wait(bar_o, (uint32_t)n & 1u, kWaitNs)) bad = 1;
        tc_fence_after();

        // ------------------------------------------------ O epilogue: lane = value channel
        {
            const int v = tid;
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + kColO, r0);
            tmem_ld32(tmem + lane_base + kColO + 32, r1);
            tmem_ld_wait();
            __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sO);
#pragma unroll
            for (int t = 0; t < 64; ++t) {
                float o = __uint_as_float(t < 32 ? r0[t] : r1[t - 32]);
                if (norm) o = o / dens[t];
                stg[t * 128 + v] = __float2bfloat16_rn(o);
            }
            if (norm) zT[v] = zU[v] + zsum[v];
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(bad)) bad = 1;
        if (GATE == 2) {
            bc_prev[tid] = bc[tid];
            beta_prev[tid] = beta[tid];
        } else if (GATE == 1 && tid == 0) {
            bc_prev[0] = bc[0];
            beta_prev[0] = beta[0];
        }
        if (bad) break;
        if (tid == 0) {
            tma_store_3d(&p.to, sO, 0, t0, bh);
            bulk_commit();
            if (n + NS < nchunks) issue_load(s, n + NS);
        }
    }

    // ------------------------------------------------ final state S = diag(r) T, z
    const int aborted = __syncthreads_or(bad);
    if (!aborted && p.final_state != nullptr) {
        tc_fence_after();
        const int i = tid;
        float f = 1.f;
        if (GATE == 2) f = __expf(bc_prev[i] - beta_prev[i]);
        if (GATE == 1) f = __expf(bc_prev[0] - beta_prev[0]);
        const size_t blk = (size_t)kD * kD + (norm ? kD : 0);
        float *dst = p.final_state + (size_t)bh * blk + (size_t)i * kD;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + kColS + 32 * j, r);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                reinterpret_cast<float4 *>(dst + 32 * j)[q4] =
                    make_float4(__uint_as_float(r[4 * q4]) * f, __uint_as_float(r[4 * q4 + 1]) * f,
                                __uint_as_float(r[4 * q4 + 2]) * f, __uint_as_float(r[4 * q4 + 3]) * f);
        }
        if (norm) p.final_state[(size_t)bh * blk + (size_t)kD * kD + i] = f * zT[i];
    }
    if (aborted) {
        // drain what is in flight before leaving: issued loads, MMAs, stores
        if (tid == 0) {
            atomicOr(&g_tc_error, 1u);
            for (int k2 = n; k2 < nchunks && k2 < n + NS; ++k2)
                mbar_wait(&full[k2 % NS], (uint32_t)(k2 / NS) & 1u, kWaitNs);
            mbar_wait(bar_o, (uint32_t)n & 1u, kWaitNs);
        }
    }
    if (tid == 0) bulk_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// [BH][L][128] bf16 viewed as a 3-D tensor {128, L, BH}; box {box_x, 64, 1}.
bool make_map(CUtensorMap *m, const void *base, int L, int BH, uint32_t box_x, bool swizzle) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
    cuuint32_t box[3] = {box_x, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int NS, int GATE>
int launch_t(const TcParams &prm, int grid, cudaStream_t s) {
    using LY = Layout<NS, GATE>;
    auto kern = la_chunk_tc_kernel<NS, GATE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::bytes) != cudaSuccess)
        return LA_ERR_CUDA;
    kern<<<grid, kThreads, LY::bytes, s>>>(prm);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // namespace

bool chunk_tc_supports(const ChunkArgs &a) {
    if ((a.mode & LA_DTYPE_F32) || a.dk != kD || a.dv != kD || a.chunk != kC || a.L < 1) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10 && get_encode();
}

int launch_chunk_tc(const ChunkArgs &a, cudaStream_t s, int *launches) {
    if (!get_encode()) return LA_ERR_CUDA;
    const int BH = a.B * a.H;
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    if (!make_map(&prm.tq, a.q, a.L, BH, 64, true) || !make_map(&prm.tk, a.k, a.L, BH, 64, true) ||
        !make_map(&prm.tv, a.v, a.L, BH, 64, true) || !make_map(&prm.to, a.out, a.L, BH, 128, false))
        return LA_ERR_CUDA;
    const bool gch = a.mode & LA_GATE_CHANNEL, ghd = a.mode & LA_GATE_HEAD;
    if (gch && !make_map(&prm.tg, a.gate, a.L, BH, 64, true)) return LA_ERR_CUDA;
    prm.gamma = ghd ? static_cast<const float *>(a.gate) : nullptr;
    prm.final_state = a.final_state;
    prm.H = a.H;
    prm.L = a.L;
    prm.mode = a.mode;
    int rc;
    if (gch)
        rc = launch_t<2, 2>(prm, BH, s);
    else if (ghd)
        rc = launch_t<3, 1>(prm, BH, s);
    else
        rc = launch_t<3, 0>(prm, BH, s);
    if (rc == LA_OK) *launches += 1;
    return rc;
}

}  // namespace la
