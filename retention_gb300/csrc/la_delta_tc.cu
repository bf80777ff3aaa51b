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
// and with L = I + A, T = L^-1 diag(beta):
//   Ut  = T (V - K S0^T)
//   out = Q S0^T + tril(Q K^T) Ut      (diagonal included)
//   S   = S0 + Ut^T K
// No page gives this form; it is the recurrence rearranged (the oracle's numpy
// restatement pins it to the recurrence).
//
// One kernel, one CTA of 384 threads per (b, h), chunks in order. T does not
// depend on the state, so T of chunk n + 1 is made while chunk n runs:
//   warps 0-7    the recurrence. The state is kept transposed in TMEM (S^T:
//                lane = key channel i, column = value channel j, fp32) with a
//                bf16 copy in shared memory. Per chunk:
//                phase 1   Y = K S0^T, P = Q K^T, then O = Q S0^T
//                          -> Vt = V - Y (bf16, over the v tile), masked P
//                phase 2   Ut = T Vt -> bf16
//                phase 3   S^T += K^T Ut, O += P Ut -> the new bf16 copy of S^T
//                The tensor pipe runs products in issue order, so the state
//                chain (Y, Vt, Ut, S^T, the bf16 copy) leads each phase; a
//                chunk's out rows are read out of O while the next chunk's Y
//                and P run, before its O starts.
//   warps 8-11   T of the next chunk. The issuer puts its K K^T into TMEM
//                lanes 64..127 during phase 1 (the A operand starts 64 rows
//                before the k tile); warps 10 and 11 (those lanes) write the
//                strictly lower part A of L; L^-1 by 16 x 16 blocks in place
//                over A (the diagonal blocks by forward substitution, a column
//                per thread, then block rows 1..3 of the lower part,
//                X_IJ = -X_II sum_{J<=K<I} A_IK X_KJ); T = L^-1 diag(beta), bf16.
// q and v come in two sets, k through a ring of three a chunk ahead of them, so
// that the next chunk's K K^T can start while this chunk is in phase 1. A set
// (and a ring slot) is refilled as soon as chunk n's state product has read it.
// Nothing goes to memory but the out rows and the final state.
//
// Accumulators with 64 valid rows are M = 128 products whose other 64 rows are
// not read; warps 0, 1, 4 and 5 (TMEM lanes 0..63) own the rows of Y, P, O and
// Ut, the two warps of a lane quarter splitting the columns.
#include <cudaTypedefs.h>
#include <cstring>
#include <mutex>

#include "la_common.cuh"
#include "sm100.cuh"

namespace la {
namespace {
using namespace sm100;

constexpr int kC = 64, kD = 128;
constexpr uint64_t kWaitNs = 2000000000ull;  // far beyond any legitimate wait
constexpr int kLd = 68;                      // fp32 row of L: 16-byte aligned, rows 4 banks apart
constexpr uint32_t cS = 0, cX = 128, cO = 256, cP = 384, kStateCols = 512;  // TMEM: S^T, Y / Ut, O, P

__device__ unsigned int g_delta_tc_error;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack8(const uint32_t *r) {
    return make_uint4(pack2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                      pack2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                      pack2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                      pack2(__uint_as_float(r[6]), __uint_as_float(r[7])));
}
// byte offset of 16-byte chunk c8 (8 bf16) of row r in a tile of 64-wide
// swizzled halves that are `half` bytes apart
__device__ __forceinline__ uint32_t chunk_off(int r, int c8, uint32_t half) {
    return (uint32_t)(c8 >> 3) * half + (uint32_t)r * 128u + ((((uint32_t)c8 & 7u) ^ ((uint32_t)r & 7u)) << 4);
}

using bf16 = __nv_bfloat16;

// descriptors: K-major tile of two halves (K = 128), K-major block (K = 64),
// MN-major operand (K rows of 128 bytes, N atoms `lbo` apart)
__device__ __forceinline__ uint64_t kmaj2(uint32_t addr, int ks) {
    return sdesc_sw128(addr + (ks >= 4 ? 8192u : 0u), 16, 1024) + (uint64_t)((ks & 3) * 2);
}
__device__ __forceinline__ uint64_t kmaj1(uint32_t addr, int ks) { return sdesc_sw128(addr, 16, 1024) + (uint64_t)(ks * 2); }
__device__ __forceinline__ uint64_t mnmaj(uint32_t addr, uint32_t lbo, int ks) {
    return sdesc_sw128(addr, lbo, 1024) + (uint64_t)(ks * 128);
}

constexpr uint32_t id64 = idesc_bf16(128, 64, false, false);   // K-major A and B
constexpr uint32_t idKM = idesc_bf16(128, 128, false, true);   // K-major A, MN-major B
constexpr uint32_t idMM = idesc_bf16(128, 128, true, true);    // MN-major A and B

constexpr int kFusedThreads = 384;
constexpr uint32_t kFSet = 32768;                      // one set: q, v tiles
constexpr uint32_t fQo = 0, fVo = 16384;               // two 8 KiB halves each; v becomes Vt in place
constexpr uint32_t fK = 2 * kFSet;                     // k ring: tile of chunk m in slot m % 3
constexpr uint32_t fP = fK + 3 * 16384;                // P, K-major [64 x 64]
constexpr uint32_t fU = fP + 8192;                     // Ut, MN-major [64 tokens x 128], two halves
constexpr uint32_t fS = fU + 16384;                    // S^T copy, MN-major, two 16 KiB halves
constexpr uint32_t fOs = fS + 32768;                   // out rows of a chunk (TMA store staging)
constexpr uint32_t fT = fOs + 16384;                   // T of chunk m in buffer m % 2, K-major bf16 [64 x 64]
constexpr uint32_t fL = fT + 16384;                    // A, then L^-1 over it, fp32 [64][kLd]
constexpr int kZb = 17;                                // Z block row: 16 + 1
constexpr uint32_t fZ = fL + 64 * kLd * 4;             // Z blocks of one block row, fp32 [3][16][kZb]
constexpr uint32_t fBeta = fZ + 3328;                  // beta of chunk m in row m % 2, fp32 [2][64]
constexpr uint32_t fBar = fBeta + 512;                 // mbarriers, TMEM address
constexpr uint32_t kFusedSmem = fBar + 160 + 1024;     // 16 mbarriers, the TMEM address; alignment
constexpr uint32_t cA = 448;                           // K K^T, 64 columns (rows in lanes 64..127)
constexpr int kSolveWarp0 = 8;                         // warps 8-11; 10 and 11 reach TMEM lanes 64..127
static_assert(kFusedSmem <= 232448, "fused kernel shared memory");
static_assert(fT + 8192 + 16384 <= fBar, "T's M = 128 operand reads 8 KiB past either buffer");
static_assert(fK >= 8192 && fP + 8192 <= fBar, "the k-tile operands read 8 KiB before and after the ring");
static_assert(3 * 16 * kZb * 4 <= 3328, "Z blocks");

// Block row I (1..3) of L^-1 in place over A (fp32 rows kLd floats apart),
// the diagonal blocks and block rows < I done: Z_J = sum_{J<=K<I} A_IK X_KJ,
// then X_IJ = -X_II Z_J over A_IJ, for every J < I. Thread s (0..127) takes the
// outputs s + 128 u, u < 2I: block J = u / 2, row r = s / 16 + 8 (u % 2),
// column s % 16. Everything is unrolled with J known, so the loads of all of a
// thread's outputs can run ahead of their arithmetic.
template <int I, typename Sync>
__device__ __forceinline__ void inverse_block_row(float *M, float *Zs, int s, Sync sync) {
    const int r0 = s >> 4, col = s & 15;
    float z[2 * I];
#pragma unroll
    for (int u = 0; u < 2 * I; ++u) {
        const int J = u >> 1, r = r0 + 8 * (u & 1);
        const float *arow = M + (16 * I + r) * kLd;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k4 = 16 * J; k4 < 16 * I; k4 += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(arow + k4);
            acc[0] = fmaf(a4.x, M[(k4 + 0) * kLd + 16 * J + col], acc[0]);
            acc[1] = fmaf(a4.y, M[(k4 + 1) * kLd + 16 * J + col], acc[1]);
            acc[2] = fmaf(a4.z, M[(k4 + 2) * kLd + 16 * J + col], acc[2]);
            acc[3] = fmaf(a4.w, M[(k4 + 3) * kLd + 16 * J + col], acc[3]);
        }
        z[u] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    }
#pragma unroll
    for (int u = 0; u < 2 * I; ++u) Zs[((u >> 1) * 16 + r0 + 8 * (u & 1)) * kZb + col] = z[u];
    sync();
#pragma unroll
    for (int u = 0; u < 2 * I; ++u) {
        const int J = u >> 1, r = r0 + 8 * (u & 1);
        const float *xrow = M + (16 * I + r) * kLd + 16 * I;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 x4 = *reinterpret_cast<const float4 *>(xrow + k4);
            acc[0] = fmaf(x4.x, Zs[(J * 16 + k4 + 0) * kZb + col], acc[0]);
            acc[1] = fmaf(x4.y, Zs[(J * 16 + k4 + 1) * kZb + col], acc[1]);
            acc[2] = fmaf(x4.z, Zs[(J * 16 + k4 + 2) * kZb + col], acc[2]);
            acc[3] = fmaf(x4.w, Zs[(J * 16 + k4 + 3) * kZb + col], acc[3]);
        }
        z[u] = -((acc[0] + acc[1]) + (acc[2] + acc[3]));
    }
#pragma unroll
    for (int u = 0; u < 2 * I; ++u) M[(16 * I + r0 + 8 * (u & 1)) * kLd + 16 * (u >> 1) + col] = z[u];
    sync();
}

// L^-1 for the unit lower-triangular L = I + A (A strictly lower, fp32 rows
// kLd floats apart) in place over A, by the 128 threads s of the solver warps,
// in 16 x 16 blocks: the diagonal blocks X_II by forward substitution (thread
// s < 64 takes column s % 16 of block s / 16; once x_r is final its share
// leaves every later row, so the dependent chain is one step per row), then
// block rows 1..3 (inverse_block_row). The blocks above the diagonal are left
// as they are, the diagonal blocks' upper halves are zero. `sync` is the
// solvers' barrier.
template <typename Sync>
__device__ __forceinline__ void invert_unit_lower(float *M, float *Zs, int s, Sync sync) {
    float x[16];
    const int b = (s >> 4) & 3, c = s & 15, o = 16 * b;
    if (s < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == c ? 1.f : 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
#pragma unroll
            for (int j = r + 1; j < 16; ++j) x[j] = fmaf(-M[(o + j) * kLd + o + r], x[r], x[j]);
        }
    }
    sync();  // every diagonal block is read before any is overwritten
    if (s < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) M[(o + r) * kLd + o + c] = x[r];
    }
    sync();
    inverse_block_row<1>(M, Zs, s, sync);
    inverse_block_row<2>(M, Zs, s, sync);
    inverse_block_row<3>(M, Zs, s, sync);
}

// T = L^-1 diag(beta) into a K-major bf16 [64 x 64] block once L^-1 is complete
// in M: thread s takes row s / 2 and every other 16-byte group of the row's
// blocks at or left of the diagonal (those to the right stay zero from the
// start). One pass of 16-byte stores after the inverse took less time than
// storing each element as it was made.
__device__ __forceinline__ void t_store(const float *M, int s, uint8_t *tb, const float *beta) {
    const int i = s >> 1, lastg = 2 * (i >> 4) + 1;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int c8 = (s & 1) + 2 * u;
        if (c8 <= lastg) {
            const float4 m0 = *reinterpret_cast<const float4 *>(M + i * kLd + 8 * c8);
            const float4 m1 = *reinterpret_cast<const float4 *>(M + i * kLd + 8 * c8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(beta + 8 * c8);
            const float4 b1 = *reinterpret_cast<const float4 *>(beta + 8 * c8 + 4);
            *reinterpret_cast<uint4 *>(tb + chunk_off(i, c8, 0)) =
                make_uint4(pack2(m0.x * b0.x, m0.y * b0.y), pack2(m0.z * b0.z, m0.w * b0.w),
                           pack2(m1.x * b1.x, m1.y * b1.y), pack2(m1.z * b1.z, m1.w * b1.w));
        }
    }
}

struct FusedParams {
    CUtensorMap tq, tk, tv, to;  // [BH][L][128] bf16 as {128, L, BH}, box {64, 64, 1}, 128-byte swizzle
    DeltaArgs a;
    int nch;
};

__global__ void __launch_bounds__(kFusedThreads, 1) delta_fused_kernel(const __grid_constant__ FusedParams p) {
    const DeltaArgs &a = p.a;
    const int nch = p.nch;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, L = a.L;
    uint64_t *mbP = reinterpret_cast<uint64_t *>(sm + fBar), *mbY = mbP + 1, *mbS = mbP + 2, *mbO = mbP + 3;
    uint64_t *mbU = mbP + 4, *mbA = mbP + 5, *drain = mbP + 6;
    uint64_t *full = mbP + 7;     // [2]: q, v tiles of chunk m in set m % 2
    uint64_t *kfull = mbP + 9;    // [3]: k tile of chunk m in ring slot m % 3
    uint64_t *ofree = mbP + 12;   // the low warps have read the previous chunk's out rows (128 arrivals)
    uint64_t *tready = mbP + 13;  // [2]: T of chunk m is in buffer m % 2 (128 arrivals)
    uint64_t *afree = mbP + 15;   // the solvers have read K K^T out of cA (64 arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + fBar + 16 * 8);
    const uint32_t sm0 = smem_u32(sm);
    const bool chain = warp < 8, solver = warp >= kSolveWarp0;
    // lane quarter of the warp (TMEM lanes 32 qw .. 32 qw + 31) and its column half
    const int qw = warp & 3, hf = (warp >> 2) & 1;
    const bool low = chain && qw < 2;  // TMEM lanes 0..63: the 64 token rows
    const int t = 32 * qw + lane;      // token row (low warps) or key channel (chain warps)
    constexpr int kIssuer = 96, kProducer = 64;  // warp 3 lane 0, warp 2 lane 0
    const bool issuer = tid == kIssuer, producer = tid == kProducer;
    auto kslot = [&](int m) { return sm0 + fK + (uint32_t)(m % 3) * 16384u; };

    // chunk m's q and v tiles into set m % 2 (full[m % 2]); its k tile into ring
    // slot m % 3 (kfull[m % 3]). TMA: rows past the sequence read as zeros.
    auto load_qv = [&](int m) {
        const uint32_t so = (uint32_t)(m & 1) * kFSet;
        uint64_t *bar = full + (m & 1);
        mbar_arrive_expect_tx(bar, kFSet);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + so + fQo + h * 8192, &p.tq, bar, 64 * h, m * kC, bh);
            tma_load_3d(sm + so + fVo + h * 8192, &p.tv, bar, 64 * h, m * kC, bh);
        }
    };
    auto load_k = [&](int m) {
        uint64_t *bar = kfull + m % 3;
        mbar_arrive_expect_tx(bar, 16384);
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_3d(sm + fK + (m % 3) * 16384 + h * 8192, &p.tk, bar, 64 * h, m * kC, bh);
    };
    int issued = 0, kissued = 0;  // loads issued (producer)

    if (warp == 0) {
        tmem_alloc(tmem_slot, kStateCols);
        tmem_relinquish();
    }
    if (issuer) {
        for (int b = 0; b < 12; ++b) mbar_init(mbP + b, 1);  // mbP .. drain, full[2], kfull[3]
        mbar_init(ofree, 128);
        mbar_init(tready, 128);
        mbar_init(tready + 1, 128);
        mbar_init(afree, 64);
        fence_mbar_init();
    }
    // S0 = 0: the bf16 copy starts at zero; so do both T buffers (the blocks
    // above the diagonal are never written)
    for (int i = tid; i < 32768 / 16; i += kFusedThreads) reinterpret_cast<uint4 *>(sm + fS)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = tid; i < 16384 / 16; i += kFusedThreads) reinterpret_cast<uint4 *>(sm + fT)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the tensor core reads the copy and T
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    int bad = 0;
    const int nchunks = nch;
    // K K^T of chunk m into cA; rows 64..127 of the M = 128 product are
    // k_t . k_s: the A descriptors start 8 KiB (64 rows) before each half of
    // the k tile
    auto issue_kk = [&](int m) {
        const uint32_t kt = kslot(m);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + cA, kmaj2(kt - 8192u, ks), kmaj2(kt, ks), id64, ks > 0);
        umma_commit(mbA);
    };

    if (solver) {
        // ============================================================ T of every chunk, in order
        const int sx = tid - 32 * kSolveWarp0;         // 0..127
        const bool reader = warp >= kSolveWarp0 + 2;  // TMEM lanes 64..127: row c of K K^T
        const int c = sx - 64;
        float *M = reinterpret_cast<float *>(sm + fL);
        float *Zs = reinterpret_cast<float *>(sm + fZ), *bs = reinterpret_cast<float *>(sm + fBeta);
        const bf16 *beta = static_cast<const bf16 *>(a.beta) + (size_t)bh * L;
        // beta_c of the next chunk, in flight (zero past the sequence)
        float bnext = reader && c < min(kC, L) ? to_f32(beta[c]) : 0.f;
        auto sync = [&]() { named_sync<3, 128>(); };
        for (int m = 0; m < nchunks; ++m) {
            const int t0 = m * kC;
            bool ok = true;
            if (reader) {
                const float bc = bnext;
                if (m + 1 < nchunks) bnext = c < min(kC, L - t0 - kC) ? to_f32(beta[t0 + kC + c]) : 0.f;
                ok = mbar_wait(mbA, (uint32_t)m & 1u, kWaitNs);
                tc_fence_after();
                __syncwarp();
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem + lane_base + cA, r0);
                tmem_ld32(tmem + lane_base + cA + 32, r1);
                tmem_ld_wait();
                tc_fence_before();
                mbar_arrive(afree);  // cA may take the next chunk's K K^T
                // row c of A: beta_c k_c . k_s for s < c (nothing reads the rest)
#pragma unroll
                for (int s4 = 0; s4 < 64; s4 += 4) {
                    if (s4 < c) {
                        float l4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = s4 + e;
                            l4[e] = bc * __uint_as_float(j < 32 ? r0[j] : r1[j - 32]);
                        }
                        *reinterpret_cast<float4 *>(M + c * kLd + s4) = make_float4(l4[0], l4[1], l4[2], l4[3]);
                    }
                }
                bs[(m & 1) * 64 + c] = bc;
            }
            __syncwarp();
            // A is complete (the previous chunk's T was read out of M before the
            // barrier that ended it)
            if (named_sync_or<3, 128>(!ok)) {
                bad = 1;
                break;
            }
            // L^-1, then T = L^-1 diag(beta) (bf16, K-major) into buffer m % 2
            invert_unit_lower(M, Zs, sx, sync);
            t_store(M, sx, sm + fT + (uint32_t)(m & 1) * 8192u, bs + (m & 1) * 64);
            fence_proxy_async_smem();
            mbar_arrive(tready + (m & 1));
            sync();  // every read of M is done before the next chunk's A goes over it
        }
    } else if (chain) {
        // ============================================================ the recurrence
        // out rows of chunk m (low warps, value channels 64 hf .. 64 hf + 63), once
        // mbO has seen its last product, into the staging tile; store_out(m) then
        // writes the tile with two TMA stores (rows past the sequence are clipped)
        auto read_out = [&](int m) -> bool {
            const bool ok = mbar_wait(mbO, (uint32_t)m & 1u, kWaitNs);
            tc_fence_after();
            __syncwarp();  // tcgen05.ld is warp-collective; the waits may leave the lanes apart
            uint32_t r[2][32];
            tmem_ld32(tmem + lane_base + cO + 64 * hf, r[0]);
            tmem_ld32(tmem + lane_base + cO + 64 * hf + 32, r[1]);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    *reinterpret_cast<uint4 *>(sm + fOs + chunk_off(t, 8 * hf + 4 * j + c4, 8192)) =
                        pack8(r[j] + 8 * c4);
            fence_proxy_async_smem();
            return ok;
        };
        auto store_out = [&](int m) {  // one thread, after the low warps' barrier
            tma_store_3d(&p.to, sm + fOs, 0, m * kC, bh);
            tma_store_3d(&p.to, sm + fOs + 8192, 64, m * kC, bh);
            bulk_commit();
        };
        if (producer) {
            tma_prefetch_desc(&p.tq);
            tma_prefetch_desc(&p.tk);
            tma_prefetch_desc(&p.tv);
            tma_prefetch_desc(&p.to);
            for (; kissued < min(3, nchunks); ++kissued) load_k(kissued);
            for (; issued < min(2, nchunks); ++issued) load_qv(issued);
        }
        if (issuer && nchunks > 0) {
            // the first chunk's K K^T, for the solvers to start on
            if (!mbar_wait(kfull, 0u, kWaitNs)) bad = 1;
            else issue_kk(0);
        }
        __syncwarp();
        for (int n = 0; n < nchunks; ++n) {
            const uint32_t ph = (uint32_t)n & 1u;
            const uint32_t set = sm0 + (uint32_t)(n & 1) * kFSet, kt = kslot(n);
            uint8_t *const setp = sm + (uint32_t)(n & 1) * kFSet;
            int fail = bad || !mbar_wait(full + (n & 1), (uint32_t)(n >> 1) & 1u, kWaitNs) ||
                       !mbar_wait(kfull + n % 3, (uint32_t)(n / 3) & 1u, kWaitNs);
            // ------------------------------------------------------------ phase 1
            // Y first (the recurrence waits on it), then P, then the next
            // chunk's K K^T (for the solvers) while Vt is formed
            bool kk_next = false;  // (issuer) K K^T of chunk n + 1 issued
            if (issuer) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(tmem + cX, kmaj2(kt, ks), mnmaj(sm0 + fS, 16384, ks), idKM, ks > 0);
                umma_commit(mbY);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(tmem + cP, kmaj2(set + fQo, ks), kmaj2(kt, ks), id64, ks > 0);
                umma_commit(mbP);
                // if its k tile has landed and the solvers have read this
                // chunk's out of cA (else after phase 3)
                if (n + 1 < nchunks && mbar_try_wait(kfull + (n + 1) % 3, (uint32_t)((n + 1) / 3) & 1u) &&
                    mbar_try_wait(afree, ph)) {
                    issue_kk(n + 1);
                    kk_next = true;
                }
            }
            if (low) {
                // Vt row t, value channels 64 hf .. 64 hf + 63: V - Y, bf16, in
                // place over the v tile (the MN-major B operand of Ut = T Vt)
                if (!mbar_wait(mbY, ph, kWaitNs)) fail = 1;
                tc_fence_after();
                __syncwarp();
                uint32_t r[2][32];
                tmem_ld32(tmem + lane_base + cX + 64 * hf, r[0]);
                tmem_ld32(tmem + lane_base + cX + 64 * hf + 32, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 2; ++j) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint8_t *pv = setp + fVo + chunk_off(t, 8 * hf + 4 * j + c4, 8192);
                        const uint4 v4 = *reinterpret_cast<const uint4 *>(pv);
                        const uint32_t vw[4] = {v4.x, v4.y, v4.z, v4.w};
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack2(__uint_as_float(vw[e] << 16) - __uint_as_float(r[j][8 * c4 + 2 * e]),
                                         __uint_as_float(vw[e] & 0xffff0000u) - __uint_as_float(r[j][8 * c4 + 2 * e + 1]));
                        *reinterpret_cast<uint4 *>(pv) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                // P row t, columns 32 hf .. 32 hf + 31: q_t . k_s (s <= t), bf16 K-major
                if (!mbar_wait(mbP, ph, kWaitNs)) fail = 1;
                tc_fence_after();
                __syncwarp();
                tmem_ld32(tmem + lane_base + cP + 32 * hf, r[0]);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int s = 32 * hf + 8 * c4 + 2 * e;
                        w[e] = pack2(s <= t ? __uint_as_float(r[0][8 * c4 + 2 * e]) : 0.f,
                                     s + 1 <= t ? __uint_as_float(r[0][8 * c4 + 2 * e + 1]) : 0.f);
                    }
                    *reinterpret_cast<uint4 *>(sm + fP + chunk_off(t, 4 * hf + c4, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
                // the staging tile is free again once the store of chunk n - 2 has read it
                if (tid == 0) bulk_wait_read<0>();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (named_sync_or<1, 256>(fail)) {
                bad = 1;
                break;
            }
            // ------------------------------------------------------------ phase 2: Ut = T Vt
            // then O = Q S0^T once the previous chunk's out rows are read out of
            // its accumulator (the low warps do that while Ut is made)
            if (issuer) {
                // (a commit with nothing before it still completes, so the wait
                // below ends either way; the failure leaves at the next barrier)
                if (!mbar_wait(tready + (n & 1), (uint32_t)(n >> 1) & 1u, kWaitNs)) fail = 1;
                tc_fence_after();
                if (!fail) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_bf16(tmem + cX, kmaj1(sm0 + fT + (uint32_t)(n & 1) * 8192u, ks),
                                  mnmaj(set + fVo, 8192, ks), idKM, ks > 0);
                }
                umma_commit(mbU);
            }
            if (low) {
                if (n > 0 && !read_out(n - 1)) fail = 1;
                tc_fence_before();
                mbar_arrive(ofree);
            }
            if (issuer || (tid == 0 && n > 0)) {
                if (!mbar_wait(ofree, ph, kWaitNs)) fail = 1;
                tc_fence_after();
                if (issuer) {
                    if (!fail) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            umma_bf16(tmem + cO, kmaj2(set + fQo, ks), mnmaj(sm0 + fS, 16384, ks), idKM, ks > 0);
                    }
                } else {
                    store_out(n - 1);
                }
            }
            if (low) {
                // Ut row t, value channels 64 hf .. 64 hf + 63, bf16 MN-major
                if (!mbar_wait(mbU, ph, kWaitNs)) fail = 1;
                tc_fence_after();
                __syncwarp();
                uint32_t r[2][32];
                tmem_ld32(tmem + lane_base + cX + 64 * hf, r[0]);
                tmem_ld32(tmem + lane_base + cX + 64 * hf + 32, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(sm + fU + chunk_off(t, 8 * hf + 4 * j + c4, 8192)) =
                            pack8(r[j] + 8 * c4);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (named_sync_or<1, 256>(fail)) {
                bad = 1;
                break;
            }
            // ------------------------------------------------------------ phase 3
            if (issuer) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + cS, mnmaj(kt, 8192, ks), mnmaj(sm0 + fU, 8192, ks), idMM, (n > 0 || ks > 0));
                umma_commit(mbS);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + cO, kmaj1(sm0 + fP, ks), mnmaj(sm0 + fU, 8192, ks), idKM, 1);
                umma_commit(mbO);
                // else the next chunk's K K^T now, behind this phase's products
                if (n + 1 < nchunks && !kk_next) {
                    if (!mbar_wait(kfull + (n + 1) % 3, (uint32_t)((n + 1) / 3) & 1u, kWaitNs) ||
                        !mbar_wait(afree, ph, kWaitNs))
                        fail = 1;
                    else
                        issue_kk(n + 1);
                }
            }
            {
                // S^T line i = t (TMEM lane), value channels 64 hf .. 64 hf + 63 ->
                // bf16 copy (every product that read the old copy came before mbS)
                if (!mbar_wait(mbS, ph, kWaitNs)) fail = 1;
                tc_fence_after();
                // every reader of this chunk's set and k slot is done (their
                // products came before mbS; Vt and the tiles were read before
                // phase 3): refill them with chunk n + 2 and n + 3
                if (producer && !fail) {
                    if (issued < nchunks) load_qv(issued++);
                    if (kissued < nchunks) load_k(kissued++);
                }
                __syncwarp();  // the issuer's and the producer's warps come out of single-lane work
                uint32_t r[2][32];
                tmem_ld32(tmem + lane_base + cS + 64 * hf, r[0]);
                tmem_ld32(tmem + lane_base + cS + 64 * hf + 32, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(sm + fS + chunk_off(t, 8 * hf + 4 * j + c4, 16384)) =
                            pack8(r[j] + 8 * c4);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (named_sync_or<1, 256>(fail)) {
                bad = 1;
                break;
            }
        }
        // the last chunk's out rows, once the store of the one before has left
        // the staging tile
        if (!bad && low && nchunks > 0) {
            if (tid == 0) bulk_wait_read<0>();
            __syncwarp();
            named_sync<2, 128>();
            if (!read_out(nchunks - 1)) bad = 1;
            named_sync<2, 128>();
            if (tid == 0) store_out(nchunks - 1);
        }
    }
    bad = __syncthreads_or(bad);
    if (!bad && chain && a.final_state) {
        // S = (S^T)^T: state block [d_v][d_k]; thread (i = t, half hf) writes
        // column i over value rows 64 hf .. 64 hf + 63
        float *fs = a.final_state + (size_t)bh * kD * kD;
        tc_fence_after();
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + cS + 64 * hf + 32 * j, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) fs[(size_t)(64 * hf + 32 * j + e) * kD + t] = __uint_as_float(r[e]);
        }
    }
    // teardown: no copy may still be landing in shared memory, and every MMA
    // issued has completed (the waits saw it, or on a time-out a final commit
    // is waited for, bounded)
    if (tid == 0) bulk_wait<0>();  // the out stores are complete
    if (bad) {
        if (issuer) {
            atomicOr(&g_delta_tc_error, 4u);
            umma_commit(drain);
        }
        if (producer) {
            // the last load of each set and slot (every earlier one was waited for)
            for (int m = max(0, issued - 2); m < issued; ++m) mbar_wait(full + (m & 1), (uint32_t)(m >> 1) & 1u, kWaitNs);
            for (int m = max(0, kissued - 3); m < kissued; ++m) mbar_wait(kfull + m % 3, (uint32_t)(m / 3) & 1u, kWaitNs);
        }
        __syncthreads();
        mbar_wait(drain, 0u, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kStateCols);
    }
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult qr;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// [BH][L][128] bf16 as {128, L, BH}; box {64 columns, 64 rows, 1}, 128-byte swizzle
bool make_tile_map(CUtensorMap *m, const void *base, int L, int BH) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

// The error word of the two delta kernels (set when a bounded wait ran out),
// read and cleared; the caller has synchronised the work that could set it.
int delta_tc_error_take(unsigned int *value) {
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(value, g_delta_tc_error, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_delta_tc_error, &zero, sizeof(unsigned int)) != cudaSuccess)
        return LA_ERR_CUDA;
    return LA_OK;
}

bool delta_tc_supports(const DeltaArgs &a) {
    if ((a.mode & LA_DTYPE_F32) || a.dk != kD || a.dv != kD || a.L < 1) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10 && get_encode();
}

int launch_delta_tc(const DeltaArgs &a, cudaStream_t s, int *launches) {
    const int nch = (a.L + kC - 1) / kC;
    const long nbh = (long)a.B * a.H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(delta_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmem) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    FusedParams fp;
    if (!get_encode() || !make_tile_map(&fp.tq, a.q, a.L, (int)nbh) || !make_tile_map(&fp.tk, a.k, a.L, (int)nbh) ||
        !make_tile_map(&fp.tv, a.v, a.L, (int)nbh) || !make_tile_map(&fp.to, a.out, a.L, (int)nbh))
        return LA_ERR_CUDA;
    fp.a = a;
    fp.nch = nch;
    delta_fused_kernel<<<(unsigned)nbh, kFusedThreads, kFusedSmem, s>>>(fp);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    ++*launches;
    return LA_OK;
}

}  // namespace la
