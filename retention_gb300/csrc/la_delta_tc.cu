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
// Two kernels. W and U do not depend on the state, so they are made for every
// chunk at once, and only the state recurrence runs chunk after chunk:
//   delta_prep_kernel   one CTA of 128 threads per (b, h, chunk), four CTAs per SM.
//       round 1  K K^T -> L = I + A (fp32, shared); L^-1 in place: the four
//                16 x 16 diagonal blocks by substitution, then two merges of
//                lower-triangular block pairs (16 -> 32 -> 64) -> T (bf16)
//       round 2  W = T K, then U = T V (one 128-column accumulator) -> bf16,
//                written to a scratch array as the shared-memory images the
//                second kernel's operands need
//   delta_state_kernel  one CTA of 256 threads per (b, h), chunks in order; the
//       state kept transposed in TMEM (S^T: lane = key channel i, column =
//       value channel j, fp32) with a bf16 copy in shared memory. Per chunk:
//       round 3  X = W S0^T, P = Q K^T, then O = Q S0^T
//                -> Ut = U - X (bf16), masked P (bf16)
//       round 4  S^T += K^T Ut, O += P Ut -> the new bf16 copy of S^T
//       The tensor pipe runs products in issue order, so the state chain
//       (X, Ut, S^T, the bf16 copy) leads each round; a chunk's out rows are
//       read out of O while the next chunk's X and P run, before its O starts.
//       q, k (TMA tiles) and the chunk's W and U images (one bulk copy) come
//       in two sets; a set is refilled with chunk n + 2 as soon as chunk n's
//       state product has read it.
// Accumulators with 64 valid rows are M = 128 products whose rows 64..127 are
// not read; warps 0, 1, 4 and 5 (TMEM lanes 0..63) own those rows, the two
// warps of a lane quarter splitting the columns.
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
constexpr uint32_t kImg = 32768;             // scratch per chunk: W image | U image, 16 KiB each

// ---- delta_prep_kernel shared memory (offsets from a 1024-byte aligned base).
// The A operand of an M = 128 product reads 64 rows past its 64-row tile;
// every such tile is followed by at least 8 KiB of other data.
constexpr int kPrepThreads = 128;
constexpr uint32_t pK = 0, pV = 16384;   // [64 x 128] bf16 tiles, two 8 KiB halves
constexpr int kLd = 68;                  // fp32 row: 16-byte aligned, rows 4 banks apart
constexpr uint32_t kM = 32768;           // L = I + A, then L^-1 in place, fp32 [64][kLd];
constexpr uint32_t pT = kM;              // then T over it, K-major bf16 [64 x 64]
constexpr int kZd = 36;                         // Z row: 32 + 4, 16-byte aligned
constexpr uint32_t kY = kM + 64 * kLd * 4;      // merge products Z, fp32 [32][kZd]
constexpr uint32_t kB = kY + 32 * kZd * 4;      // beta [64]
constexpr uint32_t pBar = kB + 64 * 4;          // mbarriers (MMA, drain, tiles), TMEM address
constexpr uint32_t kPrepSmem = pBar + 32 + 1024;
// TMEM: A (64 columns), then W, then U, each read out before the next product
constexpr uint32_t pcA = 0, pcW = 0, pcU = 0, kPrepCols = 128;
constexpr int kPrepPerSm = 4;

// ---- delta_state_kernel shared memory
constexpr int kStateThreads = 256;
constexpr uint32_t kSet = 65536;                                   // one set: q, k, W, U
constexpr uint32_t sQo = 0, sKo = 16384, sWo = 32768, sUo = 49152;  // two 8 KiB halves each
constexpr uint32_t kP = 2 * kSet;          // P, K-major [64 x 64]
constexpr uint32_t kU = kP + 8192;         // Ut, MN-major [64 tokens x 128], two halves
constexpr uint32_t kS = kU + 16384;        // S^T copy, MN-major: 128 lines x 128 values, two 16 KiB halves
constexpr uint32_t kOs = kS + 32768;       // out rows of a chunk, bf16 [64 x 128] as two swizzled halves (TMA store)
constexpr uint32_t kBar = kOs + 16384;     // mbarriers P, X, S, O, drain, full[2], ofree; TMEM address
constexpr uint32_t kStateSmem = kBar + 80 + 1024;
constexpr uint32_t cS = 0, cX = 128, cO = 256, cP = 384, kStateCols = 512;
static_assert((kPrepSmem + 1024) * kPrepPerSm <= 233472 && kPrepCols * kPrepPerSm <= 512, "four prep CTAs per SM");
static_assert(64 * kLd * 4 >= 16384, "T's M = 128 operand reads 8 KiB past T inside the fp32 block");
static_assert(kStateSmem <= 232448, "state kernel shared memory");

__device__ unsigned int g_delta_tc_error;

// bulk global -> shared copy of `bytes` (a multiple of 16, both ends 16-byte
// aligned) that completes a transaction count on `bar`
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

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

// D = (neg ? -1 : 1) A B for N x N fp32 blocks (row-major, row strides lda,
// ldb, ldd multiples of 4 floats), two rows per thread: item (0 .. N^2 / 8 - 1)
// takes rows r and r + N / 2 (r = item / (N / 4)) and columns 4 (item % (N / 4))
// .. + 3. The two rows share every load of B: the shared-memory pipe is what
// bounds this kernel.
template <int N>
__device__ __forceinline__ void blk_mm2(float *D, int ldd, const float *A, int lda, const float *B, int ldb, int item,
                                        bool neg) {
    const int r = item / (N / 4), c0 = 4 * (item % (N / 4));
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
#pragma unroll 2
    for (int k4 = 0; k4 < N; k4 += 4) {
        const float4 a0 = *reinterpret_cast<const float4 *>(A + r * lda + k4);
        const float4 a1 = *reinterpret_cast<const float4 *>(A + (r + N / 2) * lda + k4);
        const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 b = *reinterpret_cast<const float4 *>(B + (k4 + e) * ldb + c0);
            acc0.x = fmaf(av0[e], b.x, acc0.x);
            acc0.y = fmaf(av0[e], b.y, acc0.y);
            acc0.z = fmaf(av0[e], b.z, acc0.z);
            acc0.w = fmaf(av0[e], b.w, acc0.w);
            acc1.x = fmaf(av1[e], b.x, acc1.x);
            acc1.y = fmaf(av1[e], b.y, acc1.y);
            acc1.z = fmaf(av1[e], b.z, acc1.z);
            acc1.w = fmaf(av1[e], b.w, acc1.w);
        }
    }
    const float s = neg ? -1.f : 1.f;
    *reinterpret_cast<float4 *>(D + r * ldd + c0) = make_float4(s * acc0.x, s * acc0.y, s * acc0.z, s * acc0.w);
    *reinterpret_cast<float4 *>(D + (r + N / 2) * ldd + c0) =
        make_float4(s * acc1.x, s * acc1.y, s * acc1.z, s * acc1.w);
}

// ============================================================================ W, U
struct PrepParams {
    CUtensorMap tk, tv;  // [BH][L][128] bf16 as {128, L, BH}, box {64, 64, 1}, 128-byte swizzle
    DeltaArgs a;
    uint8_t *img;
    int nch;
};

__global__ void __launch_bounds__(kPrepThreads, kPrepPerSm) delta_prep_kernel(const __grid_constant__ PrepParams p) {
    const DeltaArgs &a = p.a;
    uint8_t *img = p.img;
    const int nch = p.nch;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x / nch, n = blockIdx.x % nch, L = a.L;
    const int t0 = n * kC, nt = min(kC, L - t0);
    constexpr int kThreads = kPrepThreads;
    // L and L^-1 share one array: each block of L^-1 is written over the block of
    // L that no later step reads
    float *Lm = reinterpret_cast<float *>(sm + kM), *Li = Lm;
    float *Z = reinterpret_cast<float *>(sm + kY), *bs = reinterpret_cast<float *>(sm + kB);
    uint64_t *mb = reinterpret_cast<uint64_t *>(sm + pBar), *drain = mb + 1, *tiles = mb + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + pBar + 24);
    const bf16 *beta = static_cast<const bf16 *>(a.beta) + (size_t)bh * L + t0;
    const uint32_t sm0 = smem_u32(sm);
    const float bpre = tid < nt ? to_f32(beta[tid]) : 0.f;  // in flight with the tiles

    // this chunk's k and v tiles by TMA (rows past the sequence read as zeros)
    if (tid == 0) {
        mbar_init(mb, 1);
        mbar_init(drain, 1);
        mbar_init(tiles, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(tiles, 4 * 8192);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + pK + h * 8192, &p.tk, tiles, 64 * h, t0, bh);
            tma_load_3d(sm + pV + h * 8192, &p.tv, tiles, 64 * h, t0, bh);
        }
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, kPrepCols);
        tmem_relinquish();
    }
    if (tid < kC) bs[tid] = bpre;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int bad = __syncthreads_or(!mbar_wait(tiles, 0u, kWaitNs));
    uint32_t phase = 0;
    auto wait_mma = [&]() -> bool {
        const bool ok = mbar_wait(mb, phase & 1u, kWaitNs);
        ++phase;
        tc_fence_after();
        return ok;
    };

    while (!bad) {
        // ---------------------------------------------------------------- round 1: K K^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem + pcA, kmaj2(sm0 + pK, ks), kmaj2(sm0 + pK, ks), id64, ks > 0);
            umma_commit(mb);
        }
        if (__syncthreads_or(!wait_mma())) {
            bad = 1;
            break;
        }
        if (tid < kC) {
            // row t: L[t][s] = beta_t k_t . k_s (s < t), 1 (s = t), 0 (s > t)
            const int t = tid;
            const float bt = bs[t];
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + pcA, r0);
            tmem_ld32(tmem + lane_base + pcA + 32, r1);
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
        }
        tc_fence_before();
        __syncthreads();
        // ---------------------------------------------------------------- L^-1 by 16 x 16 blocks
        {
            // diagonal block b, column c: forward substitution of a unit
            // lower-triangular system; written over L's block once all are solved
            const int b = (tid >> 4) & 3, c = tid & 15, o = 16 * b;
            float x[16];
            if (tid < kC) {
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = r == c ? 1.f : 0.f;
#pragma unroll
                    for (int s = 0; s < r; ++s) acc = fmaf(-Lm[(o + r) * kLd + o + s], x[s], acc);
                    x[r] = r < c ? 0.f : acc;
                }
            }
            __syncthreads();
            if (tid < kC) {
#pragma unroll
                for (int r = 0; r < 16; ++r) Li[(o + r) * kLd + o + c] = x[r];
            }
        }
        __syncthreads();
        // Merges: for a unit lower-triangular [[P, 0], [R, Q]] with P^-1, Q^-1
        // known, the inverse's lower-left block is -Q^-1 (R P^-1). First the
        // pairs of 16 x 16 diagonal blocks (0, 1) and (2, 3), then the two
        // 32 x 32 halves; each product is written over blocks no later step reads.
        {
            // 2 x 32 items: warp 0 takes pair 0 (rows/cols 0..31), warp 1 pair 1 (32..63)
            const int pr = tid >> 5, it = tid & 31, o = 32 * pr;
            if (tid < 64)
                blk_mm2<16>(Z + pr * 16 * kZd, kZd, Lm + (o + 16) * kLd + o, kLd, Li + o * kLd + o, kLd, it, false);
            __syncthreads();
            if (tid < 64)
                blk_mm2<16>(Li + (o + 16) * kLd + o, kLd, Li + (o + 16) * kLd + o + 16, kLd, Z + pr * 16 * kZd, kZd,
                            it, true);
            __syncthreads();
        }
        blk_mm2<32>(Z, kZd, Lm + 32 * kLd, kLd, Li, kLd, tid, false);
        __syncthreads();
        blk_mm2<32>(Li + 32 * kLd, kLd, Li + 32 * kLd + 32, kLd, Z, kZd, tid, true);
        __syncthreads();
        // T = L^-1 diag(beta), lower triangular, bf16 K-major, written over the
        // fp32 block once every thread has read its share
        {
            uint4 tw[kC * 8 / kThreads];
            // a thread's eight columns are the same in every row it takes
            const float4 b0 = *reinterpret_cast<const float4 *>(bs + 8 * (tid & 7));
            const float4 b1 = *reinterpret_cast<const float4 *>(bs + 8 * (tid & 7) + 4);
#pragma unroll
            for (int u = 0; u < kC * 8 / kThreads; ++u) {
                const int x = u * kThreads + tid, t = x >> 3, c8 = x & 7;
                const float4 l0 = *reinterpret_cast<const float4 *>(Li + t * kLd + 8 * c8);
                const float4 l1 = *reinterpret_cast<const float4 *>(Li + t * kLd + 8 * c8 + 4);
                const float lv[8] = {l0.x * b0.x, l0.y * b0.y, l0.z * b0.z, l0.w * b0.w,
                                     l1.x * b1.x, l1.y * b1.y, l1.z * b1.z, l1.w * b1.w};
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int s = c8 * 8 + 2 * e;
                    w[e] = pack2(s <= t ? lv[2 * e] : 0.f, s + 1 <= t ? lv[2 * e + 1] : 0.f);
                }
                tw[u] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < kC * 8 / kThreads; ++u) {
                const int x = u * kThreads + tid, t = x >> 3, c8 = x & 7;
                *reinterpret_cast<uint4 *>(sm + pT + chunk_off(t, c8, 0)) = tw[u];
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---------------------------------------------------------------- round 2: W = T K, then U = T V
        // into the same accumulator; each becomes a bf16 image over the tile it
        // was made from (k after W's product, v after U's)
#pragma unroll 1
        for (int wu = 0; wu < 2 && !bad; ++wu) {
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + (wu ? pcU : pcW), kmaj1(sm0 + pT, ks), mnmaj(sm0 + (wu ? pV : pK), 8192, ks),
                              idKM, ks > 0);
                umma_commit(mb);
            }
            if (__syncthreads_or(!wait_mma())) {
                bad = 1;
                break;
            }
            if (tid < kC) {
                const int t = tid;
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tmem_ld32(tmem + lane_base + (wu ? pcU : pcW) + 32 * j, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
                        *reinterpret_cast<uint4 *>(sm + (wu ? pV : pK) + chunk_off(t, 4 * j + c4, 8192)) =
                            pack8(r + 8 * c4);
                }
            }
            fence_proxy_async_smem();  // the images leave by a bulk copy
            tc_fence_before();
            __syncthreads();
        }
        if (bad) break;
        // both images, 32 KiB, to the chunk's scratch slot: one bulk copy,
        // complete before the CTA's shared memory goes
        if (tid == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             img + ((size_t)bh * nch + n) * kImg),
                         "r"(sm0 + pK), "r"(kImg)
                         : "memory");
            bulk_commit();
            bulk_wait<0>();
        }
        break;
    }
    if (bad) {
        // every MMA issued has completed before the TMEM goes: a barrier of its
        // own, committed once, so its phase is known whatever timed out; and the
        // tile loads have landed (both bounded)
        if (tid == 0) {
            atomicOr(&g_delta_tc_error, 1u);
            umma_commit(drain);
        }
        __syncthreads();
        mbar_wait(drain, 0u, kWaitNs);
        mbar_wait(tiles, 0u, kWaitNs);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kPrepCols);
    }
}

// ============================================================================ state recurrence
struct StateParams {
    CUtensorMap tq, tk, to;  // [BH][L][128] bf16 as {128, L, BH}, box {64, 64, 1}, 128-byte swizzle
    DeltaArgs a;
    const uint8_t *img;
    int nch;
};

__global__ void __launch_bounds__(kStateThreads, 1) delta_state_kernel(const __grid_constant__ StateParams p) {
    const DeltaArgs &a = p.a;
    const uint8_t *img = p.img;
    const int nch = p.nch;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    constexpr int kThreads = kStateThreads;
    uint64_t *mbP = reinterpret_cast<uint64_t *>(sm + kBar), *mbX = mbP + 1, *mbS = mbP + 2, *mbO = mbP + 3;
    uint64_t *drain = mbP + 4, *full = mbP + 5;
    uint64_t *ofree = mbP + 7;  // the low warps have read the previous chunk's out rows (128 arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kBar + 64);
    const uint8_t *wu = img + (size_t)bh * nch * kImg;
    const uint32_t sm0 = smem_u32(sm);
    // lane quarter of the warp (TMEM lanes 32 qw .. 32 qw + 31) and its column half
    const int qw = warp & 3, hf = warp >> 2;
    const bool low = qw < 2;  // TMEM lanes 0..63: the 64 token rows
    const int t = 32 * qw + lane;  // token row (low warps) or key channel (all warps)
    // one thread of a high warp issues the MMAs, one of another the loads
    constexpr int kIssuer = 96, kProducer = 64;  // warp 3 lane 0, warp 2 lane 0
    const bool issuer = tid == kIssuer, producer = tid == kProducer;

    // chunk m's q and k tiles (TMA: rows past the sequence read as zeros) and
    // its W | U images (one bulk copy) into set m % 2, counted on full[m % 2]
    auto load = [&](int m) {
        const uint32_t so = (uint32_t)(m & 1) * kSet;
        uint64_t *bar = full + (m & 1);
        mbar_arrive_expect_tx(bar, kSet);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + so + sQo + h * 8192, &p.tq, bar, 64 * h, m * kC, bh);
            tma_load_3d(sm + so + sKo + h * 8192, &p.tk, bar, 64 * h, m * kC, bh);
        }
        bulk_load(sm0 + so + sWo, wu + (size_t)m * kImg, kImg, bar);
    };
    int issued = 0;  // loads issued (producer)

    if (warp == 0) {
        tmem_alloc(tmem_slot, kStateCols);
        tmem_relinquish();
    }
    if (issuer) {
        for (int b = 0; b < 7; ++b) mbar_init(mbP + b, 1);
        mbar_init(ofree, 128);
        fence_mbar_init();
    }
    // S0 = 0: the bf16 copy starts at zero
    for (int i = tid; i < 32768 / 16; i += kThreads) reinterpret_cast<uint4 *>(sm + kS)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // the tensor core reads the copy
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)(qw * 32) << 16;
    int bad = 0;
    const int nchunks = nch;
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
                *reinterpret_cast<uint4 *>(sm + kOs + chunk_off(t, 8 * hf + 4 * j + c4, 8192)) = pack8(r[j] + 8 * c4);
        fence_proxy_async_smem();
        return ok;
    };
    auto store_out = [&](int m) {  // one thread, after the low warps' barrier
        tma_store_3d(&p.to, sm + kOs, 0, m * kC, bh);
        tma_store_3d(&p.to, sm + kOs + 8192, 64, m * kC, bh);
        bulk_commit();
    };
    if (producer) {
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.to);
        for (; issued < min(2, nchunks); ++issued) load(issued);
    }
    for (int n = 0; n < nchunks; ++n) {
        const uint32_t ph = (uint32_t)n & 1u;
        const uint32_t set = sm0 + (uint32_t)(n & 1) * kSet;
        // this chunk's tiles (the previous chunk's closing barrier already
        // ordered its bf16 state copy before this round)
        int fail = !mbar_wait(full + (n & 1), (uint32_t)(n >> 1) & 1u, kWaitNs);
        // ---------------------------------------------------------------- round 3
        // X first (the state chain waits on it), then P; O = Q S0^T follows once
        // the previous chunk's out rows are read out of its accumulator
        if (issuer) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16(tmem + cX, kmaj2(set + sWo, ks), mnmaj(sm0 + kS, 16384, ks), idKM, ks > 0);
            umma_commit(mbX);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                umma_bf16(tmem + cP, kmaj2(set + sQo, ks), kmaj2(set + sKo, ks), id64, ks > 0);
            umma_commit(mbP);
        }
        // O is free once every low thread has read chunk n - 1's out rows and
        // staged them (an mbarrier, not a named barrier: the issuer's warp is
        // diverged while its lane 0 issues)
        if (low) {
            if (n > 0 && !read_out(n - 1)) fail = 1;
            tc_fence_before();
            mbar_arrive(ofree);
        }
        if (issuer || (tid == 0 && n > 0)) {
            if (!mbar_wait(ofree, ph, kWaitNs)) fail = 1;
            tc_fence_after();
            if (issuer) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(tmem + cO, kmaj2(set + sQo, ks), mnmaj(sm0 + kS, 16384, ks), idKM, ks > 0);
            } else {
                store_out(n - 1);
            }
        }
        if (low) {
            // Ut row t, value channels 64 hf .. 64 hf + 63: U - X, bf16 MN-major
            if (!mbar_wait(mbX, ph, kWaitNs)) fail = 1;
            tc_fence_after();
            __syncwarp();
            uint32_t r[2][32];
            tmem_ld32(tmem + lane_base + cX + 64 * hf, r[0]);
            tmem_ld32(tmem + lane_base + cX + 64 * hf + 32, r[1]);
            tmem_ld_wait();
            // the eight U chunks first: the stores below could alias them as far
            // as the compiler knows
            uint4 uu[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                uu[c] = *reinterpret_cast<const uint4 *>(sm + (set - sm0) + sUo + chunk_off(t, 8 * hf + c, 8192));
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int c8 = 8 * hf + 4 * j + c4;
                    const uint4 u4 = uu[4 * j + c4];
                    const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack2(__uint_as_float(uw[e] << 16) - __uint_as_float(r[j][8 * c4 + 2 * e]),
                                     __uint_as_float(uw[e] & 0xffff0000u) - __uint_as_float(r[j][8 * c4 + 2 * e + 1]));
                    *reinterpret_cast<uint4 *>(sm + kU + chunk_off(t, c8, 8192)) = make_uint4(w[0], w[1], w[2], w[3]);
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
                *reinterpret_cast<uint4 *>(sm + kP + chunk_off(t, 4 * hf + c4, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            // the staging tile is free again once the store has read it
            if (tid == 0) bulk_wait_read<0>();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (__syncthreads_or(fail)) {
            bad = 1;
            break;
        }
        // ---------------------------------------------------------------- round 4
        if (issuer) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(tmem + cS, mnmaj(set + sKo, 8192, ks), mnmaj(sm0 + kU, 8192, ks), idMM, (n > 0 || ks > 0));
            umma_commit(mbS);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_bf16(tmem + cO, kmaj1(sm0 + kP, ks), mnmaj(sm0 + kU, 8192, ks), idKM, 1);
            umma_commit(mbO);
        }
        {
            // S^T line i = t (TMEM lane), value channels 64 hf .. 64 hf + 63 ->
            // bf16 copy (every product that read the old copy came before mbS)
            if (!mbar_wait(mbS, ph, kWaitNs)) fail = 1;
            tc_fence_after();
            // every reader of this chunk's set is done (its products came before
            // mbS, the U rows were read before round 4): refill it with chunk n + 2
            if (producer && !fail && issued < nchunks) load(issued++);
            __syncwarp();  // the issuer's and the producer's warps come out of single-lane work
            uint32_t r[2][32];
            tmem_ld32(tmem + lane_base + cS + 64 * hf, r[0]);
            tmem_ld32(tmem + lane_base + cS + 64 * hf + 32, r[1]);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
                    *reinterpret_cast<uint4 *>(sm + kS + chunk_off(t, 8 * hf + 4 * j + c4, 16384)) = pack8(r[j] + 8 * c4);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(fail)) {
            bad = 1;
            break;
        }
    }
    // the last chunk's out rows
    if (!bad && low && nchunks > 0) {
        if (!read_out(nchunks - 1)) bad = 1;
        named_sync<2, 128>();
        if (tid == 0) store_out(nchunks - 1);
    }
    bad = __syncthreads_or(bad);
    if (!bad && a.final_state) {
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
            atomicOr(&g_delta_tc_error, 2u);
            umma_commit(drain);
        }
        if (producer) {
            // the last load of each set (every earlier one was waited for)
            for (int m = max(0, issued - 2); m < issued; ++m) mbar_wait(full + (m & 1), (uint32_t)(m >> 1) & 1u, kWaitNs);
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
    if (nbh * nch > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(delta_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrepSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(delta_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStateSmem) !=
            cudaSuccess)
        return LA_ERR_CUDA;
    StateParams sp;
    if (!get_encode() || !make_tile_map(&sp.tq, a.q, a.L, (int)nbh) || !make_tile_map(&sp.tk, a.k, a.L, (int)nbh) ||
        !make_tile_map(&sp.to, a.out, a.L, (int)nbh))
        return LA_ERR_CUDA;
    void *img = nullptr;
    if (scratch_alloc(&img, (size_t)nbh * nch * kImg, s) != LA_OK) return LA_ERR_CUDA;
    sp.a = a;
    sp.img = static_cast<const uint8_t *>(img);
    sp.nch = nch;
    PrepParams pp;
    pp.tk = sp.tk;
    if (!make_tile_map(&pp.tv, a.v, a.L, (int)nbh)) {
        cudaFreeAsync(img, s);
        return LA_ERR_CUDA;
    }
    pp.a = a;
    pp.img = static_cast<uint8_t *>(img);
    pp.nch = nch;
    int rc = LA_OK;
    delta_prep_kernel<<<(unsigned)(nbh * nch), kPrepThreads, kPrepSmem, s>>>(pp);
    if (cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
    if (rc == LA_OK) {
        ++*launches;
        delta_state_kernel<<<(unsigned)nbh, kStateThreads, kStateSmem, s>>>(sp);
        if (cudaGetLastError() != cudaSuccess) rc = LA_ERR_CUDA;
        else ++*launches;
    }
    if (cudaFreeAsync(img, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

}  // namespace la
