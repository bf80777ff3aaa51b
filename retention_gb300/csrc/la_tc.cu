// la_tc.cu -- the chunkwise forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), bf16 operands, fp32 accumulation and state.
//
// Method (learnllm m22 "The Three Faces of Retention"; linear_sparse_attention.py
// linear_attn_chunkwise; the gate A_t of learnllm m22 "Interactive Exploration").
// Inside chunk n (c <= 64 tokens, local index t), with b_t[d] the inclusive
// running sum of log A over the chunk:
//
//   q~_t = phi(q_t) e^{b_t}          k~_s = phi(k_s) e^{-b_s}
//   P    = causal_mask(q~ k~^T)      (= sum_d phi(q)phi(k) e^{b_t - b_s}, s <= t)
//   O    = q~ S_{n-1} + P V
//   T_n  = S_{n-1} + k~^T V,         S_n = diag(e^{b_last}) T_n
//
// which is the chunkwise form with the decay from the chunk start to t split
// into a query factor and a key factor (exact in real arithmetic). For linear
// attention b = 0 and every factor is 1; for retention b_t = (t+1) ln gamma,
// and the rescale of the state is deferred to the end of a window of chunks
// (the accumulator holds S / gamma^(64 m), m chunks into the window, and the q
// and k rows carry the matching gamma^(+-64 m)).
//
// The normaliser z is the state's column for a value that is always 1
// (z_t = A_t z_{t-1} + phi(k_t)). With LA_NORMALIZE, V is widened by a
// constant column of ones (N = 144 instead of 128), so the same MMAs carry z in
// column 128 of the state and produce den_t = rowsum(P)_t + q~_t . z_{n-1} in
// column 128 of O: out_t = O[t][0..127] / O[t][128].
//
// Tensor-core work per chunk (all M = 128, fp32 accumulators in TMEM, NW = 128
// or 144 value columns):
//   QK    D_P [128 x 64]  = q~ (K-major, rows 64..127 unused) . k~^T (K-major)
//   state D_S [128 x NW] += k~^T (MN-major) . [V | 1] (MN-major)     -> T_n
//   inter D_O [128 x NW]  = q~ (K-major) . S' (MN-major bf16 copy of S_{n-1})
//   intra D_O            += P (K-major bf16 P) . [V | 1] (MN-major)
// q, k, v come straight from the 128-byte-swizzled TMA tiles; the threads write
// the bf16 copies of P and S_{n-1} in the same layout.
//
// One CTA per (b, h), 16 warps with fixed roles, connected by mbarriers:
//   warp 2       TMA producer: q, k, v (, g) tiles of chunk n into a ring of stages
//   warp 3       MMA issuer (one thread) and TMEM owner
//   warps 4-7, 0, 1, 14, 15  prologue (256 threads, two warps per SM
//                sub-partition): phi and decay factors in place on the q and k tiles
//   warps 8-11   state chain: S_{n-1} = diag(f) T_{n-1} (rescaled in TMEM;
//                retention only at a window's end) and its bf16 copy for the
//                inter MMA of chunk n; the final state
//   warps 12-13  outputs: P mask -> bf16; O -> 1/den -> bf16 -> TMA store
// O lives in two TMEM buffers (one with the normaliser, whose 144-column
// accumulators leave no room for a second), so chunk n+1's MMAs overlap chunk
// n's epilogue, and the state chain of chunk n+1 overlaps both.
//
// Every wait on an mbarrier is bounded (2 s of wall time); a role that runs
// out leaves its loop (inside a warpgroup the decision is made uniform with
// bar.red.or), sets a device error word and the CTA drains what it issued.
#include <cudaTypedefs.h>
#include <cstring>
#include <mutex>

#include "la_common.cuh"
#include "sm100.cuh"

namespace la {
namespace {
using namespace sm100;

constexpr int kC = 64;                   // chunk length
constexpr int kD = 128;                  // d_k = d_v
constexpr int kThreads = 512;            // 16 warps
constexpr uint32_t kTile = kC * kD * 2;  // bf16 [64 x 128] tile: 16 KiB = two 8 KiB swizzle blocks
constexpr uint32_t kHalf = 8192;
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // default wait limit: far beyond any legitimate wait
constexpr int kBarPro = 1, kBarState = 2, kBarOut = 3, kBarP = 4;  // named barrier ids
// The producer and the MMA issuer sit on the SM sub-partitions (warp % 4) that
// host the fewest busy warps, so their short instruction streams issue promptly.
constexpr int kWarpProducer = 2, kWarpMma = 3;

__device__ unsigned int g_tc_error;
__device__ unsigned int g_tc_debug;  // LA_DEBUG: source line of the first failed bounds check
#ifdef LA_DEBUG
#define TC_CHECK(cond) LA_CHECK(g_tc_debug, cond)
#else
#define TC_CHECK(cond) true
#endif

struct TcParams {
    CUtensorMap tq, tk, tv, tg, to;
    CUtensorMap tog;          // the RetNet output gate og (fused epilogue instances)
    const float *gn_w, *gn_b; // GroupNorm weight and bias [H][128] or null
    float gn_eps;
    const float *gamma;
    float *final_state;      // [BH][blk], written by the full pass's last segment of each sequence
    const float *state_in;   // [BH][nseg][blk]: state at each segment start (full pass)
    float *seg_state;        // [BH][nseg][blk]: segment-local end state (state-only pass)
    float *seg_logdecay;     // [BH][nseg][128]: log decay over each segment (state-only pass)
    int H, L, mode, nseg, seg_chunks;
    int init0;               // segment 0 starts from state_in too (a given initial state)
    uint64_t wait_ns;        // limit of every bounded wait (kWaitNs)
    int stall_chunk;         // diagnostics: the producer stops before this chunk (-1: never)
    float *e_out;             // (backward prep) e_t per token, [BH][L]
    const float *e_in;        // (bias instances) e_t per token, [BH][L]
    // extents (floats) of the global arrays, for the bounds checks of LA_DEBUG builds
    size_t n_final, n_state_in, n_seg_state, n_seg_logdecay, n_e;
};

constexpr uint32_t kSmemBudget = 232448;  // dynamic shared memory of one CTA

// Shared-memory layout. Tiles are [64 x 128] bf16, kept as two 8 KiB swizzle
// blocks (columns 0..63 and 64..127) that need not be adjacent.
//
// State-only pass (no q, P, S' or O): contiguous stages k | v | (ones) | (g),
// as many as the budget allows (at most 6).
//
// Full pass: stage s holds q, k, v as six blocks whose indices come from a
// table (one byte per stage in a 32-bit constant). Without the normaliser the
// stages are contiguous. With it, one constant ones block T serves every
// stage: [V | 1] reaches its three N atoms at v0, v0 + LBO, v0 + 2 LBO, so
// stage s puts v1 at T - d and v0 at T - 2d (d = 1, 3, 5), and q, k take the
// remaining blocks in order. The gate tiles g have a ring of their own (GR):
// the prologue is done with g after its first pass, so g is released early
// and the next chunk's g is already in place when the prologue turns to it.
template <int GATE, bool NORM, bool SO, bool OF32 = false, int EPI = 0, int BIAS = 0>
struct Layout {
    static constexpr bool GR = GATE >= 2 && !SO;
    // gated without the normaliser: three q|k|v stages and one gate slot fit;
    // with it, two stages and two gate slots
    static constexpr int NG = GR ? (NORM ? 2 : 1) : 0;          // gate ring slots
    // state-only stage: k | v | (ones) | (g)
    static constexpr uint32_t so_stage = 2 * kTile + (NORM ? kHalf : 0) + (GATE >= 2 ? kTile : 0);
    // room kept for the float arrays, barriers and alignment slack below
    static constexpr uint32_t kReserve = 8192;
    static constexpr int NS = !SO ? ((NORM && (GATE != 0 || EPI != 0)) ? 2 : 3)
                                  : ((kSmemBudget - kReserve) / so_stage < 6 ? (kSmemBudget - kReserve) / so_stage : 6);
    static constexpr int T = 6 * NS;  // the shared ones block (full pass with the normaliser)
    static constexpr uint32_t pack(int a, int b, int c) {
        return (uint32_t)a | ((uint32_t)b << 8) | ((uint32_t)c << 16);
    }
    // block table of the full pass: half h of tile tl (0 q, 1 k, 2 v), one byte per stage
    static constexpr uint32_t table(int tl, int h) {
        return !NORM    ? pack(2 * tl + h, 6 + 2 * tl + h, 12 + 2 * tl + h)
               : tl == 2 ? (h ? pack(T - 1, T - 3, T - 5) : pack(T - 2, T - 6, T - 10))
               : NS == 3 ? (tl == 0 ? (h ? pack(1, 5, 10) : pack(0, 4, 9)) : (h ? pack(3, 7, 14) : pack(2, 6, 11)))
                         : (tl == 0 ? (h ? pack(1, 5, 0) : pack(0, 4, 0)) : (h ? pack(3, 8, 0) : pack(2, 7, 0)));
    }
    static constexpr uint32_t stages = SO ? NS * so_stage : (6 * NS + (NORM ? 1 : 0)) * kHalf;
    static constexpr uint32_t Gring = stages;                              // [NG] g tiles
    static constexpr uint32_t P = Gring + NG * kTile;                      // bf16 P tile, 8 KiB
    static constexpr uint32_t S = P + (SO ? 0 : 8192);                     // bf16 S_{n-1} (+ z atom), 32 / 48 KiB
    static constexpr uint32_t O = S + (SO ? 0 : (NORM ? 49152 : 32768));   // O staging: bf16 halves or fp32 quarters
    // floats: ffinal[128], then with a gate fbuf[NF][128], with the head gate
    // fq[64] fk[64], with the channel gate tot[4][128] (normalised) or
    // tot[2][4][128] (two chunks' quarter sums). fbuf is a ring of
    // NF = NS + 1 slots: chunk n's decay factor goes to slot n % NF at the end of
    // its prologue, for the state chain to rescale T_n with.
    static constexpr int NF = NS + 1;
    // (EPI, BIAS) a second staging buffer: chunk n is staged in buffer n % 2,
    // where its og tile (EPI) or x tile (BIAS with elu+1) lands first and the
    // chunk's result is written over it
    static constexpr uint32_t O2 = O + (SO ? 0 : (OF32 ? 32768 : 16384));
    static constexpr uint32_t F = O2 + ((!SO && (EPI || BIAS)) ? 16384 : 0);
    static constexpr uint32_t nfbuf = GATE != 0 ? NF * 128 : 0, nfq = GATE == 1 ? 128 : 0;
    static constexpr uint32_t ntot = GATE >= 2 ? (NORM ? 512 : 1024) : 0;  // quarter sums (one or two chunks)
    static constexpr uint32_t nwb = EPI ? 512 : 0;  // GroupNorm weight, bias [128] each; half-row (m, M2) [2][64][2]
    // (bias instances) per-chunk column sums [NF][128], the carried vector [128],
    // e of the chunk's tokens for the prologue [64] and for the output role [64]
    static constexpr uint32_t nbias = BIAS ? (NF * 128 + 128 + 64 + 64) : 0;
    static constexpr uint32_t Bar = F + (128 + nfbuf + nfq + ntot + nwb + nbias) * 4;
    // full, empty, pro [NS]; ofull, oempty [2]; qk, pfull, pempty, sdone, sfree, sready, profinal,
    // drain; gfull, gempty [NG]; ffull [NF]; (ogfull [2]: the og or x tiles; cfull, cempty [NF])
    static constexpr uint32_t nbar = 3 * NS + 12 + 2 * NG + NF + ((EPI || BIAS) ? 2 : 0) + (BIAS ? 2 * NF : 0);
    static constexpr uint32_t Misc = Bar + nbar * 8;  // TMEM base address
    static constexpr uint32_t bytes = Misc + 16 + 1024;  // + slack for the 1024-byte alignment
    // TMEM columns (region bases 32-column aligned). With the ones column the
    // state and O accumulators are 144 wide and O has a single buffer.
    static constexpr uint32_t NW = NORM ? 144 : 128;
    static constexpr int NOB = NORM ? 1 : 2;           // O accumulator buffers
    static constexpr uint32_t colS = 0;
    static constexpr uint32_t colO0 = NORM ? 160 : 128;
    static constexpr uint32_t colO1 = NORM ? 160 : 256;
    static constexpr uint32_t colP = NORM ? 320 : 384;
};

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// The hardware base-2 exponential and logarithm (denormals flushed: the gate
// factors they make are far from the denormal range, and an underflowing e^-|g|
// only drops a term below rounding).
__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
// two fp32 values in one 64-bit register pair, for the packed fp32x2 arithmetic
typedef unsigned long long f32x2_t;
__device__ __forceinline__ f32x2_t f2(float lo, float hi) {
    f32x2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f32x2_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2_t f2_add(f32x2_t a, f32x2_t b) {
    f32x2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2_t f2_mul(f32x2_t a, f32x2_t b) {
    f32x2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f32x2_t f2_fma(f32x2_t a, f32x2_t b, f32x2_t c) {
    f32x2_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// log2 of the channel gate alpha = exp(logsigmoid(g) / 16),
//   (min(g, 0) log2(e) - log2(1 + 2^(-|g| log2(e)))) / 16,
// for both channels of one packed bf16 word, the fp32 arithmetic around the
// hardware exponential and logarithm done two channels at a time
// (g = +huge gives 0: no decay)
__device__ __forceinline__ f32x2_t log2_alpha2(uint32_t w) {
    const f32x2_t a = f2(__uint_as_float((w << 16) & 0x7fffffffu), __uint_as_float(w & 0x7fff0000u));  // |g|
    float t0, t1, u0, u1;
    f2_split(f2_mul(a, f2(-kLog2e, -kLog2e)), t0, t1);
    f2_split(f2_add(f2(ex2f(t0), ex2f(t1)), f2(1.f, 1.f)), u0, u1);
    const f32x2_t m = f2(fminf(__uint_as_float(w << 16), 0.f), fminf(__uint_as_float(w & 0xffff0000u), 0.f));
    return f2_fma(m, f2(kLog2e * 0.0625f, kLog2e * 0.0625f), f2_mul(f2(lg2f(u0), lg2f(u1)), f2(-0.0625f, -0.0625f)));
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// swish(u) = u sigmoid(u) = h + h tanh(h), h = u / 2, on two packed bf16
// values with the hardware tanh approximation (the output is bf16 either way)
__device__ __forceinline__ uint32_t swish_bf16x2(uint32_t u) {
    const uint32_t half = 0x3F003F00u;  // bf16 0.5 in both halves
    uint32_t h, th, r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(h) : "r"(u), "r"(half));
    asm("tanh.approx.bf16x2 %0, %1;" : "=r"(th) : "r"(h));
    asm("fma.rn.bf16x2 %0, %1, %2, %1;" : "=r"(r) : "r"(h), "r"(th));
    return r;
}
// two fp32 values rounded to one packed bf16 word (lo in the low half)
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// elu(x) + 1 on two packed bf16 values in bf16 arithmetic:
// max(x, 0) + 2^(min(x, 0) * log2 e). The exponent argument is rounded to bf16,
// so for x < 0 the result carries a relative error below 2^-8 |x| on top of the
// bf16 rounding the tensor-core operand needs anyway.
__device__ __forceinline__ uint32_t phi_elu1_bf16x2(uint32_t x) {
    const uint32_t zero = 0u, log2e = 0x3FB93FB9u;  // bf16(log2 e) in both halves
    uint32_t m, y, e, pos, r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(x), "r"(zero));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(m), "r"(log2e));
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(pos) : "r"(x), "r"(zero));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(pos), "r"(e));
    return r;
}

// phi'(x) = e^min(x, 0) of two bf16 values, in the arithmetic phi_elu1_bf16x2
// takes for its exponential part
__device__ __forceinline__ uint32_t dphi_elu1_bf16x2(uint32_t x) {
    const uint32_t zero = 0u, log2e = 0x3FB93FB9u;
    uint32_t m, y, e;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(x), "r"(zero));
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(m), "r"(log2e));
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(y));
    return e;
}

// SO (state only): the first pass over a split sequence. Each CTA runs one
// segment from a zero state and keeps only the state update (no QK, no
// outputs): it writes the segment's end state and its total log decay.
//
// REV (anti-causal): out_s = sum_{t >= s} A(s -> t) (q_s . k_t) v_t, the sum
// over the token and every later one, with the scalar decay gamma^(t - s).
// It is the causal form in mirrored coordinates: chunks are taken from the last
// one (so the ragged chunk comes first), the local index of row r of a chunk of
// c tokens is c - 1 - r, and the mask keeps key columns at or after the query
// row. The state carried from chunk to chunk is then the sum over all later
// tokens, decayed to the start of the chunk after the current one.
//
// EPI = 1: the RetNet output epilogue in the output role's store (learnllm m22
// "Retention": a GroupNorm per head and a swish output gate),
//   out_t = swish(og_t) * ((o_t - mean) / sqrt(var + eps) * weight[h] + bias[h]),
// mean and the biased variance over the 128 values of row t, from the fp32
// accumulator. Each output thread owns one token row, so the statistics need
// no exchange between threads; the og tile comes by TMA into the staging
// buffer, and each row is overwritten in place by its result.
//
// EPI = 2: the first step of the normalised backward, in the same store: with
// num_t (columns 0..127 of O) and den_t (column 128) of the normalised forward
// and the output gradient g_t (its tile by TMA, like og), each row writes
//   w_t = g_t / den_t            (bf16, the call's output tensor)
//   e_t = -(g_t . num_t) / den_t^2   (fp32, one value per token)
// num_t never leaves the accumulator, so e_t, a difference the later
// gradients cancel against, is formed from fp32 values.
//
// BIAS (the later steps of the normalised backward; identity features, no
// gate, no normaliser): one more term e_t on every score, carried into the
// output by a vector of value-row sums,
//   BIAS = 1 (causal):      out_t = sum_{s<=t} (q_t . k_s + e_t) v_s
//                                 = [causal form]_t + e_t (sum_{s<=t} v_s)
//   BIAS = 2 (anti-causal): out_s = sum_{t>=s} (q_s . k_t + e_t) v_t
//                                 = [anti-causal form]_s + sum_{t>=s} e_t v_t
// Inside a chunk e rides on P before the mask; the sum over earlier chunks
// (later ones with REV) is a carried vector added to each output row. The
// prologue forms each chunk's weighted column sums of the value tile while it
// holds the stage.
template <int GATE, bool ELU1, bool NORM, bool SO, bool OF32 = false, bool REV = false, int EPI = 0, int BIAS = 0>
__global__ void __launch_bounds__(kThreads, 1) la_chunk_tc_kernel(const __grid_constant__ TcParams p) {
    using LY = Layout<GATE, NORM, SO, OF32, EPI, BIAS>;
    // (the value-side gate: with ELU1 the feature map applies to the value tile,
    // the one its prologue scales, and q and k are taken as given)
    static_assert(GATE != 3 || !NORM, "the value-side gate: no normaliser");
    static_assert(!REV || (GATE <= 1 && !NORM && (!ELU1 || GATE == 0)) || (GATE >= 2 && !NORM && !OF32),
                  "the anti-causal instance: a scalar decay, or the channel gate");
    static_assert(EPI != 1 || (GATE <= 1 && !NORM && !SO && !OF32 && !REV), "the fused epilogue: bf16 output, no normaliser");
    static_assert(EPI != 2 || (GATE == 0 && NORM && !SO && !OF32 && !REV), "the backward prep: the normalised causal form");
    static_assert(BIAS == 0 || (GATE == 0 && !NORM && !OF32 && EPI == 0 && REV == (BIAS == 2)),
                  "the bias instances: no gate or normaliser, bf16 output");
    // (bias instances with ELU1) the feature map applies to the value tile, the
    // query and key tiles are taken as given, and each output row is multiplied
    // by phi'(x_t) = e^min(x_t, 0), x the tile of the map tog (the feature map's
    // input whose gradient this is), which TMA brings to the staging buffer
    constexpr bool PHIV = BIAS != 0 && ELU1;
    // SPLIT (the fused epilogue, the bias instances): P and the outputs are
    // separate roles, so P of chunk n + 1 is formed while chunk n's outputs are
    // finished. TMEM lanes 0..63 (the token rows) are reachable from SM
    // sub-partitions 0 and 1 only: warps 12 and 13 make P, warps 0, 1, 4 and 5
    // finish the outputs, half a row each, and the prologue moves to warps 6, 7,
    // 14 and 15 (sub-partitions 2 and 3). Otherwise the prologue runs on warps
    // 4-7, 0, 1, 14, 15 and warps 12 and 13 make P and the outputs in turn. (The
    // split layout measured slower for the plain forms: the prologue's work then
    // has the special function units of two sub-partitions only.)
    constexpr bool SPLIT = !SO && (EPI != 0 || BIAS != 0);
    constexpr int PT = SPLIT ? 128 : 256;  // prologue threads
    constexpr int NS = LY::NS;
    constexpr int NG = LY::GR ? LY::NG : 1;  // gate ring slots (the ring exists only if GR)
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, formed by pointer arithmetic on the shared array so
    // that every access below stays a shared-memory access (an integer round
    // trip would turn them into generic loads and stores)
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t wait_ns = p.wait_ns;  // limit of every bounded wait
    // CTA = (b, h, segment); a segment is seg_chunks consecutive chunks
    // (the state-only pass has no CTA for a sequence's last segment: the full
    // pass holds that segment's end state, which is the final state)
    const int gseg = SO ? p.nseg - 1 : p.nseg;  // this grid's segments per sequence
    const int bh = blockIdx.x / gseg, seg = blockIdx.x % gseg, h = bh % p.H, L = p.L;
    const int sgi = bh * p.nseg + seg;  // segment index in the scratch arrays
    const int c0 = seg * p.seg_chunks;
    const int nch = (L + kC - 1) / kC;
    const int N = max(0, min(p.seg_chunks, nch - c0));
    // first token of the n-th chunk this CTA takes (from the end with REV)
    auto chunk_t0 = [&](int n) { return (REV ? nch - 1 - (c0 + n) : c0 + n) * kC; };
    // first row of the gate tile of the chunk at t0: with REV and the channel
    // gate, token t of the mirrored sequence decays by the gate of token t + 1
    // (a tile wholly past the end is never read: every row of it is masked)
    auto gy = [&](int t0) { return (REV && GATE >= 2) ? min(t0 + 1, L - 1) : t0; };
    const bool init = !SO && p.state_in != nullptr && (seg > 0 || p.init0);  // start from a carried state
    // state block: S (+ z with the normaliser; + the carried vector of the bias
    // instances, for the segments of a split sequence)
    const size_t blk = (size_t)kD * kD + (NORM ? kD : 0) + (BIAS ? kD : 0);
    const size_t segblk = (size_t)sgi * blk;

    constexpr int NF = LY::NF;
    float *ffinal = reinterpret_cast<float *>(sm + LY::F);  // [128] e^{b_last} of the last chunk
    float *fbuf = ffinal + 128;                             // [NF][128] chunk n's decay factor e^{b_last(n)}
    float *fq = fbuf + LY::nfbuf;                           // [64] retention: gamma^(t+1)
    float *fk = fq + 64;                                    // [64] retention: gamma^-(t+1)
    float *tot = fq + LY::nfq;                              // [1 or 2][4][128] gated: per-quarter log2 decay sums
    float *gnw = tot + LY::ntot, *gnb = gnw + 128;          // (EPI) GroupNorm weight and bias of head h
    float *csum = gnw + LY::nwb;                            // (BIAS) [NF][128] weighted column sums of V per chunk
    float *cvec = csum + (BIAS ? NF * 128 : 0);             // (BIAS) [128] the carried vector
    float *pebuf = cvec + (BIAS ? 128 : 0);                 // (BIAS) [64] e of the prologue's chunk
    float *oebuf = pebuf + (BIAS ? 64 : 0);                 // (BIAS) [64] e of the output role's chunk
    // Shared-memory offset of half h (columns 64h..64h+63) of tile tl of stage
    // s: tl = 0 q, 1 k, 2 v, 3 g (the g tile of a state-only stage)
    auto tile_half = [&](int tl, int s, int h) -> uint32_t {
        if constexpr (SO) {
            const uint32_t base = s * LY::so_stage + h * kHalf;
            return tl == 1 ? base : tl == 2 ? base + kTile : base + 2 * kTile + (NORM ? kHalf : 0);
        } else {
            return ((LY::table(tl, h) >> (8 * s)) & 255u) * kHalf;
        }
    };
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + LY::Bar);
    uint64_t *full = bars, *empty = bars + NS, *pro = bars + 2 * NS;
    uint64_t *ofull = bars + 3 * NS, *oempty = ofull + 2;
    uint64_t *qk = oempty + 2, *pfull = qk + 1, *pempty = pfull + 1, *sdone = pempty + 1, *sfree = sdone + 1;
    uint64_t *sready = sfree + 1, *profinal = sready + 1, *drain = profinal + 1;
    uint64_t *gfull = drain + 1, *gempty = gfull + LY::NG;  // (empty arrays unless GR)
    uint64_t *ffull = gempty + LY::NG;                      // [NF]: fbuf slot written
    uint64_t *ogfull = ffull + NF;                          // (EPI, BIAS) [2]: og / x tile in staging buffer 0 / 1
    uint64_t *cfull = ogfull + ((EPI || BIAS) ? 2 : 0);     // (BIAS) [NF]: csum slot written
    uint64_t *cempty = cfull + (BIAS ? NF : 0);             // (BIAS) [NF]: csum slot read
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + LY::Misc);
    uint8_t *sP = sm + LY::P, *sS = sm + LY::S, *sO = sm + LY::O;

    // Checked accesses: in an LA_DEBUG build every shared-memory range, TMA
    // coordinate, TMEM address and global index below is compared with its
    // extent first, and a failed check skips the access (and records its line);
    // in the ordinary build each check is the constant true.
    [[maybe_unused]] const uint32_t sm_lo = smem_u32(sm), sm_hi = smem_u32(smem_raw) + LY::bytes;
    [[maybe_unused]] const int nbh_grid = (int)gridDim.x / gseg;
    auto sok = [&](const void *ptr, uint32_t n) {
        return TC_CHECK(smem_u32(ptr) >= sm_lo && smem_u32(ptr) + n <= sm_hi);
    };
    auto gok = [&](size_t i, size_t n) { return TC_CHECK(i < n); };
    // a [64 x 64] bf16 box (or [64 x 32] fp32): inner coordinate on a 16-byte boundary
    auto tma_in = [&](const void *s_ptr, int x, int y) {
        return TC_CHECK(smem_u32(s_ptr) >= sm_lo && smem_u32(s_ptr) + kHalf <= sm_hi && x >= 0 && x < kD &&
                        (x & 7) == 0 && y >= 0 && y < L && bh < nbh_grid);
    };
    auto tload = [&](void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
        if (tma_in(dst, x, y)) tma_load_3d(dst, map, bar, x, y, bh);
    };
    auto tstore = [&](const CUtensorMap *map, const void *src, int x, int y) {
        if (tma_in(src, x, y)) tma_store_3d(map, src, x, y, bh);
    };

    if (warp == kWarpMma) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&pro[s], PT);
        }
        for (int sg = 0; sg < LY::NG; ++sg) {
            mbar_init(&gfull[sg], 1);
            mbar_init(&gempty[sg], 256);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ofull[b], 1);
            mbar_init(&oempty[b], SPLIT ? 128 : 64);
        }
        mbar_init(qk, 1);
        mbar_init(pfull, 64);
        mbar_init(pempty, 64);
        mbar_init(sdone, 1);
        mbar_init(sfree, 1);
        mbar_init(sready, 128);
        mbar_init(profinal, GATE >= 2 ? 64 : 128);
        for (int j = 0; j < NF; ++j) mbar_init(&ffull[j], GATE >= 2 ? 64 : 128);
        if (EPI || BIAS) {
            mbar_init(&ogfull[0], 1);
            mbar_init(&ogfull[1], 1);
        }
        if (BIAS)
            for (int j = 0; j < NF; ++j) {
                mbar_init(&cfull[j], 16);  // one arrival per 8-column group
                mbar_init(&cempty[j], 1);
            }
        mbar_init(drain, 1);
        fence_mbar_init();
        tma_prefetch_desc(&p.tq);
        tma_prefetch_desc(&p.tk);
        tma_prefetch_desc(&p.tv);
        tma_prefetch_desc(&p.to);
        if (GATE >= 2) tma_prefetch_desc(&p.tg);
        if (EPI || PHIV) tma_prefetch_desc(&p.tog);
    }
    if (NORM) {
        // constant blocks: the [64 x 64] atom(s) whose column 0 is 1 (the ones
        // column of [V | 1]: one per state-only stage, one shared by the full
        // pass's stages); the z atom of the S' copy starts at zero
        constexpr int nones = SO ? NS : 1;
        for (int i = tid; i < nones * 512; i += kThreads) {
            const int s = i >> 9, r = (i >> 3) & 63, pc = i & 7;
            const uint32_t one = (((pc ^ r) & 7) == 0) ? 0x3f80u : 0u;  // bf16 1.0 in element 0
            const uint32_t base = SO ? s * LY::so_stage + 2 * kTile : LY::T * kHalf;
            uint8_t *pw16 = sm + base + r * 128 + pc * 16;
            if (sok(pw16, 16)) *reinterpret_cast<uint4 *>(pw16) = make_uint4(one, 0u, 0u, 0u);
        }
        if (!SO)
            for (int i = tid; i < 1024; i += kThreads)
                reinterpret_cast<uint4 *>(sS + 32768)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    int bad = 0;
    // TMEM: a warp reaches its own lane quarter only, columns inside the allocation
    auto tok = [&](uint32_t ta, uint32_t ncols) {
        return TC_CHECK((ta >> 16) == (uint32_t)((warp & 3) * 32) && (ta & 0xFFFFu) >= (tmem & 0xFFFFu) &&
                        (ta & 0xFFFFu) + ncols <= (tmem & 0xFFFFu) + kTmemCols);
    };
    auto tld32 = [&](uint32_t ta, uint32_t(&r)[32]) {
        if (tok(ta, 32)) tmem_ld32(ta, r);
    };
    auto tst32 = [&](uint32_t ta, const uint32_t(&r)[32]) {
        if (tok(ta, 32)) tmem_st32(ta, r);
    };
    auto tld8 = [&](uint32_t ta, uint32_t(&r)[8]) {
        if (tok(ta, 8)) tmem_ld8(ta, r);
    };
    auto tld1 = [&](uint32_t ta, uint32_t &r) {
        if (tok(ta, 1)) tmem_ld1(ta, r);
    };
    auto tst1 = [&](uint32_t ta, uint32_t r) {
        if (tok(ta, 1)) tmem_st1(ta, r);
    };
    // shared-memory words at computed offsets (a skipped load reads zero)
    auto ld4 = [&](const uint8_t *ptr) { return sok(ptr, 4) ? *reinterpret_cast<const uint32_t *>(ptr) : 0u; };
    auto st4 = [&](uint8_t *ptr, uint32_t v) {
        if (sok(ptr, 4)) *reinterpret_cast<uint32_t *>(ptr) = v;
    };
    auto ld16 = [&](const uint8_t *ptr) {
        return sok(ptr, 16) ? *reinterpret_cast<const uint4 *>(ptr) : make_uint4(0u, 0u, 0u, 0u);
    };
    auto st16 = [&](uint8_t *ptr, uint4 v) {
        if (sok(ptr, 16)) *reinterpret_cast<uint4 *>(ptr) = v;
    };

    if (warp == kWarpProducer) {
        // ============================================================ TMA producer
        if (lane == 0) {
            int issued = 0, gissued = 0;
            constexpr int ntl = (GATE >= 2 && !LY::GR) ? 4 : 3;  // q, k, v (, g) tiles of a stage
            for (int n = 0; n < N; ++n) {
                // diagnostics only: no tiles from chunk stall_chunk on, so that the
                // other roles' bounded waits run out
                if (p.stall_chunk >= 0 && n >= p.stall_chunk) break;
                const int s = n % NS;
                const int t0 = chunk_t0(n);
                if constexpr (LY::GR) {
                    // g of chunk n goes out before chunk n's stage is waited for
                    const int sg = n % NG;
                    if (n >= NG && !mbar_wait(&gempty[sg], (uint32_t)(n / NG - 1) & 1u, wait_ns)) {
                        bad = 1;
                        break;
                    }
                    uint8_t *dst = sm + LY::Gring + sg * kTile;
                    mbar_arrive_expect_tx(&gfull[sg], kTile);
                    tload(dst, &p.tg, &gfull[sg], 0, gy(t0));
                    tload(dst + kHalf, &p.tg, &gfull[sg], 64, gy(t0));
                    gissued = n + 1;
                }
                if (n >= NS && !mbar_wait(&empty[s], (uint32_t)(n / NS - 1) & 1u, wait_ns)) {
                    bad = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], (ntl - (SO ? 1 : 0)) * kTile);
#pragma unroll 1
                for (int tl = SO ? 1 : 0; tl < ntl; ++tl) {
                    const CUtensorMap *m = tl == 0 ? &p.tq : tl == 1 ? &p.tk : tl == 2 ? &p.tv : &p.tg;
                    const int y = tl == 3 ? gy(t0) : t0;
                    tload(sm + tile_half(tl, s, 0), m, &full[s], 0, y);
                    tload(sm + tile_half(tl, s, 1), m, &full[s], 64, y);
                }
                issued = n + 1;
            }
            // nothing may still be landing in shared memory when the CTA leaves
            for (int m = issued > NS ? issued - NS : 0; m < issued; ++m)
                if (!mbar_wait(&full[m % NS], (uint32_t)(m / NS) & 1u, wait_ns)) bad = 1;
            for (int m = gissued > NG ? gissued - NG : 0; m < gissued; ++m)
                if (!mbar_wait(&gfull[m % NG], (uint32_t)(m / NG) & 1u, wait_ns)) bad = 1;
        }
    } else if (warp == kWarpMma) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, 64, false, false);
            constexpr uint32_t id_s = idesc_bf16(128, LY::NW, true, true);
            constexpr uint32_t id_o = idesc_bf16(128, LY::NW, false, true);
            // descriptors at each operand's base; a K step adds (bytes >> 4) to the
            // start-address field, which never carries out of its 14 bits here
            const uint32_t sm0 = smem_u32(sm);
            const uint64_t dS = sdesc_sw128(smem_u32(sS), 16384, 1024);   // S' copy, MN-major
            const uint64_t dP = sdesc_sw128(smem_u32(sP), 16, 1024);      // P, K-major
            // K-major q and k: one descriptor per 64-column half; MN-major k and
            // [V | 1]: the halves (and the ones block) are the N atoms, LBO apart
            auto dkm = [&](int n) {
                const uint32_t k0 = tile_half(1, n % NS, 0), k1 = tile_half(1, n % NS, 1);
                return sdesc_sw128(sm0 + k0, k1 - k0, 1024);
            };
            auto dvm = [&](int n) {
                const uint32_t v0 = tile_half(2, n % NS, 0), v1 = tile_half(2, n % NS, 1);
                return sdesc_sw128(sm0 + v0, v1 - v0, 1024);
            };
            // operand ranges (LA_DEBUG): an M = 128 A operand reads 16 KiB from its
            // start, a 64-row operand (or N atom) 8 KiB
            auto opok = [&](uint32_t off, uint32_t span) { return sok(sm + off, span); };
            auto issue_qk = [&](int n) {
                if (!(opok(tile_half(0, n % NS, 0), 16384) && opok(tile_half(0, n % NS, 1), 16384) &&
                      opok(tile_half(1, n % NS, 0), 8192) && opok(tile_half(1, n % NS, 1), 8192)))
                    return;
                const uint64_t a0 = sdesc_sw128(sm0 + tile_half(0, n % NS, 0), 16, 1024);
                const uint64_t a1 = sdesc_sw128(sm0 + tile_half(0, n % NS, 1), 16, 1024);
                const uint64_t b0 = sdesc_sw128(sm0 + tile_half(1, n % NS, 0), 16, 1024);
                const uint64_t b1 = sdesc_sw128(sm0 + tile_half(1, n % NS, 1), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(tmem + LY::colP, (ks < 4 ? a0 : a1) + (ks & 3) * 2, (ks < 4 ? b0 : b1) + (ks & 3) * 2,
                              id_qk, ks > 0);
                umma_commit(qk);
            };
            if (SO) {
                // state only: T_n = S_{n-1} + k~^T [V | 1] per chunk
                for (int n = 0; n < N; ++n) {
                    const int s = n % NS;
                    if (!mbar_wait(&pro[s], (uint32_t)(n / NS) & 1u, wait_ns) ||
                        (n > 0 && !mbar_wait(sready, (uint32_t)(n - 1) & 1u, wait_ns))) {
                        bad = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ak = dkm(n), bv = dvm(n);
                    if (opok(tile_half(1, s, 0), 8192) && opok(tile_half(1, s, 1), 8192) && opok(tile_half(2, s, 0), 8192) &&
                        opok(tile_half(2, s, 1), 8192)) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            umma_bf16(tmem + LY::colS, ak + ks * 128, bv + ks * 128, id_s, (n > 0 || ks > 0));
                    }
                    umma_commit(sdone);
                    umma_commit(&empty[s]);
                }
            } else if (N > 0) {
                if (!mbar_wait(&pro[0], 0u, wait_ns)) bad = 1;
                tc_fence_after();
                if (!bad) issue_qk(0);
            }
            for (int n = 0; n < N && !bad && !SO; ++n) {
                const int s = n % NS, b = n % LY::NOB;
                const uint32_t dO = tmem + (b ? LY::colO1 : LY::colO0);
                const uint64_t aq0 = sdesc_sw128(sm0 + tile_half(0, s, 0), 16, 1024);
                const uint64_t aq1 = sdesc_sw128(sm0 + tile_half(0, s, 1), 16, 1024);
                const uint64_t ak = dkm(n), bv = dvm(n);
                if (!(opok(tile_half(0, s, 0), 16384) && opok(tile_half(0, s, 1), 16384) && opok(tile_half(1, s, 0), 8192) &&
                      opok(tile_half(1, s, 1), 8192) && opok(tile_half(2, s, 0), 8192) && opok(tile_half(2, s, 1), 8192) &&
                      opok(LY::P, 16384) && opok(LY::S, NORM ? 49152 : 32768))) {
                    bad = 1;
                    break;
                }
                if ((n > 0 || init) && !mbar_wait(sready, (uint32_t)(n - 1 + (init ? 1 : 0)) & 1u, wait_ns)) {
                    bad = 1;
                    break;
                }
                tc_fence_after();
                // state: T_n = S_{n-1} (rescaled in place) + k~^T [V | 1]
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(tmem + LY::colS, ak + ks * 128, bv + ks * 128, id_s, (n > 0 || init || ks > 0));
                umma_commit(sdone);
                // inter: O = q~ S_{n-1}
                if (n > 0 || init) {
                    if (n >= LY::NOB && !mbar_wait(&oempty[b], (uint32_t)((n - LY::NOB) / LY::NOB) & 1u, wait_ns)) {
                        bad = 1;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(dO, (ks < 4 ? aq0 : aq1) + (ks & 3) * 2, dS + ks * 128, id_o, ks > 0);
                }
                umma_commit(sfree);
                // intra: O += P [V | 1]
                if (!mbar_wait(pfull, (uint32_t)n & 1u, wait_ns)) {
                    bad = 1;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_bf16(dO, dP + ks * 2, bv + ks * 128, id_o, (n > 0 || init || ks > 0));
                umma_commit(&ofull[b]);
                umma_commit(&empty[s]);
                // QK of the next chunk (P is read out of TMEM by then)
                if (n + 1 < N) {
                    const int n1 = n + 1;
                    if (!mbar_wait(&pro[n1 % NS], (uint32_t)(n1 / NS) & 1u, wait_ns) ||
                        !mbar_wait(pempty, (uint32_t)n & 1u, wait_ns)) {
                        bad = 1;
                        break;
                    }
                    tc_fence_after();
                    issue_qk(n1);
                }
            }
            // every MMA this thread issued has completed before teardown
            umma_commit(drain);
            if (!mbar_wait(drain, 0u, wait_ns)) bad = 1;
        }
    } else if (SPLIT ? (warp == 6 || warp == 7 || warp >= 14) : ((warp >= 4 && warp < 8) || warp < 2 || warp >= 14)) {
        // ============================================================ prologue
        // 256 threads in eight warps, two on each SM sub-partition: prologue warp
        // pw = warps 4..7 -> 0..3, warps 0, 1 -> 4, 5, warps 14, 15 -> 6, 7
        const int pw = SPLIT ? ((warp & 1) | (warp >= 14 ? 2 : 0))
                           : (warp >= 4 && warp < 8) ? warp - 4 : warp < 2 ? warp + 4 : warp - 8;
        if constexpr (GATE >= 2) {
            // Prologue warp pw takes the channel half ch = pw % 2 and the row
            // quarter qr = pw / 2;
            // lane l owns key channels 64 ch + 2l and 64 ch + 2l + 1 (one bf16x2
            // word) of rows 16 qr .. 16 qr + 15. The 32 words a warp touches in one
            // row fill that row's 128-byte line of one swizzle block: no bank
            // conflicts, and the swizzle slot of row 16 qr + u depends on u alone.
            // Per chunk:
            //   pass 1  log2 alpha of the thread's 32 gate values, kept in registers,
            //           and their sums over the quarter -> tot[(n % 2)][qr][channel]
            //   barrier; the quarter's starting decay = sum of tot over lower quarters
            //   pass 2  running log2 decay b_t down the quarter; phi(k_t) * 2^-b_t and
            //           phi(q_t) * 2^b_t in place, two channels per packed word.
            // Rows past the end of the sequence (t >= c) get log2 alpha = 0 and keep
            // their (zero-filled) q; their k is zeroed only with the normaliser
            // (elsewhere their zero v rows cancel them). Quarter 3 ends at the
            // chunk's total decay and writes the state factors.
            // REV (the anti-causal form): the mirrored sequence's cumulative decay
            // is a suffix sum over the chunk's rows, of the gate of the next token
            // (the tile starts a row later; the sequence's last token decays
            // nothing). Step u of a quarter takes row 15 - u, the quarter sums are
            // taken over the quarters above, and quarter 0 ends at the total.
            const int ch = pw & 1, qr = pw >> 1;
            const int cw = 64 * ch + 2 * lane;  // first of the thread's two channels
            const uint32_t colw = (lane & 3) << 2, slot = lane >> 2;  // within the block of half ch
            constexpr int kLastQ = REV ? 0 : 3;
            auto rowu = [&](int u) { return REV ? 15 - u : u; };  // row of step u within the quarter
            auto offw = [&](int u) {
                const int r = rowu(u);
                return colw + (16 * qr + r) * 128 + (((slot ^ r) & 7) << 4);
            };
            // log2 decay of the two channels over the previous chunk and over the
            // segment so far (kept by quarter 3)
            float bl0 = 0.f, bl1 = 0.f, bt0 = 0.f, bt1 = 0.f;
            for (int n = 0; n < N; ++n) {
                const int s = n % NS, t0 = chunk_t0(n), c = min(kC, L - t0);
                // rows whose gate is read (REV: not the sequence's last token)
                const int cg = (REV && t0 + c >= L) ? c - 1 : c;
                // the gate tile first: from its own ring (full pass) or from the stage.
                // Without the normaliser no barrier follows: the quarter sums are
                // double-buffered, so a warp may start this chunk while others finish
                // the last one, and a failed wait is made uniform at the barrier after
                // pass 1 (what pass 1 read then is discarded). The normalised forms
                // (two stages) measured faster with the barrier kept.
                bool ok = LY::GR ? mbar_wait(&gfull[n % NG], (uint32_t)(n / NG) & 1u, wait_ns)
                                 : mbar_wait(&full[s], (uint32_t)(n / NS) & 1u, wait_ns);
                if constexpr (NORM) {
                    if (named_sync_or<kBarPro, 256>(!ok)) {
                        bad = 1;
                        break;
                    }
                }
                // the blocks of this thread's channel half
                uint8_t *sQ = sm + tile_half(0, s, ch), *sK = sm + tile_half(1, s, ch);
                const uint8_t *sG = LY::GR ? sm + LY::Gring + (n % NG) * kTile + ch * kHalf : sm + tile_half(3, s, ch);
                // gate logs of both channels in packed pairs; rows past the end
                // read as g = +huge in both halves (no decay)
                f32x2_t la[16], sq = f2(0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const uint32_t w = 16 * qr + rowu(u) < cg ? ld4(sG + offw(u)) : 0x7F7F7F7Fu;
                    la[u] = log2_alpha2(w);
                    sq = f2_add(sq, la[u]);
                }
                if (LY::GR) mbar_arrive(&gempty[n % NG]);  // g is in registers now
                float *totn = tot + (NORM ? 0 : (n & 1) * 512);
                *reinterpret_cast<f32x2_t *>(totn + qr * 128 + cw) = sq;
                // then the q, k (, v) stage; the barrier also publishes the quarter sums
                if (LY::GR && ok) ok = mbar_wait(&full[s], (uint32_t)(n / NS) & 1u, wait_ns);
                if constexpr (GATE == 3) sK = sm + tile_half(2, s, ch);
                uint32_t kw[8], qw[8], kn[8], qn[8];
                if (ok) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        kw[u] = ld4(sK + offw(u));
                        if (!SO && GATE == 2) qw[u] = ld4(sQ + offw(u));
                    }
                }
                if (named_sync_or<kBarPro, 256>(!ok)) {
                    bad = 1;
                    break;
                }
                f32x2_t bb = f2(0.f, 0.f);
                for (int r = REV ? qr + 1 : 0; r < (REV ? 4 : qr); ++r)
                    bb = f2_add(bb, *reinterpret_cast<const f32x2_t *>(totn + r * 128 + cw));
                float b0, b1;
                // pass 2 in two groups of eight rows; the second group's words are
                // loaded before the first group's results are stored. The group
                // loop is kept rolled (the prologue's code is the largest of the
                // roles and instruction fetch stalled it when unrolled), so each
                // group reads its gate logs from la[0..7] and shifts la[8..15]
                // down for the next. With the
                // gate on the value side (GATE 3) the tile scaled by 2^-b is v's,
                // and q stays as it is.
#pragma unroll(SO ? 2 : 1)
                for (int g8 = 0; g8 < 2; ++g8) {
                    if (g8 == 0) {
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            kn[u] = ld4(sK + offw(8 + u));
                            if (!SO && GATE == 2) qn[u] = ld4(sQ + offw(8 + u));
                        }
                    }
                    uint32_t ko[8], qo[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int uu = 8 * g8 + u;
                        bb = f2_add(bb, la[u]);
                        f2_split(bb, b0, b1);
                        // factors in fp32, rounded to bf16 once and applied
                        // to both channels in one packed multiply
                        uint32_t kx = kw[u];
                        if (ELU1) kx = phi_elu1_bf16x2(kx);
                        ko[u] = mul_bf16x2(kx, pack_bf16(ex2f(-b0), ex2f(-b1)));
                        // rows past the end: their v rows are zero, which cancels
                        // them everywhere but in the ones column of the normaliser
                        if (NORM && 16 * qr + rowu(uu) >= c) ko[u] = 0u;
                        if (!SO && GATE == 2) {
                            uint32_t qx = qw[u];
                            if (ELU1) qx = phi_elu1_bf16x2(qx);
                            qo[u] = mul_bf16x2(qx, pack_bf16(ex2f(b0), ex2f(b1)));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        st4(sK + offw(8 * g8 + u), ko[u]);
                        if (!SO && GATE == 2) st4(sQ + offw(8 * g8 + u), qo[u]);
                        kw[u] = kn[u];
                        if (!SO && GATE == 2) qw[u] = qn[u];
                        la[u] = la[u + 8];
                    }
                }
                if (qr == kLastQ) {
                    bl0 = b0;
                    bl1 = b1;
                    bt0 += b0;
                    bt1 += b1;
                    *reinterpret_cast<float2 *>(fbuf + (n % NF) * 128 + cw) = make_float2(ex2f(b0), ex2f(b1));
                    mbar_arrive(&ffull[n % NF]);
                }
                fence_proxy_async_smem();
                mbar_arrive(&pro[s]);
            }
            if (!bad && qr == kLastQ) {
                *reinterpret_cast<float2 *>(ffinal + cw) = make_float2(ex2f(bl0), ex2f(bl1));
                if (SO)
                    if (gok((size_t)sgi * kD + cw + 1, p.n_seg_logdecay))
                        *reinterpret_cast<float2 *>(p.seg_logdecay + (size_t)sgi * kD + cw) =
                            make_float2(bt0 * kLn2, bt1 * kLn2);
                mbar_arrive(profinal);
            }
        } else {
            // Thread pd (0..PT-1) owns the 16-byte pieces pd + PT j of each tile
            // (block, row and slot below; the eight lanes of a quarter warp share a
            // row: no bank conflicts). Threads pd < 128 also own key channel pd for
            // the decay factors.
            const int pd = 32 * pw + lane;
            const float lg = GATE == 1 && gok(h, p.H) ? __logf(p.gamma[h]) : 0.f;
            // Retention applies the state's decay once per window of R chunks instead
            // of every chunk: m chunks into a window the accumulator holds
            // S / gamma^(64 m), so q rows take an extra gamma^(64 m) and k rows
            // gamma^(-64 m), and the state chain rescales only at a window's last
            // chunk. R keeps those extra factors within e^(+-40).
            int R = 1;
            if (GATE == 1) {
                const float rl = -(float)kC * lg;
                R = rl > 0.f ? max(1, (int)fminf(40.f / rl, 1048576.f)) : 1048576;
            }
            // log decay of key channel pd over the previous chunk and over the segment so far
            float b_last = 0.f, b_total = 0.f;
            // (BIAS, state-only pass) the segment's column sums so far, held by the
            // first thread of each column group
            float crun[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            int m = 0;  // chunks into the current window
            // REV takes a ragged last chunk first: it closes a window of its own,
            // so that every window after it holds whole chunks only
            const int rag0 = (REV && c0 == 0 && (L % kC) != 0) ? 1 : 0;
            // (BIAS 2) e of token pd of a chunk, read a chunk ahead of its use
            auto e_at = [&](int m) {
                const int tm = chunk_t0(m) + pd;
                const size_t ei = (size_t)bh * L + tm;
                return (tm < L && gok(ei, p.n_e)) ? p.e_in[ei] : 0.f;
            };
            float pe_next = (BIAS == 2 && pd < kC && N > 0) ? e_at(0) : 0.f;
            if (GATE == 1) {
                // the row factors gamma^(t+1) and gamma^-(t+1) are the same in every chunk
                if (pd < 64) {
                    fq[pd] = __expf((float)(pd + 1) * lg);
                    fk[pd] = __expf(-(float)(pd + 1) * lg);
                }
                named_sync<kBarPro, PT>();
            }
            for (int n = 0; n < N; ++n) {
                const int s = n % NS, t0 = chunk_t0(n), c = min(kC, L - t0);
                const int nw = n - rag0;  // chunks counted by the windows
                m = nw < 0 ? 0 : nw % R;
                const bool wend = nw < 0 || m == R - 1;  // this chunk closes its window
                float gq = 1.f, gk = 1.f;
                if (GATE == 1 && m > 0) {
                    gq = __expf((float)(kC * m) * lg);
                    gk = __expf(-(float)(kC * m) * lg);
                }
                // (BIAS) the outputs, which may trail the MMAs, have read the column
                // sums of chunk n - NF out of the slot this chunk's go to
                const bool ok = mbar_wait(&full[s], (uint32_t)(n / NS) & 1u, wait_ns) &&
                                (BIAS == 0 || SO || n < NF || mbar_wait(&cempty[n % NF], (uint32_t)(n / NF - 1) & 1u, wait_ns));
                if (named_sync_or<kBarPro, PT>(!ok)) {
                    bad = 1;
                    break;
                }
                if (ELU1 || GATE == 1 || c < kC) {
                    // the tiles taken: q and k (k only in the state-only pass), or v
                    // alone with the feature map on the value tile
                    constexpr int TL0 = PHIV ? 2 : (SO ? 1 : 0), TL1 = PHIV ? 3 : 2;
#pragma unroll
                    for (int tl = TL0; tl < TL1; ++tl) {
                        const bool isk = tl != 0;  // rows past the end are zeroed (k, or v)
                        uint8_t *blk0 = sm + tile_half(tl, s, 0), *blk1 = sm + tile_half(tl, s, 1);
                        const float *fr_arr = isk ? fk : fq;
                        // piece x = pd + PT j: block x / 512, row (x / 8) % 64, slot x % 8
                        constexpr int NJ = 1024 / PT;
                        uint4 w[NJ];
#pragma unroll
                        for (int j = 0; j < NJ; ++j)
                            w[j] = ld16(((pd + PT * j) >> 9 ? blk1 : blk0) + (((pd + PT * j) >> 3) & 63) * 128 + (pd & 7) * 16);
#pragma unroll
                        for (int j = 0; j < NJ; ++j) {
                            const int row = ((pd + PT * j) >> 3) & 63;
                            uint4 &x = w[j];
                            if (isk && row >= c) {
                                x = make_uint4(0u, 0u, 0u, 0u);
                            } else if (ELU1 || GATE == 1) {
                                uint32_t u[4] = {x.x, x.y, x.z, x.w};
                                if (ELU1) {
#pragma unroll
                                    for (int e = 0; e < 4; ++e) u[e] = phi_elu1_bf16x2(u[e]);
                                }
                                if (GATE == 1) {
                                    // (with REV the local index is c - 1 - row; rows past the
                                    // end hold zeros and take any factor)
                                    const float fr = fr_arr[REV ? ((c - 1 - row) & (kC - 1)) : row] * (isk ? gk : gq);
                                    if constexpr (OF32) {
                                        // the fp32-output instances serve differences of nearly
                                        // equal terms: one rounding of the exact product
#pragma unroll
                                        for (int e = 0; e < 4; ++e) u[e] = pack_bf16(bf16lo(u[e]) * fr, bf16hi(u[e]) * fr);
                                    } else {
                                        // the factor rounded to bf16 once, applied to two values
                                        // by one packed multiply
                                        const uint32_t fr2 = pack_bf16(fr, fr);
#pragma unroll
                                        for (int e = 0; e < 4; ++e) u[e] = mul_bf16x2(u[e], fr2);
                                    }
                                }
                                x = make_uint4(u[0], u[1], u[2], u[3]);
                            }
                            st16(((pd + PT * j) >> 9 ? blk1 : blk0) + row * 128 + (pd & 7) * 16, x);
                        }
                    }
                }
                if (GATE == 1) b_last = (float)c * lg;
                b_total += b_last;
                if (GATE != 0 && pd < 128) {
                    // retention: 1 inside a window (the state chain leaves the
                    // accumulator alone), the decay since the window began at its end
                    float fv = __expf(b_last);
                    if (GATE == 1) fv = wend ? __expf(b_last + (float)(kC * m) * lg) : 1.f;
                    fbuf[(n % NF) * 128 + pd] = fv;
                    mbar_arrive(&ffull[n % NF]);
                }
                if constexpr (BIAS != 0) {
                    // column sums of this chunk's value tile, each row weighted by 1
                    // (BIAS 1) or by e of its token (BIAS 2): the sixteen 16-byte column
                    // groups (block bv, slot lc) take TG = PT / 16 threads each, thread
                    // pd group pd / TG over rows g, g + TG, ... (g = pd % TG); the TG
                    // threads of a group sit in one warp and reduce by shuffles
                    if (BIAS == 2 && pd < kC) {
                        pebuf[pd] = pe_next;
                        if (n + 1 < N) pe_next = e_at(n + 1);
                    }
                    // (the value tile was just rewritten with the feature map by other
                    // threads' pieces)
                    if (BIAS == 2 || PHIV) named_sync<kBarPro, PT>();
                    constexpr int TG = PT / 16;
                    const int bc = pd / TG, g = pd % TG, bv = bc >> 3, lc = bc & 7;
                    const uint8_t *vt = sm + tile_half(2, s, bv);
                    float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int rr = 0; rr < kC / TG; ++rr) {
                        const int row = g + TG * rr;
                        const float cw = BIAS == 2 ? pebuf[row] : 1.f;
                        const uint4 x = ld16(vt + row * 128 + ((lc ^ (row & 7)) << 4));
                        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            cs[2 * e] = fmaf(cw, bf16lo(xw[e]), cs[2 * e]);
                            cs[2 * e + 1] = fmaf(cw, bf16hi(xw[e]), cs[2 * e + 1]);
                        }
                    }
#pragma unroll
                    for (int off = 1; off < TG; off <<= 1)
#pragma unroll
                        for (int e = 0; e < 8; ++e) cs[e] += __shfl_xor_sync(0xffffffffu, cs[e], off);
                    if (g == 0) {
                        if constexpr (SO) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) crun[e] += cs[e];
                        } else {
                            float *dst = csum + (n % NF) * 128 + bv * 64 + lc * 8;
#pragma unroll
                            for (int e = 0; e < 8; ++e) dst[e] = cs[e];
                            mbar_arrive(&cfull[n % NF]);
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&pro[s]);
            }
            if (!bad && pd < 128) {
                ffinal[pd] = GATE == 0 ? 1.f : __expf(b_last + (GATE == 1 ? (float)(kC * m) * lg : 0.f));
                if (SO && gok((size_t)sgi * kD + pd, p.n_seg_logdecay))
                    p.seg_logdecay[(size_t)sgi * kD + pd] = b_total;
                mbar_arrive(profinal);
            }
            if constexpr (SO && BIAS != 0) {
                // the segment's column sums after its state (no decay: the scan adds
                // them up over the earlier segments)
                constexpr int TG = PT / 16;
                const int bc = pd / TG, bv = bc >> 3, lc = bc & 7;
                const size_t o = segblk + (size_t)kD * kD + bv * 64 + lc * 8;
                if (!bad && pd % TG == 0 && gok(o + 7, p.n_seg_state)) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) p.seg_state[o + e] = crun[e];
                }
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ============================================================ state chain
        const int i = tid - 256;  // TMEM lane = state row (key channel)
        const uint32_t tS = tmem + lane_base + LY::colS;
        // bf16 copy of the state row in TMEM, MN-major for the B operand: line i,
        // value columns v; z goes to element 0 of line i in the third atom
        auto write_copy = [&]() {
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tld32(tS + 32 * j, r);
                tmem_ld_wait();
                uint8_t *row = sS + (j >> 1) * 16384 + i * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int lc = 4 * (j & 1) + q4;
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(r[8 * q4 + 0]), __uint_as_float(r[8 * q4 + 1]));
                    w.y = pack_bf16(__uint_as_float(r[8 * q4 + 2]), __uint_as_float(r[8 * q4 + 3]));
                    w.z = pack_bf16(__uint_as_float(r[8 * q4 + 4]), __uint_as_float(r[8 * q4 + 5]));
                    w.w = pack_bf16(__uint_as_float(r[8 * q4 + 6]), __uint_as_float(r[8 * q4 + 7]));
                    st16(row + ((lc ^ (i & 7)) << 4), w);
                }
            }
            if (NORM) {
                uint32_t z;
                tld1(tS + 128, z);
                tmem_ld_wait();
                st16(sS + 32768 + i * 128 + ((i & 7) << 4), make_uint4(pack_bf16(__uint_as_float(z), 0.f), 0u, 0u, 0u));
            }
        };
        if (init) {
            // the state carried into this segment: into TMEM and its bf16 copy.
            // After a segment scan this launch may have started while the scan
            // still ran (programmatic dependent launch): wait for it to finish
            // before reading what it wrote (a no-op for an ordinary launch).
            griddep_wait();
            const float *src = p.state_in + segblk + (size_t)i * kD;
            if (!gok(segblk + (size_t)i * kD + kD - 1, p.n_state_in)) src = nullptr;
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 v4 = src ? reinterpret_cast<const float4 *>(src + 32 * j)[q4] : make_float4(0.f, 0.f, 0.f, 0.f);
                    r[4 * q4] = __float_as_uint(v4.x);
                    r[4 * q4 + 1] = __float_as_uint(v4.y);
                    r[4 * q4 + 2] = __float_as_uint(v4.z);
                    r[4 * q4 + 3] = __float_as_uint(v4.w);
                }
                tst32(tS + 32 * j, r);
            }
            if (NORM && gok(segblk + (size_t)kD * kD + i, p.n_state_in))
                tst1(tS + 128, __float_as_uint(p.state_in[segblk + (size_t)kD * kD + i]));
            tmem_st_wait();
            write_copy();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(sready);
        }
        for (int n = 1; n < N; ++n) {
            // T_{n-1} is complete, and so is chunk n-1's decay factor
            bool ok = mbar_wait(sdone, (uint32_t)(n - 1) & 1u, wait_ns);
            if (GATE != 0) ok = ok && mbar_wait(&ffull[(n - 1) % NF], (uint32_t)((n - 1) / NF) & 1u, wait_ns);
            if (named_sync_or<kBarState, 128>(!ok)) {
                bad = 1;
                break;
            }
            tc_fence_after();
            const float *fcol = fbuf + ((n - 1) % NF) * 128;
            const float f = GATE != 0 ? fcol[i] : 1.f;
            // (retention inside a window: factor 1, the accumulator stays as it is)
            if (GATE != 0 && !(GATE == 1 && f == 1.f)) {
                // S_{n-1} = diag(f) T_{n-1} (key-side gate) or T_{n-1} diag(f)
                // (value-side gate), in place (z rides in column 128)
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tld32(tS + 32 * j, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        r[e] = __float_as_uint(__uint_as_float(r[e]) * (GATE == 3 ? fcol[32 * j + e] : f));
                    tst32(tS + 32 * j, r);
                }
                if (NORM) {
                    uint32_t z;
                    tld1(tS + 128, z);
                    tmem_ld_wait();
                    tst1(tS + 128, __float_as_uint(__uint_as_float(z) * f));
                }
                tmem_st_wait();
            }
            if (!SO) {
                // the inter MMA of chunk n-1 has finished reading the previous copy
                ok = mbar_wait(sfree, (uint32_t)(n - 1) & 1u, wait_ns);
                if (named_sync_or<kBarState, 128>(!ok)) {
                    bad = 1;
                    break;
                }
                write_copy();
                fence_proxy_async_smem();
            }
            tc_fence_before();
            mbar_arrive(sready);
        }
        float *dst = SO ? p.seg_state + segblk : (seg == p.nseg - 1 ? p.final_state : nullptr);
        if (!SO && dst) dst += (size_t)bh * blk;
        if (dst && !gok((SO ? segblk : (size_t)bh * blk) + blk - 1, SO ? p.n_seg_state : p.n_final)) dst = nullptr;
        if (!bad && N > 0) {
            bool ok = mbar_wait(sdone, (uint32_t)(N - 1) & 1u, wait_ns) && mbar_wait(profinal, 0u, wait_ns);
            if (named_sync_or<kBarState, 128>(!ok)) {
                bad = 1;
            } else if (dst != nullptr) {
                // end state S = diag(e^{b_last}) T (with z in column 128), or
                // T diag(e^{b_last}) with the gate on the value side
                tc_fence_after();
                const float ff = ffinal[i];
                float *row = dst + (size_t)i * kD;
#pragma unroll 1
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tld32(tS + 32 * j, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        float f4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) f4[e] = GATE == 3 ? ffinal[32 * j + 4 * q4 + e] : ff;
                        reinterpret_cast<float4 *>(row + 32 * j)[q4] = make_float4(
                            __uint_as_float(r[4 * q4]) * f4[0], __uint_as_float(r[4 * q4 + 1]) * f4[1],
                            __uint_as_float(r[4 * q4 + 2]) * f4[2], __uint_as_float(r[4 * q4 + 3]) * f4[3]);
                    }
                }
                if (NORM) {
                    uint32_t z;
                    tld1(tS + 128, z);
                    tmem_ld_wait();
                    dst[(size_t)kD * kD + i] = __uint_as_float(z) * ff;
                }
            }
        }
    } else if (!SO && !SPLIT && (warp == 12 || warp == 13)) {
        // ============================================================ outputs (TMEM lanes 0..63 = rows t)
        const int t = tid - 384;
        // the mask: key columns at or before the query row (at or after it with REV)
        auto keep = [&](int j) { return REV ? j >= t : j <= t; };
        for (int n = 0; n < N; ++n) {
            const int b = n % LY::NOB, t0 = chunk_t0(n);
            bool ok = mbar_wait(qk, (uint32_t)n & 1u, wait_ns);
            if (named_sync_or<kBarOut, 64>(!ok)) {
                bad = 1;
                break;
            }
            tc_fence_after();
            {
                // P row t: causal mask (key <= t), bf16, K-major A operand of intra
                uint8_t *prow = sP + t * 128;
                if constexpr (GATE >= 2) {
                    // the channel-gated kernels carry the largest prologue; here the
                    // row goes in eight rolled steps of eight columns, which keeps
                    // this role's code small (instruction fetch stalled them otherwise)
#pragma unroll 1
                    for (int q8 = 0; q8 < 8; ++q8) {
                        uint32_t a[8];
                        tld8(tmem + lane_base + LY::colP + 8 * q8, a);
                        tmem_ld_wait();
                        uint32_t u[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int jj = q8 * 8 + 2 * e;
                            u[e] = pack_bf16(keep(jj) ? __uint_as_float(a[2 * e]) : 0.f,
                                             keep(jj + 1) ? __uint_as_float(a[2 * e + 1]) : 0.f);
                        }
                        st16(prow + (((q8 ^ t) & 7) << 4), make_uint4(u[0], u[1], u[2], u[3]));
                    }
                    tc_fence_before();
                    mbar_arrive(pempty);
                } else {
                    uint32_t r0[32], r1[32];
                    tld32(tmem + lane_base + LY::colP, r0);
                    tld32(tmem + lane_base + LY::colP + 32, r1);
                    tmem_ld_wait();
                    tc_fence_before();
                    mbar_arrive(pempty);
#pragma unroll
                    for (int q8 = 0; q8 < 8; ++q8) {
                        uint32_t u[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int jj = q8 * 8 + 2 * e;
                            const uint32_t a0 = q8 < 4 ? r0[jj] : r1[jj - 32];
                            const uint32_t a1 = q8 < 4 ? r0[jj + 1] : r1[jj - 31];
                            u[e] = pack_bf16(keep(jj) ? __uint_as_float(a0) : 0.f, keep(jj + 1) ? __uint_as_float(a1) : 0.f);
                        }
                        st16(prow + (((q8 ^ t) & 7) << 4), make_uint4(u[0], u[1], u[2], u[3]));
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(pfull);

            ok = mbar_wait(&ofull[b], (uint32_t)(n / LY::NOB) & 1u, wait_ns);
            if (t == 0) bulk_wait_read<0>();  // the previous O tile has left the staging buffer
            if (named_sync_or<kBarOut, 64>(!ok)) {
                bad = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tO = tmem + lane_base + (b ? LY::colO1 : LY::colO0);
            float rden = 1.f;
            if (NORM) {
                uint32_t dd;
                tld1(tO + 128, dd);
                tmem_ld_wait();
                rden = 1.f / __uint_as_float(dd);
            }
#pragma unroll 1
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tld32(tO + 32 * j, r);
                tmem_ld_wait();
                if constexpr (OF32) {
                    // staging: four [64 x 32] fp32 quarters with the 128-byte swizzle (box 32 x 64)
                    uint8_t *row = sO + j * 8192 + t * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st16(row + ((c ^ (t & 7)) << 4), make_uint4(
                            __float_as_uint(__uint_as_float(r[4 * c]) * rden), __float_as_uint(__uint_as_float(r[4 * c + 1]) * rden),
                            __float_as_uint(__uint_as_float(r[4 * c + 2]) * rden), __float_as_uint(__uint_as_float(r[4 * c + 3]) * rden)));
                } else {
                    // staging: two [64 x 64] halves with the 128-byte swizzle (TMA store box 64 x 64)
                    uint8_t *row = sO + (j >> 1) * 8192 + t * 128;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int lc = 4 * (j & 1) + q4;
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(r[8 * q4 + 0]) * rden, __uint_as_float(r[8 * q4 + 1]) * rden);
                        w.y = pack_bf16(__uint_as_float(r[8 * q4 + 2]) * rden, __uint_as_float(r[8 * q4 + 3]) * rden);
                        w.z = pack_bf16(__uint_as_float(r[8 * q4 + 4]) * rden, __uint_as_float(r[8 * q4 + 5]) * rden);
                        w.w = pack_bf16(__uint_as_float(r[8 * q4 + 6]) * rden, __uint_as_float(r[8 * q4 + 7]) * rden);
                        st16(row + ((lc ^ (t & 7)) << 4), w);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&oempty[b]);
            fence_proxy_async_smem();
            named_sync<kBarOut, 64>();
            if (t == 0) {
                if constexpr (OF32) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) tstore(&p.to, sO + j * 8192, 32 * j, t0);
                } else {
                    tstore(&p.to, sO, 0, t0);
                    tstore(&p.to, sO + 8192, 64, t0);
                }
                bulk_commit();
            }
        }
        if (t == 0) bulk_wait<0>();
    } else if (SPLIT && (warp == 12 || warp == 13)) {
        // ============================================================ P (split roles)
        // P row t of every chunk (TMEM lanes 0..63); the outputs are other
        // warps' work, so P of chunk n + 1 is formed while chunk n is finished
        const int t = tid - 384;
        // the mask: key columns at or before the query row (at or after it with REV)
        auto keep = [&](int j) { return REV ? j >= t : j <= t; };
        // (BIAS) e of token t of a chunk, read a chunk ahead of its use
        auto e_at = [&](int m) {
            const int tm = chunk_t0(m) + t;
            const size_t ei = (size_t)bh * L + tm;
            return (tm < L && gok(ei, p.n_e)) ? p.e_in[ei] : 0.f;
        };
        float e_next = (BIAS != 0 && N > 0) ? e_at(0) : 0.f;
        for (int n = 0; n < N; ++n) {
            // QK of this chunk, and the intra MMA of the last one has read the P tile
            bool ok = mbar_wait(qk, (uint32_t)n & 1u, wait_ns);
            if (n > 0) ok = ok && mbar_wait(&ofull[(n - 1) % LY::NOB], (uint32_t)((n - 1) / LY::NOB) & 1u, wait_ns);
            if (named_sync_or<kBarP, 64>(!ok)) {
                bad = 1;
                break;
            }
            tc_fence_after();
            // (BIAS) e on every score of the row: the query token's (1), or each
            // key column's (2, shared through oebuf)
            float e_row = 0.f;
            if constexpr (BIAS != 0) {
                const float ev = e_next;
                if (n + 1 < N) e_next = e_at(n + 1);
                if (BIAS == 1) {
                    e_row = ev;
                } else {
                    oebuf[t] = ev;
                    named_sync<kBarP, 64>();
                }
            }
            uint8_t *prow = sP + t * 128;
            uint32_t r0[32], r1[32];
            tld32(tmem + lane_base + LY::colP, r0);
            tld32(tmem + lane_base + LY::colP + 32, r1);
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(pempty);
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint32_t u[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int jj = q8 * 8 + 2 * e;
                    const uint32_t a0 = q8 < 4 ? r0[jj] : r1[jj - 32];
                    const uint32_t a1 = q8 < 4 ? r0[jj + 1] : r1[jj - 31];
                    float p0 = __uint_as_float(a0), p1 = __uint_as_float(a1);
                    if (BIAS == 1) {
                        p0 += e_row;
                        p1 += e_row;
                    } else if (BIAS == 2) {
                        p0 += oebuf[jj];
                        p1 += oebuf[jj + 1];
                    }
                    u[e] = pack_bf16(keep(jj) ? p0 : 0.f, keep(jj + 1) ? p1 : 0.f);
                }
                st16(prow + (((q8 ^ t) & 7) << 4), make_uint4(u[0], u[1], u[2], u[3]));
            }
            fence_proxy_async_smem();
            mbar_arrive(pfull);
        }
    } else if (SPLIT && (warp == 0 || warp == 1 || warp == 4 || warp == 5)) {
        // ============================================================ outputs (split roles)
        // TMEM lanes 0..63 = rows t, on SM sub-partitions 0 and 1: warps 0 and 1
        // finish columns 0..63 of O, warps 4 and 5 columns 64..127. Each thread
        // reads its half row of O out of TMEM once and keeps it in registers.
        // With the RetNet epilogue the two halves of a row combine their mean and
        // squared deviations (m, M2) through shared memory: mean = (m0 + m1) / 2,
        // M2 = M2_0 + M2_1 + (m0 - m1)^2 * 64 * 64 / 128 (the same expressions,
        // in the same order, in both halves).
        const int t = (warp & 1) * 32 + lane, oh = warp >= 4 ? 1 : 0;
        const bool lead = oh == 0 && t == 0;
        // a tile comes by TMA into each chunk's staging buffer first: og, the
        // output gradient, or (bias instances with elu+1) x
        constexpr bool TILE_IN = EPI != 0 || PHIV;
        float *part = gnb + kD;  // [2][64] per half row: (m, M2), or the partial g . num
        if constexpr (EPI == 1) {
            const int col = 64 * oh + t;
            const bool hin = gok(h, p.H);
            gnw[col] = p.gn_w && hin ? p.gn_w[(size_t)h * kD + col] : 1.f;
            gnb[col] = p.gn_b && hin ? p.gn_b[(size_t)h * kD + col] : 0.f;
        }
        if (BIAS) {
            // the carried vector: zero, or (a later segment) the scan's sum over the
            // earlier segments, after the carried state in its block (read once the
            // scan this launch may have started behind has finished)
            const size_t o = segblk + (size_t)kD * kD + 64 * oh + t;
            if (init) griddep_wait();
            cvec[64 * oh + t] = (init && gok(o, p.n_state_in)) ? p.state_in[o] : 0.f;
        }
        // (BIAS 1) e of row t's token, read a chunk ahead of its use
        auto e_at = [&](int m) {
            const int tm = chunk_t0(m) + t;
            const size_t ei = (size_t)bh * L + tm;
            return (tm < L && gok(ei, p.n_e)) ? p.e_in[ei] : 0.f;
        };
        float e_next = (BIAS == 1 && N > 0) ? e_at(0) : 0.f;
        named_sync<kBarOut, 128>();
        // staging buffer of chunk m, and the request of its og tile
        auto obuf = [&](int m) { return sm + ((m & 1) ? LY::O2 : LY::O); };
        auto og_load = [&](int m) {
            uint8_t *dst = obuf(m);
            mbar_arrive_expect_tx(&ogfull[m & 1], kTile);
            tload(dst, &p.tog, &ogfull[m & 1], 0, chunk_t0(m));
            tload(dst + kHalf, &p.tog, &ogfull[m & 1], 64, chunk_t0(m));
        };
        int ogi = 0;  // (lead) og tiles requested
        if (TILE_IN && lead && N > 0) og_load(ogi++);
        for (int n = 0; n < N; ++n) {
            const int b = n % LY::NOB, t0 = chunk_t0(n);
            bool ok = mbar_wait(&ofull[b], (uint32_t)(n / LY::NOB) & 1u, wait_ns) &&
                      (!TILE_IN || mbar_wait(&ogfull[n & 1], (uint32_t)(n >> 1) & 1u, wait_ns));
            if (TILE_IN && lead && ok && n + 1 < N) {
                // the next chunk's tile into the buffer the store of chunk n - 1
                // read from
                if (n > 0) bulk_wait_read<0>();
                og_load(ogi++);
            }
            // (no tile in) the store of chunk n - 2 has left this chunk's buffer
            if (!TILE_IN && lead && n > 1) bulk_wait_read<1>();
            if (named_sync_or<kBarOut, 128>(!ok)) {
                bad = 1;
                break;
            }
            tc_fence_after();
            // this thread's half row of O; the accumulator is free once it is read
            uint32_t x0[32], x1[32], dd = 0;
            {
                const uint32_t tO = tmem + lane_base + (b ? LY::colO1 : LY::colO0);
                if (EPI == 2) tld1(tO + 128, dd);  // den_t
                tld32(tO + 64 * oh, x0);
                tld32(tO + 64 * oh + 32, x1);
                tmem_ld_wait();
            }
            tc_fence_before();
            mbar_arrive(&oempty[b]);
            bool okc = true;  // (BIAS) the chunk's column sums arrived
            if constexpr (EPI == 2) {
                // w = g / den over this half row, in place over g; the half row's
                // share of g . num, combined with the other half's through shared memory
                const float rden = 1.f / __uint_as_float(dd);
                uint8_t *const ob = obuf(n);
                uint8_t *row = ob + oh * kHalf + t * 128;
                f32x2_t acc = f2(0.f, 0.f);
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) {
                    uint8_t *pp = row + ((lc ^ (t & 7)) << 4);
                    const uint4 g4 = ld16(pp);
                    const uint32_t gw[4] = {g4.x, g4.y, g4.z, g4.w};
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int idx = 8 * lc + 2 * e;
                        const uint32_t v0 = idx < 32 ? x0[idx] : x1[idx - 32], v1 = idx < 32 ? x0[idx + 1] : x1[idx - 31];
                        const float g0 = bf16lo(gw[e]), g1 = bf16hi(gw[e]);
                        acc = f2_fma(f2(g0, g1), f2(__uint_as_float(v0), __uint_as_float(v1)), acc);
                        w[e] = cvt_bf16x2(g0 * rden, g1 * rden);
                    }
                    st16(pp, make_uint4(w[0], w[1], w[2], w[3]));
                }
                float a0, a1;
                f2_split(acc, a0, a1);
                const float ph = a0 + a1;
                *reinterpret_cast<float2 *>(part + (oh * 64 + t) * 2) = make_float2(ph, 0.f);
                named_sync<kBarOut, 128>();
                const float other = part[((1 - oh) * 64 + t) * 2];
                const float e_t = -(oh == 0 ? ph + other : other + ph) * rden * rden;
                const size_t ei = (size_t)bh * L + t0 + t;
                if (oh == 0 && t0 + t < L && gok(ei, p.n_e)) p.e_out[ei] = e_t;
            } else if constexpr (BIAS != 0) {
                // the carried vector's share, e_t cvec (1) or cvec (2), and (PHIV)
                // the factor phi'(x) of the x value in the same place; two columns
                // at a time, in place over x
                const float e_row = e_next;
                if (BIAS == 1 && n + 1 < N) e_next = e_at(n + 1);
                const f32x2_t er = f2(e_row, e_row);
                uint8_t *const ob = obuf(n);
                uint8_t *row = ob + oh * kHalf + t * 128;
#pragma unroll
                for (int lc = 0; lc < 8; ++lc) {
                    uint8_t *pp = row + ((lc ^ (t & 7)) << 4);
                    const uint4 xv = PHIV ? ld16(pp) : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int idx = 8 * lc + 2 * e;
                        const uint32_t v0 = idx < 32 ? x0[idx] : x1[idx - 32], v1 = idx < 32 ? x0[idx + 1] : x1[idx - 31];
                        const f32x2_t cv = *reinterpret_cast<const f32x2_t *>(cvec + 64 * oh + idx);
                        f32x2_t y = f2(__uint_as_float(v0), __uint_as_float(v1));
                        y = BIAS == 1 ? f2_fma(er, cv, y) : f2_add(y, cv);
                        if (PHIV) {
                            const uint32_t d = dphi_elu1_bf16x2(xw[e]);
                            y = f2_mul(y, f2(bf16lo(d), bf16hi(d)));
                        }
                        float y0, y1;
                        f2_split(y, y0, y1);
                        w[e] = cvt_bf16x2(y0, y1);
                    }
                    st16(pp, make_uint4(w[0], w[1], w[2], w[3]));
                }
                // every row has used the carried vector: add this chunk's column sums
                named_sync<kBarOut, 128>();
                okc = mbar_wait(&cfull[n % NF], (uint32_t)(n / NF) & 1u, wait_ns);
                if (okc) cvec[64 * oh + t] += csum[(n % NF) * 128 + 64 * oh + t];
            } else {
            // half-row mean and squared deviations
            f32x2_t acc = f2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                acc = f2_add(acc, f2(__uint_as_float(x0[2 * e]), __uint_as_float(x0[2 * e + 1])));
                acc = f2_add(acc, f2(__uint_as_float(x1[2 * e]), __uint_as_float(x1[2 * e + 1])));
            }
            float a0, a1;
            f2_split(acc, a0, a1);
            const float mh = (a0 + a1) * (1.f / 64.f);
            const f32x2_t nm = f2(-mh, -mh);
            acc = f2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const f32x2_t d0 = f2_add(f2(__uint_as_float(x0[2 * e]), __uint_as_float(x0[2 * e + 1])), nm);
                const f32x2_t d1 = f2_add(f2(__uint_as_float(x1[2 * e]), __uint_as_float(x1[2 * e + 1])), nm);
                acc = f2_fma(d0, d0, acc);
                acc = f2_fma(d1, d1, acc);
            }
            f2_split(acc, a0, a1);
            const float m2h = a0 + a1;
            *reinterpret_cast<float2 *>(part + (oh * 64 + t) * 2) = make_float2(mh, m2h);
            named_sync<kBarOut, 128>();
            const float2 other = *reinterpret_cast<const float2 *>(part + ((1 - oh) * 64 + t) * 2);
            const float mean = (mh + other.x) * 0.5f;
            const float dm = mh - other.x;
            const float rstd = rsqrtf((m2h + other.y + dm * dm * 32.f) * (1.f / kD) + p.gn_eps);
            // z = (o - mean) rstd; y = z w + b; out = y swish(og), in place over og
            const f32x2_t rs = f2(rstd, rstd), mr = f2(-mean * rstd, -mean * rstd);
            uint8_t *const ob = obuf(n);
            uint8_t *row = ob + oh * kHalf + t * 128;
#pragma unroll
            for (int lc = 0; lc < 8; ++lc) {
                uint8_t *pp = row + ((lc ^ (t & 7)) << 4);
                const uint4 og4 = ld16(pp);
                const uint32_t ogw[4] = {og4.x, og4.y, og4.z, og4.w};
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int idx = 8 * lc + 2 * e, c = 64 * oh + idx;
                    const uint32_t v0 = idx < 32 ? x0[idx] : x1[idx - 32], v1 = idx < 32 ? x0[idx + 1] : x1[idx - 31];
                    const f32x2_t z = f2_fma(f2(__uint_as_float(v0), __uint_as_float(v1)), rs, mr);
                    const f32x2_t y = f2_fma(z, *reinterpret_cast<const f32x2_t *>(gnw + c),
                                             *reinterpret_cast<const f32x2_t *>(gnb + c));
                    float y0, y1;
                    f2_split(y, y0, y1);
                    w[e] = mul_bf16x2(cvt_bf16x2(y0, y1), swish_bf16x2(ogw[e]));
                }
                st16(pp, make_uint4(w[0], w[1], w[2], w[3]));
            }
            }  // (EPI == 1)
            uint8_t *const ob = obuf(n);
            fence_proxy_async_smem();
            if constexpr (BIAS != 0) {
                if (named_sync_or<kBarOut, 128>(!okc)) {
                    bad = 1;
                    break;
                }
                if (lead) mbar_arrive(&cempty[n % NF]);
            } else {
                named_sync<kBarOut, 128>();
            }
            if (lead) {
                tstore(&p.to, ob, 0, t0);
                tstore(&p.to, ob + kHalf, 64, t0);
                bulk_commit();
            }
        }
        if (lead) {
            bulk_wait<0>();
            // no og tile may still be landing when the CTA leaves (the last
            // request on each of the two barriers)
            for (int m = ogi > 2 ? ogi - 2 : 0; m < ogi; ++m)
                if (!mbar_wait(&ogfull[m & 1], (uint32_t)(m >> 1) & 1u, wait_ns)) bad = 1;
        }
    }

    // ============================================================ teardown
    // a CTA that read no carried state still leaves only after the grid it was
    // launched behind has finished (a no-op for an ordinary launch)
    if (tid == 0) griddep_wait();
    const int aborted = __syncthreads_or(bad);
    if (aborted && tid == 0) atomicOr(&g_tc_error, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
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

// [BH][L][128] bf16 viewed as a 3-D tensor {128, L, BH}; box {64, 64, 1} with
// the 128-byte swizzle (every load and store of this kernel uses that box).
bool make_map(CUtensorMap *m, const void *base, int L, int BH) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)L * kD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// fp32 [BH][L][128] as {128, L, BH}; box {32, 64, 1} (128 bytes inner) with
// the 128-byte swizzle: the output map of the fp32-output instances.
bool make_map_f32(CUtensorMap *m, const void *base, int L, int BH) {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)L * kD * 4};
    cuuint32_t box[3] = {32, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Segment scan: S_in(0) = S_0 (the initial state, or 0), S_in(p+1) =
// diag(e^{B_p}) S_in(p) + dS_p for every segment p but the last (the full
// pass writes the final state). One thread per state element (z included), a
// sequential loop over the segments.
__global__ void __launch_bounds__(256) la_seg_scan_kernel(const float *__restrict__ seg_state,
                                                          const float *__restrict__ seg_logdecay,
                                                          const float *__restrict__ initial,
                                                          float *__restrict__ state_in, int nseg, int blk,
                                                          int value_side) {
    // the full pass after this scan may start launching now: its CTAs set up
    // and begin their first chunks, and wait for this grid before reading the
    // carried states
    griddep_launch_dependents();
    const int bh = blockIdx.x;
    const int e = blockIdx.y * blockDim.x + threadIdx.x;
    if (e >= blk) return;
    // the gated channel of this element: its key channel (row), or its value
    // channel (column) with the gate on the value side
    const int d = e < kD * kD ? (value_side ? e % kD : e / kD) : e - kD * kD;
    const size_t base = (size_t)bh * nseg;
    float acc = initial ? initial[(size_t)bh * blk + e] : 0.f;
    // the state carried into each segment; the last one's end state (the final
    // state) comes from the full pass, so there is none to read for it
    for (int sgi = 0; sgi < nseg; ++sgi) {
        if (sgi > 0 || initial) state_in[(base + sgi) * blk + e] = acc;
        if (sgi + 1 < nseg) acc = __expf(seg_logdecay[(base + sgi) * kD + d]) * acc + seg_state[(base + sgi) * blk + e];
    }
}

// after_scan: launched behind the segment scan as a programmatic dependent
// launch, so that its CTAs set up and start on their first chunks while the
// scan finishes (they wait for it before reading the carried states).
template <int GATE, bool ELU1, bool NORM, bool SO, bool OF32 = false, bool REV = false, int EPI = 0, int BIAS = 0>
int launch_t(const TcParams &prm, int grid, cudaStream_t s, bool after_scan) {
    using LY = Layout<GATE, NORM, SO, OF32, EPI, BIAS>;
    static_assert(LY::NS >= 2 && LY::bytes <= kSmemBudget, "shared memory budget");
    static_assert(LY::colP + 64 <= kTmemCols && LY::colO1 + LY::NW <= LY::colP, "TMEM budget");
    auto kern = la_chunk_tc_kernel<GATE, ELU1, NORM, SO, OF32, REV, EPI, BIAS>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)LY::bytes) != cudaSuccess)
        return LA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = LY::bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_scan ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return LA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

template <int GATE, bool SO>
int launch_g(const TcParams &prm, int grid, cudaStream_t s, bool elu1, bool norm, bool pdl) {
    if (elu1)
        return norm ? launch_t<GATE, true, true, SO>(prm, grid, s, pdl) : launch_t<GATE, true, false, SO>(prm, grid, s, pdl);
    return norm ? launch_t<GATE, false, true, SO>(prm, grid, s, pdl) : launch_t<GATE, false, false, SO>(prm, grid, s, pdl);
}

template <bool SO>
int launch_mode(const TcParams &prm, int grid, cudaStream_t s, int mode, bool out_f32 = false, bool value_gate = false,
                bool pdl = false, bool rev = false, int epi = 0, int bias = 0) {
    const bool elu1 = mode & LA_PHI_ELU1, norm = mode & LA_NORMALIZE;
    if (bias != 0) {
        // the bias instances: no gate or normaliser, bf16 output; with LA_PHI_ELU1
        // the feature map applies to the value tile
        if (norm || out_f32 || value_gate || epi || (mode & (LA_GATE_HEAD | LA_GATE_CHANNEL)) || rev != (bias == 2))
            return LA_ERR_INTERNAL;
        if (bias == 1)
            return elu1 ? launch_t<0, true, false, SO, false, false, 0, 1>(prm, grid, s, pdl)
                        : launch_t<0, false, false, SO, false, false, 0, 1>(prm, grid, s, pdl);
        return elu1 ? launch_t<0, true, false, SO, false, true, 0, 2>(prm, grid, s, pdl)
                    : launch_t<0, false, false, SO, false, true, 0, 2>(prm, grid, s, pdl);
    }
    if (epi == 2 && !SO) {
        // the backward prep: the normalised causal form, no gate
        if (!norm || out_f32 || value_gate || rev || (mode & (LA_GATE_HEAD | LA_GATE_CHANNEL))) return LA_ERR_INTERNAL;
        return elu1 ? launch_t<0, true, true, false, false, false, 2>(prm, grid, s, pdl)
                    : launch_t<0, false, true, false, false, false, 2>(prm, grid, s, pdl);
    }
    if (epi == 1 && !SO) {
        // the RetNet epilogue in the store: no normaliser, no gate or the head gate
        if (norm || out_f32 || value_gate || rev || (mode & LA_GATE_CHANNEL)) return LA_ERR_INTERNAL;
        if (mode & LA_GATE_HEAD)
            return elu1 ? launch_t<1, true, false, false, false, false, 1>(prm, grid, s, pdl)
                        : launch_t<1, false, false, false, false, false, 1>(prm, grid, s, pdl);
        return elu1 ? launch_t<0, true, false, false, false, false, 1>(prm, grid, s, pdl)
                    : launch_t<0, false, false, false, false, false, 1>(prm, grid, s, pdl);
    }
    if (rev) {
        // anti-causal: no normaliser; no gate (with either feature map), the head
        // gate or the channel gate (identity feature map; the channel gate also
        // on the value side)
        if (norm) return LA_ERR_INTERNAL;
        if (mode & LA_GATE_CHANNEL) {
            if (out_f32) return LA_ERR_INTERNAL;
            if (value_gate) {
                if (elu1)
                    return SO ? launch_t<3, true, false, true, false, true>(prm, grid, s, pdl)
                              : launch_t<3, true, false, false, false, true>(prm, grid, s, pdl);
                return SO ? launch_t<3, false, false, true, false, true>(prm, grid, s, pdl)
                          : launch_t<3, false, false, false, false, true>(prm, grid, s, pdl);
            }
            if (elu1)
                return SO ? launch_t<2, true, false, true, false, true>(prm, grid, s, pdl)
                          : launch_t<2, true, false, false, false, true>(prm, grid, s, pdl);
            return SO ? launch_t<2, false, false, true, false, true>(prm, grid, s, pdl)
                      : launch_t<2, false, false, false, false, true>(prm, grid, s, pdl);
        }
        if (value_gate) return LA_ERR_INTERNAL;
        const bool gh = mode & LA_GATE_HEAD;
        if (elu1) {
            if (gh || out_f32) return LA_ERR_INTERNAL;
            return SO ? launch_t<0, true, false, true, false, true>(prm, grid, s, pdl)
                      : launch_t<0, true, false, false, false, true>(prm, grid, s, pdl);
        }
        if (SO)
            return gh ? launch_t<1, false, false, true, false, true>(prm, grid, s, pdl)
                      : launch_t<0, false, false, true, false, true>(prm, grid, s, pdl);
        if (out_f32)
            return gh ? launch_t<1, false, false, false, true, true>(prm, grid, s, pdl)
                      : launch_t<0, false, false, false, true, true>(prm, grid, s, pdl);
        return gh ? launch_t<1, false, false, false, false, true>(prm, grid, s, pdl)
                  : launch_t<0, false, false, false, false, true>(prm, grid, s, pdl);
    }
    if (value_gate) {
        // the per-channel gate on the value side: no normaliser, bf16 output; with
        // elu+1 the feature map applies to the value tile alone
        if (norm || !(mode & LA_GATE_CHANNEL) || out_f32) return LA_ERR_INTERNAL;
        if (elu1)
            return SO ? launch_t<3, true, false, true>(prm, grid, s, pdl) : launch_t<3, true, false, false>(prm, grid, s, pdl);
        return SO ? launch_t<3, false, false, true>(prm, grid, s, pdl) : launch_t<3, false, false, false>(prm, grid, s, pdl);
    }
    if (out_f32 && !SO) {
        // fp32 output: identity feature map, no normaliser, no gate or the head gate
        if (elu1 || norm || (mode & LA_GATE_CHANNEL)) return LA_ERR_INTERNAL;
        return (mode & LA_GATE_HEAD) ? launch_t<1, false, false, false, true>(prm, grid, s, pdl)
                                     : launch_t<0, false, false, false, true>(prm, grid, s, pdl);
    }
    if (mode & LA_GATE_CHANNEL) return launch_g<2, SO>(prm, grid, s, elu1, norm, pdl);
    if (mode & LA_GATE_HEAD) return launch_g<1, SO>(prm, grid, s, elu1, norm, pdl);
    return launch_g<0, SO>(prm, grid, s, elu1, norm, pdl);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

// The error word of the tensor-core forward (set when a bounded wait ran out),
// read and cleared; the caller has synchronised the work that could set it.
int tc_error_take(unsigned int *value) {
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(value, g_tc_error, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(unsigned int)) != cudaSuccess)
        return LA_ERR_CUDA;
    return LA_OK;
}

// The RetNet output epilogue runs in the tensor-core kernel's store for bf16
// output without the normaliser, with no gate or the head gate (causal).
bool chunk_tc_fuses_epilogue(const ChunkArgs &a) {
    return !(a.mode & (LA_NORMALIZE | LA_GATE_CHANNEL)) && !a.out_f32 && !a.value_gate && !a.reverse &&
           chunk_tc_supports(a);
}

// The debug word of the tensor-core forward (LA_DEBUG builds: the source line
// of the first failed bounds check; always 0 otherwise), read and cleared.
int tc_debug_take(unsigned int *line) {
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(line, g_tc_debug, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_tc_debug, &zero, sizeof(unsigned int)) != cudaSuccess)
        return LA_ERR_CUDA;
    return LA_OK;
}

bool chunk_tc_supports(const ChunkArgs &a) {
    if ((a.mode & LA_DTYPE_F32) || a.dk != kD || a.dv != kD || a.chunk != kC || a.L < 1) return false;
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10 && get_encode();
}

// Segments per sequence: one CTA per (b, h) fills the GPU when there are at
// least half as many sequences as SMs; fewer sequences are each cut into
// segments of whole chunks so that (b, h, segment) CTAs cover the SMs.
int tc_segments(int BH, int nchunks, int *seg_chunks) {
    const int sms = sm_count();
    int nseg = 1;
    if (sms > 0 && 2 * BH <= sms) nseg = sms / BH < nchunks ? sms / BH : nchunks;
    if (nseg < 1) nseg = 1;
    const int cs = (nchunks + nseg - 1) / nseg;
    *seg_chunks = cs;
    return (nchunks + cs - 1) / cs;
}

// Scratch bytes the tensor-core path needs for these arguments (0 when the
// sequences are not split).
size_t chunk_tc_scratch_bytes(const ChunkArgs &a) {
    const int BH = a.B * a.H;
    int seg_chunks = 0;
    const int nseg = tc_segments(BH, (a.L + kC - 1) / kC, &seg_chunks);
    if (nseg == 1) return 0;
    const size_t blk = (size_t)kD * kD + ((a.mode & LA_NORMALIZE) ? kD : 0) + (a.bias ? kD : 0);
    const size_t nsb = (size_t)BH * nseg;
    return (2 * nsb * blk + nsb * kD) * sizeof(float);
}

// The tensor-core path with caller-provided scratch (at least
// chunk_tc_scratch_bytes(a) bytes, 256-byte aligned). A sequence that is not
// split is one launch; split sequences take three: the state-only pass, the
// segment scan and the full pass from the carried states.
namespace {
int launch_chunk_tc_impl(const ChunkArgs &a, cudaStream_t s, int *launches, void *scratch, size_t scratch_bytes,
                         uint64_t wait_ns, int stall_chunk) {
    if (!get_encode()) return LA_ERR_CUDA;
    const int BH = a.B * a.H;
    const int nchunks = (a.L + kC - 1) / kC;
    TcParams prm;
    memset(&prm, 0, sizeof(prm));
    if (!make_map(&prm.tq, a.q, a.L, BH) || !make_map(&prm.tk, a.k, a.L, BH) || !make_map(&prm.tv, a.v, a.L, BH) ||
        !(a.out_f32 ? make_map_f32(&prm.to, a.out, a.L, BH) : make_map(&prm.to, a.out, a.L, BH)))
        return LA_ERR_CUDA;
    if ((a.mode & LA_GATE_CHANNEL) && !make_map(&prm.tg, a.gate, a.L, BH)) return LA_ERR_CUDA;
    const int epi = a.gn_ogate != nullptr ? 1 : a.bp_dout != nullptr ? 2 : 0;
    if (epi == 1) {
        if (!chunk_tc_fuses_epilogue(a) || !make_map(&prm.tog, a.gn_ogate, a.L, BH)) return LA_ERR_INTERNAL;
        prm.gn_w = a.gn_weight;
        prm.gn_b = a.gn_bias;
        prm.gn_eps = a.gn_eps;
    } else if (epi == 2) {
        // the backward prep: the output gradient's tile rides where og would
        if (a.bp_e == nullptr || !make_map(&prm.tog, a.bp_dout, a.L, BH)) return LA_ERR_INTERNAL;
        prm.e_out = a.bp_e;
        prm.n_e = (size_t)BH * a.L;
    }
    if (a.bias != 0) {
        // the carried vector adds to the state block of a split sequence's
        // segments (it has no layout in a caller's initial or final state)
        if (a.bias_e == nullptr || epi != 0 || a.initial_state || a.final_state) return LA_ERR_INTERNAL;
        prm.e_in = a.bias_e;
        prm.n_e = (size_t)BH * a.L;
        if (a.mode & LA_PHI_ELU1) {
            // phi' of the map's input multiplies the store: its tile rides where og would
            if (a.bias_x == nullptr || !make_map(&prm.tog, a.bias_x, a.L, BH)) return LA_ERR_INTERNAL;
        }
    }
    prm.gamma = (a.mode & LA_GATE_HEAD) ? static_cast<const float *>(a.gate) : nullptr;
    prm.final_state = a.final_state;
    prm.H = a.H;
    prm.L = a.L;
    prm.mode = a.mode;
    prm.nseg = tc_segments(BH, nchunks, &prm.seg_chunks);
    prm.init0 = a.initial_state != nullptr;
    prm.wait_ns = wait_ns;
    prm.stall_chunk = stall_chunk;
    const size_t blkf = (size_t)kD * kD + ((a.mode & LA_NORMALIZE) ? kD : 0);
    prm.n_final = a.final_state ? (size_t)BH * blkf : 0;
    prm.n_state_in = a.initial_state ? (size_t)BH * blkf : 0;  // (split: the carried states, below)
    if (stall_chunk >= 0 && prm.nseg != 1) return LA_ERR_UNSUPPORTED;  // the stall runs one launch only
    if (prm.nseg == 1) {
        prm.state_in = a.initial_state;  // [BH][blk]: the segment of CTA bh starts there
        const int rc = launch_mode<false>(prm, BH, s, a.mode, a.out_f32, a.value_gate, false, a.reverse, epi, a.bias);
        if (rc == LA_OK) *launches += 1;
        return rc;
    }
    const size_t blk = (size_t)kD * kD + ((a.mode & LA_NORMALIZE) ? kD : 0) + (a.bias ? kD : 0);
    const size_t nsb = (size_t)BH * prm.nseg;
    if (scratch == nullptr || scratch_bytes < (2 * nsb * blk + nsb * kD) * sizeof(float)) return LA_ERR_INTERNAL;
    float *seg_state = static_cast<float *>(scratch);
    float *state_in = seg_state + nsb * blk;
    float *seg_logdecay = state_in + nsb * blk;
    prm.seg_state = seg_state;
    prm.seg_logdecay = seg_logdecay;
    prm.n_seg_state = nsb * blk;
    prm.n_seg_logdecay = nsb * kD;
    // the state-only pass: every segment but each sequence's last
    int rc = launch_mode<true>(prm, BH * (prm.nseg - 1), s, a.mode, false, a.value_gate, false, a.reverse, 0, a.bias);
    if (rc != LA_OK) return rc;
    *launches += 1;
    la_seg_scan_kernel<<<dim3((unsigned)BH, (unsigned)((blk + 255) / 256)), 256, 0, s>>>(
        seg_state, seg_logdecay, a.initial_state, state_in, prm.nseg, (int)blk, a.value_gate);
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    *launches += 1;
    prm.state_in = state_in;
    prm.n_state_in = nsb * blk;
    prm.seg_state = nullptr;
    prm.seg_logdecay = nullptr;
    prm.n_seg_state = prm.n_seg_logdecay = 0;
    rc = launch_mode<false>(prm, (int)nsb, s, a.mode, a.out_f32, a.value_gate, true, a.reverse, epi, a.bias);
    if (rc == LA_OK) *launches += 1;
    return rc;
}
}  // namespace

int launch_chunk_tc_into(const ChunkArgs &a, cudaStream_t s, int *launches, void *scratch,
                         size_t scratch_bytes) {
    return launch_chunk_tc_impl(a, s, launches, scratch, scratch_bytes, kWaitNs, -1);
}

// Diagnostics: one unsplit launch whose producer issues no tiles from chunk
// stall_chunk on and whose bounded waits give up after wait_ns, so that the
// time-out path (error word, drain, TMEM freed) runs on purpose.
int launch_chunk_tc_stalled(const ChunkArgs &a, cudaStream_t s, int *launches, int stall_chunk,
                            unsigned long long wait_ns) {
    return launch_chunk_tc_impl(a, s, launches, nullptr, 0, wait_ns, stall_chunk);
}

// The tensor-core path with its scratch (if any) allocated and freed in
// stream order around the launches.
int launch_chunk_tc(const ChunkArgs &a, cudaStream_t s, int *launches) {
    const size_t bytes = chunk_tc_scratch_bytes(a);
    if (bytes == 0) return launch_chunk_tc_into(a, s, launches, nullptr, 0);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, bytes, s) != LA_OK) return LA_ERR_CUDA;
    int rc = launch_chunk_tc_into(a, s, launches, scratch, bytes);
    if (cudaFreeAsync(scratch, s) != cudaSuccess && rc == LA_OK) rc = LA_ERR_CUDA;
    return rc;
}

}  // namespace la
