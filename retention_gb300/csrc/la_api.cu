// la_api.cu -- the C ABI of include/la.h: argument validation, kernel choice,
// status strings, and the scratch memory of the multi-kernel paths (the
// library's own stream-ordered pool, and the fixed array of
// la_chunk_fwd_noalloc). Every check runs before any launch.
#include <atomic>
#include <cuda.h>
#include <cmath>
#include <mutex>
#include <stdint.h>

#include "la_common.cuh"

namespace {

std::atomic<unsigned long long> g_launches{0};

constexpr int kKnownModeBits = LA_PHI_ELU1 | LA_NORMALIZE | LA_GATE_HEAD | LA_GATE_CHANNEL |
                               LA_DTYPE_F32 | LA_KERNEL_SIMT | LA_REVERSE;
// what the anti-causal form does not run with (and elu+1 together with the head gate)
constexpr int kNotWithReverse = LA_NORMALIZE | LA_DTYPE_F32 | LA_KERNEL_SIMT;
bool reverse_unsupported(int mode) {
    return (mode & kNotWithReverse) || ((mode & LA_PHI_ELU1) && (mode & LA_GATE_HEAD));
}

bool dim_ok(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// `chunk`: a chunk-forward call (the only kind that takes LA_REVERSE)
int check_mode(int mode, const void *gate, bool decode, bool chunk = false) {
    if (mode & ~kKnownModeBits) return LA_ERR_INVALID_ARG;
    if (decode && (mode & LA_KERNEL_SIMT)) return LA_ERR_INVALID_ARG;
    if (mode & LA_REVERSE) {
        if (!chunk) return LA_ERR_INVALID_ARG;
        if (reverse_unsupported(mode)) return LA_ERR_UNSUPPORTED;
    }
    const bool gh = mode & LA_GATE_HEAD, gc = mode & LA_GATE_CHANNEL;
    if (gh && gc) return LA_ERR_INVALID_ARG;
    if ((gh || gc) && gate == nullptr) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

// The output epilogue's own arguments (ogate null: no epilogue).
struct Epilogue {
    const void *ogate;
    const float *weight, *bias;
    float eps;
};

int check_epilogue(const Epilogue &ep) {
    if (!(ep.eps >= 0.f) || std::isinf(ep.eps)) return LA_ERR_INVALID_ARG;
    if (!aligned16(ep.ogate)) return LA_ERR_MISALIGNED;
    if ((ep.weight && !aligned16(ep.weight)) || (ep.bias && !aligned16(ep.bias))) return LA_ERR_MISALIGNED;
    return LA_OK;
}

int chunk_fwd(const void *q, const void *k, const void *v, const void *gate, const float *initial_state,
              void *out, float *final_state, int B, int H, int L, int dk, int dv, int mode, int chunk,
              la_stream_t stream, const Epilogue &ep = Epilogue{nullptr, nullptr, nullptr, 0.f}) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (chunk < 1 || chunk > 128) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    int rc = check_mode(mode, gate, false, true);
    if (rc != LA_OK) return rc;
    const long nbh = (long)B * H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool norm = mode & LA_NORMALIZE;
    if (nbh == 0) return LA_OK;
    if (initial_state && !aligned16(initial_state)) return LA_ERR_MISALIGNED;
    if (L == 0) {
        // an empty sequence leaves the starting state: S_0 = 0 (and z_0 = 0) or the given one
        if (final_state) {
            if (!aligned16(final_state)) return LA_ERR_MISALIGNED;
            const size_t bytes = (size_t)nbh * ((size_t)dk * dv + (norm ? dk : 0)) * sizeof(float);
            const cudaError_t e = initial_state
                ? cudaMemcpyAsync(final_state, initial_state, bytes, cudaMemcpyDeviceToDevice, s)
                : cudaMemsetAsync(final_state, 0, bytes, s);
            if (e != cudaSuccess) return LA_ERR_CUDA;
        }
        return LA_OK;
    }
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_MISALIGNED;
    if (final_state && !aligned16(final_state)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_CHANNEL) && !aligned16(gate)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_HEAD) && ((uintptr_t)gate & 3u)) return LA_ERR_MISALIGNED;
    if (ep.ogate && (rc = check_epilogue(ep)) != LA_OK) return rc;

    const bool rev = mode & LA_REVERSE;
    la::ChunkArgs a{q, k, v, gate, out, final_state, B, H, L, dk, dv, mode & ~LA_REVERSE, chunk, initial_state,
                    0, 0, rev ? 1 : 0};
    int launches = 0;
    const bool tc = !(mode & LA_KERNEL_SIMT) && la::chunk_tc_supports(a);
    // the output epilogue goes into the tensor-core kernel's store where it can
    bool fused = false;
    if (ep.ogate && tc && la::chunk_tc_fuses_epilogue(a)) {
        a.gn_ogate = ep.ogate;
        a.gn_weight = ep.weight;
        a.gn_bias = ep.bias;
        a.gn_eps = ep.eps;
        fused = true;
    }
    if (tc)
        rc = la::launch_chunk_tc(a, s, &launches);
    else if (rev)
        return LA_ERR_UNSUPPORTED;  // the anti-causal form runs on the tensor-core kernel only
    else
        rc = la::launch_chunk_simt(a, s, &launches);
    if (rc == LA_OK && ep.ogate && !fused) {
        // the output epilogue: a streaming pass of its own, in place on out
        la::GnArgs g{out, ep.ogate, ep.weight, ep.bias, ep.eps, out, B, H, L, dv, mode & LA_DTYPE_F32};
        rc = la::launch_gn_swish(g, s, &launches);
    }
    g_launches += (unsigned long long)launches;
    return rc;
}

}  // namespace

extern "C" {

int la_chunk_fwd(const void *q, const void *k, const void *v, const void *gate, void *out,
                 float *final_state, int B, int H, int L, int dk, int dv, int mode, int chunk,
                 la_stream_t stream) {
    return chunk_fwd(q, k, v, gate, nullptr, out, final_state, B, H, L, dk, dv, mode, chunk, stream);
}

int la_chunk_fwd_from_state(const void *q, const void *k, const void *v, const void *gate,
                            const float *initial_state, void *out, float *final_state, int B, int H,
                            int L, int dk, int dv, int mode, int chunk, la_stream_t stream) {
    return chunk_fwd(q, k, v, gate, initial_state, out, final_state, B, H, L, dk, dv, mode, chunk, stream);
}

int la_chunk_fwd_gn_swish(const void *q, const void *k, const void *v, const void *gate,
                          const float *initial_state, const void *ogate, const float *gn_weight,
                          const float *gn_bias, float gn_eps, void *out, float *final_state, int B, int H,
                          int L, int dk, int dv, int mode, int chunk, la_stream_t stream) {
    if (ogate == nullptr && L > 0 && (long)B * H > 0) return LA_ERR_INVALID_ARG;
    return chunk_fwd(q, k, v, gate, initial_state, out, final_state, B, H, L, dk, dv, mode, chunk, stream,
                     Epilogue{ogate, gn_weight, gn_bias, gn_eps});
}

int la_group_norm_swish(const void *x, const void *ogate, const float *gn_weight, const float *gn_bias,
                        float gn_eps, void *out, int B, int H, int L, int dv, int mode, la_stream_t stream) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    if (mode & ~LA_DTYPE_F32) return LA_ERR_INVALID_ARG;
    if ((long)B * H * L == 0) return LA_OK;
    if (!x || !ogate || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return LA_ERR_MISALIGNED;
    int rc = check_epilogue(Epilogue{ogate, gn_weight, gn_bias, gn_eps});
    if (rc != LA_OK) return rc;
    la::GnArgs g{x, ogate, gn_weight, gn_bias, gn_eps, out, B, H, L, dv, mode};
    int launches = 0;
    rc = la::launch_gn_swish(g, reinterpret_cast<cudaStream_t>(stream), &launches);
    g_launches += (unsigned long long)launches;
    return rc;
}

int la_chunk_bwd(const void *q, const void *k, const void *v, const void *gate, const void *dout, void *dq,
                 void *dk_, void *dv_, void *dgate, int B, int H, int L, int dk, int dv, int mode,
                 la_stream_t stream) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    int rc = check_mode(mode, gate, false);
    if (rc != LA_OK) return rc;
    const long nbh = (long)B * H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (nbh == 0 || L == 0) return LA_OK;
    if (!q || !k || !v || !dout || !dq || !dk_ || !dv_) return LA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, dout, dq, dk_, dv_};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_CHANNEL) && (!aligned16(gate) || (dgate && !aligned16(dgate)))) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_HEAD) && ((uintptr_t)gate & 3u)) return LA_ERR_MISALIGNED;
    la::BwdArgs a{q, k, v, gate, dout, dq, dk_, dv_,
                  (mode & LA_GATE_CHANNEL) ? dgate : nullptr, B, H, L, dk, dv, mode & ~LA_KERNEL_SIMT};
    int launches = 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    rc = (!(mode & LA_KERNEL_SIMT) && la::bwd_tc_supports(a)) ? la::launch_bwd_tc(a, s, &launches)
                                                               : la::launch_bwd(a, s, &launches);
    g_launches += (unsigned long long)launches;
    return rc;
}

int la_decode_step(const void *q, const void *k, const void *v, const void *gate, float *state,
                   void *out, int B, int H, int dk, int dv, int mode, la_stream_t stream) {
    if (B < 0 || H < 0) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    int rc = check_mode(mode, gate, true);
    if (rc != LA_OK) return rc;
    const long nbh = (long)B * H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (nbh == 0) return LA_OK;
    if (!q || !k || !v || !state || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(state))
        return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_CHANNEL) && !aligned16(gate)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_HEAD) && ((uintptr_t)gate & 3u)) return LA_ERR_MISALIGNED;
    la::DecodeArgs a{q, k, v, gate, state, out, B, H, dk, dv, mode};
    int launches = 0;
    rc = la::launch_decode(a, reinterpret_cast<cudaStream_t>(stream), &launches);
    g_launches += (unsigned long long)launches;
    return rc;
}

int la_delta_fwd(const void *q, const void *k, const void *v, const void *beta, void *out,
                 float *final_state, int B, int H, int L, int dk, int dv, int mode, la_stream_t stream) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    if (mode & ~(LA_DTYPE_F32 | LA_KERNEL_SIMT)) return LA_ERR_INVALID_ARG;
    const long nbh = (long)B * H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (nbh == 0) return LA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (final_state && !aligned16(final_state)) return LA_ERR_MISALIGNED;
    if (L == 0) {
        // no token: the state stays S_0 = 0
        if (final_state &&
            cudaMemsetAsync(final_state, 0, (size_t)nbh * dk * dv * sizeof(float), s) != cudaSuccess)
            return LA_ERR_CUDA;
        return LA_OK;
    }
    if (!q || !k || !v || !beta || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_MISALIGNED;
    if ((uintptr_t)beta & ((mode & LA_DTYPE_F32) ? 3u : 1u)) return LA_ERR_MISALIGNED;
    la::DeltaArgs a{q, k, v, beta, out, final_state, B, H, L, dk, dv, mode & LA_DTYPE_F32};
    int launches = 0;
    const int rc = (!(mode & LA_KERNEL_SIMT) && la::delta_tc_supports(a)) ? la::launch_delta_tc(a, s, &launches)
                                                                          : la::launch_delta(a, s, &launches);
    g_launches += (unsigned long long)launches;
    return rc;
}

int la_chunk_fwd_path(int B, int H, int L, int dk, int dv, int mode, int chunk) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (chunk < 1 || chunk > 128) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    if (mode & ~kKnownModeBits) return LA_ERR_INVALID_ARG;
    if ((mode & LA_GATE_HEAD) && (mode & LA_GATE_CHANNEL)) return LA_ERR_INVALID_ARG;
    if ((mode & LA_REVERSE) && reverse_unsupported(mode)) return LA_ERR_UNSUPPORTED;
    la::ChunkArgs a{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, H, L, dk, dv, mode & ~LA_REVERSE, chunk};
    const bool tc = !(mode & LA_KERNEL_SIMT) && la::chunk_tc_supports(a);
    if ((mode & LA_REVERSE) && !tc) return LA_ERR_UNSUPPORTED;
    return tc ? 1 : 0;
}

const char *la_status_string(int status) {
    switch (status) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: shape or mode not supported by the library";
        case LA_ERR_MISALIGNED: return "LA_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case LA_ERR_CUDA: return "LA_ERR_CUDA: a CUDA call or kernel launch failed";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device-side wait ran out";
        case LA_ERR_INTERNAL: return "LA_ERR_INTERNAL: internal consistency check failed";
        default: return "unknown la_status";
    }
}

unsigned long long la_kernel_launches(void) { return g_launches.load(); }

int la_chunk_fwd_stall_test(const void *q, const void *k, const void *v, const void *gate, void *out, int B,
                            int H, int L, int mode, int stall_chunk, long long wait_ns, la_stream_t stream) {
    if (B < 1 || H < 1 || L < 1 || stall_chunk < 0) return LA_ERR_INVALID_ARG;
    if (wait_ns < 100000LL || wait_ns > 2000000000LL) return LA_ERR_INVALID_ARG;
    int rc = check_mode(mode, gate, false);
    if (rc != LA_OK) return rc;
    if ((long)B * H > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_CHANNEL) && !aligned16(gate)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_HEAD) && ((uintptr_t)gate & 3u)) return LA_ERR_MISALIGNED;
    la::ChunkArgs a{q, k, v, gate, out, nullptr, B, H, L, 128, 128, mode, 64, nullptr};
    if ((mode & LA_KERNEL_SIMT) || !la::chunk_tc_supports(a)) return LA_ERR_UNSUPPORTED;
    int launches = 0;
    rc = la::launch_chunk_tc_stalled(a, reinterpret_cast<cudaStream_t>(stream), &launches, stall_chunk,
                                     (unsigned long long)wait_ns);
    g_launches += (unsigned long long)launches;
    return rc;
}

int la_device_status(la_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return LA_ERR_CUDA;
    unsigned int tc = 0, delta = 0, dbg_tc = 0, dbg_dec = 0;
    const int rcs[4] = {la::tc_error_take(&tc), la::delta_tc_error_take(&delta), la::tc_debug_take(&dbg_tc),
                        la::decode_debug_take(&dbg_dec)};
    for (int rc : rcs)
        if (rc != LA_OK) return rc;
    if (dbg_tc | dbg_dec) return LA_ERR_INTERNAL;  // a bounds check of an LA_DEBUG build failed
    return (tc | delta) ? LA_ERR_TIMEOUT : LA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scratch of the multi-kernel paths: stream-ordered allocations from a memory
// pool of the library's own, one per device, created on first use. Its release
// threshold is raised so that memory freed at the end of one call stays
// mapped for the next instead of being returned at the next synchronisation
// and mapped again (which costs a large fraction of a call's time at these
// sizes); the pool therefore keeps up to the largest scratch any call used
// until the process exits. The device's default pool, which belongs to the
// whole process, is neither used nor changed.
namespace la {
namespace {
constexpr int kMaxPoolDevices = 64, kPoolSlots = 4;
std::mutex g_pool_mu;
// per device, a few (context id, pool) pairs: a pool dies with its context
// (e.g. at cudaDeviceReset), and a context made again gets a new id, so a dead
// pool is never used; a caller alternating between contexts on one device
// keeps one pool in each
struct PoolSlot {
    unsigned long long ctx;
    cudaMemPool_t pool;
};
PoolSlot g_pool[kMaxPoolDevices][kPoolSlots] = {};
unsigned int g_pool_next[kMaxPoolDevices] = {};  // slot to replace when all are taken

typedef CUresult (*PfnCtxGetCurrent)(CUcontext *);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long *);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the current context (0 when it cannot be had). The driver calls
// come through the runtime's entry-point query, so nothing links the driver.
unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(f);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&c) != CUDA_SUCCESS || c == nullptr || g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

int scratch_pool(cudaMemPool_t *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxPoolDevices) return LA_ERR_UNSUPPORTED;
    const unsigned long long ctx = current_context_id();  // 0: unknown (e.g. no context current yet)
    std::lock_guard<std::mutex> lock(g_pool_mu);
    PoolSlot *slots = g_pool[dev];
    for (int i = 0; i < kPoolSlots; ++i) {
        // with the context id unknown the first pool made on the device serves
        if (slots[i].pool != nullptr && (slots[i].ctx == ctx || ctx == 0)) {
            *out = slots[i].pool;
            return LA_OK;
        }
    }
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return LA_ERR_CUDA;
    uint64_t keep = UINT64_MAX;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
        cudaMemPoolDestroy(pool);
        return LA_ERR_CUDA;
    }
    // an empty slot, else the oldest (most likely of a context that is gone)
    int slot = -1;
    for (int i = 0; i < kPoolSlots && slot < 0; ++i)
        if (slots[i].pool == nullptr) slot = i;
    if (slot < 0) slot = (int)(g_pool_next[dev]++ % kPoolSlots);
    slots[slot] = PoolSlot{ctx, pool};
    *out = pool;
    return LA_OK;
}
}  // namespace

int scratch_alloc(void **p, size_t bytes, cudaStream_t s) {
    cudaMemPool_t pool = nullptr;
    const int rc = scratch_pool(&pool);
    if (rc != LA_OK) return rc == LA_ERR_UNSUPPORTED ? LA_ERR_CUDA : rc;
    return cudaMallocFromPoolAsync(p, bytes, pool, s) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
}  // namespace la

// ---------------------------------------------------------------------------
// la_chunk_fwd_noalloc: la_chunk_fwd for callers that must not allocate device
// memory. When a short batch makes the tensor-core path split sequences into
// segments, its scratch comes from this fixed device array instead of
// cudaMallocAsync. The array exists once per GPU that loads the library and
// stays allocated until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current device's context. The
// host-side name of the array is only a stand-in, so the address is looked up
// with the device current. It is looked up on every call rather than cached:
// a cache keyed by device would keep a dead address after the context is
// destroyed and created again (cudaDeviceReset), and the lookup allocates
// nothing. The first lookup in a context loads the module that holds the
// array, which is when the driver maps it.
int noalloc_scratch(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return LA_ERR_CUDA;
    *out = p;
    return LA_OK;
}

}  // namespace

extern "C" int la_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *gate, void *out,
                                    float *final_state, int B, int H, int L, int dk, int dv, int mode,
                                    int chunk, la_stream_t stream) {
    if (B < 0 || H < 0 || L < 0) return LA_ERR_INVALID_ARG;
    if (chunk < 1 || chunk > 128) return LA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    int rc = check_mode(mode, gate, false, true);
    if (rc != LA_OK) return rc;
    const long nbh = (long)B * H;
    if (nbh > 0x7fffffffL) return LA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (nbh == 0) return LA_OK;
    if (L == 0) {
        if (final_state) {
            if (!aligned16(final_state)) return LA_ERR_MISALIGNED;
            const size_t blk = (size_t)dk * dv + ((mode & LA_NORMALIZE) ? dk : 0);
            if (cudaMemsetAsync(final_state, 0, (size_t)nbh * blk * sizeof(float), s) != cudaSuccess)
                return LA_ERR_CUDA;
        }
        return LA_OK;
    }
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return LA_ERR_MISALIGNED;
    if (final_state && !aligned16(final_state)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_CHANNEL) && !aligned16(gate)) return LA_ERR_MISALIGNED;
    if ((mode & LA_GATE_HEAD) && ((uintptr_t)gate & 3u)) return LA_ERR_MISALIGNED;

    const bool rev = mode & LA_REVERSE;
    la::ChunkArgs a{q, k, v, gate, out, final_state, B, H, L, dk, dv, mode & ~LA_REVERSE, chunk, nullptr, 0, 0,
                    rev ? 1 : 0};
    int launches = 0;
    if (rev && ((mode & LA_KERNEL_SIMT) || !la::chunk_tc_supports(a))) return LA_ERR_UNSUPPORTED;
    if (!(mode & LA_KERNEL_SIMT) && la::chunk_tc_supports(a)) {
        void *scratch = nullptr;
        if (la::chunk_tc_scratch_bytes(a) > (size_t)LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_UNSUPPORTED;
        if (la::chunk_tc_scratch_bytes(a) > 0) {
            rc = noalloc_scratch(&scratch);
            if (rc != LA_OK) return rc;
        }
        rc = la::launch_chunk_tc_into(a, s, &launches, scratch, LA_NOALLOC_SCRATCH_BYTES);
    } else {
        rc = la::launch_chunk_simt(a, s, &launches);
    }
    g_launches += (unsigned long long)launches;
    return rc;
}
