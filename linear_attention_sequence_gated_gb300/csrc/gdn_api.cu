// C-ABI front end of libgdn.so: argument validation, path selection,
// workspace handling and the device status word.  Every compute step runs in
// the kernels of gdn_recurrent.cu and gdn_chunked.cu; this file launches
// nothing else.  Declarations and the full contract are in include/gdn.h.
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

// Device status word: kernels whose waits are bounded write GDN_ERR_TIMEOUT
// here when a wait gives up.  One per device that loads the library.
__device__ int g_device_status = 0;

using gdn::kMaxDevices;
int *g_status_ptr[kMaxDevices] = {};
std::mutex g_status_mu;

int *status_word_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

// Stream-ordered workspace allocations (when the caller passes none) come
// from one library-owned memory pool per device that keeps up to
// kPoolKeepBytes reserved across calls, so that a call does not map fresh
// device memory each time.  Each call still gets its own allocation, freed in
// stream order, so calls on different streams never share a workspace.
constexpr unsigned long long kPoolKeepBytes = 1ull << 30;
cudaMemPool_t g_pool[kMaxDevices] = {};
std::mutex g_pool_mu;

cudaMemPool_t pool_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        unsigned long long keep = kPoolKeepBytes;
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return nullptr;
        }
        g_pool[dev] = pool;
    }
    return g_pool[dev];
}

using gdn::host::aligned;
using gdn::host::mul_ok;
using gdn::host::overlap;
using gdn::host::Range;
using gdn::host::range_of;
using gdn::host::span_bytes;

// Tokens from which AUTO prefers the chunked path, measured on GB300 with
// bf16 q/k/v: both paths timed per call over T = 16..128, 20 calls captured
// in a CUDA graph, for 8 to 2048 (sequence, head) pairs.  The recurrent path
// costs a near-constant time per token; the chunked path a near-constant time
// per 64-token chunk (plus, below 80 pairs at head_dim 128 and at head_dim
// 256, a chunk-transform pass), so the switch sits where one chunk's time
// equals the tokens' time.  With few pairs the recurrent kernel has more of
// the GPU per pair and stays ahead longer; with very many, head_dim 64 fills
// the GPU with the recurrent kernel as well and the switch moves up again.
int chunked_min_tokens(long long pairs, int head_dim) {
    switch (head_dim) {
        case 64: return pairs < 64 ? 56 : (pairs < 256 ? 32 : (pairs < 1024 ? 40 : 56));
        // fewer than 80 pairs run the two-kernel chunked path, 80 or more the
        // one-kernel path
        case 128:
            return pairs < 32 ? 56 : (pairs < 48 ? 48 : (pairs < 64 ? 40 : (pairs < 80 ? 32 : 24)));
        case 256: return pairs < 16 ? 40 : (pairs < 24 ? 32 : 16);
        default: return INT_MAX;
    }
}

int select_path(long long pairs, int n_tokens, int head_dim, int dtype) {
    const int caps = gdn_supports(head_dim);
    if (!caps) return GDN_ERR_HEADDIM;
    if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_ARG;
    if ((caps & 2) && dtype == GDN_DTYPE_BF16 && n_tokens >= chunked_min_tokens(pairs, head_dim))
        return GDN_PATH_CHUNKED;
    return GDN_PATH_RECURRENT;
}

struct Sizes {
    unsigned long long qk_bytes, v_bytes, gb_bytes, state_bytes, out_bytes;
};

// Host-side validation; fills `sz`.  Launches nothing.
int validate(const void *q, const void *k, const void *v, const float *g, const float *beta,
             const float *state_in, const float *out, const float *state_out, int B, int T,
             int H, int Hk, int d, int dtype, int path, bool out_bf16, Sizes *sz) {
    if (B < 0 || T < 0 || H < 0 || d <= 0) return GDN_ERR_ARG;
    // key heads: value head i reads key head i % Hk; Hk must divide H
    if (H > 0 && (Hk < 1 || Hk > H || H % Hk != 0)) return GDN_ERR_ARG;
    if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return GDN_ERR_ARG;
    if (path != GDN_PATH_AUTO && path != GDN_PATH_RECURRENT && path != GDN_PATH_CHUNKED)
        return GDN_ERR_ARG;
    const int caps = gdn_supports(d);
    if (!caps) return GDN_ERR_HEADDIM;
    if (path == GDN_PATH_RECURRENT && !(caps & 1)) return GDN_ERR_HEADDIM;
    if (path == GDN_PATH_CHUNKED && !(caps & 2)) return GDN_ERR_HEADDIM;
    if (path == GDN_PATH_CHUNKED && dtype != GDN_DTYPE_BF16) return GDN_ERR_DTYPE;

    unsigned long long bth, bthd, bthkd, bh, bhdd;
    if (!mul_ok((unsigned long long)B * (unsigned long long)T, (unsigned long long)H, &bth))
        return GDN_ERR_ARG;
    if (!mul_ok(bth, (unsigned long long)d, &bthd)) return GDN_ERR_ARG;
    bthkd = H > 0 ? bthd / (unsigned long long)H * (unsigned long long)Hk : 0;
    bh = (unsigned long long)B * (unsigned long long)H;
    if (!mul_ok(bh, (unsigned long long)d * (unsigned long long)d, &bhdd)) return GDN_ERR_ARG;
    if (bh > (unsigned long long)INT_MAX) return GDN_ERR_ARG;  // one block row per (b, h)
    const unsigned long long elt = dtype == GDN_DTYPE_BF16 ? 2 : 4;
    if (!span_bytes(bthkd, elt, &sz->qk_bytes) || !span_bytes(bthd, elt, &sz->v_bytes) ||
        !span_bytes(bth, 4, &sz->gb_bytes) ||
        !span_bytes(bhdd, 4, &sz->state_bytes) ||
        !span_bytes(bthd, out_bf16 ? 2 : 4, &sz->out_bytes))
        return GDN_ERR_ARG;

    if (bh == 0) return GDN_OK;  // nothing to do, nothing to check
    if (!state_out) return GDN_ERR_ARG;
    if (bth > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;

    const uintptr_t A16 = 16;
    if (!aligned(state_out, A16) || (state_in && !aligned(state_in, A16))) return GDN_ERR_ALIGN;
    if (bth > 0) {
        if (!aligned(q, A16) || !aligned(k, A16) || !aligned(v, A16) || !aligned(out, A16))
            return GDN_ERR_ALIGN;
        if (!aligned(g, 4) || !aligned(beta, 4)) return GDN_ERR_ALIGN;
    }

    const Range rq = range_of(q, sz->qk_bytes), rk = range_of(k, sz->qk_bytes),
                rv = range_of(v, sz->v_bytes), rg = range_of(g, sz->gb_bytes),
                rb = range_of(beta, sz->gb_bytes), rsi = range_of(state_in, sz->state_bytes),
                ro = range_of(out, bth > 0 ? sz->out_bytes : 0),
                rso = range_of(state_out, sz->state_bytes);
    for (Range in : {rq, rk, rv, rg, rb, rsi, rso})
        if (overlap(ro, in)) return GDN_ERR_ALIAS;
    for (Range in : {rq, rk, rv, rg, rb})
        if (overlap(rso, in)) return GDN_ERR_ALIAS;
    if (state_in && state_in != state_out && overlap(rso, rsi)) return GDN_ERR_ALIAS;
    return GDN_OK;
}

constexpr int kPathMask = 0xff;
constexpr int kKnownOptions = GDN_OPT_L2NORM_QK | GDN_OPT_OUT_BF16;

int run(const void *q, const void *k, const void *v, const float *g, const float *beta,
        const float *state_in, float *out, float *state_out, int B, int T, int H, int Hk, int d,
        int dtype, int path_opts, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (path_opts < 0 || (path_opts & ~kPathMask & ~kKnownOptions)) return GDN_ERR_ARG;
    int path = path_opts & kPathMask;
    const bool l2norm = (path_opts & GDN_OPT_L2NORM_QK) != 0;
    const bool out_bf16 = (path_opts & GDN_OPT_OUT_BF16) != 0;
    Sizes sz{};
    int rc = validate(q, k, v, g, beta, state_in, out, state_out, B, T, H, Hk, d, dtype, path,
                      out_bf16, &sz);
    if (rc != GDN_OK) return rc;
    if ((long long)B * H == 0) return GDN_OK;

    if (T == 0) {  // no steps: the final state is the initial state
        cudaError_t e;
        if (!state_in)
            e = cudaMemsetAsync(state_out, 0, sz.state_bytes, stream);
        else if (state_in != state_out)
            e = cudaMemcpyAsync(state_out, state_in, sz.state_bytes, cudaMemcpyDeviceToDevice,
                                stream);
        else
            e = cudaSuccess;
        return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }

    if (path == GDN_PATH_AUTO) path = select_path((long long)B * H, T, d, dtype);
    const size_t need =
        path == GDN_PATH_CHUNKED ? gdn::chunked_workspace_bytes(B, T, H, d, dtype) : 0;
    if (need > 0 && workspace && (workspace_bytes < need || !aligned(workspace, 256)))
        return GDN_ERR_WORKSPACE;

    // Everything above is host-only validation; CUDA is touched from here on.
    int *status = status_word_for_current_device();
    if (!status) return GDN_ERR_CUDA;

    gdn::Problem p{q, k, v, g, beta, state_in, out, state_out, B, T, H, Hk, d, dtype,
                   (float)(1.0 / std::sqrt((double)d)), status, l2norm, out_bf16};

    if (path == GDN_PATH_RECURRENT) {
        return gdn::launch_recurrent(p, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }

    void *ws = workspace;
    bool owned = false;
    if (need > 0 && !ws) {
        cudaMemPool_t pool = pool_for_current_device();
        if (!pool) return GDN_ERR_CUDA;
        if (cudaMallocFromPoolAsync(&ws, need, pool, stream) != cudaSuccess) return GDN_ERR_NOMEM;
        owned = true;
    }
    const cudaError_t e = gdn::launch_chunked(p, ws, need, stream);
    if (owned) {
        const cudaError_t f = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess && f != cudaSuccess) return GDN_ERR_CUDA;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_forward(const float *q, const float *k, const float *v, const float *g,
                const float *beta, const float *state_in, float *out, float *state_out,
                int n_seqs, int n_tokens, int n_heads, int head_dim, gdn_stream_t stream) {
    return run(q, k, v, g, beta, state_in, out, state_out, n_seqs, n_tokens, n_heads, n_heads,
               head_dim, GDN_DTYPE_F32, GDN_PATH_AUTO, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

int gdn_forward_bf16(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, const float *state_in, float *out, float *state_out,
                     int n_seqs, int n_tokens, int n_heads, int head_dim, gdn_stream_t stream) {
    return run(q, k, v, g, beta, state_in, out, state_out, n_seqs, n_tokens, n_heads, n_heads,
               head_dim, GDN_DTYPE_BF16, GDN_PATH_AUTO, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

int gdn_forward_ex(const void *q, const void *k, const void *v, const float *g,
                   const float *beta, const float *state_in, float *out, float *state_out,
                   int n_seqs, int n_tokens, int n_heads, int n_k_heads, int head_dim, int dtype,
                   int path, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    if (n_k_heads < 0) return GDN_ERR_ARG;
    return run(q, k, v, g, beta, state_in, out, state_out, n_seqs, n_tokens, n_heads,
               n_k_heads == 0 ? n_heads : n_k_heads, head_dim, dtype, path, workspace,
               workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t gdn_workspace_bytes(int n_seqs, int n_tokens, int n_heads, int head_dim, int dtype,
                           int path_opts) {
    if (n_seqs < 0 || n_tokens < 0 || n_heads < 0 || head_dim <= 0) return 0;
    if (path_opts < 0 || (path_opts & ~kPathMask & ~kKnownOptions)) return 0;
    int path = path_opts & kPathMask;
    if (dtype != GDN_DTYPE_F32 && dtype != GDN_DTYPE_BF16) return 0;
    if (n_tokens == 0 || (long long)n_seqs * n_heads == 0) return 0;
    if (path == GDN_PATH_AUTO)
        path = select_path((long long)n_seqs * n_heads, n_tokens, head_dim, dtype);
    if (path != GDN_PATH_CHUNKED || dtype != GDN_DTYPE_BF16) return 0;
    if (!(gdn_supports(head_dim) & 2)) return 0;
    return gdn::chunked_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, dtype);
}

int gdn_select_path(int n_seqs, int n_tokens, int n_heads, int head_dim, int dtype) {
    if (n_seqs < 0 || n_tokens < 0 || n_heads < 0) return GDN_ERR_ARG;
    return select_path((long long)n_seqs * n_heads, n_tokens, head_dim, dtype);
}

int gdn_supports(int head_dim) {
    int caps = 0;
    if (head_dim == 32 || head_dim == 64 || head_dim == 96 || head_dim == 128 || head_dim == 256)
        caps |= 1;
    if (gdn::chunked_supports(head_dim)) caps |= 2;
    return caps;
}

int gdn_get_device_status(gdn_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GDN_ERR_CUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_device_status, sizeof(int)) != cudaSuccess)
        return GDN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess)
        return GDN_ERR_CUDA;
    return value;
}

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_ARG: return "invalid argument (null pointer, negative size or size overflow)";
        case GDN_ERR_HEADDIM: return "head_dim not supported on the requested path";
        case GDN_ERR_ALIGN: return "misaligned pointer (16 B for tensors, 4 B for g/beta)";
        case GDN_ERR_ALIAS: return "an output overlaps an input or the other output";
        case GDN_ERR_CUDA: return "CUDA launch or enqueue failed";
        case GDN_ERR_TIMEOUT: return "a bounded device wait gave up";
        case GDN_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case GDN_ERR_NOMEM: return "stream-ordered workspace allocation failed";
        case GDN_ERR_DTYPE: return "dtype not supported on the requested path (chunked: bf16 only)";
        case GDN_ERR_SHAPE: return "shape outside the op's scope (flash_attn: 20 or more queries)";
        case GDN_ERR_SCRATCH:
            return "the call needs more scratch than gdn_forward_noalloc's fixed 64 MiB array";
        default: return "unknown status";
    }
}

int gdn_version(void) { return 100; }

int gdn_selftest_wait_timeout(gdn_stream_t stream) {
    int *status = status_word_for_current_device();
    if (!status) return GDN_ERR_CUDA;
    return gdn::launch_wait_selftest(status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.  Some callers must not allocate device memory
// at all once they are running: a serving process whose framework has
// reserved the whole device up front for its own arena, or a decode loop in
// which an allocation (and the device synchronisation cudaMalloc can imply)
// would stall the step.  For them the chunked calls that need scratch --
// head_dim 256, and head_dim 128 with few (sequence, head) pairs, which keep
// a 32 KiB transform tile per (sequence, head, 64-token chunk) -- take it
// from this fixed array instead.  The array is part of the library image: every GPU that loads the
// library holds these 64 MiB until the process exits.  Calls share it, so two
// calls that overlap on the GPU (different streams, no ordering between them)
// race on it.  Nothing in it has to start at zero: the transform kernel writes
// every tile a call reads before the state kernel of that call reads it.

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

namespace {

void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device (with that device current) on the first call that needs it.  The
// array's name in host code is only a stand-in; kernels get this address.
void *noalloc_scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int gdn_forward_noalloc(const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, const float *state_in, float *out,
                                   float *state_out, int n_seqs, int n_tokens, int n_heads,
                                   int n_k_heads, int head_dim, int dtype, int path,
                                   gdn_stream_t stream) {
    if (n_k_heads < 0) return GDN_ERR_ARG;
    // scratch the call needs (0 for invalid sizes: run() reports those)
    const size_t need = gdn_workspace_bytes(n_seqs, n_tokens, n_heads, head_dim, dtype, path);
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_SCRATCH;
    void *ws = nullptr;
    if (need > 0) {
        ws = noalloc_scratch_for_current_device();
        if (!ws) return GDN_ERR_CUDA;
    }
    return run(q, k, v, g, beta, state_in, out, state_out, n_seqs, n_tokens, n_heads,
               n_k_heads == 0 ? n_heads : n_k_heads, head_dim, dtype, path, ws,
               ws ? (size_t)GDN_NOALLOC_SCRATCH_BYTES : 0, reinterpret_cast<cudaStream_t>(stream));
}
